// TMA throughput probe: each CTA streams K tiles [64 rows x 512 B] of a [1, S, 2, 256] bf16
// tensor (L2-resident) through an NS-stage ring, no compute.  Box forms: 4 x 4-D (64 x 128 B)
// or one 5-D box.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdint.h>
#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s line %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ unsigned int g_err;
template <int NS, bool FIVE>
__global__ void __launch_bounds__(32, 1) probe(const __grid_constant__ CUtensorMap map, int tiles, int S) {
  extern __shared__ unsigned char raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bar = (uint64_t*)(sm + NS * 32768);
  if (threadIdx.x != 0) return;
  for (int i = 0; i < NS; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(sa(&bar[i])));
  asm volatile("fence.mbarrier_init.release.cluster;");
  const int ntile_rows = S / 64;
  auto issue = [&](int t) {
    const int st = t % NS;
    const int row = ((t * 7 + blockIdx.x * 13) % ntile_rows) * 64;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(sa(&bar[st])), "r"(32768));
    if (FIVE) {
      asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
                   :: "r"(sa(sm + st * 32768)), "l"((uint64_t)&map), "r"(0), "r"(row), "r"(0), "r"(0), "r"(0), "r"(sa(&bar[st])) : "memory");
    } else {
      for (int c = 0; c < 4; ++c)
        asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
                     :: "r"(sa(sm + st * 32768 + c * 8192)), "l"((uint64_t)&map), "r"(64 * c), "r"(0), "r"(row), "r"(0), "r"(sa(&bar[st])) : "memory");
    }
  };
  for (int t = 0; t < NS && t < tiles; ++t) issue(t);
  for (int t = 0; t < tiles; ++t) {
    const int st = t % NS;
    const uint32_t par = (t / NS) & 1;
    uint32_t done = 0;
    long long t0 = clock64();
    while (!done) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(sa(&bar[st])), "r"(par) : "memory");
      if (!done && clock64() - t0 > 2000000000LL) { atomicOr(&g_err, 1u); return; }
    }
    if (t + NS < tiles) issue(t + NS);
  }
}
typedef CUresult (*EncFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                          const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                          CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
template <int NS, bool FIVE>
int run(EncFn enc, void* base, int S, int sms) {
  CUtensorMap m;
  const int H = 2, D = 256;
  CUresult r;
  if (FIVE) {
    cuuint64_t dims[5] = {64, (cuuint64_t)S, 4, (cuuint64_t)H, 1};
    cuuint64_t str[4] = {(cuuint64_t)H * D * 2, 128, (cuuint64_t)D * 2, (cuuint64_t)S * H * D * 2};
    cuuint32_t box[5] = {64, 64, 4, 1, 1}, es[5] = {1, 1, 1, 1, 1};
    r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, 1};
    cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S * H * D * 2};
    cuuint32_t box[4] = {64, 1, 64, 1}, es[4] = {1, 1, 1, 1};
    r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); return 1; }
  const size_t smem = NS * 32768 + 1024 + 64;
  CK(cudaFuncSetAttribute(probe<NS, FIVE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const int tiles = 2000;
  probe<NS, FIVE><<<sms, 32, smem>>>(m, tiles, S);
  CK(cudaDeviceSynchronize());
  cudaEvent_t a, b;
  cudaEventCreate(&a); cudaEventCreate(&b);
  cudaEventRecord(a);
  probe<NS, FIVE><<<sms, 32, smem>>>(m, tiles, S);
  cudaEventRecord(b);
  CK(cudaEventSynchronize(b));
  float ms; cudaEventElapsedTime(&ms, a, b);
  unsigned int err = 0; CK(cudaMemcpyFromSymbol(&err, g_err, 4));
  const double bytes = (double)sms * tiles * 32768;
  printf("%s NS=%d  %.1f GB/s total, %.1f B/clk/SM at 2.07 GHz  err=%u\n", FIVE ? "5D" : "4x4D", NS, bytes / ms / 1e6,
         bytes / (ms * 1e-3) / sms / 2.07e9, err);
  return 0;
}
int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  void* fn = nullptr; cudaDriverEntryPointQueryResult q;
  CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
  EncFn enc = (EncFn)fn;
  const int S = 4096;
  void* base; CK(cudaMalloc(&base, (size_t)S * 2 * 256 * 2)); CK(cudaMemset(base, 1, (size_t)S * 2 * 256 * 2));
  if (run<2, false>(enc, base, S, sms)) return 1;
  if (run<4, false>(enc, base, S, sms)) return 1;
  if (run<6, false>(enc, base, S, sms)) return 1;
  if (run<2, true>(enc, base, S, sms)) return 1;
  if (run<4, true>(enc, base, S, sms)) return 1;
  if (run<6, true>(enc, base, S, sms)) return 1;
  return 0;
}
