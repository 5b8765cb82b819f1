// tcgen05.mma throughput probe: one CTA per SM, one thread issues R back-to-back
// kind::f16 MMAs (M = 128, K = 16, BF16, FP32 accumulate) into one TMEM accumulator,
// A from TMEM (ts) or shared memory (ss), B from shared memory (128-byte swizzle,
// zero data); clock64 from first issue to the commit's mbarrier.
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdint.h>
#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s line %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ long long g_cyc[1024];
__device__ unsigned g_err;
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
template <int N, bool TS, int BMN>
__global__ void __launch_bounds__(128, 1) probe(int R) {
  extern __shared__ unsigned char raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x;
  // zero the operand area (64 KiB A + 64 KiB B)
  for (int i = tid; i < 131072 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(sa(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  asm volatile("fence.proxy.async.shared::cta;");
  if (tid < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(sa(&tbase)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tm = tbase;
  if (tid == 0) {
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)BMN << 16) | ((uint32_t)(N >> 3) << 17) | (8u << 24);
    const uint32_t sA = sa(sm), sB = sa(sm + 65536);
    long long t0 = clock64();
    for (int i = 0; i < R; ++i) {
      const int kk = i & 3;
      const uint64_t bd = BMN ? desc(sB + kk * 2048, 8192, 1024) : desc(sB + kk * 32, 16, 1024);
      const uint32_t acc = i > 0;
      if (TS) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                     :: "r"(tm + 256), "r"(tm + 8 * kk), "l"(bd), "r"(idesc), "r"(acc) : "memory");
      } else {
        const uint64_t ad = desc(sA + kk * 32, 16, 1024);
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                     :: "r"(tm + 256), "l"(ad), "l"(bd), "r"(idesc), "r"(acc) : "memory");
      }
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(sa(&bar)) : "memory");
    uint32_t done = 0;
    while (!done) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(sa(&bar)) : "memory");
      if (!done && clock64() - t0 > 4000000000LL) { atomicOr(&g_err, 1u); break; }
    }
    g_cyc[blockIdx.x] = clock64() - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (tid < 32) {
    asm volatile("tcgen05.fence::after_thread_sync;");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tm));
  }
}
template <int N, bool TS, int BMN>
int run(int sms) {
  const int R = 4096;
  const size_t smem = 131072 + 1024;
  CK(cudaFuncSetAttribute(probe<N, TS, BMN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  probe<N, TS, BMN><<<sms, 128, smem>>>(R);
  CK(cudaDeviceSynchronize());
  probe<N, TS, BMN><<<sms, 128, smem>>>(R);
  CK(cudaDeviceSynchronize());
  long long cyc[1024];
  CK(cudaMemcpyFromSymbol(cyc, g_cyc, sizeof(long long) * sms));
  unsigned err; CK(cudaMemcpyFromSymbol(&err, g_err, 4));
  double avg = 0; for (int i = 0; i < sms; ++i) avg += cyc[i]; avg /= sms;
  const double flop = 2.0 * 128 * N * 16 * R;
  printf("N=%3d %s B-%s: %.1f cycles per MMA, %.0f FLOP/clk/SM  err=%u\n", N, TS ? "A-tmem" : "A-smem", BMN ? "MN-major" : "K-major",
         avg / R, flop / avg, err);
  return 0;
}
int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  if (run<64, true, 0>(sms)) return 1;
  if (run<64, false, 0>(sms)) return 1;
  if (run<128, true, 0>(sms)) return 1;
  if (run<128, false, 0>(sms)) return 1;
  if (run<256, true, 0>(sms)) return 1;
  if (run<256, false, 0>(sms)) return 1;
  if (run<256, true, 1>(sms)) return 1;
  if (run<64, true, 1>(sms)) return 1;
  return 0;
}
