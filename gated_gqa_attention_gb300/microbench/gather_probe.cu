// gather_probe.cu -- how fast can one GB300 stream scattered K/V-sized rows?
//
// Measures the gather of 512 MiB of rows at random row indices from a 1 GiB pool
// (one persistent CTA per SM, or many warps per SM) with four mechanisms:
//   TMA   one cp.async.bulk (1-D bulk copy) per row into a shared-memory ring,
//         row sizes 512 B .. 16 KiB
//   LDG   16-byte vector loads into registers, many warps per SM
//   CPA   cp.async 16-byte copies into a CTA-wide shared-memory ring
//   WARP  per-warp patterns on 16-row x 512 B tiles: a register tile per warp,
//         and a per-warp cp.async ring of 2 or 3 stages
// These numbers decided the stage-1 load path: scattered 512-byte rows need
// 16-byte loads or cp.async from many warps; one bulk copy per row is limited by
// the copy-request rate.
//
//   python -m gated_gqa_attention_gb300.microbench     (builds and runs it)
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <random>
#include <cuda_runtime.h>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool tryw(uint64_t* b, uint32_t ph) { uint32_t ok; asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0,1,0,p; }" : "=r"(ok) : "r"(sa(b)), "r"(ph) : "memory"); return ok; }
__device__ __forceinline__ bool waitb(uint64_t* b, uint32_t ph) { long long t0 = clock64(); while (!tryw(b, ph)) { if (clock64() - t0 > 2000000000LL) return false; } return true; }

// ---- per-warp tile patterns (see header)
// A/B: register loads; each warp handles 16-row tiles; lane loads 16 x 16 B (T tensors) per tile
template <int NB>   // register buffers (1 or 2)
__global__ void __launch_bounds__(256) k_warp_reg(const uint8_t* pool, const int* idx, int ntile_total, unsigned* out) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31, nw = (gridDim.x * blockDim.x) >> 5;
  unsigned acc = 0;
  uint4 buf[NB][16];
  int t = gw;
  auto issue = [&](int b, int tile) {
    int slot = idx[tile * 16 + (lane & 15)];
#pragma unroll
    for (int r = 0; r < 16; ++r) { int s = __shfl_sync(0xffffffffu, slot, r); buf[b][r] = __ldcs((const uint4*)(pool + (size_t)s * 512) + lane); }
  };
  if (t < ntile_total) issue(0, t);
  if (NB == 2 && t + nw < ntile_total) issue(NB - 1, t + nw);
  int b = 0;
  for (; t < ntile_total; t += nw) {
#pragma unroll
    for (int r = 0; r < 16; ++r) acc ^= buf[b][r].x ^ buf[b][r].w;
    int nt = t + NB * nw;
    if (nt < ntile_total) issue(b, nt);
    if (NB == 2) b ^= 1;
  }
  if (acc == 0x12345678) out[0] = acc;
}

// C: per-warp cp.async ring with NV stages of 16 rows x 512 B
template <int NV>
__global__ void __launch_bounds__(256) k_warp_cpa(const uint8_t* pool, const int* idx, int ntile_total, unsigned* out) {
  extern __shared__ __align__(128) uint8_t sm[];
  int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = sm + (size_t)w * NV * 16 * 528;
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  unsigned acc = 0;
  auto issue = [&](int st, int tile) {
    if (tile < ntile_total) {
      int slot = idx[tile * 16 + (lane & 15)];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        int s = __shfl_sync(0xffffffffu, slot, r);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(sa(ring + (st * 16 + r) * 528 + lane * 16)), "l"(pool + (size_t)s * 512 + lane * 16) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (int k = 0; k < NV - 1; ++k) issue(k, gw + k * nw);
  int st = 0;
  for (int t = gw; t < ntile_total; t += nw) {
    issue((st + NV - 1) % NV, t + (NV - 1) * nw);
    asm volatile("cp.async.wait_group %0;" :: "n"(NV - 1) : "memory");
    __syncwarp();
    const uint8_t* src = ring + st * 16 * 528;
#pragma unroll
    for (int r = 0; r < 16; ++r) acc ^= *(const unsigned*)(src + r * 528 + lane * 16);
    __syncwarp();
    st = (st + 1) % NV;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (acc == 0x12345678) out[0] = acc;
}


// mode TMA: producer warp issues one bulk copy per row; consumer warps read one word per row.
template <int RB, int TILE, int NST>
__global__ void __launch_bounds__(160, 1) k_tma(const uint8_t* pool, const int* idx, int rows_per_cta, int nrows, unsigned* out, unsigned* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* ring = sm;
  uint64_t* full = (uint64_t*)(sm + (size_t)NST * TILE * RB);
  uint64_t* empty = full + NST;
  int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) { for (int s = 0; s < NST; ++s) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(sa(&full[s])), "r"(1)); asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(sa(&empty[s])), "r"(4)); } asm volatile("fence.mbarrier_init.release.cluster;"); }
  __syncthreads();
  int r0 = blockIdx.x * rows_per_cta, r1 = min(nrows, r0 + rows_per_cta);
  int ntiles = (r1 - r0 + TILE - 1) / TILE;
  if (w == 4) {
    int st = 0; uint32_t ph = 0; int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!waitb(&empty[st], ph ^ 1)) {
        atomicOr(err, 1);
        // drain: wait (bounded) for the copies already issued
        int s2 = st; uint32_t p2 = ph;
        for (int k = 0; k < min(issued, NST); ++k) { if (--s2 < 0) { s2 = NST - 1; p2 ^= 1; } waitb(&full[s2], p2); }
        break;
      }
      ++issued;
      int base = r0 + t * TILE; int n = min(TILE, r1 - base);
      if (lane == 0) asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(sa(&full[st])), "r"(n * RB) : "memory");
      __syncwarp();
      for (int r = lane; r < n; r += 32) {
        const uint8_t* src = pool + (size_t)idx[base + r] * RB;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" :: "r"(sa(ring + ((size_t)st * TILE + r) * RB)), "l"(src), "r"(RB), "r"(sa(&full[st])) : "memory");
      }
      if (++st == NST) { st = 0; ph ^= 1; }
    }
  } else {
    unsigned acc = 0; int st = 0; uint32_t ph = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!waitb(&full[st], ph)) { atomicOr(err, 2); break; }
      int base = r0 + t * TILE; int n = min(TILE, r1 - base);
      for (int r = w * 32 + lane; r < n; r += 128) acc ^= *(const unsigned*)(ring + ((size_t)st * TILE + r) * RB + 4 * (r & 7));
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(sa(&empty[st])) : "memory");
      if (++st == NST) { st = 0; ph ^= 1; }
    }
    if (acc == 0x12345678) out[0] = acc;
  }
}

// mode LDG: each warp streams rows into registers with 16-byte loads, U rows in flight per warp.
template <int RB, int U>
__global__ void __launch_bounds__(512) k_ldg(const uint8_t* pool, const int* idx, int nrows, unsigned* out) {
  constexpr int V = RB / 16;             // uint4 per row
  constexpr int PER = (V + 31) / 32;      // per lane per row
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  int nw = (gridDim.x * blockDim.x) >> 5;
  unsigned acc = 0;
  for (int r = gw * U; r < nrows; r += nw * U) {
    uint4 v[U][PER];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int rr = r + u;
      const uint4* src = (const uint4*)(pool + (size_t)idx[rr < nrows ? rr : r] * RB);
#pragma unroll
      for (int p = 0; p < PER; ++p) { int c = lane + 32 * p; v[u][p] = c < V ? __ldcs(src + c) : make_uint4(0,0,0,0); }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int p = 0; p < PER; ++p) acc ^= v[u][p].x ^ v[u][p].w;
  }
  if (acc == 0x12345678) out[0] = acc;
}

// mode CPASYNC: 4 warps load tiles with cp.async 16B, NST stages, then read one word per row.
template <int RB, int TILE, int NST>
__global__ void __launch_bounds__(128, 1) k_cpa(const uint8_t* pool, const int* idx, int rows_per_cta, int nrows, unsigned* out) {
  extern __shared__ __align__(128) uint8_t sm[];
  constexpr int V = RB / 16;
  int r0 = blockIdx.x * rows_per_cta, r1 = min(nrows, r0 + rows_per_cta);
  int ntiles = (r1 - r0 + TILE - 1) / TILE;
  unsigned acc = 0;
  auto issue = [&](int t) {
    if (t < ntiles) {
      int base = r0 + t * TILE; int n = min(TILE, r1 - base); uint8_t* dst = sm + (size_t)(t % NST) * TILE * RB;
      for (int e = threadIdx.x; e < n * V; e += 128) {
        int r = e / V, c = e % V;
        const uint8_t* src = pool + (size_t)idx[base + r] * RB + c * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(sa(dst + r * RB + c * 16)), "l"(src) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  for (int t = 0; t < NST - 1; ++t) issue(t);
  for (int t = 0; t < ntiles; ++t) {
    issue(t + NST - 1);
    asm volatile("cp.async.wait_group %0;" :: "n"(NST - 1) : "memory");
    __syncthreads();
    int base = r0 + t * TILE; int n = min(TILE, r1 - base); const uint8_t* src = sm + (size_t)(t % NST) * TILE * RB;
    for (int r = threadIdx.x; r < n; r += 128) acc ^= *(const unsigned*)(src + r * RB + 4 * (r & 7));
    __syncthreads();
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (acc == 0x12345678) out[0] = acc;
}

template <class F> float timeit(F f, int reps) {
  cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
  f(); cudaDeviceSynchronize();
  cudaEventRecord(a); for (int i = 0; i < reps; ++i) f(); cudaEventRecord(b); cudaEventSynchronize(b);
  float ms; cudaEventElapsedTime(&ms, a, b); return ms / reps;
}

template <int RB, int TILE, int NST>
int run_tma(const uint8_t* pool, const int* idx, int nrows, unsigned* out, unsigned* err, int sms) {
  size_t smem = (size_t)NST * TILE * RB + 2 * NST * 8;
  if (smem > 227 * 1024) return 0;
  auto k = k_tma<RB, TILE, NST>;
  CK(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per = (nrows + sms - 1) / sms;
  float ms = timeit([&] { k<<<sms, 160, smem>>>(pool, idx, per, nrows, out, err); }, 10);
  CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
  unsigned ev = 0; CK(cudaMemcpy(&ev, err, 4, cudaMemcpyDeviceToHost));
  printf("TMA   RB=%5d TILE=%3d NST=%d  inflight<=%6zu B  %7.1f GB/s %s\n", RB, TILE, NST, (size_t)NST * TILE * RB, (double)nrows * RB / ms / 1e6, ev ? "ERR" : "");
  return 0;
}
template <int RB, int U>
int run_ldg(const uint8_t* pool, const int* idx, int nrows, unsigned* out, int sms, int blocks_per_sm, int threads) {
  float ms = timeit([&] { k_ldg<RB, U><<<sms * blocks_per_sm, threads>>>(pool, idx, nrows, out); }, 10);
  CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
  printf("LDG   RB=%5d U=%d warps/SM=%2d  %7.1f GB/s\n", RB, U, blocks_per_sm * threads / 32, (double)nrows * RB / ms / 1e6);
  return 0;
}
template <int RB, int TILE, int NST>
int run_cpa(const uint8_t* pool, const int* idx, int nrows, unsigned* out, int sms) {
  size_t smem = (size_t)NST * TILE * RB;
  if (smem > 227 * 1024) return 0;
  auto k = k_cpa<RB, TILE, NST>;
  CK(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  int per = (nrows + sms - 1) / sms;
  float ms = timeit([&] { k<<<sms, 128, smem>>>(pool, idx, per, nrows, out); }, 10);
  CK(cudaGetLastError()); CK(cudaDeviceSynchronize());
  printf("CPA   RB=%5d TILE=%3d NST=%d  %7.1f GB/s\n", RB, TILE, NST, (double)nrows * RB / ms / 1e6);
  return 0;
}

int main_warp() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t POOL = (size_t)1 << 30, READ = (size_t)512 << 20;
  const int nrows = (int)(READ / 512), prow = (int)(POOL / 512), ntiles = nrows / 16;
  uint8_t* pool; CK(cudaMalloc(&pool, POOL)); CK(cudaMemset(pool, 1, POOL));
  unsigned* out; CK(cudaMalloc(&out, 64));
  int* idx; CK(cudaMalloc(&idx, (size_t)nrows * 4));
  std::vector<int> p(prow); for (int i = 0; i < prow; ++i) p[i] = i; std::mt19937 rng(1); std::shuffle(p.begin(), p.end(), rng);
  CK(cudaMemcpy(idx, p.data(), (size_t)nrows * 4, cudaMemcpyHostToDevice));
  for (int bps : {1, 2}) {
    float ms = timeit([&] { k_warp_reg<1><<<sms * bps, 256>>>(pool, idx, ntiles, out); }, 10); CK(cudaGetLastError());
    printf("WARP  register tile (8 KB per warp)  warps/SM=%2d  %7.1f GB/s\n", 8 * bps, (double)READ / ms / 1e6);
  }
  auto run_warp_cpa = [&](auto kern, int nv) -> int {
    size_t smem = (size_t)8 * nv * 16 * 528;
    CK(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    float ms = timeit([&] { kern<<<sms, 256, smem>>>(pool, idx, ntiles, out); }, 10); CK(cudaGetLastError());
    printf("WARP  cp.async ring NV=%d            warps/SM= 8  %7.1f GB/s\n", nv, (double)READ / ms / 1e6);
    return 0;
  };
  run_warp_cpa(k_warp_cpa<2>, 2); run_warp_cpa(k_warp_cpa<3>, 3);
  CK(cudaDeviceSynchronize());
  CK(cudaFree(pool)); CK(cudaFree(out)); CK(cudaFree(idx));
  return 0;
}

int main() {
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t POOL_BYTES = (size_t)1 << 30;   // 1 GiB pool
  const size_t READ_BYTES = (size_t)512 << 20; // 512 MiB gathered per launch
  uint8_t* pool; CK(cudaMalloc(&pool, POOL_BYTES)); CK(cudaMemset(pool, 1, POOL_BYTES));
  unsigned *out, *err; CK(cudaMalloc(&out, 64)); CK(cudaMalloc(&err, 4)); CK(cudaMemset(err, 0, 4));
  int* idx; CK(cudaMalloc(&idx, (READ_BYTES / 256) * 4));   // room for the 256-byte rows
  std::mt19937 rng(1);
  auto make = [&](int RB) -> int {
    int nrows = (int)(READ_BYTES / RB), prow = (int)(POOL_BYTES / RB);
    std::vector<int> p(prow); for (int i = 0; i < prow; ++i) p[i] = i; std::shuffle(p.begin(), p.end(), rng);
    cudaMemcpy(idx, p.data(), (size_t)nrows * 4, cudaMemcpyHostToDevice);
    return nrows;
  };
  // rows in runs of `page` consecutive rows (a paged pool), the pages in random order
  auto make_paged = [&](int RB, int page) -> int {
    int nrows = (int)(READ_BYTES / RB), npages = (int)(POOL_BYTES / RB) / page;
    std::vector<int> pg(npages); for (int i = 0; i < npages; ++i) pg[i] = i; std::shuffle(pg.begin(), pg.end(), rng);
    std::vector<int> p(nrows); for (int i = 0; i < nrows; ++i) p[i] = pg[i / page] * page + i % page;
    cudaMemcpy(idx, p.data(), (size_t)nrows * 4, cudaMemcpyHostToDevice);
    return nrows;
  };
  // stream copy reference
  { float ms = timeit([&] { cudaMemcpyAsync(pool + POOL_BYTES / 2, pool, POOL_BYTES / 2, cudaMemcpyDeviceToDevice); }, 10);
    printf("memcpy D2D %.1f GB/s (read+write)\n", (double)POOL_BYTES / ms / 1e6); }
  int n;
  n = make(256);
  printf("-- 256-byte rows (one FP8 K or V row), random\n");
  run_ldg<256, 8>(pool, idx, n, out, sms, 2, 512); run_ldg<256, 16>(pool, idx, n, out, sms, 2, 512);
  run_ldg<256, 8>(pool, idx, n, out, sms, 4, 512);
  run_cpa<256, 128, 3>(pool, idx, n, out, sms); run_cpa<256, 256, 3>(pool, idx, n, out, sms);
  n = make_paged(256, 16);
  printf("-- 256-byte rows in random 16-row pages\n");
  run_ldg<256, 8>(pool, idx, n, out, sms, 2, 512); run_ldg<256, 16>(pool, idx, n, out, sms, 2, 512);
  n = make_paged(512, 16);
  printf("-- 512-byte rows in random 16-row pages\n");
  run_ldg<512, 4>(pool, idx, n, out, sms, 2, 512);
  printf("-- 512-byte rows, random\n");
  n = make(512);
  run_tma<512, 64, 3>(pool, idx, n, out, err, sms);  run_tma<512, 128, 3>(pool, idx, n, out, err, sms);
  run_tma<512, 64, 6>(pool, idx, n, out, err, sms);  run_tma<512, 128, 3>(pool, idx, n, out, err, sms);
  run_ldg<512, 4>(pool, idx, n, out, sms, 2, 512); run_ldg<512, 8>(pool, idx, n, out, sms, 2, 512); run_ldg<512, 4>(pool, idx, n, out, sms, 4, 512);
  run_cpa<512, 64, 4>(pool, idx, n, out, sms); run_cpa<512, 128, 3>(pool, idx, n, out, sms);
  n = make(1024);
  run_tma<1024, 32, 6>(pool, idx, n, out, err, sms); run_tma<1024, 64, 3>(pool, idx, n, out, err, sms); run_tma<1024, 32, 3>(pool, idx, n, out, err, sms);
  run_ldg<1024, 4>(pool, idx, n, out, sms, 2, 512); run_ldg<1024, 2>(pool, idx, n, out, sms, 4, 512);
  run_cpa<1024, 32, 6>(pool, idx, n, out, sms); run_cpa<1024, 64, 3>(pool, idx, n, out, sms);
  n = make(2048);
  run_tma<2048, 16, 6>(pool, idx, n, out, err, sms); run_tma<2048, 32, 3>(pool, idx, n, out, err, sms);
  run_ldg<2048, 2>(pool, idx, n, out, sms, 2, 512);
  n = make(4096);
  run_tma<4096, 8, 6>(pool, idx, n, out, err, sms); run_tma<4096, 16, 3>(pool, idx, n, out, err, sms);
  n = make(16384);
  run_tma<16384, 4, 3>(pool, idx, n, out, err, sms); run_tma<16384, 2, 6>(pool, idx, n, out, err, sms);
  printf("-- per-warp tile patterns\n");
  if (main_warp()) return 1;
  printf("done\n");
  return 0;
}
