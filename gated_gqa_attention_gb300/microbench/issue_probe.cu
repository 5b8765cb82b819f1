// tcgen05.mma issue probe: how synchronisation in the issuing thread affects the tensor
// pipe.  One CTA per SM; one thread issues the per-tile MMA stream of an attention
// mainloop (operands in shared memory and TMEM, zero data) for T tiles, and clock64
// from the first issue to the final commit gives cycles per 64 keys.
//   stream:   S = 16 x (M 128, N 64, K 16) + PV = 4 x (N 256), four commits per tile;
//             the same with one mbarrier.try_wait (on a completed barrier) or one
//             volatile shared load after each group;
//   sched64:  the 64-key stream with its real dependencies (S runs two tiles ahead of
//             PV, each group waits on the commit barrier of the group it depends on);
//   sched128: 128-key tiles (S = 16 x N 128, PV = 16 x N 128 over two halves of O) with
//             two S buffers and a helper warp that stands in for the softmax (it waits
//             for S, spins 1000 cycles, releases P); one issuer (S(j+1) then PV(j)) or
//             two issuers (S warp and PV warp).
// Every wait is bounded; a timeout sets an error bit that the host prints.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#define CK(x)                                                                   \
  do {                                                                          \
    cudaError_t e_ = (x);                                                       \
    if (e_ != cudaSuccess) {                                                    \
      printf("CUDA %s line %d\n", cudaGetErrorString(e_), __LINE__);            \
      return 1;                                                                 \
    }                                                                           \
  } while (0)

__device__ long long g_cyc[1024];
__device__ unsigned g_err;

__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 128-byte swizzle shared-memory descriptor (version 1): start, LBO, SBO (all >> 4)
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: FP32 accumulate, BF16 A and B, A K-major
__host__ __device__ constexpr uint32_t idesc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d), "l"(a), "l"(b), "r"(id),
               "r"(acc)
               : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d), "r"(a), "l"(b), "r"(id),
               "r"(acc)
               : "memory");
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
               : "memory");
}
__device__ __forceinline__ void bar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(bar)), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(bar)) : "memory");
}
// bounded parity wait: false (and an error bit) after ~2 s of cycles
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, long long t0) {
  uint32_t done = 0;
  while (!done) {
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(sa(bar)), "r"(parity)
                 : "memory");
    if (!done && clock64() - t0 > 4000000000LL) {
      atomicOr(&g_err, 1u);
      return false;
    }
  }
  return true;
}

constexpr int kSmem = 196608;  // Q [64 KiB] | K [64 KiB] | V [64 KiB], zero-filled

// common prologue: zero the operands, allocate all 512 TMEM columns
__device__ __forceinline__ unsigned char* setup(unsigned char* raw, uint32_t* tbase) {
  unsigned char* sm = (unsigned char*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
  for (int i = threadIdx.x; i < kSmem / 16; i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(sa(tbase)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  return sm;
}
__device__ __forceinline__ void teardown(uint32_t tm) {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm));
  }
}

// SYNC = 0: nothing between groups; 1: try_wait on a completed barrier; 2: volatile shared load
template <int SYNC>
__global__ void __launch_bounds__(128, 1) stream64(int T) {
  extern __shared__ unsigned char raw[];
  __shared__ uint64_t bar[5], done_bar;
  __shared__ uint32_t tbase;
  __shared__ volatile int flag;
  unsigned char* sm = setup(raw, &tbase);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 5; ++i) bar_init(&bar[i], 1);
    bar_init(&done_bar, 1);
    bar_arrive(&done_bar);  // phase 0 complete
    flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    const uint32_t sQ = sa(sm), sK = sa(sm + 65536), sV = sa(sm + 131072);
    const uint32_t idS = idesc(128, 64, 0), idO = idesc(128, 256, 1);
    const long long t0 = clock64();
    for (int j = 0; j < T; ++j) {
      const int ks = j & 1, sb = (j & 3) * 64;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        mma_ss(tm + sb, desc(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
               desc(sK + ks * 32768 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      commit(&bar[0]);
      commit(&bar[1]);
      if (SYNC == 1) bar_wait(&done_bar, 0, t0);
      if (SYNC == 2 && flag == 12345) atomicOr(&g_err, 2u);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts(tm + 256, tm + sb + 8 * kk, desc(sV + ks * 32768 + kk * 2048, 8192, 1024), idO, 1);
      commit(&bar[2]);
      commit(&bar[3]);
      if (SYNC == 1) bar_wait(&done_bar, 0, t0);
      if (SYNC == 2 && flag == 12345) atomicOr(&g_err, 2u);
    }
    commit(&bar[4]);
    bar_wait(&bar[4], 0, t0);
    g_cyc[blockIdx.x] = clock64() - t0;
  }
  teardown(tm);
}

// 64-key tiles with the real dependencies: S(j) into buffer j % 4 waits for PV(j - 4),
// PV(j) waits for S(j); S runs two tiles ahead of PV; one issuer
__global__ void __launch_bounds__(128, 1) sched64(int T) {
  extern __shared__ unsigned char raw[];
  __shared__ uint64_t s_full[4], p_empty[4], fin;
  __shared__ uint32_t tbase;
  unsigned char* sm = setup(raw, &tbase);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; ++i) {
      bar_init(&s_full[i], 1);
      bar_init(&p_empty[i], 1);
    }
    bar_init(&fin, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    const uint32_t sQ = sa(sm), sK = sa(sm + 65536), sV = sa(sm + 131072);
    const uint32_t idS = idesc(128, 64, 0), idO = idesc(128, 256, 1);
    const long long t0 = clock64();
    bool ok = true;
    auto issue_s = [&](int j) {
      const int sb = j & 3;
      if (j >= 4) ok = ok && bar_wait(&p_empty[sb], ((j >> 2) - 1) & 1, t0);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        mma_ss(tm + sb * 64, desc(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
               desc(sK + (j & 1) * 32768 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
      commit(&s_full[sb]);
    };
    auto issue_pv = [&](int j) {
      const int pb = j & 3;
      ok = ok && bar_wait(&s_full[pb], (j >> 2) & 1, t0);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts(tm + 256, tm + pb * 64 + 8 * kk, desc(sV + (j & 1) * 32768 + kk * 2048, 8192, 1024), idO, 1);
      commit(&p_empty[pb]);
    };
    issue_s(0);
    issue_s(1);
    for (int j = 0; j < T && ok; ++j) {
      if (j + 2 < T) issue_s(j + 2);
      issue_pv(j);
    }
    commit(&fin);
    bar_wait(&fin, 0, t0);
    g_cyc[blockIdx.x] = clock64() - t0;
  }
  teardown(tm);
}

// 128-key tiles, two S buffers of 128 columns, O in columns [256, 512); a helper warp
// stands in for the softmax.  TWO = 0: one issuer (S(j+1), then PV(j)); TWO = 1: S
// issued by thread 0, PV by thread 64.
template <int TWO>
__global__ void __launch_bounds__(128, 1) sched128(int T, int softmax_cycles) {
  extern __shared__ unsigned char raw[];
  __shared__ uint64_t s_full[2], p_full[2], p_empty[2], fin[2];
  __shared__ uint32_t tbase;
  unsigned char* sm = setup(raw, &tbase);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      bar_init(&s_full[i], 1);
      bar_init(&p_full[i], 1);
      bar_init(&p_empty[i], 1);
      bar_init(&fin[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  const uint32_t sQ = sa(sm), sK = sa(sm + 65536), sV = sa(sm + 131072);
  const uint32_t idS = idesc(128, 128, 0), idO = idesc(128, 128, 1);
  const long long t0 = clock64();
  auto issue_s = [&](int j) -> bool {
    const int sb = j & 1;
    if (j >= 2 && !bar_wait(&p_empty[sb], ((j >> 1) - 1) & 1, t0)) return false;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
      mma_ss(tm + sb * 128, desc(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
             desc(sK + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), idS, kk > 0);
    commit(&s_full[sb]);
    return true;
  };
  auto issue_pv = [&](int j) -> bool {
    const int pb = j & 1;
    if (!bar_wait(&p_full[pb], (j >> 1) & 1, t0)) return false;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ts(tm + 256 + 128 * hh, tm + pb * 128 + 8 * kk, desc(sV + hh * 32768 + kk * 2048, 16384, 1024), idO,
               1);
    commit(&p_empty[pb]);
    return true;
  };
  if (threadIdx.x == 0) {
    bool ok = true;
    if (TWO) {
      for (int j = 0; j < T && ok; ++j) ok = issue_s(j);
    } else {
      ok = issue_s(0);
      for (int j = 0; j < T && ok; ++j) {
        if (j + 1 < T) ok = issue_s(j + 1);
        if (ok) ok = issue_pv(j);
      }
    }
    commit(&fin[0]);
    bar_wait(&fin[0], 0, t0);
    if (!TWO) g_cyc[blockIdx.x] = clock64() - t0;
  } else if (TWO && threadIdx.x == 64) {
    bool ok = true;
    for (int j = 0; j < T && ok; ++j) ok = issue_pv(j);
    commit(&fin[1]);
    bar_wait(&fin[1], 0, t0);
    g_cyc[blockIdx.x] = clock64() - t0;
  } else if (threadIdx.x == 32) {
    for (int j = 0; j < T; ++j) {
      if (!bar_wait(&s_full[j & 1], (j >> 1) & 1, t0)) break;
      const long long a = clock64();
      while (clock64() - a < softmax_cycles) {
      }
      bar_arrive(&p_full[j & 1]);
    }
  }
  teardown(tm);
}

template <typename F>
static int run(F launch, int sms, int keys_per_call, const char* name) {
  launch();
  CK(cudaDeviceSynchronize());
  launch();
  CK(cudaDeviceSynchronize());
  long long cyc[1024];
  CK(cudaMemcpyFromSymbol(cyc, g_cyc, sizeof(long long) * sms));
  unsigned err;
  CK(cudaMemcpyFromSymbol(&err, g_err, 4));
  double avg = 0;
  for (int i = 0; i < sms; ++i) avg += (double)cyc[i];
  avg /= sms;
  printf("%-62s %7.1f cycles per 64 keys  err=%u\n", name, avg / keys_per_call * 64.0, err);
  return 0;
}

int main() {
  int sms = 0;
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  if (sms > 1024) sms = 1024;
  const size_t smem = kSmem + 1024;
  CK(cudaFuncSetAttribute(stream64<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  CK(cudaFuncSetAttribute(stream64<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  CK(cudaFuncSetAttribute(stream64<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  CK(cudaFuncSetAttribute(sched64, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  CK(cudaFuncSetAttribute(sched128<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  CK(cudaFuncSetAttribute(sched128<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const int T = 512;
  if (run([&] { stream64<0><<<sms, 128, smem>>>(T); }, sms, 64 * T, "stream, 64-key tiles, no waits")) return 1;
  if (run([&] { stream64<1><<<sms, 128, smem>>>(T); }, sms, 64 * T,
          "stream + try_wait on a completed barrier after each group"))
    return 1;
  if (run([&] { stream64<2><<<sms, 128, smem>>>(T); }, sms, 64 * T, "stream + volatile shared load after each group"))
    return 1;
  if (run([&] { sched64<<<sms, 128, smem>>>(T); }, sms, 64 * T, "64-key tiles, real dependencies, one issuer")) return 1;
  if (run([&] { sched128<0><<<sms, 128, smem>>>(T / 2, 1000); }, sms, 128 * (T / 2),
          "128-key tiles, softmax stand-in 1000 cycles, one issuer"))
    return 1;
  if (run([&] { sched128<1><<<sms, 128, smem>>>(T / 2, 1000); }, sms, 128 * (T / 2),
          "128-key tiles, softmax stand-in 1000 cycles, two issuers"))
    return 1;
  return 0;
}
