// gda_small.cu -- single-pass gated decode for small batches on sm_103a.
//
// The same result as stage 1 + stage 2 (FreeToken PR #781, Summary: split-KV
// partial softmax per split, FP32 log-sum-exp merge, the BF16 gate in the merge's
// epilogue; cuDNN FE-OSS "Gated Attention Block (SM107)", Overview stages (4)-(5)),
// computed in one launch for batches whose latency, not bandwidth, sets the time.
//
// One thread-block cluster of C = 8, 4, 2 or 1 CTAs per (sequence b, KV head) (the host
// takes the largest C whose clusters all run at once and leave each CTA at most 128
// positions): CTA r takes the r-th of C
// parts of the sequence's attended positions, in chunks of 64 whose K and V rows
// the CTA's 256 threads bring into shared memory (cp.async, two buffers, the next
// chunk in flight during the current one).  Per chunk, on the tensor cores
// (mma.sync m16n8k16, BF16 in, FP32 accumulate; the G <= 8 query heads are the rows):
//   S = Q K^T     warp w takes positions 8w .. 8w + 7 (16 k-steps over the 256 dims);
//   softmax       the chunk's max per head through shared memory, an online update of
//                 the running max (log2 units) and sum, P = 2^(S - max) as BF16;
//   O += P V      warp w owns head dimensions 32w .. 32w + 31 of every head.
// Each CTA then stores its state of query head G*kvh + g into the shared memory of
// CTA g % C of the cluster (distributed shared memory); after one cluster barrier,
// that CTA merges the C states (with the attention sink), divides by the sum, rounds
// to BF16, applies the BF16 gate, and writes out and lse.  No partials go through HBM and no
// second kernel runs.
#include <atomic>
#include "gda_device.cuh"
#include "gda_small.h"

namespace gda {

namespace {

constexpr int kSW = 8;              // warps per CTA
constexpr int kChunk = 64;          // positions per shared-memory chunk (8 per warp in S)

struct SmallSmem {
  unsigned char k[2][kChunk][kSmemRow];  // K rows of a chunk (padded rows: conflict-free
  unsigned char v[2][kChunk][kSmemRow];  // ldmatrix), V rows; two buffers
  uint32_t p[kG][kChunk / 2];            // P of the chunk: BF16 pairs [head][position pair]
  float wmax[kSW][kG];                   // per warp and head: max of the warp's 8 scores
  float wsum[kSW][kG];                   // per warp and head: sum of its BF16 probabilities
  // incoming states, slot (g / C) * C + x: CTA x's unnormalised O of query head g of the
  // group (finalised by CTA g % C), its running max (log2 units) and sum
  float o[kG][kD];
  float m[kG];
  float l[kG];
};
constexpr size_t kSmallSmem = sizeof(SmallSmem);

// all threads of all CTAs of the cluster: writes before it (also into other CTAs'
// shared memory) are visible after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the address that p (in this CTA's shared memory) has in CTA `rank`'s shared memory
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
  return remote;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_v2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
// 16 bytes global -> shared; src_bytes = 0 zero-fills the destination
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// FP16 counterparts of the BF16 tensor-core helpers (the e4m3 cache's operands)
__device__ __forceinline__ void mma_f16_16816(float* c, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float f16_lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu))); }
__device__ __forceinline__ float f16_hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }
// four e4m3 codes (bytes 0..3 of w) -> two f16 pairs (bytes 0, 1 and bytes 2, 3); exact
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}

}  // namespace

// F8: the pools hold e4m3 codes; K and V are widened to FP16 while being staged, Q
// goes to FP16 with one power-of-two factor per group, the MMAs run in FP16, and
// v_descale scales the merged O (k_descale is in scale_log2)
template <int C, bool F8>
__global__ void __launch_bounds__(kSW * 32, 1) small_decode_kernel(SmallParams p) {
  static_assert(C == 1 || C == 2 || C == 4 || C == 8, "cluster sizes");
  constexpr int kFin = kG / C;  // query heads each CTA finalises
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SmallSmem& sm = *reinterpret_cast<SmallSmem*>(smem_raw);
  const int r = blockIdx.x;  // rank in the cluster (the grid's x extent is the cluster)
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = lane >> 2, qd = lane & 3;  // fragment row (query head of the group) and quad lane
  const int G = p.G;

  // launched as a programmatic dependent of the previous kernel in the stream: its
  // results are visible after this wait, which comes before any global read; the next
  // call's kernel may then launch (and set up) while this one runs
  pdl_wait_prior_grid();
  pdl_launch_dependents();
  // independent loads first: the range, Q as A fragments (rows 8..15 and heads >= G
  // are zero), the gate element this CTA finalises (its sigmoid comes later)
  int L;
  long long base;
  seq_range(p.indptr, b, p.window, &L, &base);
  uint32_t qa[16][2];  // k-step ks: a0 = q[h][16 ks + 2 qd ..], a2 = q[h][16 ks + 8 + 2 qd ..]
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((size_t)b * p.Hq + kvh * G + h) * kD);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks) {
      qa[ks][0] = (h < G) ? __ldg(qrow + 8 * ks + qd) : 0u;
      qa[ks][1] = (h < G) ? __ldg(qrow + 8 * ks + 4 + qd) : 0u;
    }
  }
  float sl2 = p.scale_log2;
  if (F8) {
    // every warp holds the whole group's Q: its largest magnitude sets 2^e, which puts
    // it in [2^14, 2^15) (every BF16 value down to 2^-14 below it stays exact in FP16)
    float mx = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 16; ++ks)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(qa[ks][i] << 16)), fabsf(__uint_as_float(qa[ks][i] & 0xFFFF0000u))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const uint32_t qm = __float_as_uint(mx);
    int e = (qm == 0u) ? 0 : 141 - (int)((qm >> 23) & 0xFFu);
    e = max(-126, min(127, e));
    const float qs = __uint_as_float((uint32_t)(e + 127) << 23);
    sl2 = ldexpf(p.scale_log2, -e);
#pragma unroll
    for (int ks = 0; ks < 16; ++ks)
#pragma unroll
      for (int i = 0; i < 2; ++i)
        qa[ks][i] = f16x2_rn(__uint_as_float(qa[ks][i] << 16) * qs, __uint_as_float(qa[ks][i] & 0xFFFF0000u) * qs);
  }
  // the query heads this CTA finalises: r + C k of the group (when below G)
  uint16_t gbits[kFin];
#pragma unroll
  for (int k = 0; k < kFin; ++k) {
    const int hl = r + C * k;
    gbits[k] = (hl < G && p.fuse_gate)
                   ? __bfloat16_as_ushort(p.gate[((size_t)b * p.Hq + kvh * G + hl) * kD + tid])
                   : (uint16_t)0;
  }

  const int c = (L + C - 1) / C;
  const int lo = min(L, r * c), hi = min(L, lo + c);
  const int nch = (hi - lo + kChunk - 1) / kChunk;
  const size_t row_stride = (size_t)p.Hkv * kD;  // elements between slots

  // e4m3 rows (256 B): thread t loads the 64-byte piece t % 4 of the K and V rows of
  // position t / 4 into registers; store_chunk widens them to FP16 into buffer c & 1
  // (the same row layout as BF16 rows).  Positions past the range read as zeros.
  uint4 rk[4], rv[4];
  auto fetch_raw = [&](int cidx) {
    const int pos = lo + cidx * kChunk + (tid >> 2);
    const bool ok = cidx < nch && pos < hi;
    const int slot = ok ? __ldg(p.indices + base + pos) : 0;
    const size_t off = ((size_t)slot * row_stride + (size_t)kvh * kD) + (size_t)qd * 64;  // bytes (1 per code)
    const uint4* ks = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(p.k_pool) + off);
    const uint4* vs = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(p.v_pool) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      rk[i] = ok ? __ldg(ks + i) : make_uint4(0u, 0u, 0u, 0u);
      rv[i] = ok ? __ldg(vs + i) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  auto store_chunk = [&](int cidx) {
    const int j = tid >> 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t wk[4] = {rk[i].x, rk[i].y, rk[i].z, rk[i].w}, wv[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
      uint32_t fk[8], fv[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        e4m3x4_to_f16(wk[u], fk[2 * u], fk[2 * u + 1]);
        e4m3x4_to_f16(wv[u], fv[2 * u], fv[2 * u + 1]);
      }
      // codes 64 qd + 16 i .. + 15 -> FP16 elements at byte 2 (64 qd + 16 i)
      uint4* dk = reinterpret_cast<uint4*>(&sm.k[cidx & 1][j][2 * (64 * qd + 16 * i)]);
      uint4* dv = reinterpret_cast<uint4*>(&sm.v[cidx & 1][j][2 * (64 * qd + 16 * i)]);
      dk[0] = make_uint4(fk[0], fk[1], fk[2], fk[3]);
      dk[1] = make_uint4(fk[4], fk[5], fk[6], fk[7]);
      dv[0] = make_uint4(fv[0], fv[1], fv[2], fv[3]);
      dv[1] = make_uint4(fv[4], fv[5], fv[6], fv[7]);
    }
  };
  // BF16 rows: chunk c into buffer c & 1 by cp.async: thread t copies pieces t % 4 + 4 k
  // (k < 8) of the K and V rows of position t / 4; positions past the range are zero-filled
  auto load_chunk = [&](int cidx) {
    const int j = tid >> 2, pos = lo + cidx * kChunk + j;
    const bool ok = pos < hi;
    const int slot = ok ? __ldg(p.indices + base + pos) : 0;
    const size_t off = (size_t)slot * row_stride + (size_t)kvh * kD;
    const unsigned char* ks =
        reinterpret_cast<const unsigned char*>(static_cast<const __nv_bfloat16*>(p.k_pool) + (ok ? off : 0));
    const unsigned char* vs =
        reinterpret_cast<const unsigned char*>(static_cast<const __nv_bfloat16*>(p.v_pool) + (ok ? off : 0));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int piece = qd + 4 * k;
      cp_async16(&sm.k[cidx & 1][j][piece * 16], ks + piece * 16, ok ? 16u : 0u);
      cp_async16(&sm.v[cidx & 1][j][piece * 16], vs + piece * 16, ok ? 16u : 0u);
    }
    cp_async_commit();
  };
  if (F8) {
    fetch_raw(0);
    if (nch > 0) store_chunk(0);
    fetch_raw(1);  // in flight during chunk 0
  } else {
    if (nch > 0) load_chunk(0);
    if (nch > 1) load_chunk(1);
  }

  float m_run = -INFINITY, l_run = 0.0f;  // head h (identical in every thread of row h)
  float oacc[4][4];                        // O of head h, dims 32 warp + 8 nt + 2 qd .. (c0, c1)
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[nt][e] = 0.0f;

  for (int cidx = 0; cidx < nch; ++cidx) {
    if (!F8) {
      if (cidx + 1 < nch) cp_async_wait<1>(); else cp_async_wait<0>();
    }
    __syncthreads();
    const int buf = cidx & 1;
    const int n = min(kChunk, hi - lo - cidx * kChunk);  // positions in this chunk

    // S = Q K^T for positions 8 warp .. 8 warp + 7
    float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    {
      // ldmatrix x4: matrix i = dims 8 i .. of rows 8 warp + lane % 8 -> b0, b1 of two k-steps
      const uint32_t kaddr = smem_u32(&sm.k[buf][8 * warp + (lane & 7)][0]) + (lane >> 3) * 16;
#pragma unroll
      for (int kp = 0; kp < 8; ++kp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kaddr + kp * 64, b0, b1, b2, b3);
        if (F8) {
          mma_f16_16816(sacc, qa[2 * kp][0], qa[2 * kp][1], b0, b1);
          mma_f16_16816(sacc, qa[2 * kp + 1][0], qa[2 * kp + 1][1], b2, b3);
        } else {
          mma_bf16_16816(sacc, qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, b0, b1);
          mma_bf16_16816(sacc, qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, b2, b3);
        }
      }
    }
    // scores (log2 units) of positions 8 warp + 2 qd, + 1; past the chunk's end -inf
    const int j0 = 8 * warp + 2 * qd;
    const float s0 = (j0 < n) ? sacc[0] * sl2 : -INFINITY;
    const float s1 = (j0 + 1 < n) ? sacc[1] * sl2 : -INFINITY;
    const float wm = quad_max(fmaxf(s0, s1));
    if (qd == 0) sm.wmax[warp][h] = wm;
    __syncthreads();
    float cmax = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSW; ++w) cmax = fmaxf(cmax, sm.wmax[w][h]);
    const float m_new = fmaxf(m_run, cmax);
    const float alpha = (m_new == -INFINITY) ? 1.0f : safe_exp2_diff(m_run, m_new);
    float p0 = 0.0f, p1 = 0.0f;
    if (m_new != -INFINITY) {
      p0 = safe_exp2_diff(s0, m_new);
      p1 = safe_exp2_diff(s1, m_new);
    }
    // P rounded to the MMA's type; the sum adds the rounded values the MMA uses
    const uint32_t pp = F8 ? f16x2_rn(p0, p1) : pack_bf16x2(p0, p1);
    sm.p[h][4 * warp + qd] = pp;
    const float ws = quad_sum(F8 ? (f16_lo(pp) + f16_hi(pp))
                                 : (__uint_as_float(pp << 16) + __uint_as_float(pp & 0xFFFF0000u)));
    if (qd == 0) sm.wsum[warp][h] = ws;
    __syncthreads();
    float csum = 0.0f;
#pragma unroll
    for (int w = 0; w < kSW; ++w) csum += sm.wsum[w][h];
    l_run = l_run * alpha + csum;
    m_run = m_new;

    // O += P V over the chunk's 64 positions, this warp's 32 dims (4 n-tiles)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      oacc[nt][0] *= alpha;
      oacc[nt][1] *= alpha;
    }
#pragma unroll
    for (int kt = 0; kt < kChunk / 16; ++kt) {
      const uint32_t a0 = sm.p[h][8 * kt + qd], a2 = sm.p[h][8 * kt + 4 + qd];
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        // x4.trans: positions 16 kt + lane % 8 (+ 8 for matrices 1, 3), dims of n-tiles 2 np, 2 np + 1
        const int pos = 16 * kt + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int dim = 32 * warp + 16 * np + 8 * (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(smem_u32(&sm.v[buf][pos][dim * 2]), b0, b1, b2, b3);
        if (F8) {
          mma_f16_16816(oacc[2 * np], a0, a2, b0, b1);
          mma_f16_16816(oacc[2 * np + 1], a0, a2, b2, b3);
        } else {
          mma_bf16_16816(oacc[2 * np], a0, 0u, a2, 0u, b0, b1);
          mma_bf16_16816(oacc[2 * np + 1], a0, 0u, a2, 0u, b2, b3);
        }
      }
    }
    __syncthreads();  // buffer buf and the P tile are free
    if (F8) {
      if (cidx + 1 < nch) {
        store_chunk(cidx + 1);  // its codes arrived during this chunk
        fetch_raw(cidx + 2);
      }
    } else if (cidx + 2 < nch) {
      load_chunk(cidx + 2);
    }
  }

  // this CTA's state of head h into slot (h / C) * C + r of CTA h % C, which finalises it
  if (h < G) {
    const int slot = (h / C) * C + r;
    const uint32_t dst = (uint32_t)(h % C);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int dim = 32 * warp + 8 * nt + 2 * qd;
      st_cluster_v2(cluster_addr(&sm.o[slot][dim], dst), oacc[nt][0], oacc[nt][1]);
    }
    if (warp == 0 && qd == 0) {
      st_cluster_f32(cluster_addr(&sm.m[slot], dst), m_run);
      st_cluster_f32(cluster_addr(&sm.l[slot], dst), l_run);
    }
  }
  uint16_t sig[kFin];
#pragma unroll
  for (int k = 0; k < kFin; ++k) sig[k] = (r + C * k < G && p.fuse_gate) ? sigmoid_bf16(gbits[k]) : (uint16_t)0;

  // every state has arrived where it is merged after this; afterwards each CTA reads
  // only its own shared memory, so no second barrier is needed before leaving
  cluster_sync_all();

#pragma unroll
  for (int k = 0; k < kFin; ++k) {
    const int hl = r + C * k;
    if (hl >= G) break;
    // query head hf: merge the C states (and the sink), normalise, round, gate
    const int hf = kvh * G + hl;
    const float sink2 = (p.sinks != nullptr) ? __ldg(p.sinks + hf) * 1.44269504088896340736f : -INFINITY;
    float M = sink2;
#pragma unroll
    for (int x = 0; x < C; ++x) M = fmaxf(M, sm.m[k * C + x]);
    float acc = 0.0f, W = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int x = 0; x < C; ++x) {
        const float f = safe_exp2_diff(sm.m[k * C + x], M);
        acc = fmaf(sm.o[k * C + x][tid], f, acc);
        W = fmaf(sm.l[k * C + x], f, W);
      }
      if (sink2 != -INFINITY) W += exp2f(sink2 - M);
      acc = F8 ? acc * p.v_descale / W : acc / W;
    }
    const uint16_t ob = float_to_bf16_bits(acc);
    const size_t row = ((size_t)b * p.Hq + hf) * kD;
    reinterpret_cast<uint16_t*>(p.out)[row + tid] = p.fuse_gate ? gate_product_bf16(ob, sig[k]) : ob;
    if (p.lse_out != nullptr && tid == 0)
      p.lse_out[(size_t)b * p.Hq + hf] = (M == -INFINITY) ? -INFINITY : (M + log2f(W)) * 0.69314718055994530942f;
  }
}

namespace {

template <int C>
cudaError_t small_attr_c() {
  const cudaError_t e =
      cudaFuncSetAttribute(small_decode_kernel<C, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(small_decode_kernel<C, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmallSmem);
}

// cluster index 0, 1, 2, 3 for C = 8, 4, 2, 1
int cidx_of(int C) { return C == 8 ? 0 : (C == 4 ? 1 : (C == 2 ? 2 : 3)); }

// per device and cluster size (idempotent; atomics, as calls may come from any thread)
std::atomic<bool> g_small_attr[64][4];
std::atomic<int> g_small_clusters[64][4];

cudaError_t small_attr(int dev, int C) {
  std::atomic<bool>& done = g_small_attr[dev][cidx_of(C)];
  if (!done) {
    const cudaError_t e = (C == 8)   ? small_attr_c<8>()
                          : (C == 4) ? small_attr_c<4>()
                          : (C == 2) ? small_attr_c<2>()
                                     : small_attr_c<1>();
    if (e != cudaSuccess) return e;
    done = true;
  }
  return cudaSuccess;
}

void cluster_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int C, dim3 grid, cudaStream_t stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = grid;
  cfg->blockDim = dim3(kSW * 32, 1, 1);
  cfg->dynamicSmemBytes = kSmallSmem;
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

}  // namespace

int small_max_clusters(int C) {
  if (C != 8 && C != 4 && C != 2 && C != 1) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::atomic<int>& n = g_small_clusters[dev][cidx_of(C)];
  if (n == 0) {
    if (small_attr(dev, C) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    cluster_config(&cfg, attr, C, dim3((unsigned)C, 1, 1), nullptr);
    int got = 0;
    // (the e4m3 instances have the same launch shape and shared memory)
    const cudaError_t e = (C == 8)   ? cudaOccupancyMaxActiveClusters(&got, small_decode_kernel<8, false>, &cfg)
                          : (C == 4) ? cudaOccupancyMaxActiveClusters(&got, small_decode_kernel<4, false>, &cfg)
                          : (C == 2) ? cudaOccupancyMaxActiveClusters(&got, small_decode_kernel<2, false>, &cfg)
                                     : cudaOccupancyMaxActiveClusters(&got, small_decode_kernel<1, false>, &cfg);
    if (e != cudaSuccess || got <= 0) {
      (void)cudaGetLastError();
      return 0;
    }
    n = got;
  }
  return n;
}

int small_cluster_for(long long pairs, int max_len) {
  if (max_len <= 0 || max_len > kSmallMaxLen) return 0;
  for (int C = 8; C >= 1; C /= 2)
    if (max_len <= 128 * C && pairs <= (long long)small_max_clusters(C)) return C;
  return 0;
}

cudaError_t launch_small(const SmallParams& p, int C, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = small_attr(dev, C);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  cluster_config(&cfg, attr, C, dim3((unsigned)C, (unsigned)p.Hkv, (unsigned)p.B), stream);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  if (p.kv_fp8) {
    if (C == 8) return cudaLaunchKernelEx(&cfg, small_decode_kernel<8, true>, p);
    if (C == 4) return cudaLaunchKernelEx(&cfg, small_decode_kernel<4, true>, p);
    if (C == 2) return cudaLaunchKernelEx(&cfg, small_decode_kernel<2, true>, p);
    if (C == 1) return cudaLaunchKernelEx(&cfg, small_decode_kernel<1, true>, p);
  } else {
    if (C == 8) return cudaLaunchKernelEx(&cfg, small_decode_kernel<8, false>, p);
    if (C == 4) return cudaLaunchKernelEx(&cfg, small_decode_kernel<4, false>, p);
    if (C == 2) return cudaLaunchKernelEx(&cfg, small_decode_kernel<2, false>, p);
    if (C == 1) return cudaLaunchKernelEx(&cfg, small_decode_kernel<1, false>, p);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gda
