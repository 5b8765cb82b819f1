// gda_stage1_tma.cu -- split-KV decode stage 1 fed by a TMA bulk-copy ring (sm_103a).
//
// This is the first stage-1 design, kept as a selectable variant for comparison.
// Measured on GB300 it is bound by the rate of 512-byte bulk copies (about 1.75
// TB/s for scattered 512-byte rows, against 6.7 TB/s for 16-byte vector loads
// from many warps), so the default stage 1 (gda_stage1.cu) loads K/V rows
// straight into registers instead.
//
// Per piece (sequence b, KV head kvh, positions [j0, j1)) and for the G = 8 query
// heads that share kvh, stage 1 computes the normalised partial
//   O_piece = sum_j softmax_piece(scale * q K_j^T) V_j      and     LSE_piece (log2 units)
// with a running max and running sum, as split-KV decode stage 1 does (FreeToken
// PR #781 "Fuse the BF16 attention output sigmoid gate into the existing Triton
// decode stage2", Summary: stage1 and the stage2 FP32 reduction are kept).
//
// GB300 design:
//  * Persistent grid, one CTA per SM; the work schedule (gda_device.cuh) gives each
//    CTA an equal share of the batch's KV stream, so ragged batches stay balanced.
//  * One producer warp gathers the K and V rows of each 64-token tile behind the
//    CSR slot index with 1-D bulk copies (the TMA bulk engine, 512 B per row,
//    L2 evict-first) into a 3-stage shared-memory ring guarded by mbarriers; the
//    next tile's slot indices are prefetched while the current tile is issued.
//  * Consumer warps each take a fixed slice of every tile.  Each K/V byte is read
//    from HBM once and used by all 8 query heads of its group.
//  * Consumer arithmetic MathMma: QK^T and PV on mma.sync m16n8k16 bf16 tiles,
//    FP32 accumulate: S^T = K Q^T with the 8 heads as N, O^T += V^T P^T.
//  * At the end of a piece the consumer warps merge their states in shared memory
//    and write one partial; stage 2 merges partials across pieces.
//  * Every wait is bounded; a timeout (a kernel bug) sets an error bit and the CTA
//    winds down along the same control flow, so nothing can hang.
#include <atomic>
#include "gda_device.cuh"
#include "gda_kernels.h"

namespace gda {

__device__ __align__(16) unsigned char g_zero_row[kRowBytes];

template <int NCW, int WTOK, int NSTAGE>
struct Stage1Smem {
  static constexpr int kTile = NCW * WTOK;
  alignas(128) unsigned char k[NSTAGE][kTile][kSmemRow];
  alignas(128) unsigned char v[NSTAGE][kTile][kSmemRow];
  float obuf[kG][kD];
  float mbuf[NCW][kG];
  float lbuf[kG];
  alignas(8) uint64_t full[NSTAGE];
  alignas(8) uint64_t empty[NSTAGE];
  int abort_flag;
};

// ------------------------------------------------------------------ small helpers

// ------------------------------------------------------------------ MathMma
//
// Per 16-token slice (one warp): S^T[16 tok x 8 heads] = K[16 x 256] Q^T[256 x 8]
// as 16 m16n8k16 steps (K from shared memory by ldmatrix, Q^T fragments held in
// registers), the online softmax on the accumulator fragments (lane holds tokens
// lane/4 and lane/4+8 of heads 2(lane%4), 2(lane%4)+1), P rounded to BF16 and
// turned into the B operand by movmatrix.trans, then O^T[256 x 8] += V^T P^T as
// 16 m16n8k16 steps (V^T from shared memory by ldmatrix.trans).  The running sum
// adds the same BF16-rounded probabilities that multiply V.

template <int WTOK>
struct MathMma {
  static_assert(WTOK == 16, "one m16 tile per warp");
  uint32_t qb[16][2];
  float o[16][4];
  float m0, m1;  // heads 2(lane%4), 2(lane%4)+1
  float l0, l1;  // per-lane partial sums, reduced at the merge

  __device__ __forceinline__ void load_q(const __nv_bfloat16* qg, int gv, int lane) {
    const int h = lane >> 2, dq = 2 * (lane & 3);
    const uint32_t* base = reinterpret_cast<const uint32_t*>(qg + min(h, gv - 1) * kD);  // stays in the group
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      qb[kk][0] = (h < gv) ? __ldg(base + (kk * 16 + dq) / 2) : 0u;
      qb[kk][1] = (h < gv) ? __ldg(base + (kk * 16 + dq + 8) / 2) : 0u;
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[dt][i] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
  }

  __device__ __forceinline__ void tile(const unsigned char* kb, const unsigned char* vb, int nv, float sl2,
                                       int lane) {
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t kaddr = smem_u32(kb) + (lane & 15) * kSmemRow + (lane >> 4) * 16;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 2) {
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      ldsm_x4(kaddr + kk * 32, a0, a1, a2, a3);
      ldsm_x4(kaddr + (kk + 1) * 32, c0, c1, c2, c3);
      mma_bf16_16816(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      mma_bf16_16816(sb, c0, c1, c2, c3, qb[kk + 1][0], qb[kk + 1][1]);
    }
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = (sa[i] + sb[i]) * sl2;
    const int t0 = lane >> 2;
    if (t0 >= nv) s[0] = s[1] = -INFINITY;
    if (t0 + 8 >= nv) s[2] = s[3] = -INFINITY;
    float xa = fmaxf(s[0], s[2]), xb = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, off));
    }
    const float na = fmaxf(m0, xa), nb = fmaxf(m1, xb);
    const float aa = safe_exp2_diff(m0, na), ab = safe_exp2_diff(m1, nb);
    const uint32_t P0 = pack_bf16x2(safe_exp2_diff(s[0], na), safe_exp2_diff(s[1], nb));
    const uint32_t P1 = pack_bf16x2(safe_exp2_diff(s[2], na), safe_exp2_diff(s[3], nb));
    l0 = l0 * aa + (__uint_as_float(P0 << 16) + __uint_as_float(P1 << 16));
    l1 = l1 * ab + (__uint_as_float(P0 & 0xFFFF0000u) + __uint_as_float(P1 & 0xFFFF0000u));
    m0 = na;
    m1 = nb;
    if (__any_sync(0xffffffffu, (aa != 1.0f) || (ab != 1.0f))) {
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        o[dt][0] *= aa;
        o[dt][1] *= ab;
        o[dt][2] *= aa;
        o[dt][3] *= ab;
      }
    }
    const uint32_t b0 = movmatrix_trans(P0), b1 = movmatrix_trans(P1);
    const int mj = lane >> 3, mr = lane & 7;
    const uint32_t vaddr = smem_u32(vb) + (mr + 8 * (mj >> 1)) * kSmemRow + 16 * (mj & 1);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(vaddr + dt * 32, a0, a1, a2, a3);
      mma_bf16_16816(o[dt], a0, a1, a2, a3, b0, b1);
    }
  }

  template <int NCW>
  __device__ __forceinline__ void publish_max(float (*mbuf)[kG], int w, int lane) {
    if (lane < 4) {
      mbuf[w][2 * lane] = m0;
      mbuf[w][2 * lane + 1] = m1;
    }
  }

  // Reduce the per-lane running sums over the 8 lanes that share a head pair
  // (done by every warp before the ordered accumulation).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }

  template <int NCW>
  __device__ __forceinline__ void accumulate(const float (*mbuf)[kG], float (*obuf)[kD], float* lbuf, int w,
                                             int lane, bool first) {
    const int ha = 2 * (lane & 3), hb = ha + 1, g = lane >> 2;
    float Ma = mbuf[0][ha], Mb = mbuf[0][hb];
#pragma unroll
    for (int x = 1; x < NCW; ++x) {
      Ma = fmaxf(Ma, mbuf[x][ha]);
      Mb = fmaxf(Mb, mbuf[x][hb]);
    }
    const float fa = (Ma == -INFINITY) ? 0.0f : safe_exp2_diff(m0, Ma);
    const float fb = (Mb == -INFINITY) ? 0.0f : safe_exp2_diff(m1, Mb);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      const int d = dt * 16 + g;
      float v0 = o[dt][0] * fa, v2 = o[dt][2] * fa, v1 = o[dt][1] * fb, v3 = o[dt][3] * fb;
      if (!first) {
        v0 += obuf[ha][d];
        v2 += obuf[ha][d + 8];
        v1 += obuf[hb][d];
        v3 += obuf[hb][d + 8];
      }
      obuf[ha][d] = v0;
      obuf[ha][d + 8] = v2;
      obuf[hb][d] = v1;
      obuf[hb][d + 8] = v3;
    }
    if (lane < 4) {
      lbuf[ha] = first ? l0 * fa : lbuf[ha] + l0 * fa;
      lbuf[hb] = first ? l1 * fb : lbuf[hb] + l1 * fb;
    }
  }
};

// ------------------------------------------------------------------ the kernel

template <class Math, int NCW, int WTOK, int NSTAGE>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) stage1_kernel(Stage1Params p) {
  using Smem = Stage1Smem<NCW, WTOK, NSTAGE>;
  constexpr int kTile = Smem::kTile;
  constexpr int kConsumers = NCW * 32;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], NCW);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kG * kD; i += blockDim.x) (&sm.obuf[0][0])[i] = 0.0f;
  if (threadIdx.x < kG) sm.lbuf[threadIdx.x] = 0.0f;
  __syncthreads();

  Sched sched;
  sched.begin(p.indptr, p.B, p.Hkv * p.npass, p.num_splits, gridDim.x, blockIdx.x, p.min_chunk, p.window, p.piece_cost, p.rule_kv8);
  // Stage 2 may start its prologue (gate loads and sigmoids) once this CTA knows it has
  // work: an idle CTA (the automatic plan launches a full grid) exits without the
  // trigger, which counts as one, so stage 2's CTAs are placed after the idle CTAs have
  // left.  (Measured: idle CTAs that stay resident while stage 2 is placed slowed stage
  // 2's merge by ~3 us on B1 L32768.)
  {
    Sched peek = sched;
    Piece first;
    if (peek.next(first)) pdl_launch_dependents();
  }
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == NCW) {
    // ---------------------------------------------------------------- producer
    const uint64_t pol = l2_policy_evict_first();
    constexpr int kPer = (kTile + 31) / 32;
    const size_t slot_stride = (size_t)p.Hkv * kRowBytes;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int issued = 0;

    // tile cursor over the CTA's pieces
    Piece pc;
    bool have = sched.next(pc);
    int t0 = have ? pc.j0 : 0;
    int cur_slot[kPer];
    int cur_n = 0, cur_kvh = 0;
    auto load_slots = [&](const Piece& pp, int tt0, int* slots) -> int {
      const int n = min(kTile, pp.j1 - tt0);
      const int* idx = p.indices + pp.base + tt0;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int rr = lane + 32 * r;
        slots[r] = (rr < n) ? __ldg(idx + rr) : -1;
      }
      return n;
    };
    if (have) {
      cur_n = load_slots(pc, t0, cur_slot);
      cur_kvh = pc.kvh / p.npass;
    }
    while (have) {
      if (*abort_flag) {
        ok = false;
        break;
      }
      // advance the cursor and prefetch the next tile's slots
      int nxt_slot[kPer];
      int nxt_n = 0, nxt_kvh = 0;
      t0 += kTile;
      if (t0 >= pc.j1) {
        have = sched.next(pc);
        if (have) t0 = pc.j0;
      }
      if (have) {
        nxt_n = load_slots(pc, t0, nxt_slot);
        nxt_kvh = pc.kvh / p.npass;
      }
      // issue the current tile
      if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, p.wait_limit)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&sm.full[stage], kTile * 2 * kRowBytes);
      __syncwarp();
      const size_t head_off = (size_t)cur_kvh * kRowBytes;
#pragma unroll
      for (int r = 0; r < kPer; ++r) {
        const int rr = lane + 32 * r;
        if (rr < kTile) {
          const unsigned char* ks = g_zero_row;
          const unsigned char* vs = g_zero_row;
          const int slot = cur_slot[r];
          if (rr < cur_n) {
            const bool bad = p.check_indices && (slot < 0 || (long long)slot >= p.num_slots);
            if (bad) {
              atomicOr(&p.hdr->error, kErrIndex);
            } else {
              ks = p.k_pool + (size_t)slot * slot_stride + head_off;
              vs = p.v_pool + (size_t)slot * slot_stride + head_off;
            }
          }
          bulk_g2s(&sm.k[stage][rr][0], ks, kRowBytes, &sm.full[stage], pol);
          bulk_g2s(&sm.v[stage][rr][0], vs, kRowBytes, &sm.full[stage], pol);
        }
      }
      ++issued;
      if (++stage == NSTAGE) {
        stage = 0;
        phase ^= 1u;
      }
#pragma unroll
      for (int r = 0; r < kPer; ++r) cur_slot[r] = nxt_slot[r];
      cur_n = nxt_n;
      cur_kvh = nxt_kvh;
    }
    if (!ok || *abort_flag) {
      if (lane == 0) {
        atomicOr(&p.hdr->error, kErrTimeout);
        sm.abort_flag = 1;
      }
      // let the copies already issued land before the CTA can exit
      const int inflight = min(issued, NSTAGE);
      int s = stage;
      uint32_t ph = phase;
      for (int k = 0; k < inflight; ++k) {
        if (--s < 0) {
          s = NSTAGE - 1;
          ph ^= 1u;
        }
        const long long t_start = clock64();
        while (!mbar_try_wait(&sm.full[s], ph) && clock64() - t_start < kWaitLimitCycles) {
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  Math math;
  int stage = 0;
  uint32_t phase = 0;
  bool aborted = false;
  Piece pc;
  while (sched.next(pc)) {
    {
      // query heads of virtual head pc.kvh: up to 8 of KV head pc.kvh / npass
      const int kvh = pc.kvh / p.npass, pass = pc.kvh - kvh * p.npass;
      const int gv = min(kG, p.G - kG * pass);
      math.load_q(p.q + ((size_t)pc.b * p.Hq + (size_t)kvh * p.G + (size_t)kG * pass) * kD, gv, lane);
    }
    math.reset();
    for (int t0 = pc.j0; t0 < pc.j1; t0 += kTile) {
      const int n = min(kTile, pc.j1 - t0);
      const int nv = max(0, min(WTOK, n - warp * WTOK));
      if (!aborted && !mbar_wait(&sm.full[stage], phase, abort_flag, p.wait_limit)) {
        aborted = true;
        if (lane == 0) {
          atomicOr(&p.hdr->error, kErrTimeout);
          sm.abort_flag = 1;
        }
      }
      if (!aborted && nv > 0)
        math.tile(&sm.k[stage][warp * WTOK][0], &sm.v[stage][warp * WTOK][0], nv, p.scale_log2, lane);
      __syncwarp();
      // a warp that gave up frees no stage: its copies may still be landing, and the
      // producer (which then sees the abort) must not refill it
      if (lane == 0 && !aborted) mbar_arrive(&sm.empty[stage]);
      if (++stage == NSTAGE) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // ---- merge the consumer warps' states and write the piece's partial
    math.finish_sums();
    math.template publish_max<NCW>(sm.mbuf, warp, lane);
    named_bar_sync(1, kConsumers);
    // ordered accumulation: deterministic summation order across warps
#pragma unroll 1
    for (int x = 0; x < NCW; ++x) {
      if (warp == x) math.template accumulate<NCW>(sm.mbuf, sm.obuf, sm.lbuf, warp, lane, x == 0);
      named_bar_sync(1, kConsumers);
    }
    float* op = p.o_part + pc.id * (kG * kD);
    const int tid = threadIdx.x;
    for (int e = tid * 4; e < kG * kD; e += kConsumers * 4) {
      const int h = e / kD;
      const float lsum = sm.lbuf[h];
      const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
      float4 v = *reinterpret_cast<const float4*>(&sm.obuf[0][0] + e);
      v.x *= inv;
      v.y *= inv;
      v.z *= inv;
      v.w *= inv;
      *reinterpret_cast<float4*>(op + e) = v;
    }
    if (tid < kG) {
      float M = sm.mbuf[0][tid];
#pragma unroll
      for (int x = 1; x < NCW; ++x) M = fmaxf(M, sm.mbuf[x][tid]);
      const float lsum = sm.lbuf[tid];
      p.lse_part[pc.id * kG + tid] = (lsum > 0.0f) ? M + log2f(lsum) : -INFINITY;
    }
    named_bar_sync(1, kConsumers);
  }
}

// ------------------------------------------------------------------ launchers

template <class Math, int NCW, int WTOK, int NSTAGE>
static cudaError_t launch_variant(const Stage1Params& p, int grid, cudaStream_t stream) {
  using Smem = Stage1Smem<NCW, WTOK, NSTAGE>;
  auto kern = stage1_kernel<Math, NCW, WTOK, NSTAGE>;
  const size_t smem = sizeof(Smem);
  // the shared-memory opt-in is per device; set it once per device
  static std::atomic<bool> attr_set[64];  // zero-initialised: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<grid, (NCW + 1) * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_stage1_tma(const Stage1Params& p, int grid, cudaStream_t stream) {
  return launch_variant<MathMma<16>, 4, 16, 3>(p, grid, stream);
}

}  // namespace gda
