// gda_stage1.cu -- split-KV decode stage 1 on sm_103a, K/V rows loaded straight
// into registers.
//
// Per piece (sequence b, KV head kvh, positions [j0, j1)) and for a group of up to
// 8 query heads that share kvh (with G = 9..16 on the MMA kernel, both groups at
// once), stage 1 computes the normalised partial
//   O_piece = sum_j softmax_piece(scale * q K_j^T) V_j     and     LSE_piece (log2 units)
// with a running max and running sum, as split-KV decode stage 1 does (FreeToken
// PR #781 "Fuse the BF16 attention output sigmoid gate into the existing Triton
// decode stage2", Summary: stage1 and the stage2 FP32 reduction are kept).
//
// GB300 design.  The K/V rows behind the CSR slot index are 512-byte rows at
// scattered addresses (page size 1).  Measured on GB300, 16-byte vector loads
// issued by many warps stream such rows at ~6.7 TB/s, while one 1-D bulk copy per
// row is limited by the copy-request rate (~1.75 TB/s), so:
//  * Persistent grid, one CTA of 8 warps per SM; the work schedule (gda_device.cuh)
//    gives each CTA an equal share of the batch's KV stream.
//  * Warp w takes 16-token tiles w, w+8, ... of the CTA's piece.  K rows are
//    loaded with 16-byte streaming loads straight into mma.sync fragment
//    registers one tile ahead (and prefetched into L2 two tiles ahead); V rows go
//    through a per-warp 3-stage cp.async ring in shared memory, two tiles ahead,
//    with an L2 evict-first hint so the streamed rows do not push the indices,
//    q and the partials out of L2.
//  * The first loads of the next piece (its Q^T fragments, slots and first K
//    tile) are issued before the current piece's merge, so a piece boundary does
//    not restart the pipeline from an empty memory queue.
//  * MMA arithmetic: S^T[16 tok x 8 heads] = K Q^T and O^T[256 x 8] += V^T P^T on
//    m16n8k16 bf16 tiles with FP32 accumulation.  For QK the head dimension is
//    permuted (consistently for Q and K) so every 16-byte K load lands in fragment
//    slots: lane (g, t) holds dims {32c + 8t .. +7} of tokens g and g+8.  V^T
//    fragments come from the ring through ldmatrix.trans.  P is rounded to BF16
//    and turned into the B operand with movmatrix.trans; the running sum adds
//    the same rounded values.
//  * SIMT arithmetic (variant): lane l owns dims [8l, 8l+8) of every row; 64 FP32
//    FMAs per token and a transposing warp-shuffle reduction for the 8 scores.
//  * At the end of a piece each warp writes its rescaled O into its (idle) ring
//    and all threads add the 8 slices in a fixed order (deterministic); one
//    partial is written per piece.
#include <atomic>
#include "gda_device.cuh"
#include "gda_kernels.h"

namespace gda {

constexpr int kDirectWarps = 8;

// Query heads of virtual head vh (a group of up to 8 query heads sharing KV head
// vh / npass): their first row in q and how many of the 8 slots are real.
__device__ __forceinline__ const __nv_bfloat16* group_q(const Stage1Params& p, int b, int vh, int* gv) {
  const int kvh = vh / p.npass, pass = vh - kvh * p.npass;
  *gv = min(kG, p.G - kG * pass);
  return p.q + ((size_t)b * p.Hq + (size_t)kvh * p.G + (size_t)kG * pass) * kD;
}

__device__ __forceinline__ uint4 ld_stream(const unsigned char* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void unpack8(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

struct DirectSmem {
  float obuf[kG][kD];             // merge: O of the piece
  float mbuf[kDirectWarps][kG];   // merge: each warp's running max
  float lbuf[kG];                 // merge: running sums
};

// ------------------------------------------------------------------ MMA arithmetic
//
// Warp tile: 16 tokens.  K rows go straight into registers (one tile ahead) in a
// permuted head-dim order that matches the mma.sync A fragments: lane (g, t)
// holds dims {32c + 8t .. +7} of tokens g and g+8, and k-step kk = 2c + h uses
// dims 32c + 8t + 4h + {0,1} for k-slots (2t, 2t+1) and + {2,3} for (2t+8, 2t+9);
// the Q^T fragments use the same order.  V rows go through a per-warp cp.async
// ring in shared memory (two tiles ahead) and reach the V^T fragments through
// ldmatrix.trans.  O^T accumulators: o[dt] = {O[2t][16dt+g], O[2t+1][16dt+g],
// O[2t][16dt+g+8], O[2t+1][16dt+g+8]}.

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int NWARP, int NV, int NG>
struct MmaSmem {
  uint2 qf[NG][16][32];                                  // Q^T fragments per group, lane order
  unsigned char vring[NWARP][NV][16][kSmemRow];          // per-warp V rings
  float mbuf[NWARP][kG];                                 // each warp's running max
  float lsum[NWARP][kG];                                 // each warp's rescaled sum
  // NG > 1: each warp's S^T of its tile for the other NG - 1 groups of its team
  // (slot i for group i, or i - 1 past the warp's own group), double-buffered
  float4 xs[NG > 1 ? NWARP : 1][2][NG > 1 ? NG - 1 : 1][32];
};

// Lazy-rescale threshold of the MMA softmax, in log2 units.
constexpr float kLazyLog2 = 8.0f;

struct MmaWarpState {
  uint4 kr[16];
  float o[16][4];
  float m0, m1, l0, l1;
  uint32_t P0, P1;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[i][j] = 0.0f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.0f;
  }

  __device__ __forceinline__ void load_k(const unsigned char* kb, size_t stride, int slot_lane, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const int s0 = __shfl_sync(0xffffffffu, slot_lane, g);
    const int s1 = __shfl_sync(0xffffffffu, slot_lane, g + 8);
    const unsigned char* p0 = kb + (size_t)max(s0, 0) * stride + 16 * t;
    const unsigned char* p1 = kb + (size_t)max(s1, 0) * stride + 16 * t;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int c = 0; c < 8; ++c) kr[c] = (s0 >= 0) ? ld_stream(p0 + 64 * c) : z;
#pragma unroll
    for (int c = 0; c < 8; ++c) kr[8 + c] = (s1 >= 0) ? ld_stream(p1 + 64 * c) : z;
  }

  __device__ __forceinline__ void qk_softmax(const uint2 (*qf)[32], int nv, float sl2, int lane) {
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const int c = kk >> 1, h = kk & 1;
      const uint4& r0 = kr[c];
      const uint4& r1 = kr[8 + c];
      const uint32_t a0 = h ? r0.z : r0.x, a2 = h ? r0.w : r0.y;
      const uint32_t a1 = h ? r1.z : r1.x, a3 = h ? r1.w : r1.y;
      const uint2 b = qf[kk][lane];
      mma_bf16_16816((kk & 1) ? sb : sa, a0, a1, a2, a3, b.x, b.y);
    }
    float s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = (sa[i] + sb[i]) * sl2;
    const int tg = lane >> 2;
    if (tg >= nv) s[0] = s[1] = -INFINITY;
    if (tg + 8 >= nv) s[2] = s[3] = -INFINITY;
    // Lazy rescale: the reference maxima m0/m1 move only when a score exceeds
    // them by more than kLazyLog2 (probabilities then stay below 2^kLazyLog2);
    // otherwise no max reduction and no rescale of O are needed.  The result is
    // the same softmax: every probability and sum is relative to one reference.
    const bool grow = fmaxf(s[0], s[2]) > m0 + kLazyLog2 || fmaxf(s[1], s[3]) > m1 + kLazyLog2;
    if (__any_sync(0xffffffffu, grow)) {
      float xa = fmaxf(s[0], s[2]), xb = fmaxf(s[1], s[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, off));
      }
      const float na = fmaxf(m0, xa), nb = fmaxf(m1, xb);
      const float aa = safe_exp2_diff(m0, na), ab = safe_exp2_diff(m1, nb);
      l0 *= aa;
      l1 *= ab;
      m0 = na;
      m1 = nb;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= aa;
        o[i][1] *= ab;
        o[i][2] *= aa;
        o[i][3] *= ab;
      }
    }
    P0 = pack_bf16x2(safe_exp2_diff(s[0], m0), safe_exp2_diff(s[1], m1));
    P1 = pack_bf16x2(safe_exp2_diff(s[2], m0), safe_exp2_diff(s[3], m1));
    l0 += __uint_as_float(P0 << 16) + __uint_as_float(P1 << 16);
    l1 += __uint_as_float(P0 & 0xFFFF0000u) + __uint_as_float(P1 & 0xFFFF0000u);
  }

  // Unscaled S^T of the register K tile against the Q^T fragments of NG groups (one
  // A fragment, two MMA chains per group; the same summation order as qk_softmax).
  template <int NG>
  __device__ __forceinline__ void qk_rawN(const uint2 (*const qf)[16][32], float (*s_out)[4], int lane) {
    float a[NG][2][4];
#pragma unroll
    for (int x = 0; x < NG; ++x)
#pragma unroll
      for (int i = 0; i < 4; ++i) a[x][0][i] = a[x][1][i] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const int c = kk >> 1, h = kk & 1;
      const uint4& r0 = kr[c];
      const uint4& r1 = kr[8 + c];
      const uint32_t x0 = h ? r0.z : r0.x, x2 = h ? r0.w : r0.y;
      const uint32_t x1 = h ? r1.z : r1.x, x3 = h ? r1.w : r1.y;
#pragma unroll
      for (int x = 0; x < NG; ++x) {
        const uint2 f = qf[x][kk][lane];
        mma_bf16_16816(a[x][h], x0, x1, x2, x3, f.x, f.y);
      }
    }
#pragma unroll
    for (int x = 0; x < NG; ++x)
#pragma unroll
      for (int i = 0; i < 4; ++i) s_out[x][i] = a[x][0][i] + a[x][1][i];
  }

  // Online softmax over NT 16-token tiles of the same 8 heads: tile x has n[x] valid
  // rows and unscaled scores s[x].  Same lazy rescale as qk_softmax; returns the BF16 P
  // fragments of each tile and adds their rounded values to the sums, tile by tile.
  template <int NT>
  __device__ __forceinline__ void softmaxN(float (*s)[4], const int* n, float sl2, int lane, uint32_t (*P)[2]) {
    const int tg = lane >> 2;
    float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
    for (int x = 0; x < NT; ++x) {
#pragma unroll
      for (int i = 0; i < 4; ++i) s[x][i] *= sl2;
      if (tg >= n[x]) s[x][0] = s[x][1] = -INFINITY;
      if (tg + 8 >= n[x]) s[x][2] = s[x][3] = -INFINITY;
      xa = fmaxf(xa, fmaxf(s[x][0], s[x][2]));
      xb = fmaxf(xb, fmaxf(s[x][1], s[x][3]));
    }
    const bool grow = xa > m0 + kLazyLog2 || xb > m1 + kLazyLog2;
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, off));
      }
      const float na_ = fmaxf(m0, xa), nb_ = fmaxf(m1, xb);
      const float aa = safe_exp2_diff(m0, na_), ab = safe_exp2_diff(m1, nb_);
      l0 *= aa;
      l1 *= ab;
      m0 = na_;
      m1 = nb_;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= aa;
        o[i][1] *= ab;
        o[i][2] *= aa;
        o[i][3] *= ab;
      }
    }
    float la = 0.0f, lb = 0.0f;
#pragma unroll
    for (int x = 0; x < NT; ++x) {
      P[x][0] = pack_bf16x2(safe_exp2_diff(s[x][0], m0), safe_exp2_diff(s[x][1], m1));
      P[x][1] = pack_bf16x2(safe_exp2_diff(s[x][2], m0), safe_exp2_diff(s[x][3], m1));
      la += __uint_as_float(P[x][0] << 16) + __uint_as_float(P[x][1] << 16);
      lb += __uint_as_float(P[x][0] & 0xFFFF0000u) + __uint_as_float(P[x][1] & 0xFFFF0000u);
    }
    l0 += la;
    l1 += lb;
  }

  // O^T += V^T P^T with V^T fragments from a 16-row shared-memory tile
  __device__ __forceinline__ void pv(const unsigned char* vtile, int lane) { pv_with(vtile, P0, P1, lane); }

  __device__ __forceinline__ void pv_with(const unsigned char* vtile, uint32_t p0, uint32_t p1, int lane) {
    const uint32_t b0 = movmatrix_trans(p0), b1 = movmatrix_trans(p1);
    const int mj = lane >> 3, mr = lane & 7;
    const uint32_t vaddr = smem_u32(vtile) + (mr + 8 * (mj >> 1)) * kSmemRow + 16 * (mj & 1);
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(vaddr + dt * 32, a0, a1, a2, a3);
      mma_bf16_16816(o[dt], a0, a1, a2, a3, b0, b1);
    }
  }
};

// Prefetch into L2 the K rows of a 16-token tile (two lanes per 512-byte row,
// two 128-byte lines each): the whole row is requested from HBM at once, and the
// later register loads of that tile (64 bytes per row per instruction) hit L2.
__device__ __forceinline__ void prefetch_k_tile(const unsigned char* kb, size_t stride, int slot_lane, int lane) {
  const int s = __shfl_sync(0xffffffffu, slot_lane, lane >> 1);
  if (s >= 0) {
    const unsigned char* row = kb + (size_t)s * stride + 256 * (lane & 1);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 128));
  }
}

// Issue the cp.async copies of one V tile (16 rows; rows >= n and bad slots are
// zero-filled) into a ring stage and commit them as one group.
__device__ __forceinline__ void issue_v_tile(unsigned char* stage, const unsigned char* vb, size_t stride,
                                             int slot_lane, int n, int lane, uint64_t policy) {
  const uint32_t dst0 = smem_u32(stage) + 16 * lane;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int s = __shfl_sync(0xffffffffu, slot_lane, r);
    const bool ok = (r < n) && (s >= 0);
    const unsigned char* src = vb + (ok ? (size_t)s * stride : (size_t)0) + 16 * lane;
    cp_async16(dst0 + r * kSmemRow, src, ok ? 16u : 0u, policy);
  }
  cp_async_commit();
}

// Teams (NG > 1, G > 8: the groups of 8 query heads of a KV head in teams of NG):
// one piece per (sequence, KV head, team) serves the NG groups of the team, and every
// K/V row is loaded once per team (NG = 2: once for G = 9..16; NG = 3: once for
// G = 17..24).  Warp w loads tiles w + NWARP*k as with NG = 1 and computes S^T of its
// tile for all NG groups (one K fragment, NG MMA chains).  Warp w is member w / WPG
// of team w % WPG and owns group w / WPG.  Each step a warp leaves the other groups'
// S^T in shared memory, the team meets at a named barrier, and each warp then runs
// the softmax and PV of its own group over the team's NG tiles: its own (its V ring)
// and its partners' (their V rings).  The partial of (piece, group) is written at
// piece * NG + group.  With NG = 1, one piece per (sequence, virtual head).
template <int NWARP, int NV, int NG>
__global__ void __launch_bounds__(NWARP * 32, 1) stage1_mma_kernel(Stage1Params p) {
  constexpr bool TEAM = NG > 1;
  constexpr int WPG = NWARP / NG;        // warps per group (= teams per CTA)
  constexpr int QPT = NG * 16 / NWARP;   // Q^T fragments per thread
  using Smem = MmaSmem<NWARP, NV, NG>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WPG;   // this warp's group (its member index in the team)
  const int team = warp % WPG;  // its team: warps team + WPG * j, j = 0 .. NG - 1
  static_assert(NWARP % NG == 0 && (NG * 16) % NWARP == 0, "whole teams, whole Q fragments per thread");
  static_assert(WPG <= 15, "named barriers 1 .. WPG");

  Sched sched;
  sched.begin(p.indptr, p.B, TEAM ? p.Hkv * p.nteam : p.Hkv * p.npass, p.num_splits, gridDim.x, blockIdx.x,
              p.min_chunk, p.window, p.piece_cost, p.rule_kv8);
  const size_t stride = (size_t)p.Hkv * kRowBytes;
  const uint64_t pol_v = l2_policy_evict_first();
  // KV head of a piece (in teams the scheduled head is kvh * nteam + the team)
  auto kv_head = [&](const Piece& pp) -> int { return TEAM ? pp.kvh / p.nteam : pp.kvh / p.npass; };

  // Warp w's tiles of a piece of `len` positions: tile w + NWARP*k.
  auto nmine_for = [&](int w, int len) -> int {
    const int ntiles = (len + 15) >> 4;
    return (ntiles > w) ? (ntiles - w + NWARP - 1) / NWARP : 0;
  };
  auto tile_n_for = [&](int w, int k, int len, int nm) -> int {
    return (k < nm) ? min(16, len - 16 * (w + NWARP * k)) : 0;
  };
  auto nmine_of = [&](int len) -> int { return nmine_for(warp, len); };
  auto tile_n = [&](int k, int len, int nmine) -> int { return tile_n_for(warp, k, len, nmine); };
  auto fetch = [&](const int* idx, int k, int len, int nmine) -> int {
    const int n = tile_n(k, len, nmine);
    int s = -1;
    if (lane < n) {
      s = __ldg(idx + 16 * (warp + NWARP * k) + lane);
      if (p.check_indices && (s < 0 || (long long)s >= p.num_slots)) {
        atomicOr(&p.hdr->error, kErrIndex);
        s = -1;
      }
    }
    return s;
  };

  MmaWarpState st;
  uint2 qfrag[QPT];
  int s0 = -1, s1 = -1, s2 = -1;
  // Head of a piece: its Q^T fragments (requested first), the slots of this
  // warp's first three tiles and the K rows of its first tile.  For every piece
  // after the first this runs before the previous piece's merge, so the loads
  // are in flight while the warps merge.
  auto piece_head = [&](const Piece& pp) {
    // teams: the piece's KV head and the first group of its team
    const int pkv = TEAM ? pp.kvh / p.nteam : 0, pg0 = TEAM ? NG * (pp.kvh - pkv * p.nteam) : 0;
#pragma unroll
    for (int r = 0; r < QPT; ++r) {
      const int e = threadIdx.x + r * NWARP * 32;
      const int fg = e >> 9, kk = (e >> 5) & 15, ln = e & 31;  // group, k-step, lane
      int gv;
      const __nv_bfloat16* qg;
      if (TEAM) {
        // group NG * team + fg of the KV head; past the last group (npass not a
        // multiple of NG) the group is empty: its Q is zero and its partial is never read
        const int gi = pg0 + fg;
        qg = group_q(p, pp.b, pkv * p.npass + min(gi, p.npass - 1), &gv);
        if (gi >= p.npass) gv = 0;
      } else {
        qg = group_q(p, pp.b, pp.kvh, &gv);
      }
      const int g = ln >> 2, t = ln & 3, c = kk >> 1, h = kk & 1;
      const __nv_bfloat16* row = qg + max(0, min(g, gv - 1)) * kD;  // never addresses a row beyond the group
      qfrag[r] = (g < gv) ? __ldg(reinterpret_cast<const uint2*>(row + 32 * c + 8 * t + 4 * h)) : make_uint2(0u, 0u);
    }
    const int* idx = p.indices + pp.base + pp.j0;
    const int len = pp.j1 - pp.j0, nmine = nmine_of(len);
    s0 = fetch(idx, 0, len, nmine);
    s1 = fetch(idx, 1, len, nmine);
    s2 = fetch(idx, 2, len, nmine);
    if (nmine > 0) st.load_k(p.k_pool + (size_t)kv_head(pp) * kRowBytes, stride, s0, lane);
  };

  // Stage 2 may start its prologue (gate loads and sigmoids) once this CTA knows it has
  // work: an idle CTA (the automatic plan launches a full grid) exits without the
  // trigger, which counts as one, so stage 2's CTAs are placed after the idle CTAs have
  // left.  (Measured: idle CTAs that stay resident while stage 2 is placed slowed stage
  // 2's merge by ~3 us on B1 L32768.)
  Piece pc;
  bool have = sched.next(pc);
  if (have) pdl_launch_dependents();
  if (have) piece_head(pc);
  while (have) {
    const unsigned char* kb = p.k_pool + (size_t)kv_head(pc) * kRowBytes;
    const unsigned char* vb = p.v_pool + (size_t)kv_head(pc) * kRowBytes;
    const int* idx = p.indices + pc.base + pc.j0;
    const int len = pc.j1 - pc.j0;
    const int nmine = nmine_of(len);

    st.reset();  // O, max and sum; the K rows of tile 0 are already in flight
    unsigned char(*ring)[16][kSmemRow] = sm.vring[warp];
    // steps of this warp's loop: its tiles, or in teams those of the team's first
    // warp (the one with the most tiles), so that all members meet at every barrier
    const int nsteps = TEAM ? nmine_for(team, len) : nmine;
    if (nsteps > 0) {
      issue_v_tile(&ring[0][0][0], vb, stride, s0, tile_n(0, len, nmine), lane, pol_v);
      issue_v_tile(&ring[1 % NV][0][0], vb, stride, s1, tile_n(1, len, nmine), lane, pol_v);
      prefetch_k_tile(kb, stride, s1, lane);
    }
    // the previous piece's merge ended with a barrier: the fragment buffer is free
#pragma unroll
    for (int r = 0; r < QPT; ++r) {
      const int e = threadIdx.x + r * NWARP * 32;
      sm.qf[e >> 9][(e >> 5) & 15][e & 31] = qfrag[r];
    }
    __syncthreads();

    int stage = 0;
    if constexpr (TEAM) {
      // tile x of a step: x = 0 this warp's own, then its partners in member order
      int pw[NG];  // warp of tile x
      int nmp[NG];
#pragma unroll
      for (int x = 0; x < NG; ++x) {
        const int j = (x == 0) ? grp : (x - 1 < grp ? x - 1 : x);
        pw[x] = team + WPG * j;
        nmp[x] = nmine_for(pw[x], len);
      }
      const int bar = 1 + team;
      for (int k = 0; k < nsteps; ++k) {
        // K rows of tile k+2 into L2 and the slots of tile k+3; tile k's S^T for all
        // groups (the other groups' to shared memory); the K rows of tile k+1
        prefetch_k_tile(kb, stride, s2, lane);
        const int s3 = fetch(idx, k + 3, len, nmine);
        const int nown = tile_n(k, len, nmine);
        float sg[NG][4];
#pragma unroll
        for (int x = 0; x < NG; ++x) sg[x][0] = sg[x][1] = sg[x][2] = sg[x][3] = 0.0f;
        if (nown > 0) st.qk_rawN<NG>(sm.qf, sg, lane);
#pragma unroll
        for (int i = 0; i < NG; ++i)
          if (i != grp) sm.xs[warp][k & 1][i < grp ? i : i - 1][lane] = make_float4(sg[i][0], sg[i][1], sg[i][2], sg[i][3]);
        if (k + 1 < nmine) st.load_k(kb, stride, s1, lane);
        cp_async_wait<1>();  // this warp's V tile k has landed (tile k+1 may be in flight)
        // The team meets: all V tiles k and all S^T are visible, and every member has
        // finished step k-1, so ring stage (k+2) % NV (read as stage (k-1) % NV) and
        // the S^T buffer of step k+2 are free.
        named_bar_sync(bar, NG * 32);
        issue_v_tile(&ring[(k + 2) % NV][0][0], vb, stride, s2, tile_n(k + 2, len, nmine), lane, pol_v);
        float sc[NG][4];
        int nt[NG];
#pragma unroll
        for (int x = 0; x < NG; ++x) {
          if (x == 0) {
            // this warp's group's S^T (a select per group: no dynamic register index)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[0][i] = sg[0][i];
#pragma unroll
            for (int y = 1; y < NG; ++y)
              if (grp == y) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sc[0][i] = sg[y][i];
              }
            nt[0] = nown;
          } else {
            // the partner's slot for this warp's group
            const int j = pw[x] / WPG;
            const float4 sp = sm.xs[pw[x]][k & 1][grp < j ? grp : grp - 1][lane];
            sc[x][0] = sp.x;
            sc[x][1] = sp.y;
            sc[x][2] = sp.z;
            sc[x][3] = sp.w;
            nt[x] = tile_n_for(pw[x], k, len, nmp[x]);
          }
        }
        uint32_t P[NG][2];
        st.softmaxN<NG>(sc, nt, p.scale_log2, lane, P);
#pragma unroll
        for (int x = 0; x < NG; ++x)
          if (nt[x] > 0) st.pv_with(&sm.vring[pw[x]][stage][0][0], P[x][0], P[x][1], lane);
        stage = (stage + 1 == NV) ? 0 : stage + 1;
        s1 = s2;
        s2 = s3;
      }
    } else {
      for (int k = 0; k < nmine; ++k) {
        // V two tiles ahead (an empty group when there is no such tile), K rows of
        // that tile into L2, the slots three tiles ahead; then tile k's QK
        issue_v_tile(&ring[(k + 2) % NV][0][0], vb, stride, s2, tile_n(k + 2, len, nmine), lane, pol_v);
        prefetch_k_tile(kb, stride, s2, lane);
        const int s3 = fetch(idx, k + 3, len, nmine);
        st.qk_softmax(sm.qf[0], tile_n(k, len, nmine), p.scale_log2, lane);
        if (k + 1 < nmine) st.load_k(kb, stride, s1, lane);
        cp_async_wait<2>();
        __syncwarp();
        st.pv(&ring[stage][0][0], lane);
        __syncwarp();
        stage = (stage + 1 == NV) ? 0 : stage + 1;
        s1 = s2;
        s2 = s3;
      }
    }
    cp_async_wait<0>();
    __syncwarp();

    // look ahead: the next piece's first loads go out before this piece's merge
    Piece nx;
    const bool have_next = sched.next(nx);
    if (have_next) piece_head(nx);

    // ---- merge: per-warp slices in the (now idle) V rings, summed in a fixed order
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
      st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
    }
    if (lane < 4) {
      sm.mbuf[warp][2 * lane] = st.m0;
      sm.mbuf[warp][2 * lane + 1] = st.m1;
    }
    __syncthreads();
    {
      const int ha = 2 * (lane & 3), hb = ha + 1, g = lane >> 2;
      const int x0 = grp * WPG;  // this group's warps: x0 .. x0 + WPG - 1
      float Ma = sm.mbuf[x0][ha], Mb = sm.mbuf[x0][hb];
#pragma unroll
      for (int x = 1; x < WPG; ++x) {
        Ma = fmaxf(Ma, sm.mbuf[x0 + x][ha]);
        Mb = fmaxf(Mb, sm.mbuf[x0 + x][hb]);
      }
      const float fa = (Ma == -INFINITY) ? 0.0f : safe_exp2_diff(st.m0, Ma);
      const float fb = (Mb == -INFINITY) ? 0.0f : safe_exp2_diff(st.m1, Mb);
      float* slice = reinterpret_cast<float*>(&sm.vring[warp][0][0][0]);
#pragma unroll
      for (int dt = 0; dt < 16; ++dt) {
        const int d = dt * 16 + g;
        slice[ha * kD + d] = st.o[dt][0] * fa;
        slice[hb * kD + d] = st.o[dt][1] * fb;
        slice[ha * kD + d + 8] = st.o[dt][2] * fa;
        slice[hb * kD + d + 8] = st.o[dt][3] * fb;
      }
      if (lane < 4) {
        sm.lsum[warp][ha] = st.l0 * fa;
        sm.lsum[warp][hb] = st.l1 * fb;
      }
    }
    __syncthreads();
    // partial (piece, group) at piece * NG + group: NG * 8 heads from pc.id * NG
    float* op = p.o_part + pc.id * (NG * kG * kD);
    for (int e = threadIdx.x * 4; e < NG * kG * kD; e += blockDim.x * 4) {
      const int x0 = (e / (kG * kD)) * WPG, el = e % (kG * kD), h = el / kD;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float lt = 0.0f;
#pragma unroll
      for (int x = x0; x < x0 + WPG; ++x) {
        const float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(&sm.vring[x][0][0][0]) + el);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
        lt += sm.lsum[x][h];
      }
      const float inv = (lt > 0.0f) ? 1.0f / lt : 0.0f;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      *reinterpret_cast<float4*>(op + e) = acc;
    }
    if (threadIdx.x < NG * kG) {
      const int x0 = (threadIdx.x / kG) * WPG, h = threadIdx.x % kG;
      float M = sm.mbuf[x0][h], lt = 0.0f;
#pragma unroll
      for (int x = 1; x < WPG; ++x) M = fmaxf(M, sm.mbuf[x0 + x][h]);
#pragma unroll
      for (int x = 0; x < WPG; ++x) lt += sm.lsum[x0 + x][h];
      p.lse_part[pc.id * (NG * kG) + threadIdx.x] = (lt > 0.0f) ? M + log2f(lt) : -INFINITY;
    }
    __syncthreads();  // rings, Q fragments and merge buffers free for the next piece
    pc = nx;
    have = have_next;
  }
}

// ------------------------------------------------------------------ SIMT arithmetic

struct DirectSimt {
  static constexpr int kTok = 8;
  float q[kG][8];     // head h, dims 8l .. 8l+7
  float acc[kG][8];
  float m, l;         // head (lane >> 2)
  float p[kTok];
  float alpha;
  uint4 kr[kTok], vr[kTok];

  __device__ __forceinline__ void load_q_regs(const __nv_bfloat16* qg, int gv, int lane) {
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      const __nv_bfloat16* row = qg + min(h, gv - 1) * kD;  // never addresses a row beyond the group
      const uint4 r = (h < gv) ? __ldg(reinterpret_cast<const uint4*>(row + lane * 8)) : make_uint4(0u, 0u, 0u, 0u);
      unpack8(r, q[h]);
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < kG; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
    m = -INFINITY;
    l = 0.0f;
  }

  __device__ __forceinline__ void load_k(const unsigned char* kb, size_t stride, int slot_lane, int lane) {
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
      const int s = __shfl_sync(0xffffffffu, slot_lane, u);
      kr[u] = (s >= 0) ? ld_stream(kb + (size_t)max(s, 0) * stride + 16 * lane) : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  __device__ __forceinline__ void load_v(const unsigned char* vb, size_t stride, int slot_lane, int lane) {
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
      const int s = __shfl_sync(0xffffffffu, slot_lane, u);
      vr[u] = (s >= 0) ? ld_stream(vb + (size_t)max(s, 0) * stride + 16 * lane) : make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // Score of head (lane >> 2) for one K row: 64 FMAs, then a transposing
  // butterfly (4 + 2 + 1 exchanges halve the live head set while summing, two
  // more finish the sum).
  __device__ __forceinline__ float score(const uint4& kraw, int lane) const {
    float k[8];
    unpack8(kraw, k);
    float part[kG];
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) s = fmaf(q[h][i], k[i], s);
      part[h] = s;
    }
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float r4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float keep = b4 ? part[j + 4] : part[j];
      const float send = b4 ? part[j] : part[j + 4];
      r4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float r2[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float keep = b3 ? r4[j + 2] : r4[j];
      const float send = b3 ? r4[j] : r4[j + 2];
      r2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float r1 = (b2 ? r2[1] : r2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? r2[0] : r2[1], 4);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    return r1;
  }

  __device__ __forceinline__ void qk_softmax(const DirectSmem&, int nv, float sl2, int lane) {
    float s[kTok];
#pragma unroll
    for (int u = 0; u < kTok; ++u) s[u] = (u < nv) ? score(kr[u], lane) * sl2 : -INFINITY;
    float tmax = s[0];
#pragma unroll
    for (int u = 1; u < kTok; ++u) tmax = fmaxf(tmax, s[u]);
    const float mnew = fmaxf(m, tmax);
    alpha = safe_exp2_diff(m, mnew);
    float psum = 0.0f;
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
      p[u] = safe_exp2_diff(s[u], mnew);
      psum += p[u];
    }
    l = l * alpha + psum;
    m = mnew;
  }

  __device__ __forceinline__ void pv_lane(int lane) {
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      const float a = __shfl_sync(0xffffffffu, alpha, 4 * h);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] *= a;
    }
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
      float v[8];
      unpack8(vr[u], v);
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        const float ph = __shfl_sync(0xffffffffu, p[u], 4 * h);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(ph, v[i], acc[h][i]);
      }
    }
  }

  __device__ __forceinline__ void finish_sums() {}

  __device__ __forceinline__ void publish_max(DirectSmem& sm, int w, int lane) const {
    if ((lane & 3) == 0) sm.mbuf[w][lane >> 2] = m;
  }

  __device__ __forceinline__ void accumulate(DirectSmem& sm, int w, int lane, bool first) const {
#pragma unroll
    for (int h = 0; h < kG; ++h) {
      float M = sm.mbuf[0][h];
#pragma unroll
      for (int x = 1; x < kDirectWarps; ++x) M = fmaxf(M, sm.mbuf[x][h]);
      const float f = (M == -INFINITY) ? 0.0f : safe_exp2_diff(sm.mbuf[w][h], M);
      float4* dst = reinterpret_cast<float4*>(&sm.obuf[h][lane * 8]);
      float4 a = make_float4(acc[h][0] * f, acc[h][1] * f, acc[h][2] * f, acc[h][3] * f);
      float4 b = make_float4(acc[h][4] * f, acc[h][5] * f, acc[h][6] * f, acc[h][7] * f);
      if (!first) {
        const float4 a0 = dst[0], b0 = dst[1];
        a.x += a0.x; a.y += a0.y; a.z += a0.z; a.w += a0.w;
        b.x += b0.x; b.y += b0.y; b.z += b0.z; b.w += b0.w;
      }
      dst[0] = a;
      dst[1] = b;
      if ((lane & 3) == 0 && (lane >> 2) == h) sm.lbuf[h] = first ? l * f : sm.lbuf[h] + l * f;
    }
  }
};

// ------------------------------------------------------------------ the kernel

template <class Math>
__global__ void __launch_bounds__(kDirectWarps * 32, 1) stage1_direct_kernel(Stage1Params p) {
  constexpr int kTok = Math::kTok;
  __shared__ __align__(16) DirectSmem sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Sched sched;
  sched.begin(p.indptr, p.B, p.Hkv * p.npass, p.num_splits, gridDim.x, blockIdx.x, p.min_chunk, p.window, p.piece_cost, p.rule_kv8);
  const size_t stride = (size_t)p.Hkv * kRowBytes;
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

  auto fetch_slot = [&](const int* idx, int tok0, int n) -> int {
    int s = -1;
    if (lane < n) {
      s = __ldg(idx + tok0 + lane);
      if (p.check_indices && (s < 0 || (long long)s >= p.num_slots)) {
        atomicOr(&p.hdr->error, kErrIndex);
        s = -1;
      }
    }
    return s;
  };

  Piece pc;
  while (sched.next(pc)) {
    int gv;
    const __nv_bfloat16* qg = group_q(p, pc.b, pc.kvh, &gv);
    Math math;
    math.load_q_regs(qg, gv, lane);
    math.reset();

    const unsigned char* kb = p.k_pool + (size_t)(pc.kvh / p.npass) * kRowBytes;
    const unsigned char* vb = p.v_pool + (size_t)(pc.kvh / p.npass) * kRowBytes;
    const int* idx = p.indices + pc.base + pc.j0;
    const int len = pc.j1 - pc.j0;
    const int ntiles = (len + kTok - 1) / kTok;
    int tile = warp;
    if (tile < ntiles) {
      int n = min(kTok, len - tile * kTok);
      int slot = fetch_slot(idx, tile * kTok, n);
      math.load_k(kb, stride, slot, lane);
      math.load_v(vb, stride, slot, lane);
      int ntile = tile + kDirectWarps;
      int nn = (ntile < ntiles) ? min(kTok, len - ntile * kTok) : 0;
      int nslot = fetch_slot(idx, ntile * kTok, nn);
      while (true) {
        math.qk_softmax(sm, n, p.scale_log2, lane);
        if (nn > 0) math.load_k(kb, stride, nslot, lane);
        math.pv_lane(lane);
        if (nn > 0) math.load_v(vb, stride, nslot, lane);
        if (nn == 0) break;
        n = nn;
        ntile += kDirectWarps;
        nn = (ntile < ntiles) ? min(kTok, len - ntile * kTok) : 0;
        nslot = fetch_slot(idx, ntile * kTok, nn);
      }
    }

    // ---- merge the warps' states (fixed order) and write the piece's partial
    math.finish_sums();
    math.publish_max(sm, warp, lane);
    __syncthreads();
#pragma unroll 1
    for (int x = 0; x < kDirectWarps; ++x) {
      if (warp == x) math.accumulate(sm, warp, lane, x == 0);
      __syncthreads();
    }
    float* op = p.o_part + pc.id * (kG * kD);
    for (int e = threadIdx.x * 4; e < kG * kD; e += blockDim.x * 4) {
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
    if (threadIdx.x < kG) {
      float M = sm.mbuf[0][threadIdx.x];
#pragma unroll
      for (int x = 1; x < kDirectWarps; ++x) M = fmaxf(M, sm.mbuf[x][threadIdx.x]);
      const float lsum = sm.lbuf[threadIdx.x];
      p.lse_part[pc.id * kG + threadIdx.x] = (lsum > 0.0f) ? M + log2f(lsum) : -INFINITY;
    }
    __syncthreads();  // shared buffers free for the next piece
  }
}

cudaError_t launch_stage1_tma(const Stage1Params& p, int grid, cudaStream_t stream);

template <int NWARP, int NV, int NG>
cudaError_t launch_mma(const Stage1Params& p, int grid, cudaStream_t stream) {
  using Smem = MmaSmem<NWARP, NV, NG>;
  auto kern = stage1_mma_kernel<NWARP, NV, NG>;
  static std::atomic<bool> attr_set[64];  // zero-initialised: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<grid, NWARP * 32, sizeof(Smem), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_stage1(const Stage1Params& p, int variant, int grid, cudaStream_t stream) {
  if (variant == kVariantTma) return launch_stage1_tma(p, grid, stream);
  if (variant == kVariantSimt) {
    stage1_direct_kernel<DirectSimt><<<grid, kDirectWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
  }
  constexpr int kW = 8, kNV = 3;
  // teams of three groups run on 6 warps (two teams per CTA)
  return p.team == 3   ? launch_mma<6, kNV, 3>(p, grid, stream)
         : p.team == 2 ? launch_mma<kW, kNV, 2>(p, grid, stream)
                       : launch_mma<kW, kNV, 1>(p, grid, stream);
}

}  // namespace gda
