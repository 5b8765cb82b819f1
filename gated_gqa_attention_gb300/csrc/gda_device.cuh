// gda_device.cuh -- device helpers shared by the gated decode kernels (sm_103a).
//
// * PTX wrappers: mbarrier (init / arrive / expect_tx / bounded parity wait),
//   1-D bulk copies global -> shared (the TMA bulk engine), L2 eviction
//   policies, programmatic dependent launch, named barriers.
// * The work schedule that stage 1 and stage 2 both derive from kv_indptr: which
//   (sequence, KV head, position range) "pieces" each stage-1 CTA computes and
//   where each piece's partial result lives.
// * The BF16 gate arithmetic of FreeToken PR #781 "Fuse the BF16 attention output
//   sigmoid gate into the existing Triton decode stage2" (Summary): O rounded to
//   BF16, sigmoid of the gate rounded to BF16, product rounded to nearest even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gda {

// Geometry the kernels are built for (FreeToken PR #781, Automatic dispatch:
// query [1,16,256] with two KV heads -> D = 256, G = 8 query heads per KV head).
constexpr int kD = 256;
constexpr int kG = 8;
constexpr int kRowBytes = kD * 2;          // one (slot, KV head) row of K or V
constexpr int kSmemRow = kRowBytes + 16;   // padded shared-memory row: conflict-free ldmatrix
constexpr int kAutoMaxCtas = 1024;         // bound on the automatic-mode stage-1 grid
constexpr int kHeaderBytes = 256;          // workspace header
constexpr uint32_t kErrIndex = 0x1u;
constexpr uint32_t kErrTimeout = 0x2u;
// A pipeline wait gives up after this many SM cycles (~2 s): only a kernel bug
// can get there; the kernel then records kErrTimeout and winds down.
constexpr long long kWaitLimitCycles = 4000000000LL;

struct WsHeader {
  unsigned int error;   // kErr* bits, sticky until read and cleared by the host
  unsigned int pad[63];
};
static_assert(sizeof(WsHeader) == kHeaderBytes, "header size");

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up (returns
// false) when *abort_flag becomes nonzero or after `limit` SM cycles.  A limit below
// kWaitLimitCycles is the failure-path test's: the wait then polls without
// suspending and checks the clock on every poll, so any wait that does not
// complete within that many cycles gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          long long limit = kWaitLimitCycles) {
  if (limit < kWaitLimitCycles) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity)) {
      if (*abort_flag || clock64() - t0 > limit) return false;
    }
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > limit) return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrive on a named barrier without waiting (the other side waits with bar.sync).
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait for the previous kernel's results.  No-ops without PDL.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ warp-level tensor-core helpers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

__device__ __forceinline__ float safe_exp2_diff(float a, float m) {
  // exp2(a - m) with -inf handling: a == -inf -> 0; m == -inf (so a == -inf) -> 0
  return (a == -INFINITY) ? 0.0f : exp2f(a - m);
}

// ------------------------------------------------------------------ work schedule
//
// Stage 1 runs a persistent grid of `grid` CTAs.  The KV stream of the batch is
// ordered by (sequence b, KV head kvh, position j); segment sigma = b*Hkv + kvh
// holds L_b positions.  A "piece" is the part of one segment one CTA computes; it
// yields one partial (normalised O for the G query heads, and their LSE).
//
// Explicit mode (num_splits S > 0): every segment is cut into S splits, split s
//   covering positions [s*c, min(L, (s+1)*c)), c = ceil(L/S).  Unit u = sigma*S + s
//   goes to CTA u % grid; the partial lives at index u.  Empty splits are skipped
//   by both stages.
// Automatic mode (S <= 0), decided on the device from kv_indptr alone:
//   * small batches -- when cutting every segment into ceil(L_max / min_chunk)
//     equal splits still gives at most one split per CTA (B*Hkv*S <= grid) -- use
//     those uniform splits exactly as the explicit mode does: every CTA then has
//     one piece and no piece boundary to cross (the latency-bound regime);
//   * otherwise the whole stream of total = Hkv * nnz positions is cut into grid
//     chunks of equal cost, chunk c to CTA c: a position costs 1 and, when there are
//     more segments than CTAs, every segment start after the first kPieceCost more
//     (the measured price of one more piece), so T = max(ceil(cost / grid),
//     min_chunk) cost units per CTA and a CTA that crosses more segment starts takes
//     fewer positions (equal time per CTA for any length mix); the piece (segment
//     sigma, chunk c) lives at index c + sigma.
//     That index is unique (a later chunk can only meet a later-or-equal segment)
//     and below grid + B*Hkv, which bounds the workspace.

struct Piece {
  int b, kvh, sigma;  // kvh: the (virtual) head of the piece, sigma = b * heads + kvh
  int j0, j1;         // positions [j0, j1) of the sequence's attended range
  long long base;     // kv_indices offset of position 0 of that range
  long long id;       // partial index
};

// Attended range of sequence b: all L positions, or the last `window` of them.
__device__ __forceinline__ void seq_range(const int* indptr, int b, int window, int* L, long long* base) {
  const int i0 = __ldg(indptr + b), i1 = __ldg(indptr + b + 1);
  int len = i1 - i0;
  int off = 0;
  if (window > 0 && len > window) {
    off = len - window;
    len = window;
  }
  *L = len;
  *base = (long long)i0 + off;
}

// Automatic mode: per-CTA stream length from which the chunked schedule is used
// even for batches that fit one wave of uniform splits: 3072 positions of a BF16
// cache, twice as many of an e4m3 cache (the same streaming time; measured: one-wave
// uniform splits win at 3450 .. 5174 e4m3 positions per CTA, tie at 6899 and lose from
// ~13800).
constexpr int kStreamMinPerCta = 3072;

// Stream schedule: what starting one more (sequence, KV head) segment costs a CTA, in
// positions of streaming.  Measured on GB300 (per-CTA end times on b224_ragged, ~3
// segment starts per CTA): a CTA ends ~5 us later per extra piece -- the piece's
// merge, its partial tile round and the restart of its loads -- while it streams ~42
// positions per us of a BF16 cache (twice as many of an e4m3 cache, half the bytes);
// the chunks are then cut in a cost space where each segment start adds this much.
// A sweep of the cost on that batch put the best at 300 (BF16; 200 and 400 ~1 %
// slower) and 600 (e4m3; 400 1 %, 1000 3 % slower).  With fewer segments than CTAs
// (b64_l4096: every CTA meets one or two) the weighting measured slower, and the cost
// is 0 (the host passes the cost it picks).
constexpr int kPieceCost = 300;
constexpr int kPieceCostE4m3 = 600;

struct Sched {
  const int* indptr;
  int B, Hkv, S, grid, cta, window;
  long long T, total, X;
  // iteration state
  long long pos, end;  // automatic
  int b;
  long long u;         // explicit

  // Hkv_ here is the number of (virtual) heads that split the batch into segments.
  // window > 0 requires S_ > 0 (the host picks the split count then).
  __device__ __forceinline__ void begin(const int* indptr_, int B_, int Hkv_, int S_, int grid_,
                                        int cta_, int min_chunk, int window_, int piece_cost_, int kv8) {
    indptr = indptr_;
    B = B_;
    Hkv = Hkv_;
    grid = grid_;
    cta = cta_;
    window = window_;
    // the first round of the sequence search and the batch total are loaded
    // together (and, for small batches, the longest-sequence scan): one round trip
    const int step0 = (B - 1 + 32) / 32;
    const int cand0 = min(B - 1, (int)(threadIdx.x & 31) * step0);
    const int v0 = __ldg(indptr + cand0 + 1);
    const int ntot = __ldg(indptr + B);
    S = (S_ > 0) ? S_ : auto_uniform_splits(indptr_, B_, Hkv_, grid_, min_chunk, kv8);
    if (S > 0) {
      u = cta;
      return;
    }
    // the stream of total = Hkv * nnz positions in a cost space where every segment
    // start after the first adds kPieceCost: CTA c takes the costs [c T, (c + 1) T) and
    // so the positions between the first ones costing at least c T and (c + 1) T
    total = (long long)Hkv * (long long)ntot;
    X = piece_cost_;
    const long long ctot = stream_cost(total, B, Hkv, X);
    T = auto_chunk(ctot, grid, min_chunk);
    const long long t0 = (long long)cta * T, t1 = t0 + T;
    b = 0;
    pos = end = total;
    if (t0 < ctot) {
      int b0, b1;
      if (X == 0) {
        // costs are positions: no second search, no mapping back (every dependent
        // load here delays the CTA's first tile)
        pos = t0;
        end = min(total, t1);
        b0 = first_seq_ending_after(indptr, B, Hkv, pos, v0);
      } else {
        first_seqs_costing_beyond(indptr, B, Hkv, X, t0, t1, v0, &b0, &b1);
        pos = position_at_cost(indptr, Hkv, X, b0, t0);
        end = (t1 >= ctot) ? total : position_at_cost(indptr, Hkv, X, b1, t1);
      }
      b = b0;
    }
  }

  // First sequence b whose (Hkv-scaled) end Hkv*indptr[b+1] lies beyond pos (one
  // exists).  Called by every lane of a full warp: a 32-way search, each round
  // one load per lane, so ceil(log32 B) dependent loads instead of log2 B.
  // v0: this lane's value of the first round, indptr[min(B-1, lane*step0) + 1].
  static __device__ __forceinline__ int first_seq_ending_after(const int* indptr, int B, int Hkv,
                                                               long long pos, int v0) {
    const int lane = (int)(threadIdx.x & 31);
    int lo = 0, hi = B - 1;  // the answer lies in [lo, hi]
    bool first = true;
    while (lo < hi) {
      const int step = (hi - lo + 32) / 32;  // 32 candidates cover [lo, hi]
      const int cand = min(hi, lo + lane * step);
      const int v = first ? v0 : __ldg(indptr + cand + 1);
      first = false;
      const bool past = (long long)Hkv * v > pos;
      const unsigned ball = __ballot_sync(0xffffffffu, past);
      // candidates are non-decreasing in the lane index; hi itself satisfies `past`
      if (ball == 0u) {
        lo = min(hi, lo + 31 * step) + 1;
      } else {
        const int f = __ffs(ball) - 1;
        const int cf = min(hi, lo + f * step);
        lo = (f == 0) ? lo : min(hi, lo + (f - 1) * step) + 1;
        hi = cf;
      }
    }
    return lo;
  }

  // Cost of the whole stream (positions plus X per segment start after the first).
  static __device__ __forceinline__ long long stream_cost(long long total, int B, int Hkv, long long X) {
    const long long nseg = (long long)B * Hkv;
    return total + X * (nseg > 0 ? nseg - 1 : 0);
  }

  // Cost at which sequence b's first segment starts: Hkv * indptr[b] + X * b * Hkv.
  static __device__ __forceinline__ long long seq_cost_start(long long ib, int b, int Hkv, long long X) {
    return (long long)Hkv * ib + X * b * Hkv;
  }

  // The first position whose cost is at least t (t < the stream cost), with b the
  // sequence whose cost range holds t.  Segment (b, k) covers positions
  // Hkv indptr[b] + k L + [0, L) at costs seq_cost_start + k (L + X) + [0, L), followed
  // by X of cost with no positions (a t there maps to the next segment's first position).
  static __device__ __forceinline__ long long position_at_cost(const int* indptr, int Hkv, long long X, int b,
                                                               long long t) {
    const long long ib = __ldg(indptr + b);
    const long long L = __ldg(indptr + b + 1) - ib;
    const long long cs = seq_cost_start(ib, b, Hkv, X);
    long long k = (L + X > 0) ? (t - cs) / (L + X) : 0;
    k = k < 0 ? 0 : (k > Hkv - 1 ? Hkv - 1 : k);
    const long long into = t - (cs + k * (L + X));
    return (long long)Hkv * ib + k * L + (into < 0 ? 0 : (into > L ? L : into));
  }

  // The first sequences whose cost range ends beyond ta and beyond tb (both below the
  // stream cost, so sequence B - 1 qualifies): the end of sequence b's range is
  // seq_cost_start(indptr[b + 1], b + 1, Hkv, X).  Called by every lane of a full warp: two
  // 32-way searches in lockstep, each round one load per lane and search, so ceil(log32
  // B) dependent loads instead of log2 B.  v0: this lane's value of the first round
  // (shared by both), indptr[min(B-1, lane*step0) + 1].
  static __device__ __forceinline__ void first_seqs_costing_beyond(const int* indptr, int B, int Hkv, long long X,
                                                                   long long ta, long long tb, int v0, int* ba,
                                                                   int* bb) {
    const int lane = (int)(threadIdx.x & 31);
    int lo[2] = {0, 0}, hi[2] = {B - 1, B - 1};  // each answer lies in [lo, hi]
    const long long tt[2] = {ta, tb};
    bool first = true;
    while (lo[0] < hi[0] || lo[1] < hi[1]) {
      int step[2], cand[2], v[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        step[x] = (hi[x] - lo[x] + 32) / 32;  // 32 candidates cover [lo, hi]
        cand[x] = min(hi[x], lo[x] + lane * step[x]);
        v[x] = first ? v0 : ((lo[x] < hi[x]) ? __ldg(indptr + cand[x] + 1) : 0);
      }
      first = false;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const bool past = seq_cost_start(v[x], cand[x] + 1, Hkv, X) > tt[x];
        const unsigned ball = __ballot_sync(0xffffffffu, past);
        if (lo[x] >= hi[x]) continue;  // (warp-uniform) this search is done
        // candidates are non-decreasing in the lane index; hi itself satisfies `past`
        if (ball == 0u) {
          lo[x] = min(hi[x], lo[x] + 31 * step[x]) + 1;
        } else {
          const int f = __ffs(ball) - 1;
          const int cf = min(hi[x], lo[x] + f * step[x]);
          lo[x] = (f == 0) ? lo[x] : min(hi[x], lo[x] + (f - 1) * step[x]) + 1;
          hi[x] = cf;
        }
      }
    }
    *ba = lo[0];
    *bb = lo[1];
  }

  // Automatic mode: the uniform split count S (every segment cut into S equal
  // pieces), or 0 for the chunked (stream) schedule.  Called by every lane of a
  // full warp: the longest sequence is found with the lanes striding over the batch.
  // The rule comes from split sweeps on GB300 (equal lengths, B = 1 .. 128, L = 512
  // .. 32768, every S in 1 .. 128):
  //  * a call costs about a + b L/S (stage 1, one piece per CTA) + c S (stage 2
  //    merges S partials per head), c/b ~ 2 positions (stage 2 keeps four partials'
  //    loads in flight), so the best S is near sqrt(lmax / 2): S_opt, the smallest
  //    power of two with 4 S^2 > lmax, and at most ceil(lmax / min_chunk).  An e4m3
  //    cache (kv8) streams a position in half the time, c/b ~ 8: 16 S^2 > lmax;
  //  * at most one wave of CTAs (B Hkv S <= grid); when the wave bounds S, the
  //    power of two below the bound if it keeps >= 80 % of the CTAs busy (pieces
  //    aligned to the warps' tiles), else the bound itself, and with < 80 % busy
  //    the stream schedule;
  //  * the stream schedule once each CTA would stream >= 3072 positions (6144 of an
  //    e4m3 cache; it then wins by 1-3 %: no idle SMs) or when the lengths are far
  //    from equal
  //    (lmax > 1.25 x the mean: S pieces of the longest sequence bound the call).
  static __device__ __forceinline__ int auto_uniform_splits(const int* indptr, int B, int Hkv, int grid,
                                                            int min_chunk, int kv8) {
    if ((long long)B * Hkv > grid) return 0;
    const int units1 = B * Hkv;  // one piece per segment; <= grid
    if (units1 == 0) return 1;
    // the longest length and the total from the same loads (kv_indptr[0] = 0): no
    // further round trip, which every CTA's start and stage 2's prologue would wait on
    int lmax = 0, n = 0;
    for (int b = (int)(threadIdx.x & 31); b < B; b += 32) {
      const int len = __ldg(indptr + b + 1) - __ldg(indptr + b);
      lmax = max(lmax, len);
      n += len;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
      n += __shfl_xor_sync(0xffffffffu, n, off);
    }
    if ((long long)Hkv * n >= (long long)kStreamMinPerCta * (kv8 ? 2 : 1) * grid) return 0;
    if (4LL * lmax * B > 5LL * n) return 0;
    // (closed forms, short dependent chains: every CTA's start waits on this)
    // s_opt: the smallest power of two p with 4 p^2 > lmax, 2^(h / 2) with h the index
    // of lmax's top bit (kv8: 16 p^2 > lmax, 2^max(0, h / 2 - 1))
    const int s_opt = (lmax > 0) ? (1 << max(0, ((31 - __clz(lmax)) >> 1) - (kv8 ? 1 : 0))) : 1;
    const int s_len = max(1, (lmax + min_chunk - 1) / min_chunk);
    int s = min(s_opt, s_len);
    const int s_wave = grid / units1;
    if (s >= s_wave) {
      const int p2 = 1 << (31 - __clz(s_wave));  // the largest power of two <= s_wave
      s = (5 * p2 * units1 >= 4 * grid) ? p2 : s_wave;
      if (5 * s * units1 < 4 * grid) return 0;
    }
    return s;
  }

  static __device__ __forceinline__ long long auto_chunk(long long total, int grid, int min_chunk) {
    long long t = (total + grid - 1) / grid;
    return t > min_chunk ? t : (long long)min_chunk;
  }

  __device__ __forceinline__ bool next(Piece& p) {
    if (S > 0) {
      const long long units = (long long)B * Hkv * S;
      while (u < units) {
        const long long uu = u;
        u += grid;
        const int sigma = (int)(uu / S), s = (int)(uu % S);
        const int bb = sigma / Hkv;
        int L;
        long long base;
        seq_range(indptr, bb, window, &L, &base);
        const int c = (L + S - 1) / S;
        const int j0 = s * c;
        const int j1 = min(L, j0 + c);
        if (j0 >= j1) continue;
        p.b = bb;
        p.kvh = sigma % Hkv;
        p.sigma = sigma;
        p.j0 = j0;
        p.j1 = j1;
        p.base = base;
        p.id = uu;
        return true;
      }
      return false;
    }
    if (pos >= end) return false;
    while ((long long)Hkv * __ldg(indptr + b + 1) <= pos) ++b;
    const int ib = __ldg(indptr + b);
    const long long base = (long long)Hkv * ib;
    const int L = __ldg(indptr + b + 1) - ib;
    const long long off = pos - base;
    const int kvh = (int)(off / L);
    const int j0 = (int)(off - (long long)kvh * L);
    const long long seg_end = base + (long long)(kvh + 1) * L;
    const long long stop = min(end, seg_end);
    p.b = b;
    p.kvh = kvh;
    p.sigma = b * Hkv + kvh;
    p.j0 = j0;
    p.j1 = j0 + (int)(stop - pos);
    p.base = ib;
    p.id = (long long)cta + p.sigma;
    pos = stop;
    return true;
  }
};

// Partials of segment (b, kvh) for stage 2: ids first + k, k in [0, n) (automatic
// mode: first = c_first + sigma), or sigma*S + k (explicit mode), in position order.
// (With a window the split count is explicit and L is the windowed length.)
__device__ __forceinline__ void segment_pieces(const int* indptr, int b, int kvh, int Hkv, int B, int S,
                                               int grid, int min_chunk, int window, int piece_cost, int kv8,
                                               long long* first, int* n) {
  const int ib = __ldg(indptr + b);
  int L;
  long long base;
  seq_range(indptr, b, window, &L, &base);
  const int sigma = b * Hkv + kvh;
  if (L <= 0) {
    *first = 0;
    *n = 0;
    return;
  }
  if (S <= 0) S = Sched::auto_uniform_splits(indptr, B, Hkv, grid, min_chunk, kv8);
  if (S > 0) {
    const int c = (L + S - 1) / S;
    *first = (long long)sigma * S;
    *n = (L + c - 1) / c;
    return;
  }
  const long long total = (long long)Hkv * (long long)__ldg(indptr + B);
  const long long X = piece_cost;
  const long long T = Sched::auto_chunk(Sched::stream_cost(total, B, Hkv, X), grid, min_chunk);
  // the segment's positions in the stream's cost space (Sched::begin): they start at
  // cost Hkv indptr[b] + kvh L + X (b Hkv + kvh), one cost unit each
  const long long start = (long long)Hkv * ib + (long long)kvh * L + X * sigma;
  const long long c0 = start / T, c1 = (start + L - 1) / T;
  *first = c0 + sigma;
  *n = (int)(c1 - c0 + 1);
}

// ------------------------------------------------------------------ BF16 gate arithmetic

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Round a double to BF16 (nearest, ties to even) without double rounding: first
// to float with round-to-odd (truncate, then set the last bit if anything was
// dropped), which keeps 16 more bits than BF16 has, then float -> BF16 RNE.
// (Round-to-odd as an intermediate step is exact for any target with at least
// two fewer bits: Boldo & Melquiond, "Emulation of FMA and correctly rounded
// sums: proved algorithms using rounding to odd", IEEE TC 2008.)
__device__ __forceinline__ uint16_t bf16_rne_from_double(double x) {
  float f = __double2float_rz(x);
  if ((double)f != x && !isnan(x)) f = __uint_as_float(__float_as_uint(f) | 1u);
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// BF16 bits of RNE(sigmoid(g)) for a BF16 gate g, exact for all 65 536 codes.
// Fast path in float: e = expf(-|g|) (documented max error 2 ulp), 1 + e and the
// division correctly rounded, so the float sigmoid is within a few ulp of the
// real value.  When its low 16 bits lie within 16 ulp of a BF16 rounding tie the
// decision is retaken in double (exp with max error 1 ulp); |g| > 80, the
// infinities and NaN go the double way too.  Exhaustively tested on the GPU
// against the FP64 oracle.
__device__ __forceinline__ uint16_t sigmoid_bf16(uint16_t gbits) {
  const float g = bf16_bits_to_float(gbits);
  const float a = fabsf(g);
  if (a <= 80.0f) {
    const float e = expf(-a);
    const float den = __fadd_rn(1.0f, e);
    const float s = (g >= 0.0f) ? __fdiv_rn(1.0f, den) : __fdiv_rn(e, den);
    const uint32_t low = __float_as_uint(s) & 0xFFFFu;
    if (low - 0x7FF0u > 0x20u) return __bfloat16_as_ushort(__float2bfloat16_rn(s));
  }
  const double gd = (double)g;
  return bf16_rne_from_double(1.0 / (1.0 + exp(-gd)));
}

// RNE_bf16(o * s) for BF16 o and s.  The float product is exact unless it falls
// below the float normal range, where it is redone exactly in double.
__device__ __forceinline__ uint16_t gate_product_bf16(uint16_t obits, uint16_t sbits) {
  const float o = bf16_bits_to_float(obits);
  const float s = bf16_bits_to_float(sbits);
  const float p = __fmul_rn(o, s);
  if (fabsf(p) < 1.17549435e-38f && p != 0.0f) return bf16_rne_from_double((double)o * (double)s);
  return __bfloat16_as_ushort(__float2bfloat16_rn(p));
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

}  // namespace gda
