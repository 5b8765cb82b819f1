// gda_prefill.cu -- prefill / extend gated SDPA on sm_103a with tcgen05 MMAs, TMEM
// operands and accumulators, and TMA loads.
//
// Computes, per sequence b, query i and query head h (cuDNN FE-OSS "Gated Attention
// Block (SM107)", Overview stage (4) SDPA O = softmax(Q K^T * scale + mask) V with
// GQA H_q / H_kv, and stage (5) fused into the SDPA epilogue, Fusion knobs,
// fuse_gate: O *= sigmoid(GATE) after the dead-row select):
//   keys visible to query i: j < L (L = kv_lens[b], or Skv) and, causal, j <= i + (L - Sq)
//   O   = sum_j softmax_j(scale * q_i . k_j) v_j            (a dead row gives O = 0)
//   out = RNE_bf16(RNE_bf16(O) * RNE_bf16(sigmoid(gate)))   (the decode path's gate)
//   lse = natural-log log-sum-exp of the visible scaled scores ([B, Hq, Sq], optional)
//
// GB300 design: one CTA per (128-query block, query head, sequence), roles that hand
// tiles to each other through mbarriers (full / empty pairs, every wait bounded):
//  * Keys go in tiles of 128, so every MMA has N = 128 and runs at the full tensor
//    rate.  Shared memory: the Q tile [128 x 256] (128-byte swizzle, [column block]
//    [row][128 B]), and K and V each as two half tiles, a half being 128 keys x 128
//    head dimensions ([2 column blocks][128 rows][128 B], 32 KiB): half h of tile
//    j + 1 is loaded as soon as the MMAs of tile j that read half h have completed.
//    At the end the Q buffer takes the gate tile and the V halves the output tile.
//  * TMEM (512 columns): two S / P buffers (columns [128 n, 128 n + 128), FP32
//    scores, their first half then overwritten by P as BF16 pairs) and O (columns
//    [256, 512)).
//  * warps 8 and 10, TMA producers (cp.async.bulk.tensor, one 5-D box per half):
//    Q, then K halves, then the gate tile (warp 8); V halves (warp 10).
//  * two MMA issuers (one lane each; tcgen05.mma kind::f16, BF16 operands, FP32
//    accumulation, M = 128, N = 128): warp 9 (which also owns the TMEM allocation)
//    issues S(j) = Q K(j)^T (16 k-steps, A and B from shared memory), warp 11 issues
//    O += P(j) V(j) (per 128-dimension half of O, 8 k-steps, A = P from TMEM, B = V
//    MN-major).  Any wait in an issuing thread lets the tensor pipe drain behind it;
//    with the two products in separate warps, one keeps the pipe fed while the
//    other waits, and each waits once per tile.
//  * warps 0-7, softmax and epilogue: warps w and w + 4 share query rows 32 w .. + 31
//    (TMEM lanes), each reading 64 of a tile's 128 scores (tcgen05.ld); per tile they
//    agree on the row max through shared memory, keep a running max (moved lazily,
//    by more than 2^8, as the decode kernels do; O in TMEM is rescaled then) and sum,
//    and write P (BF16) over their S buffer with tcgen05.st.  Epilogue: O row from
//    TMEM, divided by the sum, rounded to BF16, gated with the BF16 sigmoid of the
//    staged gate row (an SFU fast path, and a per-device table of all 65 536 BF16
//    sigmoids near rounding ties), staged in shared memory, written by TMA stores.
// On a timeout the CTA records kErrTimeout, every role stops, waits (bounded) for the
// copies and MMAs it started, the TMEM is freed and the CTA returns.  TMEM accesses
// stay warp-convergent (decisions combined with __all_sync).
#include <cuda.h>

#include <mutex>

#include "gda_device.cuh"
#include "gda_kernels.h"
#include "gda_prefill.h"

namespace gda {

namespace {

constexpr int kPM = 128;            // query rows per CTA (MMA M)
constexpr int kPN = 128;            // keys per tile (MMA N of S)
constexpr int kNSB = 2;             // S / P buffers in TMEM
constexpr int kSoftmaxWarps = 8;    // warps 0-7: softmax and epilogue
constexpr int kLoadWarp = 8;        // TMA producer: Q, K halves, then the gate tile
constexpr int kMmaWarp = 9;         // S = Q K^T issuer; allocates and frees TMEM
constexpr int kLoadWarpV = 10;      // TMA producer: V halves
constexpr int kPvWarp = 11;         // O += P V issuer
constexpr int kPThreads = 12 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;      // S / P buffers: columns [128 n, 128 n + 128), n < kNSB
constexpr uint32_t kTmemO = 256;    // O accumulator: columns [256, 512)

// shared memory plan (offsets from a 1024-byte aligned base)
constexpr uint32_t kBlk = 128 * 128;               // one 64-column block of 128 rows: 16 KiB
constexpr uint32_t kHalf = 2 * kBlk;               // a half tile: 2 column blocks, 32 KiB
constexpr uint32_t kOffQ = 0;                      // Q tile [4 blocks][128 rows][128 B]; the gate tile at the end
constexpr int kKSlots = 3;                         // K ring: three half slots (half n of the K stream in slot n % 3)
constexpr uint32_t kOffK = kOffQ + 4 * kBlk;       // K ring
constexpr uint32_t kOffV = kOffK + kKSlots * kHalf; // V halves (slot h: head dimensions [128 h, 128 h + 128));
                                                   // the output tile is staged here at the end
constexpr uint32_t kOffX = kOffV + 2 * kHalf;      // row max exchange [parity][half][row]; the sums reuse a slot
constexpr uint32_t kOffBar = kOffX + 2048;         // mbarriers and the TMEM address
constexpr uint32_t kSmemBytes = kOffBar + 512;     // the dynamic shared memory base is 1024-byte aligned (checked)
static_assert(kPM == 128 && kPN == 128, "one 64-column block is 128 rows of 128 B");
static_assert(2 * kHalf >= 4 * kBlk, "the output tile fits the V halves");
static_assert(kNSB * kPN <= kTmemO, "S / P buffers below O");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// ---- PTX wrappers (tcgen05, TMA) ----

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (TMEM) += A (shared memory descriptor) * B (shared memory descriptor)
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (TMEM) += A (TMEM) * B (shared memory descriptor)
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// all prior tcgen05 MMAs of this thread arrive on `bar` when complete
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 columns of 32 bits: thread t of the warp gets lane (warp base + t), columns col .. col+31
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x on the SFU (ex2.approx, subnormal results flushed): P is rounded to BF16 right
// after, far coarser than the instruction's error.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// {lo, hi} -> BF16x2, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// TMA: a 5-D tile into shared memory, completing on `bar`
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// TMA: a 4-D tile from shared memory to global (rows past the tensor's end are
// dropped); completion tracked by the bulk-group mechanism
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, int x, int y, int z, int w, const void* src) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (descriptor version 1):
// start address, leading and stride byte offsets, all encoded >> 4.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// BF16 sigmoid table: entry g = RNE_bf16(sigmoid(g)) for every BF16 code g, filled
// once per device with the certified sigmoid_bf16 (FreeToken PR #781, Summary: a
// per-device table of BF16 sigmoid values, 128 KiB).  The prefill epilogue gates
// Sq * Hq * D elements, where one table load is far cheaper than the computation.
__device__ uint16_t g_sigmoid_table[65536];

// RNE_bf16(o * s) for BF16 o and s, as gate_product_bf16 computes it, with the exact
// double-precision path for products below the float normal range kept out of line:
// inlined, the compiler may evaluate it for every element, and FP64 on this part is
// far slower than the rest of the epilogue.
__device__ __noinline__ uint16_t gate_product_tiny(float o, float s) {
  return bf16_rne_from_double((double)o * (double)s);
}
__device__ __forceinline__ uint16_t gate_product_fast(uint16_t obits, uint16_t sbits) {
  const float o = __uint_as_float((uint32_t)obits << 16);
  const float s = __uint_as_float((uint32_t)sbits << 16);
  const float p = __fmul_rn(o, s);
  if (fabsf(p) < 1.17549435e-38f && p != 0.0f) return gate_product_tiny(o, s);
  return __bfloat16_as_ushort(__float2bfloat16_rn(p));
}

__global__ void sigmoid_table_kernel() {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 65536) g_sigmoid_table[i] = sigmoid_bf16((uint16_t)i);
}

struct PrefillBars {
  uint64_t qf, g;                                   // Q tile landed; gate tile landed
  uint64_t k_full[kKSlots], k_empty[kKSlots], v_full[2], v_empty[2];  // per half slot
  uint64_t s_full[kNSB], p_full[kNSB], p_empty[kNSB];  // per S / P buffer
  uint64_t xm[4][2];                                // per row quarter and tile parity: both maxima stored
  uint64_t xl[4];                                   // per row quarter: both sums stored
  uint64_t ost;                                     // output tile staged (8 softmax warps)
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(PrefillBars) <= 512, "barrier block");

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap tg, const __grid_constant__ CUtensorMap to,
                   PrefillParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* sm = smem_raw;
  // the 128-byte swizzled tiles need a 1024-byte aligned base, which the layout takes
  // without slack: a misaligned base is reported, not used (the same for every CTA)
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(p.error, kErrTimeout);
    return;
  }
  PrefillBars& bars = *reinterpret_cast<PrefillBars*>(sm + kOffBar);
  float* xbuf = reinterpret_cast<float*>(sm + kOffX);  // [parity][half][row]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqb = (p.Sq + kPM - 1) / kPM;
  // CTAs start in linear order (x fastest): x enumerates (query block, head) with the
  // head fastest, so every head's longest causal blocks come first (longest-first
  // scheduling keeps the last wave short)
  const int qb = nqb - 1 - (int)blockIdx.x / p.Hq;
  const int h = (int)blockIdx.x % p.Hq, b = blockIdx.y;
  const int kvh = h / (p.Hq / p.Hkv);
  const int L = p.kv_lens ? __ldg(p.kv_lens + b) : p.Skv;
  const int i0 = qb * kPM;
  const int off = L - p.Sq;  // causal: key j visible to query i when j <= i + off
  int last_key = L - 1;
  if (p.causal) last_key = min(last_key, i0 + kPM - 1 + off);
  const int ntiles = (last_key >= 0) ? (last_key / kPN + 1) : 0;

  if (tid == 0) {
    mbar_init(&bars.qf, 1);
    mbar_init(&bars.g, 1);
    for (int x = 0; x < kKSlots; ++x) {
      mbar_init(&bars.k_full[x], 1);
      mbar_init(&bars.k_empty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars.v_full[x], 1);
      mbar_init(&bars.v_empty[x], 1);
    }
    for (int x = 0; x < kNSB; ++x) {
      mbar_init(&bars.s_full[x], 1);
      mbar_init(&bars.p_full[x], kSoftmaxWarps);
      mbar_init(&bars.p_empty[x], 1);
    }
    for (int q4 = 0; q4 < 4; ++q4) {
      mbar_init(&bars.xm[q4][0], 2);
      mbar_init(&bars.xm[q4][1], 2);
      mbar_init(&bars.xl[q4], 2);
    }
    mbar_init(&bars.ost, kPThreads / 32);
    bars.abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem;
  volatile int* abort_flag = &bars.abort;
  auto fail = [&]() {
    if (bars.abort == 0) atomicOr(p.error, kErrTimeout);
    bars.abort = 1;
  };

  float m_run = -INFINITY, l_run = 0.0f;  // softmax warps: running row max (log2 units) and sum

  if (warp == kLoadWarp || warp == kLoadWarpV) {
    // ---------------- TMA producers (one lane each): K halves (then the gate tile) from
    // warp kLoadWarp, V halves from warp kLoadWarpV.  Half n = 2 j + h of the stream
    // (head dimensions [128 h, 128 h + 128) of tile j) goes into slot n % nslot once
    // the MMAs that read the slot's previous half have completed.
    const bool is_k = warp == kLoadWarp;
    if (lane == 0 && ntiles > 0) {
      int arm_g = 0, arm_gate = 0, arm[kKSlots] = {};
      uint64_t* full = is_k ? bars.k_full : bars.v_full;
      uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
      const CUtensorMap* map = is_k ? &tk : &tv;
      const uint32_t base = is_k ? kOffK : kOffV;
      const int nslot = is_k ? kKSlots : 2;
      bool ok = true;
      if (is_k) {
        ++arm_g;
        mbar_arrive_expect_tx(&bars.qf, 4 * kBlk);
        tma_load_5d(sm + kOffQ, &tq, 0, i0, 0, h, b, &bars.qf);
      }
      for (int n = 0; n < 2 * ntiles; ++n) {
        const int x = n % nslot, u = n / nslot;  // slot and its use count
        if (u > 0 && !mbar_wait(&empty[x], (u - 1) & 1, abort_flag, p.wait_limit)) { ok = false; break; }
        ++arm[x];
        mbar_arrive_expect_tx(&full[x], kHalf);
        // box {64 elements, 128 rows, 2 column blocks}: keys 128 j .., head dimensions 128 h ..
        tma_load_5d(sm + base + x * kHalf, map, 0, (n >> 1) * kPN, 2 * (n & 1), kvh, b, &full[x]);
      }
      if (ok && is_k && p.fuse_gate) {
        // the gate tile goes into the Q buffer once the last S product has read Q (its
        // last commit covers every earlier MMA of the S issuer)
        const int nl = 2 * ntiles - 1;  // the last K half
        if (!mbar_wait(&bars.k_empty[nl % kKSlots], (nl / kKSlots) & 1, abort_flag, p.wait_limit)) ok = false;
        if (ok) {
          ++arm_gate;
          mbar_arrive_expect_tx(&bars.g, 4 * kBlk);
          tma_load_5d(sm + kOffQ, &tg, 0, i0, 0, h, b, &bars.g);
        }
      }
      if (!ok) {
        fail();
        // wait (bounded) for every copy this producer started before its memory goes away
        int dummy = 0;
        volatile int* none = &dummy;
        if (arm_g > 0) mbar_wait(&bars.qf, 0, none);
        if (arm_gate > 0) mbar_wait(&bars.g, 0, none);
        for (int x = 0; x < nslot; ++x)
          if (arm[x] > 0) mbar_wait(&full[x], (arm[x] - 1) & 1, none);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- S issuer (one lane): S(j) = Q K(j)^T into S buffer j % 2, which
    // P(j - 2) occupied; one wait point per tile
    if (lane == 0 && ntiles > 0) {
      const uint32_t sQ = smem_u32(sm + kOffQ), sK = smem_u32(sm + kOffK);
      const uint32_t idS = idesc_bf16(kPM, kPN, 0);
      uint64_t* last_bar = nullptr;  // the barrier of the last commit and its phase parity
      int last_par = 0;
      bool ok = mbar_wait(&bars.qf, 0, abort_flag, p.wait_limit);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int sb = j & 1;
        const int x0 = (2 * j) % kKSlots, x1 = (2 * j + 1) % kKSlots;  // the slots of K(j)'s halves
        ok = mbar_wait(&bars.k_full[x0], ((2 * j) / kKSlots) & 1, abort_flag, p.wait_limit) &&
             mbar_wait(&bars.k_full[x1], ((2 * j + 1) / kKSlots) & 1, abort_flag, p.wait_limit);
        if (ok && j >= kNSB) ok = mbar_wait(&bars.p_empty[sb], ((j >> 1) - 1) & 1, abort_flag, p.wait_limit);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8) {
            const int kk = 8 * hh + k8;  // k-step: head dimensions 16 kk .. 16 kk + 15
            const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * kBlk + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sK + (hh ? x1 : x0) * kHalf + ((kk >> 2) & 1) * kBlk + (kk & 3) * 32, 16, 1024);
            umma_bf16_ss(tmem + kTmemS + sb * kPN, ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars.k_empty[hh ? x1 : x0]);
        }
        umma_commit(&bars.s_full[sb]);
        last_bar = &bars.s_full[sb];
        last_par = (j >> 1) & 1;
      }
      if (!ok) {
        fail();
        // the last commit covers every MMA issued before it: wait for it (bounded)
        int dummy = 0;
        volatile int* none = &dummy;
        if (last_bar != nullptr) mbar_wait(last_bar, last_par, none);
      }
    }
  } else if (warp == kPvWarp) {
    // ---------------- PV issuer (one lane): O += P(j) V(j), per 128-dimension half of O
    if (lane == 0 && ntiles > 0) {
      const uint32_t sV = smem_u32(sm + kOffV);
      const uint32_t idO = idesc_bf16(kPM, 128, 1);
      uint64_t* last_bar = nullptr;
      int last_par = 0;
      bool ok = true;
      for (int j = 0; j < ntiles && ok; ++j) {
        const int pb = j & 1;
        ok = mbar_wait(&bars.p_full[pb], (j >> 1) & 1, abort_flag, p.wait_limit) &&
             mbar_wait(&bars.v_full[0], j & 1, abort_flag, p.wait_limit) && mbar_wait(&bars.v_full[1], j & 1, abort_flag, p.wait_limit);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // V half hh is MN-major (dims contiguous): LBO = stride between its two 64-dim
            // blocks, SBO = 8 key rows; k-step kk = keys 16 kk .. 16 kk + 15, whose P is
            // in columns 8 kk .. 8 kk + 7 of the S buffer
            const uint64_t bd = sdesc_sw128(sV + hh * kHalf + kk * 16 * 128, kBlk, 1024);
            umma_bf16_ts(tmem + kTmemO + 128 * hh, tmem + kTmemS + pb * kPN + 8 * kk, bd, idO,
                         (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars.v_empty[hh]);
        }
        umma_commit(&bars.p_empty[pb]);
        last_bar = &bars.p_empty[pb];
        last_par = (j >> 1) & 1;
      }
      if (!ok) {
        fail();
        int dummy = 0;
        volatile int* none = &dummy;
        if (last_bar != nullptr) mbar_wait(last_bar, last_par, none);
      }
    }
  } else {
    // ---------------- softmax and epilogue: warp w owns rows 32 (w % 4) .. + 31 (its
    // TMEM lane quarter) and keys [64 h, 64 h + 64) of each tile, h = w / 4
    const int rg = warp & 3, hc = warp >> 2;
    const int r = 32 * rg + lane;
    const int qi = i0 + r;
    const uint32_t t_row = tmem + ((uint32_t)(rg * 32) << 16);
    bool ok = true;

    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1, x2 = j & 1;  // S / P buffer; parity slot of the max exchange
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars.s_full[sb], (j >> 1) & 1, abort_flag, p.wait_limit));
      if (!ok) break;
      tc_fence_after();
      float s[64];
      tmem_ld32(t_row + kTmemS + sb * kPN + 64 * hc, s);
      tmem_ld32(t_row + kTmemS + sb * kPN + 64 * hc + 32, s + 32);
      tmem_wait_ld();

      const int k0 = j * kPN + 64 * hc;  // key of s[0]
      const bool need_mask = (k0 + 64 > L) || (p.causal && k0 + 63 > i0 + off);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int kj = k0 + c;
          if (kj >= L || (p.causal && kj > qi + off)) s[c] = -INFINITY;
        }
      }
      float hm;
      {
        float e4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 64; ++c) e4[c & 3] = fmaxf(e4[c & 3], s[c]);
        hm = fmaxf(fmaxf(e4[0], e4[1]), fmaxf(e4[2], e4[3]));
      }
      // the two halves of the row agree on the tile max (parity-buffered shared slots);
      // after this both have read their S, so P may overwrite it
      xbuf[(x2 * 2 + hc) * kPM + r] = hm;
      tc_fence_before();  // this warp's S reads are ordered before the partner's P writes
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.xm[rg][x2]);
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.xm[rg][x2], (j >> 1) & 1, abort_flag, p.wait_limit));
      if (!ok) break;
      tc_fence_after();
      const float mx = fmaxf(hm, xbuf[(x2 * 2 + (1 - hc)) * kPM + r]) * p.scale_log2;

      // lazy max: it moves only by more than 2^8, so probabilities stay below 2^8
      // (both halves of a row take the same decisions from the same values)
      float alpha = 1.0f;
      if (mx > m_run + 8.0f) {
        alpha = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - mx);
        l_run *= alpha;
        m_run = mx;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // O must hold PV(j - 1) before it is rescaled; this warp rescales its half of O
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.wait_limit));
        if (!ok) break;
        tc_fence_after();
        for (int c0 = 128 * hc; c0 < 128 * hc + 128; c0 += 32) {
          float o[32];
          tmem_ld32(t_row + kTmemO + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(t_row + kTmemO + c0, o);
        }
        tmem_wait_st();
      }
      // p = 2^(s * scale_log2 - m): one FFMA and one SFU op per score (a masked score
      // gives 2^-inf = 0; a row with no visible key yet uses m = 0); P (BF16 pairs)
      // over the first half of the S buffer: keys 64 h .. at columns 32 h ..
      const float mneg = (m_run == -INFINITY) ? 0.0f : -m_run;
      uint32_t w[32];
      float la = 0.0f, lb = 0.0f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = ex2_approx(fmaf(s[2 * e], p.scale_log2, mneg));
        const float p1 = ex2_approx(fmaf(s[2 * e + 1], p.scale_log2, mneg));
        w[e] = bf16x2_rn(p0, p1);
        la += __uint_as_float(w[e] << 16);
        lb += __uint_as_float(w[e] & 0xFFFF0000u);
      }
      l_run += la + lb;
      tmem_st16(t_row + kTmemS + sb * kPN + 32 * hc, w);
      tmem_st16(t_row + kTmemS + sb * kPN + 32 * hc + 16, w + 16);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[sb]);
    }
    if (!ok) fail();
  }

  // ---------------- epilogue, all twelve warps: warp w reads TMEM lane quarter w % 4
  // (rows 32 (w % 4) ..) and 32-column chunks {0, 1, 2} (warps 0-3), {4, 5, 6} (4-7) or
  // {3, 7} (8-11) of O; O / l, BF16, gate, staged in the V halves (free once the last
  // PV has completed) in the swizzled [column block][row][128 B] layout, TMA stores
  __syncwarp();
  {
    const int eq = warp & 3;
    const int r = 32 * eq + lane;
    const int qi = i0 + r;
    const uint32_t t_row = tmem + ((uint32_t)(eq * 32) << 16);
    bool ok = (*abort_flag == 0);
    const int xs = ntiles & 1;  // exchange slot for the row sums (last used at tile ntiles - 2)
    if (ok && ntiles > 0) {
      const int jl = ntiles - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_empty[jl & 1], (jl >> 1) & 1, abort_flag, p.wait_limit));
      // the row's sum is the two halves' sums
      if (ok) {
        if (warp < kSoftmaxWarps) {
          xbuf[(xs * 2 + (warp >> 2)) * kPM + r] = l_run;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.xl[eq]);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.xl[eq], 0, abort_flag, p.wait_limit));
      }
      if (ok && p.fuse_gate) ok = __all_sync(0xffffffffu, mbar_wait(&bars.g, 0, abort_flag, p.wait_limit));
      if (!ok) fail();
      tc_fence_after();
    }
    if (ok) {
      const float l_row = (ntiles > 0) ? xbuf[xs * 2 * kPM + r] + xbuf[(xs * 2 + 1) * kPM + r] : 0.0f;
      const float inv = (l_row > 0.0f) ? 1.0f / l_row : 0.0f;
      unsigned char* ostage = sm + kOffV;
      unsigned char* orow = ostage + r * 128;             // output row r of block c at + c * kBlk
      const unsigned char* grow = sm + kOffQ + r * 128;  // gate row r of block c at + c * kBlk
      const int nch = (warp < kSoftmaxWarps) ? 3 : 2;
      uint32_t needs[3] = {0u, 0u, 0u};  // per chunk: elements whose exact product is still to do
#pragma unroll
      for (int ci = 0; ci < 3; ++ci) {
        if (ci >= nch) break;
        const int c0 = 32 * ((warp < kSoftmaxWarps) ? (4 * (warp >> 2) + ci) : (ci ? 7 : 3));
        float o[32];
        if (ntiles > 0) {
          tmem_ld32(t_row + kTmemO + c0, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.0f;
        }
        uint32_t res[16];  // BF16 pairs: elements c0 + 2 e (low half) and c0 + 2 e + 1
#pragma unroll
        for (int e = 0; e < 16; ++e) res[e] = 0u;
        // a row past the end (after the warp-collective load) is not computed; TMA drops it
        if (qi < p.Sq) {
          // every BF16 rounding here is done two values at a time (cvt.rn.bf16x2.f32)
          uint32_t ob[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) ob[e] = bf16x2_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
          if (p.fuse_gate) {
            // RNE_bf16(sigmoid(g)) from the SFU: for |g| <= 16, 1 / (1 + 2^(-g log2 e))
            // (2^x and 1/x approximations) is within 24 float ulp of the real value
            // (argument rounding |g| log2 e * 2^-24, 2^x ~2^-22, the add and 1/x ~2^-23),
            // so its BF16 rounding is the correct one unless its low 16 bits lie within 32
            // of the tie.  Branch-free over the 32 elements (so their SFU chains
            // interleave); an element that needs the exact path (|g| > 16 or NaN, a
            // sigmoid near a tie, a product below the float normal range) is staged
            // ungated, marked, and redone after the chunk from the table of all 65 536
            // BF16 sigmoids.  Exhaustively checked against the FP64 oracle on all 65 536
            // gate codes through this epilogue.
            uint32_t gp[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int d = c0 + 2 * e;  // gate elements d, d + 1 of row r
              if (ntiles > 0) {
                const int cb = d >> 6, ch = (d & 63) >> 3;
                gp[e] = *reinterpret_cast<const uint32_t*>(grow + cb * kBlk + 16 * (ch ^ (r & 7)) + 2 * (d & 7));
              } else {
                gp[e] = __ldg(reinterpret_cast<const uint32_t*>(p.gate + (((size_t)b * p.Sq + qi) * p.Hq + h) * kD + d));
              }
            }
            uint32_t need = 0u;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float sg[2], pr[2];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const float g = __uint_as_float(t ? (gp[e] & 0xFFFF0000u) : (gp[e] << 16));
                float ex, rc;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ex) : "f"(g * -1.44269504088896341f));
                asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(1.0f + ex));
                sg[t] = rc;
                const uint32_t low = __float_as_uint(rc) & 0xFFFFu;
                need |= (!(fabsf(g) <= 16.0f) || (low - 0x7FE0u <= 0x40u)) ? (1u << (2 * e + t)) : 0u;
              }
              const uint32_t sv = bf16x2_rn(sg[0], sg[1]);
              pr[0] = __fmul_rn(__uint_as_float(ob[e] << 16), __uint_as_float(sv << 16));
              pr[1] = __fmul_rn(__uint_as_float(ob[e] & 0xFFFF0000u), __uint_as_float(sv & 0xFFFF0000u));
#pragma unroll
              for (int t = 0; t < 2; ++t)
                need |= (fabsf(pr[t]) < 1.17549435e-38f && pr[t] != 0.0f) ? (1u << (2 * e + t)) : 0u;
              res[e] = bf16x2_rn(pr[0], pr[1]);
              // a marked element is staged as O (BF16) and finished below
              const uint32_t m2 = (need >> (2 * e)) & 3u;
              if (m2) res[e] = (res[e] & ~((m2 & 1u) * 0xFFFFu) & ~((m2 >> 1) * 0xFFFF0000u)) |
                               (ob[e] & (((m2 & 1u) * 0xFFFFu) | ((m2 >> 1) * 0xFFFF0000u)));
            }
            needs[ci] = need;
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) res[e] = ob[e];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cb = (c0 + 8 * u) >> 6, ch = ((c0 + 8 * u) & 63) >> 3;
          *reinterpret_cast<uint4*>(orow + cb * kBlk + 16 * (ch ^ (r & 7))) =
              make_uint4(res[4 * u], res[4 * u + 1], res[4 * u + 2], res[4 * u + 3]);
        }
      }
      // the marked elements: exact sigmoid from the table, exact product (each lane only
      // touches its own row)
#pragma unroll
      for (int ci = 0; ci < 3; ++ci) {
        uint32_t m = needs[ci];
        const int c0 = 32 * ((warp < kSoftmaxWarps) ? (4 * (warp >> 2) + ci) : (ci ? 7 : 3));
        while (m != 0u) {
          const int d = c0 + __ffs(m) - 1;
          m &= m - 1u;
          const int cb = d >> 6, ch = (d & 63) >> 3;
          uint16_t* op = reinterpret_cast<uint16_t*>(orow + cb * kBlk + 16 * (ch ^ (r & 7)) + 2 * (d & 7));
          const uint16_t gb = (ntiles > 0)
              ? *reinterpret_cast<const uint16_t*>(grow + cb * kBlk + 16 * (ch ^ (r & 7)) + 2 * (d & 7))
              : __ldg(reinterpret_cast<const uint16_t*>(p.gate + (((size_t)b * p.Sq + qi) * p.Hq + h) * kD + d));
          *op = gate_product_fast(*op, __ldg(g_sigmoid_table + gb));
        }
      }
      if (p.lse && qi < p.Sq && warp < 4) {
        p.lse[((size_t)b * p.Hq + h) * p.Sq + qi] =
            (l_row > 0.0f) ? (m_run + log2f(l_row)) * 0.69314718055994530942f : -INFINITY;
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.ost);
      if (tid == 0) {
        // every warp has staged its part: four TMA stores, then wait until they have read
        // the staging buffer before the CTA's shared memory goes away
        if (mbar_wait(&bars.ost, 0, abort_flag, p.wait_limit)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_store_4d(&to, 64 * c, h, i0, b, ostage + c * kBlk);
          tma_store_commit_and_wait_read();
        } else {
          fail();
        }
      }
    }
  }

  // ---- teardown: every role is done (or gave up and waited for what it started)
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [B, S, H, D] BF16, box {64, 1, rows, 1}, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int B, int S, int H, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, (cuuint64_t)S * H * kD * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q, K, V or the gate [B, S, H, D] BF16 as a 5-D tensor {64 elements, S, 4 column
// blocks, H, B} with box {64, rows, blocks, 1, 1}: one copy fills a tile laid out
// [block][row][128 B] (128-byte swizzle), the layout the MMA descriptors read
bool make_map_kv(CUtensorMap* m, const void* base, int B, int S, int H, int rows, int blocks) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[5] = {64, (cuuint64_t)S, 4, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[4] = {(cuuint64_t)H * kD * 2, 128, (cuuint64_t)kD * 2, (cuuint64_t)S * H * kD * 2};
  const cuuint32_t box[5] = {64, (cuuint32_t)rows, (cuuint32_t)blocks, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// First use on a device: the kernel's shared-memory limit and the sigmoid table.
// The table is built on a private stream that is waited for before the device is
// marked ready, so every later call, on any stream or thread, finds it complete.
// Refused while `stream` is capturing: the table must exist outside any graph.
static cudaError_t prefill_init(int dev, cudaStream_t stream) {
  static std::mutex mu;
  static bool ready[64] = {};
  std::lock_guard<std::mutex> lk(mu);
  if (ready[dev]) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  if (cs != cudaStreamCaptureStatusNone) return cudaErrorStreamCaptureUnsupported;
  e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaStream_t own = nullptr;
  e = cudaStreamCreateWithFlags(&own, cudaStreamNonBlocking);
  if (e != cudaSuccess) return e;
  sigmoid_table_kernel<<<256, 256, 0, own>>>();
  e = cudaGetLastError();
  const cudaError_t es = cudaStreamSynchronize(own);
  cudaStreamDestroy(own);
  if (e != cudaSuccess) return e;
  if (es != cudaSuccess) return es;
  ready[dev] = true;
  return cudaSuccess;
}

cudaError_t launch_prefill(const PrefillParams& p, const void* q, const void* k, const void* v, const void* gate,
                           cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tg, to;
  // S = 0 still needs a valid map: use extent 1 (nothing is loaded then)
  if (!make_map_kv(&tq, q, p.B, p.Sq > 0 ? p.Sq : 1, p.Hq, kPM, 4) ||
      !make_map_kv(&tk, k, p.B, p.Skv > 0 ? p.Skv : 1, p.Hkv, kPN, 2) ||
      !make_map_kv(&tv, v, p.B, p.Skv > 0 ? p.Skv : 1, p.Hkv, kPN, 2) ||
      !make_map_kv(&tg, gate ? gate : q, p.B, p.Sq > 0 ? p.Sq : 1, p.Hq, kPM, 4) ||
      !make_map(&to, p.out, p.B, p.Sq > 0 ? p.Sq : 1, p.Hq, kPM))
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = prefill_init(dev, stream);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(((p.Sq + kPM - 1) / kPM) * p.Hq), (unsigned)p.B, 1u);
  prefill_kernel<<<grid, kPThreads, kSmemBytes, stream>>>(tq, tk, tv, tg, to, p);
  return cudaGetLastError();
}

}  // namespace gda
