// gda_stage1_fp8.cu -- split-KV decode stage 1 over an FP8 (e4m3) KV cache, sm_103a.
//
// The K and V pools hold e4m3 codes (one byte per element) with one per-tensor
// descale each: K = k_descale * e4m3(code), V = v_descale * e4m3(code)
// (cuDNN FE-OSS "Gated Attention Block (SM107)", API, QuantSpec: static
// per-tensor scales for torch.float8_e4m3fn).  Q stays BF16.  The partial O and
// LSE it writes are the same as the BF16-cache stage 1's, so stage 2 (FP32 merge
// and the gate epilogue) is shared.
//
// GB300 design.  The BF16 kernel's structure with 32-token warp tiles, so one
// iteration moves the same 16 KiB (K + V) as a 16-token BF16 tile: the memory
// pipeline per iteration is unchanged while the arithmetic per byte doubles.
//  * Persistent grid, one CTA of 8 warps per SM; warp w takes tiles w, w+8, ...
//    of its CTA's piece.  K rows (256 bytes) are loaded with 16-byte streaming
//    loads straight into registers about one tile ahead and prefetched into L2
//    two tiles ahead; V rows go through a per-warp 3-stage cp.async ring two tiles
//    ahead (L2 evict-first hint).
//  * e4m3 values are exact in FP16, so the codes are widened with
//    cvt.rn.f16x2.e4m3x2 and the tiles run as m16n8k16 f16 MMAs with FP32
//    accumulation.  Q is moved into FP16 with one power-of-two factor per piece
//    (its largest magnitude lands in [2^14, 2^15)); that factor and k_descale
//    are folded into the score scale, v_descale into the partial's normalisation.
//  * QK: S^T[32 tok x 8 heads] = K Q^T, two m-tiles.  Lane (g, t) loads dims
//    {64c + 16t .. +15} (c = 0..3) of tokens g, g+8, g+16, g+24 (chunk c of the
//    next tile is loaded once QK has used chunk c + 1 of this one, chunk 3 after
//    the last MMA, so each load is about one tile ahead of its use); k-step
//    kk = 4c + h uses dims 64c + 16t + 4h + {0,1} for k-slots (2t, 2t+1) and
//    + {2,3} for (2t+8, 2t+9); the Q^T fragments use the same order.
//  * PV: O^T[256 x 8] += V^T P^T, two k-steps of 16 tokens.  The V^T fragment
//    pairs two tokens per register, so lane (g, t) reads from the ring tokens
//    2t, 2t+1, 2t+8, 2t+9 (+16 for the second k-step), bytes {128h + 16g .. +15}
//    (h = 0, 1), and byte permutes pair the tokens before the widening.  Row g of
//    m-tile mt is dim d0 = 128 (mt / 8) + 16 g + 2 (mt % 8), row g+8 is d0 + 1.
//    P is rounded to FP16 (it lies in [0, 2^8]) and transposed with movmatrix.
//  * Merge: each warp writes its rescaled O^T fragments into its idle ring in
//    fragment order (conflict-free float4 stores); all threads add the 8 warps'
//    slices in a fixed order and write one partial per piece.
#include <atomic>
#include <cuda_fp16.h>

#include "gda_device.cuh"
#include "gda_kernels.h"

namespace gda {

namespace {

constexpr int kRowBytes8 = kD;  // one (slot, KV head) row of e4m3 codes
constexpr int kW8 = 8;          // warps per CTA
constexpr float kLazyLog2F8 = 8.0f;

// Widen the four e4m3 codes of w: lo = f16x2(byte 0, byte 1), hi = f16x2(byte 2, byte 3)
// (the lower byte of each pair goes to the lower half).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ void mma_f16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t x) {
  return __half22float2(*reinterpret_cast<const __half2*>(&x));
}

__device__ __forceinline__ uint4 ld_stream16(const unsigned char* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

constexpr int kTok8 = 32;                  // tokens per warp tile
constexpr int kNV8 = 3;                    // V ring stages per warp
constexpr int kRing8Row = kRowBytes8 + 16; // padded ring row: conflict-free 16-byte reads

struct Fp8Smem {
  uint2 qf[16][32];                                  // Q^T fragments (FP16, scaled), lane order
  unsigned char vring[kW8][kNV8][kTok8][kRing8Row];  // per-warp V rings; stage 0 also holds the merge slice
  float mbuf[kW8][kG];                               // each warp's running max
  float lsum[kW8][kG];                               // each warp's rescaled sum
  unsigned int qmax;                                 // largest |q| of the piece's group (float bits)
};
// Pairs of groups: both groups' Q^T fragments and each warp's S^T of its tile for its
// partner's group (one buffer; the partner signals a read-done barrier once it has
// taken it).
struct Fp8PairSmem {
  uint2 qf[2][16][32];
  unsigned char vring[kW8][kNV8][kTok8][kRing8Row];
  float mbuf[kW8][kG];
  float lsum[kW8][kG];
  float4 xs[kW8][2][32];
  unsigned int qmax[2];                              // largest |q| of each group of the piece (float bits)
};
static_assert(sizeof(float4) * 16 * 32 <= kTok8 * kRing8Row, "merge slice fits a ring stage");

__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

struct Fp8WarpState {
  uint4 kr[16];  // K of the next tile: kr[4j + c] = token g + 8j, dims 64c + 16t .. +15
  float o[16][4];
  float m0, m1, l0, l1;
  uint32_t P[4];  // one group: FP16 probabilities, P[j] = tokens g + 8j, heads (2t, 2t+1)

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
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = __shfl_sync(0xffffffffu, slot_lane, g + 8 * j);
      const unsigned char* row = kb + (size_t)max(s, 0) * stride + 16 * t;
#pragma unroll
      for (int c = 0; c < 4; ++c) kr[4 * j + c] = (s >= 0) ? ld_stream16(row + 64 * c) : z;
    }
  }

  // QK of the tile in kr, then the softmax update (one group: the probabilities go to P).  After the K registers of chunk
  // c have had their last use, chunk c of the next tile (slots slot_next) is
  // loaded into them one chunk later (measured: one chunk later than the earliest
  // point is faster on randomly placed rows), so every K load is about one tile
  // ahead of its use.
  __device__ __forceinline__ void qk_softmax(const uint2 (*qf)[32], int nv, float sl2, int lane,
                                             const unsigned char* kb, size_t stride, int slot_next, bool more) {
    const int g = lane >> 2, t = lane & 3;
    const unsigned char* rn[4];
    bool okn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int sn = __shfl_sync(0xffffffffu, slot_next, g + 8 * j);
      okn[j] = more && sn >= 0;
      rn[j] = kb + (size_t)max(sn, 0) * stride + 16 * t;
    }
    float acc[4][4];  // [m-tile * 2 + (kk & 1)][4]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int kk = 4 * c + h;
        const uint2 b = qf[kk][lane];
#pragma unroll
        for (int mtile = 0; mtile < 2; ++mtile) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + c], h), a0, a2);
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + 4 + c], h), a1, a3);
          mma_f16_16816(acc[2 * mtile + (kk & 1)], a0, a1, a2, a3, b.x, b.y);
        }
      }
      if (more && c >= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) kr[4 * j + c - 1] = okn[j] ? ld_stream16(rn[j] + 64 * (c - 1)) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (more) {
#pragma unroll
      for (int j = 0; j < 4; ++j) kr[4 * j + 3] = okn[j] ? ld_stream16(rn[j] + 64 * 3) : make_uint4(0u, 0u, 0u, 0u);
    }
    float s[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[i] = (acc[0][i] + acc[1][i]) * sl2;
      s[4 + i] = (acc[2][i] + acc[3][i]) * sl2;
    }
    const int tg = lane >> 2;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (tg + 8 * j >= nv) s[2 * j] = s[2 * j + 1] = -INFINITY;
    // Lazy rescale (as in the BF16 kernel): the reference maxima move only when a
    // score exceeds them by more than kLazyLog2F8, so probabilities stay <= 2^8.
    const float xa0 = fmaxf(fmaxf(s[0], s[2]), fmaxf(s[4], s[6]));
    const float xb0 = fmaxf(fmaxf(s[1], s[3]), fmaxf(s[5], s[7]));
    const bool grow = xa0 > m0 + kLazyLog2F8 || xb0 > m1 + kLazyLog2F8;
    if (__any_sync(0xffffffffu, grow)) {
      float xa = xa0, xb = xb0;
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
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      P[j] = pack_f16x2(safe_exp2_diff(s[2 * j], m0), safe_exp2_diff(s[2 * j + 1], m1));
      const float2 pf = unpack_f16x2(P[j]);
      l0 += pf.x;
      l1 += pf.y;
    }
  }

  // Unscaled S^T of the tile in kr against one group's Q^T fragments: s[4 mt + i] is
  // accumulator i of m-tile mt (tokens g + 16 mt and g + 16 mt + 8, heads 2t, 2t + 1).
  // With REFILL, after the K registers of chunk c have had their last use, chunk c of
  // the next tile (slots slot_next) is loaded into them one chunk later (measured: one
  // chunk later than the earliest point is faster on randomly placed rows), so every K
  // load is about one tile ahead of its use.
  template <bool REFILL>
  __device__ __forceinline__ void qk_raw(const uint2 (*qf)[32], int lane, const unsigned char* kb, size_t stride,
                                         int slot_next, bool more, float* s) {
    const int g = lane >> 2, t = lane & 3;
    const unsigned char* rn[4];
    bool okn[4];
    if (REFILL) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int sn = __shfl_sync(0xffffffffu, slot_next, g + 8 * j);
        okn[j] = more && sn >= 0;
        rn[j] = kb + (size_t)max(sn, 0) * stride + 16 * t;
      }
    }
    float acc[4][4];  // [m-tile * 2 + (kk & 1)][4]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int kk = 4 * c + h;
        const uint2 b = qf[kk][lane];
#pragma unroll
        for (int mtile = 0; mtile < 2; ++mtile) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + c], h), a0, a2);
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + 4 + c], h), a1, a3);
          mma_f16_16816(acc[2 * mtile + (kk & 1)], a0, a1, a2, a3, b.x, b.y);
        }
      }
      if (REFILL && more && c >= 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) kr[4 * j + c - 1] = okn[j] ? ld_stream16(rn[j] + 64 * (c - 1)) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (REFILL && more) {
#pragma unroll
      for (int j = 0; j < 4; ++j) kr[4 * j + 3] = okn[j] ? ld_stream16(rn[j] + 64 * 3) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[i] = acc[0][i] + acc[1][i];
      s[4 + i] = acc[2][i] + acc[3][i];
    }
  }

  // Unscaled S^T of the tile in kr for two groups at once (qk_raw's layout and summation
  // order for each): every converted K fragment feeds both groups' MMAs.  One m-tile
  // (16 tokens) at a time, so the two groups' accumulators stay within qk_raw's
  // register count; the next tile's K chunks are loaded as in qk_raw, per m-tile.  The
  // second group's scores go straight to shared memory: m-tile mt at xb[mt][lane].
  __device__ __forceinline__ void qk_raw_pair(const uint2 (*qa)[32], const uint2 (*qb)[32], int lane,
                                              const unsigned char* kb, size_t stride, int slot_next, bool more,
                                              float* sa, float4 (*xb)[32]) {
    const int g = lane >> 2, t = lane & 3;
    const unsigned char* rn[4];
    bool okn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int sn = __shfl_sync(0xffffffffu, slot_next, g + 8 * j);
      okn[j] = more && sn >= 0;
      rn[j] = kb + (size_t)max(sn, 0) * stride + 16 * t;
    }
#pragma unroll
    for (int mtile = 0; mtile < 2; ++mtile) {
      float acc[2][2][4];  // [group][kk & 1][4]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[x][0][i] = acc[x][1][i] = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int kk = 4 * c + h;
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + c], h), a0, a2);
          e4m3x4_to_f16x2x2(word(kr[8 * mtile + 4 + c], h), a1, a3);
          const uint2 ba = qa[kk][lane], bb = qb[kk][lane];
          mma_f16_16816(acc[0][kk & 1], a0, a1, a2, a3, ba.x, ba.y);
          mma_f16_16816(acc[1][kk & 1], a0, a1, a2, a3, bb.x, bb.y);
        }
        if (more && c >= 1) {
#pragma unroll
          for (int j = 2 * mtile; j < 2 * mtile + 2; ++j)
            kr[4 * j + c - 1] = okn[j] ? ld_stream16(rn[j] + 64 * (c - 1)) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (more) {
#pragma unroll
        for (int j = 2 * mtile; j < 2 * mtile + 2; ++j)
          kr[4 * j + 3] = okn[j] ? ld_stream16(rn[j] + 64 * 3) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sa[4 * mtile + i] = acc[0][0][i] + acc[0][1][i];
      xb[mtile][lane] = make_float4(acc[1][0][0] + acc[1][1][0], acc[1][0][1] + acc[1][1][1],
                                    acc[1][0][2] + acc[1][1][2], acc[1][0][3] + acc[1][1][3]);
    }
  }

  // Online softmax over NT 32-token tiles of the same 8 heads: tile x has nv[x] valid
  // tokens and unscaled scores s[x] (qk_raw's layout).  Lazy rescale (as in the BF16
  // kernel): the reference maxima move only when a score exceeds them by more than
  // kLazyLog2F8, so probabilities stay <= 2^8.  P[x][j]: FP16 probabilities of tile x,
  // tokens g + 8j, heads (2t, 2t+1); their rounded values join the sums tile by tile.
  template <int NT>
  __device__ __forceinline__ void softmax_tiles(float (*s)[8], const int* nv, float sl2, int lane,
                                                uint32_t (*P)[4]) {
    const int tg = lane >> 2;
    float xa0 = -INFINITY, xb0 = -INFINITY;
#pragma unroll
    for (int x = 0; x < NT; ++x) {
      // s[x][2j], s[x][2j + 1]: token g + 8j (j = 0 .. 3), heads 2t, 2t + 1
#pragma unroll
      for (int i = 0; i < 8; ++i) s[x][i] *= sl2;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (tg + 8 * j >= nv[x]) s[x][2 * j] = s[x][2 * j + 1] = -INFINITY;
      xa0 = fmaxf(xa0, fmaxf(fmaxf(s[x][0], s[x][2]), fmaxf(s[x][4], s[x][6])));
      xb0 = fmaxf(xb0, fmaxf(fmaxf(s[x][1], s[x][3]), fmaxf(s[x][5], s[x][7])));
    }
    const bool grow = xa0 > m0 + kLazyLog2F8 || xb0 > m1 + kLazyLog2F8;
    if (__any_sync(0xffffffffu, grow)) {
      float xa = xa0, xb = xb0;
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
#pragma unroll
    for (int x = 0; x < NT; ++x)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        P[x][j] = pack_f16x2(safe_exp2_diff(s[x][2 * j], m0), safe_exp2_diff(s[x][2 * j + 1], m1));
        const float2 pf = unpack_f16x2(P[x][j]);
        l0 += pf.x;
        l1 += pf.y;
      }
  }

  // O^T += V^T P^T from a 32-row ring stage: per k-step of 16 tokens, the lane's
  // four tokens are read (two 16-byte halves each), paired by byte permutes and
  // widened to FP16.
  __device__ __forceinline__ void pv(const unsigned char* vtile, int lane) { pv_with(vtile, P, lane); }

  __device__ __forceinline__ void pv_with(const unsigned char* vtile, const uint32_t* P, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t base = smem_u32(vtile) + 16 * g;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const uint32_t b0 = movmatrix_trans(P[2 * ks]), b1 = movmatrix_trans(P[2 * ks + 1]);
      uint4 vr[8];  // vr[2i + h]: token T_i = 16ks + (2t, 2t+1, 2t+8, 2t+9)[i], bytes 128h + 16g
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int tok = 16 * ks + 2 * t + (i & 1) + 8 * (i >> 1);
        vr[2 * i] = lds128(base + tok * kRing8Row);
        vr[2 * i + 1] = lds128(base + tok * kRing8Row + 128);
      }
#pragma unroll
      for (int mt = 0; mt < 16; ++mt) {
        const int hs = mt >> 3, wi = (mt & 7) >> 1;
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t x01 = __byte_perm(word(vr[0 + hs], wi), word(vr[2 + hs], wi), sel);
        const uint32_t x23 = __byte_perm(word(vr[4 + hs], wi), word(vr[6 + hs], wi), sel);
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2x2(x01, a0, a1);  // (d0: T0, T1), (d1: T0, T1)
        e4m3x4_to_f16x2x2(x23, a2, a3);  // (d0: T2, T3), (d1: T2, T3)
        mma_f16_16816(o[mt], a0, a1, a2, a3, b0, b1);
      }
    }
  }
};

// Prefetch into L2 the K rows of a 32-token tile: lane l takes both 128-byte lines
// of token l's row.
__device__ __forceinline__ void prefetch_k_tile8(const unsigned char* kb, size_t stride, int slot_lane) {
  if (slot_lane >= 0) {
    const unsigned char* row = kb + (size_t)slot_lane * stride;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 128));
  }
}

// Issue the cp.async copies of one V tile (32 rows of 256 bytes; rows >= n and bad
// slots are zero-filled) into a ring stage and commit them as one group: each
// instruction moves two rows, 16 lanes per row.
__device__ __forceinline__ void issue_v_tile8(unsigned char* stage, const unsigned char* vb, size_t stride,
                                              int slot_lane, int n, int lane, uint64_t policy) {
  const int half = lane >> 4, chunk = lane & 15;
  const uint32_t dst0 = smem_u32(stage) + 16 * chunk;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = 2 * i + half;
    const int s = __shfl_sync(0xffffffffu, slot_lane, r);
    const bool ok = (r < n) && (s >= 0);
    const unsigned char* src = vb + (ok ? (size_t)s * stride : (size_t)0) + 16 * chunk;
    cp_async16_hint(dst0 + r * kRing8Row, src, ok ? 16u : 0u, policy);
  }
  cp_async_commit_group();
}

__global__ void __launch_bounds__(kW8 * 32, 1) stage1_fp8_kernel(Stage1Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Fp8Smem& sm = *reinterpret_cast<Fp8Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) sm.qmax = 0u;
  Sched sched;
  sched.begin(p.indptr, p.B, p.Hkv * p.npass, p.num_splits, gridDim.x, blockIdx.x, p.min_chunk, p.window, p.piece_cost, p.rule_kv8);
  const size_t stride = (size_t)p.Hkv * kRowBytes8;
  const uint64_t pol_v = l2_policy_evict_first();

  auto nmine_of = [&](int len) -> int {
    const int ntiles = (len + kTok8 - 1) / kTok8;
    return (ntiles > warp) ? (ntiles - warp + kW8 - 1) / kW8 : 0;
  };
  auto tile_n = [&](int k, int len, int nmine) -> int {
    return (k < nmine) ? min(kTok8, len - kTok8 * (warp + kW8 * k)) : 0;
  };
  // slot of token `lane` of this warp's tile k (-1 past the tile's end or for a bad index)
  auto fetch = [&](const int* idx, int k, int len, int nmine) -> int {
    const int n = tile_n(k, len, nmine);
    int s = -1;
    if (lane < n) {
      s = __ldg(idx + kTok8 * (warp + kW8 * k) + lane);
      if (p.check_indices && (s < 0 || (long long)s >= p.num_slots)) {
        atomicOr(&p.hdr->error, kErrIndex);
        s = -1;
      }
    }
    return s;
  };

  Fp8WarpState st;
  uint2 qraw[2];  // this thread's two BF16 Q^T fragments of the next piece
  int s0 = -1, s1 = -1, s2 = -1;
  // Head of a piece: its Q rows (BF16, converted at the piece start), the slots of
  // this warp's first three tiles and the K rows of its first tile.  For every
  // piece after the first this runs before the previous piece's merge.
  auto piece_head = [&](const Piece& pp) {
    const int kvh = pp.kvh / p.npass, pass = pp.kvh - kvh * p.npass;
    const int gv = min(kG, p.G - kG * pass);
    const __nv_bfloat16* qg = p.q + ((size_t)pp.b * p.Hq + (size_t)kvh * p.G + (size_t)kG * pass) * kD;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int e = threadIdx.x + r * kW8 * 32;
      const int kk = e >> 5, ln = e & 31;
      const int g = ln >> 2, t = ln & 3, c = kk >> 2, h = kk & 3;
      const __nv_bfloat16* row = qg + min(g, gv - 1) * kD;  // never addresses a row beyond the group
      qraw[r] = (g < gv) ? __ldg(reinterpret_cast<const uint2*>(row + 64 * c + 16 * t + 4 * h)) : make_uint2(0u, 0u);
    }
    const int* idx = p.indices + pp.base + pp.j0;
    const int len = pp.j1 - pp.j0, nmine = nmine_of(len);
    s0 = fetch(idx, 0, len, nmine);
    s1 = fetch(idx, 1, len, nmine);
    s2 = fetch(idx, 2, len, nmine);
    if (nmine > 0) st.load_k(p.k_pool + (size_t)kvh * kRowBytes8, stride, s0, lane);
  };

  __syncthreads();  // qmax initialised
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
    const size_t head_off = (size_t)(pc.kvh / p.npass) * kRowBytes8;
    const unsigned char* kb = p.k_pool + head_off;
    const unsigned char* vb = p.v_pool + head_off;
    const int* idx = p.indices + pc.base + pc.j0;
    const int len = pc.j1 - pc.j0;
    const int nmine = nmine_of(len);

    st.reset();
    unsigned char(*ring)[kTok8][kRing8Row] = sm.vring[warp];
    if (nmine > 0) {
      issue_v_tile8(&ring[0][0][0], vb, stride, s0, tile_n(0, len, nmine), lane, pol_v);
      issue_v_tile8(&ring[1 % kNV8][0][0], vb, stride, s1, tile_n(1, len, nmine), lane, pol_v);
      prefetch_k_tile8(kb, stride, s1);
    }

    // Q into FP16: one power-of-two factor 2^e for the group puts its largest
    // magnitude in [2^14, 2^15) (every BF16 value at most 2^28 below it is exact).
    {
      float mx = 0.0f;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t w2[2] = {qraw[r].x, qraw[r].y};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mx = fmaxf(mx, fabsf(__uint_as_float(w2[j] << 16)));
          mx = fmaxf(mx, fabsf(__uint_as_float(w2[j] & 0xFFFF0000u)));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (lane == 0) atomicMax(&sm.qmax, __float_as_uint(mx));
    }
    __syncthreads();  // also: the previous piece's merge is done with the rings and Q fragments
    const unsigned int qm = sm.qmax;
    int e = (qm == 0u) ? 0 : 141 - (int)((qm >> 23) & 0xFFu);  // 2^e * max in [2^14, 2^15)
    e = max(-126, min(127, e));
    const float qs = __uint_as_float((uint32_t)(e + 127) << 23);
    const float sl2 = ldexpf(p.scale_log2, -e);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int idxq = threadIdx.x + r * kW8 * 32;
      const uint32_t x = qraw[r].x, y = qraw[r].y;
      uint2 f;
      f.x = pack_f16x2(__uint_as_float(x << 16) * qs, __uint_as_float(x & 0xFFFF0000u) * qs);
      f.y = pack_f16x2(__uint_as_float(y << 16) * qs, __uint_as_float(y & 0xFFFF0000u) * qs);
      sm.qf[idxq >> 5][idxq & 31] = f;
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.qmax = 0u;  // every thread has read it; the next write follows a barrier

    int stage = 0;
    for (int k = 0; k < nmine; ++k) {
      // V two tiles ahead (an empty group when there is no such tile), K rows of
      // that tile into L2, the slots three tiles ahead; then tile k's QK
      issue_v_tile8(&ring[(k + 2) % kNV8][0][0], vb, stride, s2, tile_n(k + 2, len, nmine), lane, pol_v);
      prefetch_k_tile8(kb, stride, s2);
      const int s3 = fetch(idx, k + 3, len, nmine);
      st.qk_softmax(sm.qf, tile_n(k, len, nmine), sl2, lane, kb, stride, s1, k + 1 < nmine);
      cp_async_wait_group<2>();
      __syncwarp();
      st.pv(&ring[stage][0][0], lane);
      __syncwarp();
      stage = (stage + 1 == kNV8) ? 0 : stage + 1;
      s1 = s2;
      s2 = s3;
    }
    cp_async_wait_group<0>();
    __syncwarp();

    // look ahead: the next piece's first loads go out before this piece's merge
    Piece nx;
    const bool have_next = sched.next(nx);
    if (have_next) piece_head(nx);

    // ---- merge: fragment-order slices in the (now idle) rings, summed in a fixed order
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
      const int ha = 2 * (lane & 3), hb = ha + 1;
      float Ma = sm.mbuf[0][ha], Mb = sm.mbuf[0][hb];
#pragma unroll
      for (int x = 1; x < kW8; ++x) {
        Ma = fmaxf(Ma, sm.mbuf[x][ha]);
        Mb = fmaxf(Mb, sm.mbuf[x][hb]);
      }
      const float fa = (Ma == -INFINITY) ? 0.0f : safe_exp2_diff(st.m0, Ma);
      const float fb = (Mb == -INFINITY) ? 0.0f : safe_exp2_diff(st.m1, Mb);
      float4* slice = reinterpret_cast<float4*>(&sm.vring[warp][0][0][0]);
#pragma unroll
      for (int mt = 0; mt < 16; ++mt)
        slice[mt * 32 + lane] = make_float4(st.o[mt][0] * fa, st.o[mt][1] * fb, st.o[mt][2] * fa, st.o[mt][3] * fb);
      if (lane < 4) {
        sm.lsum[warp][ha] = st.l0 * fa;
        sm.lsum[warp][hb] = st.l1 * fb;
      }
    }
    __syncthreads();
    float* op = p.o_part + pc.id * (kG * kD);
    for (int f = threadIdx.x; f < 16 * 32; f += blockDim.x) {
      const int mt = f >> 5, ln = f & 31;
      const int g = ln >> 2, ha = 2 * (ln & 3), hb = ha + 1;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float la = 0.0f, lb = 0.0f;
#pragma unroll
      for (int x = 0; x < kW8; ++x) {
        const float4 v = reinterpret_cast<const float4*>(&sm.vring[x][0][0][0])[f];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
        la += sm.lsum[x][ha];
        lb += sm.lsum[x][hb];
      }
      const float ia = (la > 0.0f) ? p.v_descale / la : 0.0f;
      const float ib = (lb > 0.0f) ? p.v_descale / lb : 0.0f;
      const int d0 = 128 * (mt >> 3) + 16 * g + 2 * (mt & 7);
      *reinterpret_cast<float2*>(op + ha * kD + d0) = make_float2(acc.x * ia, acc.z * ia);
      *reinterpret_cast<float2*>(op + hb * kD + d0) = make_float2(acc.y * ib, acc.w * ib);
    }
    if (threadIdx.x < kG) {
      float M = sm.mbuf[0][threadIdx.x], lt = 0.0f;
#pragma unroll
      for (int x = 1; x < kW8; ++x) M = fmaxf(M, sm.mbuf[x][threadIdx.x]);
#pragma unroll
      for (int x = 0; x < kW8; ++x) lt += sm.lsum[x][threadIdx.x];
      p.lse_part[pc.id * kG + threadIdx.x] = (lt > 0.0f) ? M + log2f(lt) : -INFINITY;
    }
    __syncthreads();  // rings, Q fragments and merge buffers free for the next piece
    pc = nx;
    have = have_next;
  }
}

// PAIR (G > 8): the groups of 8 query heads of a KV head in pairs, one piece per
// (sequence, KV head, pair) serving both groups, so every K/V row is read once per
// pair.  Warp w loads its tiles as without PAIR and computes S^T of its tile for both
// groups (the partner group's first, then its own with the next tile's K loads);
// warps w and w ^ 4 form a pair, warps 0-3 owning group 0 and 4-7 group 1.  Each step
// a warp leaves the partner group's S^T in shared memory, the pair meets at a named
// barrier, and each warp runs the softmax and PV of its own group over both tiles:
// its own (its V ring) and the partner's (the partner's V ring).  The S^T buffer is
// single: its reader arrives on the writer's read-done barrier once it has taken it,
// and the writer waits on that barrier before the next write.  The partial of
// (piece, group) is written at piece * 2 + group.
__global__ void __launch_bounds__(kW8 * 32, 1) stage1_fp8_pair_kernel(Stage1Params p) {
  constexpr bool PAIR = true;
  constexpr int NG = 2;
  constexpr int WPG = kW8 / NG;  // warps per group
  constexpr int QPT = 2 * NG;    // Q^T fragments per thread
  using Smem = Fp8PairSmem;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / WPG;              // this warp's group
  const int partner = warp ^ (kW8 / 2);    // PAIR: the warp of the other group on the same tiles
  const int team = warp & (kW8 / 2 - 1);   // PAIR: the pair (named barrier 1 + team)
  // PAIR: read-done barrier of warp x's S^T buffer (named barriers 5 .. 12)
  auto read_bar = [](int x) -> int { return 5 + x; };

  if (threadIdx.x < 2) sm.qmax[threadIdx.x] = 0u;
  Sched sched;
  sched.begin(p.indptr, p.B, PAIR ? p.Hkv * p.nteam : p.Hkv * p.npass, p.num_splits, gridDim.x, blockIdx.x,
              p.min_chunk, p.window, p.piece_cost, p.rule_kv8);
  const size_t stride = (size_t)p.Hkv * kRowBytes8;
  const uint64_t pol_v = l2_policy_evict_first();
  auto kv_head = [&](const Piece& pp) -> int { return PAIR ? pp.kvh / p.nteam : pp.kvh / p.npass; };

  auto nmine_for = [&](int w, int len) -> int {
    const int ntiles = (len + kTok8 - 1) / kTok8;
    return (ntiles > w) ? (ntiles - w + kW8 - 1) / kW8 : 0;
  };
  auto tile_n_for = [&](int w, int k, int len, int nm) -> int {
    return (k < nm) ? min(kTok8, len - kTok8 * (w + kW8 * k)) : 0;
  };
  auto nmine_of = [&](int len) -> int { return nmine_for(warp, len); };
  auto tile_n = [&](int k, int len, int nmine) -> int { return tile_n_for(warp, k, len, nmine); };
  // slot of token `lane` of this warp's tile k (-1 past the tile's end or for a bad index)
  auto fetch = [&](const int* idx, int k, int len, int nmine) -> int {
    const int n = tile_n(k, len, nmine);
    int s = -1;
    if (lane < n) {
      s = __ldg(idx + kTok8 * (warp + kW8 * k) + lane);
      if (p.check_indices && (s < 0 || (long long)s >= p.num_slots)) {
        atomicOr(&p.hdr->error, kErrIndex);
        s = -1;
      }
    }
    return s;
  };

  Fp8WarpState st;
  uint2 qraw[QPT];  // this thread's BF16 Q^T fragments of the next piece
  int s0 = -1, s1 = -1, s2 = -1;
  // Head of a piece: its Q rows (BF16, converted at the piece start), the slots of
  // this warp's first three tiles and the K rows of its first tile.  For every
  // piece after the first this runs before the previous piece's merge.
  auto piece_head = [&](const Piece& pp) {
    // PAIR: the piece's KV head and the first group of its pair
    const int pkv = kv_head(pp), pg0 = PAIR ? 2 * (pp.kvh - pkv * p.nteam) : 0;
#pragma unroll
    for (int r = 0; r < QPT; ++r) {
      const int e = threadIdx.x + r * kW8 * 32;
      const int fg = e >> 9, kk = (e >> 5) & 15, ln = e & 31;  // group, k-step, lane
      const int g = ln >> 2, t = ln & 3, c = kk >> 2, h = kk & 3;
      // group pg0 + fg of the KV head (PAIR; past the last group it is empty: Q = 0, its
      // partial never read), else the piece's virtual head
      const int pass = PAIR ? min(pg0 + fg, p.npass - 1) : pp.kvh - pkv * p.npass;
      const int gv = (PAIR && pg0 + fg >= p.npass) ? 0 : min(kG, p.G - kG * pass);
      const __nv_bfloat16* qg = p.q + ((size_t)pp.b * p.Hq + (size_t)pkv * p.G + (size_t)kG * pass) * kD;
      const __nv_bfloat16* row = qg + max(0, min(g, gv - 1)) * kD;  // never addresses a row beyond the group
      qraw[r] = (g < gv) ? __ldg(reinterpret_cast<const uint2*>(row + 64 * c + 16 * t + 4 * h)) : make_uint2(0u, 0u);
    }
    const int* idx = p.indices + pp.base + pp.j0;
    const int len = pp.j1 - pp.j0, nmine = nmine_of(len);
    s0 = fetch(idx, 0, len, nmine);
    s1 = fetch(idx, 1, len, nmine);
    s2 = fetch(idx, 2, len, nmine);
    if (nmine > 0) st.load_k(p.k_pool + (size_t)pkv * kRowBytes8, stride, s0, lane);
  };

  __syncthreads();  // qmax initialised
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
    const size_t head_off = (size_t)kv_head(pc) * kRowBytes8;
    const unsigned char* kb = p.k_pool + head_off;
    const unsigned char* vb = p.v_pool + head_off;
    const int* idx = p.indices + pc.base + pc.j0;
    const int len = pc.j1 - pc.j0;
    const int nmine = nmine_of(len);
    // steps of this warp's loop: its tiles, or with PAIR those of the pair's first
    // warp (the one with more tiles), so that both partners meet at every barrier
    const int nsteps = PAIR ? nmine_for(team, len) : nmine;

    st.reset();
    unsigned char(*ring)[kTok8][kRing8Row] = sm.vring[warp];
    if (nsteps > 0) {
      issue_v_tile8(&ring[0][0][0], vb, stride, s0, tile_n(0, len, nmine), lane, pol_v);
      issue_v_tile8(&ring[1 % kNV8][0][0], vb, stride, s1, tile_n(1, len, nmine), lane, pol_v);
      prefetch_k_tile8(kb, stride, s1);
    }

    // Q into FP16: per group, one power-of-two factor 2^e puts the group's largest
    // magnitude in [2^14, 2^15) (every BF16 value at most 2^28 below it is exact).  Each
    // group has its own factor, so a group of ordinary magnitude beside a much larger
    // one keeps its scores; a warp's scores are those of its own group, scaled by its
    // group's factor.  Fragments r = 0, 1 of a thread are group 0's, r = 2, 3 group 1's.
    {
      float mx[2] = {0.0f, 0.0f};
#pragma unroll
      for (int r = 0; r < QPT; ++r) {
        const uint32_t w2[2] = {qraw[r].x, qraw[r].y};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mx[r >> 1] = fmaxf(mx[r >> 1], fabsf(__uint_as_float(w2[j] << 16)));
          mx[r >> 1] = fmaxf(mx[r >> 1], fabsf(__uint_as_float(w2[j] & 0xFFFF0000u)));
        }
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx[x] = fmaxf(mx[x], __shfl_xor_sync(0xffffffffu, mx[x], off));
        if (lane == 0) atomicMax(&sm.qmax[x], __float_as_uint(mx[x]));
      }
    }
    __syncthreads();  // also: the previous piece's merge is done with the rings and Q fragments
    float qs[2];
    float sl2 = 0.0f;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const unsigned int qm = sm.qmax[x];
      int e = (qm == 0u) ? 0 : 141 - (int)((qm >> 23) & 0xFFu);  // 2^e * max in [2^14, 2^15)
      e = max(-126, min(127, e));
      qs[x] = __uint_as_float((uint32_t)(e + 127) << 23);
      if (x == grp) sl2 = ldexpf(p.scale_log2, -e);
    }
#pragma unroll
    for (int r = 0; r < QPT; ++r) {
      const int idxq = threadIdx.x + r * kW8 * 32;
      const uint32_t x = qraw[r].x, y = qraw[r].y;
      const float f_s = qs[r >> 1];
      uint2 f;
      f.x = pack_f16x2(__uint_as_float(x << 16) * f_s, __uint_as_float(x & 0xFFFF0000u) * f_s);
      f.y = pack_f16x2(__uint_as_float(y << 16) * f_s, __uint_as_float(y & 0xFFFF0000u) * f_s);
      sm.qf[idxq >> 9][(idxq >> 5) & 15][idxq & 31] = f;
    }
    __syncthreads();
    if (threadIdx.x < 2) sm.qmax[threadIdx.x] = 0u;  // every thread has read them; the next writes follow a barrier

    int stage = 0;
    if constexpr (PAIR) {
      const int nmp = nmine_for(partner, len);
      for (int k = 0; k < nsteps; ++k) {
        // K rows of tile k+2 into L2, the slots of tile k+3; tile k's S^T for the
        // partner's group (to shared memory), then for this warp's own group with the
        // next tile's K loads
        prefetch_k_tile8(kb, stride, s2);
        const int s3 = fetch(idx, k + 3, len, nmine);
        const int nown = tile_n(k, len, nmine);
        float sc[2][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) sc[0][i] = sc[1][i] = 0.0f;
        if (k > 0) named_bar_sync(read_bar(warp), 64);  // the partner has taken step k-1's
        if (nown > 0) {
          st.qk_raw_pair(sm.qf[grp], sm.qf[grp ^ 1], lane, kb, stride, s1, k + 1 < nmine, sc[0], sm.xs[warp]);
        } else {
          sm.xs[warp][0][lane] = make_float4(0.f, 0.f, 0.f, 0.f);
          sm.xs[warp][1][lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        cp_async_wait_group<1>();  // this warp's V tile k has landed (tile k+1 may be in flight)
        // The pair meets: both V tiles k and both S^T are visible, and the partner has
        // finished step k-1, so ring stage (k+2) % 3 (read as stage (k-1) % 3) is free.
        named_bar_sync(1 + team, 64);
        issue_v_tile8(&ring[(k + 2) % kNV8][0][0], vb, stride, s2, tile_n(k + 2, len, nmine), lane, pol_v);
        {
          const float4 u0 = sm.xs[partner][0][lane], u1 = sm.xs[partner][1][lane];
          sc[1][0] = u0.x;
          sc[1][1] = u0.y;
          sc[1][2] = u0.z;
          sc[1][3] = u0.w;
          sc[1][4] = u1.x;
          sc[1][5] = u1.y;
          sc[1][6] = u1.z;
          sc[1][7] = u1.w;
        }
        __syncwarp();
        named_bar_arrive(read_bar(partner), 64);
        const int nt[2] = {nown, tile_n_for(partner, k, len, nmp)};
        uint32_t P[2][4];
        st.softmax_tiles<2>(sc, nt, sl2, lane, P);
        if (nt[0] > 0) st.pv_with(&ring[stage][0][0], P[0], lane);
        if (nt[1] > 0) st.pv_with(&sm.vring[partner][stage][0][0], P[1], lane);
        stage = (stage + 1 == kNV8) ? 0 : stage + 1;
        s1 = s2;
        s2 = s3;
      }
      if (nsteps > 0) named_bar_sync(read_bar(warp), 64);  // the partner's last read-done
    } else {
      for (int k = 0; k < nmine; ++k) {
        // V two tiles ahead (an empty group when there is no such tile), K rows of
        // that tile into L2, the slots three tiles ahead; then tile k's QK
        issue_v_tile8(&ring[(k + 2) % kNV8][0][0], vb, stride, s2, tile_n(k + 2, len, nmine), lane, pol_v);
        prefetch_k_tile8(kb, stride, s2);
        const int s3 = fetch(idx, k + 3, len, nmine);
        st.qk_softmax(sm.qf[0], tile_n(k, len, nmine), sl2, lane, kb, stride, s1, k + 1 < nmine);
        cp_async_wait_group<2>();
        __syncwarp();
        st.pv(&ring[stage][0][0], lane);
        __syncwarp();
        stage = (stage + 1 == kNV8) ? 0 : stage + 1;
        s1 = s2;
        s2 = s3;
      }
    }
    cp_async_wait_group<0>();
    __syncwarp();

    // look ahead: the next piece's first loads go out before this piece's merge
    Piece nx;
    const bool have_next = sched.next(nx);
    if (have_next) piece_head(nx);

    // ---- merge: fragment-order slices in the (now idle) rings, summed in a fixed order
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
      const int ha = 2 * (lane & 3), hb = ha + 1;
      const int x0 = grp * WPG;  // this group's warps: x0 .. x0 + WPG - 1
      float Ma = sm.mbuf[x0][ha], Mb = sm.mbuf[x0][hb];
#pragma unroll
      for (int x = 1; x < WPG; ++x) {
        Ma = fmaxf(Ma, sm.mbuf[x0 + x][ha]);
        Mb = fmaxf(Mb, sm.mbuf[x0 + x][hb]);
      }
      const float fa = (Ma == -INFINITY) ? 0.0f : safe_exp2_diff(st.m0, Ma);
      const float fb = (Mb == -INFINITY) ? 0.0f : safe_exp2_diff(st.m1, Mb);
      float4* slice = reinterpret_cast<float4*>(&sm.vring[warp][0][0][0]);
#pragma unroll
      for (int mt = 0; mt < 16; ++mt)
        slice[mt * 32 + lane] = make_float4(st.o[mt][0] * fa, st.o[mt][1] * fb, st.o[mt][2] * fa, st.o[mt][3] * fb);
      if (lane < 4) {
        sm.lsum[warp][ha] = st.l0 * fa;
        sm.lsum[warp][hb] = st.l1 * fb;
      }
    }
    __syncthreads();
    // partial (piece, group) at piece * NG + group
    for (int f = threadIdx.x; f < NG * 16 * 32; f += blockDim.x) {
      const int fg = f >> 9, fl = f & 511;
      const int mt = fl >> 5, ln = fl & 31;
      const int g = ln >> 2, ha = 2 * (ln & 3), hb = ha + 1;
      const int x0 = fg * WPG;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float la = 0.0f, lb = 0.0f;
#pragma unroll
      for (int x = x0; x < x0 + WPG; ++x) {
        const float4 v = reinterpret_cast<const float4*>(&sm.vring[x][0][0][0])[fl];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
        la += sm.lsum[x][ha];
        lb += sm.lsum[x][hb];
      }
      const float ia = (la > 0.0f) ? p.v_descale / la : 0.0f;
      const float ib = (lb > 0.0f) ? p.v_descale / lb : 0.0f;
      const int d0 = 128 * (mt >> 3) + 16 * g + 2 * (mt & 7);
      float* op = p.o_part + (pc.id * NG + fg) * (kG * kD);
      *reinterpret_cast<float2*>(op + ha * kD + d0) = make_float2(acc.x * ia, acc.z * ia);
      *reinterpret_cast<float2*>(op + hb * kD + d0) = make_float2(acc.y * ib, acc.w * ib);
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


}  // namespace

template <typename Smem>
cudaError_t launch_fp8(void (*kern)(Stage1Params), const Stage1Params& p, int grid, cudaStream_t stream,
                       std::atomic<bool>* attr_set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<grid, kW8 * 32, sizeof(Smem), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_stage1_fp8(const Stage1Params& p, int grid, cudaStream_t stream) {
  static std::atomic<bool> single_set[64], pair_set[64];  // zero-initialised: false
  return p.team == 2 ? launch_fp8<Fp8PairSmem>(stage1_fp8_pair_kernel, p, grid, stream, pair_set)
                     : launch_fp8<Fp8Smem>(stage1_fp8_kernel, p, grid, stream, single_set);
}

}  // namespace gda
