// gda_prep.cu -- the step before attention, for one decode token per sequence:
// per-head RMSNorm of Q and K, rotary embedding of their first rope_dim dims
// (rotate-half convention), and the write of the token's K and V rows into the
// paged pools at their slots (cuDNN FE-OSS "Gated Attention Block (SM107)",
// Overview stages (2)+(3) "QK-RMSNorm per head (optional) + partial RoPE on the
// first rope_dim, one kernel"; Weights and tables: w_q_norm, w_k_norm [D], cos,
// sin [B, rope_dim]).  The projection output of a token is the flat row
// [q (Hq*D) | gate (Hq*D) | k (Hkv*D) | v (Hkv*D)] (W_qkvg column blocks
// Q | GATE | K | V); the gate is copied out contiguously for the decode call.
//
// One warp per (token, row): lane l owns dims [8l, 8l+8) of the 256 (one 16-byte
// load and store).  The sum of squares is a warp all-reduce; the RoPE partner of
// dim d < rope_dim/2 is dim d + rope_dim/2, held by lane l + rope_dim/16 at the
// same position, fetched by shuffle.  FP32 arithmetic, one BF16 rounding (RNE).
// HBM-bound: 2 bytes read and 2 written per element of every row.
#include "gda_device.cuh"
#include "gda_kernels.h"

namespace gda {

__device__ __forceinline__ void unpack_bf16x8(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__global__ void __launch_bounds__(256) prep_kernel(PrepParams p) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int rows = 2 * p.Hq + 2 * p.Hkv;
  if (gw >= (long long)p.B * rows) return;  // whole warps
  const int b = (int)(gw / rows), r = (int)(gw % rows);
  const __nv_bfloat16* src = p.qgkv + (size_t)b * p.row_stride + (size_t)r * kD;
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + lane);

  const int slot = (r >= 2 * p.Hq) ? __ldg(p.slots + b) : 0;
  const bool slot_ok = slot >= 0 && (long long)slot < p.num_slots;
  if (r >= p.Hq && r < 2 * p.Hq) {  // gate: copied out
    if (p.gate_out != nullptr)
      reinterpret_cast<uint4*>(p.gate_out + ((size_t)b * p.Hq + (r - p.Hq)) * kD)[lane] = raw;
    return;
  }
  if (r >= 2 * p.Hq + p.Hkv) {  // v: written to its slot
    if (slot_ok)
      reinterpret_cast<uint4*>(p.v_pool + ((size_t)slot * p.Hkv + (r - 2 * p.Hq - p.Hkv)) * kD)[lane] = raw;
    return;
  }
  const bool is_q = r < p.Hq;
  float x[8];
  unpack_bf16x8(raw, x);
  const __nv_bfloat16* w = is_q ? p.w_q : p.w_k;
  if (w != nullptr) {
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float rinv = 1.0f / sqrtf(ss * (1.0f / kD) + p.eps);
    float wv[8];
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(w) + lane), wv);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = x[i] * rinv * wv[i];
  }
  if (p.rope_dim > 0) {
    const int hl = p.rope_dim / 16;  // lanes holding the first half of the rotated dims
    const int partner = (lane < hl) ? lane + hl : lane - hl;
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __shfl_sync(0xffffffffu, x[i], partner & 31);
    if (lane < 2 * hl) {
      float c[8], s[8];
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.cos_t + (size_t)b * p.rope_dim) + lane), c);
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p.sin_t + (size_t)b * p.rope_dim) + lane), s);
      const float sign = (lane < hl) ? -1.0f : 1.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = x[i] * c[i] + sign * (y[i] * s[i]);
    }
  }
  const uint4 outv = pack_bf16x8(x);
  if (is_q) {
    reinterpret_cast<uint4*>(p.q_out + ((size_t)b * p.Hq + r) * kD)[lane] = outv;
  } else if (slot_ok) {
    reinterpret_cast<uint4*>(p.k_pool + ((size_t)slot * p.Hkv + (r - 2 * p.Hq)) * kD)[lane] = outv;
  }
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  const long long warps = (long long)p.B * (2 * p.Hq + 2 * p.Hkv);
  if (warps == 0) return cudaSuccess;
  const long long blocks = (warps + 7) / 8;
  prep_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gda
