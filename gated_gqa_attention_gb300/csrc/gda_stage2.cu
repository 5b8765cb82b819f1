// gda_stage2.cu -- split-KV decode stage 2 (FP32 LSE merge + fused BF16 gate) and
// the standalone gate, on sm_103a.
//
// Stage 2 follows FreeToken PR #781 "Fuse the BF16 attention output sigmoid gate
// into the existing Triton decode stage2" (Summary): the partials of every split
// are merged in FP32 by their log-sum-exp, and the epilogue applies the output
// gate with the BF16 rounding of the unfused Torch path -- O rounded to BF16, the
// sigmoid of the gate rounded to BF16, their product rounded to nearest even --
// so no separate sigmoid or multiply kernel runs.  A zero-length sequence gives
// O = 0 (cuDNN FE-OSS "Gated Attention Block (SM107)": a dead row produces zeros).
// Optional per-head attention sinks join the merged denominator here (FreeToken
// PR #781, Automatic dispatch lists sinks among the cases of the general path).
//
// One CTA per (sequence, query head), 4 warps.  The prologue -- loading the gate
// and computing its BF16 sigmoid -- runs before griddepcontrol.wait, overlapping
// the tail of stage 1 under programmatic dependent launch.  Warp w merges
// partials w, w+4, ... online (lane = 8 dims, two 16-byte loads per partial),
// up to four partials' loads in flight at a time; the four warp states are
// then combined through shared memory.
#include "gda_device.cuh"
#include "gda_kernels.h"

namespace gda {

constexpr int kS2Warps = 4;

// kBatch: partials whose loads a warp has in flight at a time (1 or 4; 4 takes 80
// registers a thread against 46, so the host picks it only when the grid fits one wave
// at that size and there are several partials per warp).
template <int kBatch>
__global__ void __launch_bounds__(kS2Warps * 32) stage2_kernel(Stage2Params p) {
  __shared__ float s_acc[kS2Warps][kD];
  __shared__ float s_m[kS2Warps];
  __shared__ float s_w[kS2Warps];

  const int bh = blockIdx.x;
  const int b = bh / p.Hq, h = bh % p.Hq;
  // query head h belongs to KV head h / G; its slot g in group `pass` (groups of 8).
  // Stage 1 scheduled pieces per (KV head, team of `team` groups) kvh * nteam +
  // pass / team, with the partial of (piece, group of the team) at piece * team +
  // pass % team (team = 1: per virtual head kvh * npass + pass).
  const int kvh = h / p.G, r = h - kvh * p.G;
  const int pass = r / kG, g = r % kG;
  const int sched_h = kvh * p.nteam + pass / p.team;
  const int sched_n = p.Hkv * p.nteam;
  const int id_mul = p.team, id_add = pass % p.team;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the next call's one-kernel decode (a programmatic dependent) may launch and set up
  // now; it waits for this grid before it reads anything
  pdl_launch_dependents();

  // prologue: this thread's two gate values and their BF16 sigmoids
  const size_t row = (size_t)bh * kD;
  uint32_t sig2 = 0;
  if (p.fuse_gate) {
    const uint32_t g2 = __ldg(reinterpret_cast<const uint32_t*>(p.gate + row) + tid);
    sig2 = (uint32_t)sigmoid_bf16((uint16_t)(g2 & 0xFFFFu)) |
           ((uint32_t)sigmoid_bf16((uint16_t)(g2 >> 16)) << 16);
  }

  // which partials hold this segment: from kv_indptr, an input, so before the wait
  long long first;
  int n;
  segment_pieces(p.indptr, b, sched_h, sched_n, p.B, p.num_splits, p.grid1, p.min_chunk, p.window, p.piece_cost, p.rule_kv8,
                 &first, &n);
  // attention sink (a logit in the softmax denominator with no value row), log2 units
  const float sink2 = (p.sinks != nullptr) ? __ldg(p.sinks + h) * 1.44269504088896340736f : -INFINITY;

  pdl_wait_prior_grid();

  float M = -INFINITY, W = 0.0f;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // Warp w merges partials w, w + 4, w + 8, ... in that order, online.  The LSE and O
  // rows of kBatch of them are requested before any is merged, so a warp waits for
  // one round trip per kBatch partials instead of one per partial (the same order,
  // so the same bits, for either kBatch).
  for (int k0 = warp; k0 < n; k0 += kBatch * kS2Warps) {
    float lse[kBatch];
    float4 x0[kBatch], x1[kBatch];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      const int k = k0 + t * kS2Warps;
      lse[t] = -INFINITY;
      if (k < n) {
        const long long id = (first + k) * id_mul + id_add;
        lse[t] = __ldcg(p.lse_part + id * kG + g);
        const float4* src = reinterpret_cast<const float4*>(p.o_part + (id * kG + g) * kD + lane * 8);
        x0[t] = __ldcg(src);
        x1[t] = __ldcg(src + 1);
      }
    }
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      if (lse[t] == -INFINITY) continue;
      const float Mn = fmaxf(M, lse[t]);
      const float fo = (M == -INFINITY) ? 0.0f : exp2f(M - Mn);
      const float fn = exp2f(lse[t] - Mn);
      const float xv[8] = {x0[t].x, x0[t].y, x0[t].z, x0[t].w, x1[t].x, x1[t].y, x1[t].z, x1[t].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = acc[i] * fo + xv[i] * fn;
      W = W * fo + fn;
      M = Mn;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) s_acc[warp][lane * 8 + i] = acc[i];
  if (lane == 0) {
    s_m[warp] = M;
    s_w[warp] = W;
  }
  __syncthreads();

  float Mt = sink2;
#pragma unroll
  for (int x = 0; x < kS2Warps; ++x) Mt = fmaxf(Mt, s_m[x]);
  float o0 = 0.0f, o1 = 0.0f, Wt = 0.0f;
  if (Mt != -INFINITY) {
#pragma unroll
    for (int x = 0; x < kS2Warps; ++x) {
      const float f = (s_m[x] == -INFINITY) ? 0.0f : exp2f(s_m[x] - Mt);
      o0 += s_acc[x][2 * tid] * f;
      o1 += s_acc[x][2 * tid + 1] * f;
      Wt += s_w[x] * f;
    }
    if (sink2 != -INFINITY) Wt += exp2f(sink2 - Mt);
    o0 /= Wt;
    o1 /= Wt;
  }
  const uint16_t ob0 = float_to_bf16_bits(o0), ob1 = float_to_bf16_bits(o1);
  uint32_t res;
  if (p.fuse_gate) {
    res = (uint32_t)gate_product_bf16(ob0, (uint16_t)(sig2 & 0xFFFFu)) |
          ((uint32_t)gate_product_bf16(ob1, (uint16_t)(sig2 >> 16)) << 16);
  } else {
    res = (uint32_t)ob0 | ((uint32_t)ob1 << 16);
  }
  reinterpret_cast<uint32_t*>(p.out + row)[tid] = res;
  if (p.lse_out != nullptr && tid == 0) {
    // log2 units -> natural log
    p.lse_out[bh] = (Mt == -INFINITY) ? -INFINITY : (Mt + log2f(Wt)) * 0.69314718055994530942f;
  }
}

cudaError_t launch_stage2(const Stage2Params& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.Hq));
  cfg.blockDim = dim3(kS2Warps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.batched ? cudaLaunchKernelEx(&cfg, stage2_kernel<4>, p) : cudaLaunchKernelEx(&cfg, stage2_kernel<1>, p);
}

// ------------------------------------------------------------------ standalone gate
//
// out[i] = RNE_bf16(o[i] * RNE_bf16(sigmoid(gate[i]))), eight elements (16 bytes)
// per thread, grid-stride; the last n % 8 elements one by one.

__global__ void gate_kernel(const uint4* __restrict__ o, const uint4* __restrict__ gt, uint4* __restrict__ out,
                            long long nvec, const uint16_t* __restrict__ o_s, const uint16_t* __restrict__ g_s,
                            uint16_t* __restrict__ out_s, long long n) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    const uint4 a = o[i], c = gt[i];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
    uint32_t r[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint16_t lo = gate_product_bf16((uint16_t)(av[j] & 0xFFFFu), sigmoid_bf16((uint16_t)(cv[j] & 0xFFFFu)));
      const uint16_t hi = gate_product_bf16((uint16_t)(av[j] >> 16), sigmoid_bf16((uint16_t)(cv[j] >> 16)));
      r[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    out[i] = make_uint4(r[0], r[1], r[2], r[3]);
  }
  const long long tail0 = nvec * 8;
  const long long t = tail0 + (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n && t < tail0 + 8) out_s[t] = gate_product_bf16(o_s[t], sigmoid_bf16(g_s[t]));
}

cudaError_t launch_gate(const __nv_bfloat16* o, const __nv_bfloat16* gate, __nv_bfloat16* out, long long n,
                        cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long nvec = n / 8;
  const int threads = 256;
  long long blocks = (nvec + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  gate_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      reinterpret_cast<const uint4*>(o), reinterpret_cast<const uint4*>(gate), reinterpret_cast<uint4*>(out), nvec,
      reinterpret_cast<const uint16_t*>(o), reinterpret_cast<const uint16_t*>(gate), reinterpret_cast<uint16_t*>(out),
      n);
  return cudaGetLastError();
}

}  // namespace gda
