// gda_kernels.h -- launch interface between the C ABI (gda_api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gda {

struct WsHeader;

constexpr int kVariantMma = 1;    // register-direct loads, mma.sync tiles (default)
constexpr int kVariantSimt = 2;   // register-direct loads, FP32 FMAs + warp shuffles
constexpr int kVariantTma = 3;    // TMA bulk-copy ring, mma.sync tiles

struct Stage1Params {
  const __nv_bfloat16* q;
  const unsigned char* k_pool;
  const unsigned char* v_pool;
  const int* indptr;
  const int* indices;
  float* o_part;       // [pieces][G][D]
  float* lse_part;     // [pieces][G], log2 units
  WsHeader* hdr;
  long long num_slots;
  int B, Hq, Hkv;
  int G;               // query heads per KV head (Hq / Hkv)
  int npass;           // ceil(G / 8): groups of 8 query heads per KV head ("virtual heads")
  int team;            // groups per piece: 1, or on the MMA kernel with npass >= 2 the groups
                       // go in teams of 2 or 3, one piece per (sequence, KV head, team)
                       // serving every group of the team
  int nteam;           // ceil(npass / team): teams per KV head
  int window;          // > 0: attend to the last `window` positions only
  float scale_log2;    // scale * log2(e) (e4m3 pools: scale * k_descale * log2(e))
  int num_splits;      // > 0 explicit, else automatic
  int min_chunk;       // automatic mode
  int piece_cost;      // automatic stream schedule: cost of a segment start in positions (0: none)
  int rule_kv8;        // automatic rule, e4m3 variant: the per-CTA bound for the stream
                       // schedule doubled, S_opt from 16 S^2 > lmax (BF16: 4 S^2)
  int check_indices;
  float v_descale;     // e4m3 pools: V = v_descale * e4m3(code)
  long long wait_limit;  // SM cycles after which a pipeline wait gives up (kWaitLimitCycles;
                         // shorter only in the failure-path test)
};

struct Stage2Params {
  const __nv_bfloat16* gate;
  const int* indptr;
  const float* o_part;
  const float* lse_part;
  __nv_bfloat16* out;
  float* lse_out;      // [B, Hq] natural log, or nullptr
  const float* sinks;  // [Hq] sink logits (natural units), or nullptr
  int B, Hq, Hkv;
  int G, npass, window;
  int team;            // stage 1's groups per piece: partial (piece, group of the team) is at
                       // piece * team + group
  int nteam;           // ceil(npass / team)
  int num_splits;
  int grid1;           // stage-1 grid (automatic-mode chunking)
  int min_chunk;
  int piece_cost;      // the stage-1 schedule's cost of a segment start
  int rule_kv8;        // the stage-1 rule's e4m3 variant
  int fuse_gate;
  int batched;         // merge with four partials' loads in flight per warp (small grids)
};

struct PrepParams {
  const __nv_bfloat16* qgkv;   // [B, row_stride] rows [q | gate | k | v]
  long long row_stride;        // elements between tokens
  const __nv_bfloat16* w_q;    // [D] or nullptr (no Q norm)
  const __nv_bfloat16* w_k;    // [D] or nullptr (no K norm)
  float eps;
  const __nv_bfloat16* cos_t;  // [B, rope_dim]
  const __nv_bfloat16* sin_t;  // [B, rope_dim]
  int rope_dim;                // 0 or a multiple of 16 up to D
  const int* slots;            // [B]
  long long num_slots;
  __nv_bfloat16* q_out;        // [B, Hq, D]
  __nv_bfloat16* gate_out;     // [B, Hq, D] or nullptr
  __nv_bfloat16* k_pool;       // [num_slots, Hkv, D]
  __nv_bfloat16* v_pool;
  int B, Hq, Hkv;
};

// The step before attention (Q/K RMSNorm, partial RoPE, KV write).
cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);

// Stage 1: grid CTAs, persistent.  Returns the launch status.
cudaError_t launch_stage1(const Stage1Params& p, int variant, int grid, cudaStream_t stream);
// Stage 1 over e4m3 K/V pools (same partials, same schedule).
cudaError_t launch_stage1_fp8(const Stage1Params& p, int grid, cudaStream_t stream);
// Stage 2: FP32 LSE merge + gate epilogue, launched as a programmatic dependent of stage 1.
cudaError_t launch_stage2(const Stage2Params& p, cudaStream_t stream);
// Standalone gate over n elements.
cudaError_t launch_gate(const __nv_bfloat16* o, const __nv_bfloat16* gate, __nv_bfloat16* out, long long n,
                        cudaStream_t stream);

}  // namespace gda
