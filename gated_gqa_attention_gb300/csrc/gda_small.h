// gda_small.h -- the single-pass small-batch decode kernel's launch interface.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gda {

constexpr int kSmallCluster = 8;    // CTAs per (sequence, KV head): one cluster
constexpr int kSmallMaxLen = 2048;  // longest sequence (host bound) the path takes

struct SmallParams {
  const __nv_bfloat16* q;       // [B, Hq, D]
  const __nv_bfloat16* gate;    // [B, Hq, D] (fuse_gate)
  const __nv_bfloat16* k_pool;  // [num_slots, Hkv, D]
  const __nv_bfloat16* v_pool;  // [num_slots, Hkv, D]
  const int32_t* indptr;        // [B + 1]
  const int32_t* indices;       // [indptr[B]]
  __nv_bfloat16* out;           // [B, Hq, D]
  float* lse_out;               // [B, Hq] natural log, or null
  const float* sinks;           // [Hq] sink logits, or null
  int B, Hq, Hkv, G;            // G = Hq / Hkv <= 8
  float scale_log2;             // scale * log2(e)
  int window;                   // > 0: the last `window` positions only
  int fuse_gate;
};

// grid (kSmallCluster, Hkv, B) in clusters of kSmallCluster CTAs
cudaError_t launch_small(const SmallParams& p, cudaStream_t stream);

// How many of the kernel's clusters the current device runs at once (one CTA per SM
// and 8 SMs of one GPC per cluster: fewer than SMs / 8); 0 when the query fails.
// The path is only worth it when every (sequence, KV head) cluster fits in one wave.
int small_max_clusters();

}  // namespace gda
