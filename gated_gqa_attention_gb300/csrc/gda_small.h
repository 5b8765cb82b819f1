// gda_small.h -- the single-pass small-batch decode kernel's launch interface.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gda {

constexpr int kSmallMaxLen = 1024;  // longest sequence (host bound) the path takes

struct SmallParams {
  const __nv_bfloat16* q;       // [B, Hq, D]
  const __nv_bfloat16* gate;    // [B, Hq, D] (fuse_gate)
  const void* k_pool;           // [num_slots, Hkv, D] bf16, or e4m3 codes (kv_fp8)
  const void* v_pool;           // [num_slots, Hkv, D] likewise
  const int32_t* indptr;        // [B + 1]
  const int32_t* indices;       // [indptr[B]]
  __nv_bfloat16* out;           // [B, Hq, D]
  float* lse_out;               // [B, Hq] natural log, or null
  const float* sinks;           // [Hq] sink logits, or null
  int B, Hq, Hkv, G;            // G = Hq / Hkv <= 8
  float scale_log2;             // scale * log2(e) (times k_descale for e4m3 pools)
  int kv_fp8;                   // the pools hold e4m3 codes
  float v_descale;              // e4m3 pools: V = v_descale * e4m3(code)
  int window;                   // > 0: the last `window` positions only
  int fuse_gate;
};

// grid (C, Hkv, B) in clusters of C = 8, 4, 2 or 1 CTAs, one per (sequence, KV head)
cudaError_t launch_small(const SmallParams& p, int C, cudaStream_t stream);

// How many of the kernel's C-CTA clusters the current device runs at once (one CTA
// per SM and the C SMs of a cluster in one GPC); 0 when the query fails.
int small_max_clusters(int C);

// The cluster size for `pairs` (sequence, KV head) pairs whose lengths are at most
// max_len, or 0 for the split path: the largest C whose clusters all run at once (one
// wave) and give each CTA at most 128 positions (max_len <= 128 C).  Measured on
// GB300 against the split path with its split count chosen on the host: 0.67-0.9x
// its time inside these bounds; with 256 positions per CTA mostly slower.
int small_cluster_for(long long pairs, int max_len);

}  // namespace gda
