// gda_prefill.h -- launch interface between the C ABI (gda_api.cu) and the prefill kernel.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gda {

struct PrefillParams {
  __nv_bfloat16* out;          // [B, Sq, Hq, D]
  float* lse;                  // [B, Hq, Sq] natural log, or nullptr
  const __nv_bfloat16* gate;   // [B, Sq, Hq, D] (read directly only for rows with no visible key)
  const int* kv_lens;          // [B] or nullptr (all Skv)
  unsigned int* error;         // device error word (kErr* bits)
  int B, Sq, Skv, Hq, Hkv;
  float scale_log2;            // scale * log2(e)
  int causal;
  int fuse_gate;
  long long wait_limit;        // SM cycles after which a pipeline wait gives up (kWaitLimitCycles;
                               // shorter only in the failure-path test)
};

// Prefill / extend gated SDPA (tcgen05); q, k, v, gate are [B, S, H, 256] BF16.
cudaError_t launch_prefill(const PrefillParams& p, const void* q, const void* k, const void* v, const void* gate,
                           cudaStream_t stream);

}  // namespace gda
