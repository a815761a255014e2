// Standalone cache-append kernel (see append.cu).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pagedattn {

struct AppendParams {
  const __nv_bfloat16* k_new;   // [num_seqs, H_kv, D]
  const __nv_bfloat16* v_new;   // [num_seqs, H_kv, D]
  __nv_bfloat16* k_cache;       // [num_blocks, H_kv, BS, D]
  __nv_bfloat16* v_cache;
  const int32_t* block_tables;  // [num_seqs, maxb]
  const int32_t* seq_lens;      // [num_seqs]
  int num_seqs, H_kv, D, maxb, BS;
  long long num_blocks;         // > 0: skip rows whose block id is outside the pool
};

cudaError_t launch_append(const AppendParams& a, int sms, cudaStream_t stream);

}  // namespace pagedattn
