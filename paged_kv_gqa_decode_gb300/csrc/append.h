// Standalone cache-append kernels (see append.cu).
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace pagedattn {

struct AppendParams {
  const __nv_bfloat16* k_new;   // [rows, H_kv, D]: one row per sequence, or total_q rows
  const __nv_bfloat16* v_new;
  void* k_cache;                // [num_blocks, H_kv, BS, D]: bf16, or e4m3 bytes (fp8)
  void* v_cache;
  float* k_scale;               // fp8: [num_blocks, H_kv, BS] dequant floats; else null
  float* v_scale;
  const int32_t* block_tables;  // [num_seqs, maxb]
  const int32_t* seq_lens;      // [num_seqs]
  const int32_t* qo_indptr;     // [num_seqs + 1]: rows of each sequence; null: one each
  int num_seqs, total_q, H_kv, D, maxb, BS;
  long long num_blocks;         // > 0: rows whose block id is outside the pool are skipped
  int32_t* status;              // with num_blocks > 0: bit 0 set for such a row
};

// bf16 caches; one new token per sequence, or qo_indptr's rows.
cudaError_t launch_append(const AppendParams& a, int sms, cudaStream_t stream);
// FP8 caches: each new row is quantized to e4m3 with its own dequant float.
cudaError_t launch_append_fp8(const AppendParams& a, int sms, cudaStream_t stream);

}  // namespace pagedattn
