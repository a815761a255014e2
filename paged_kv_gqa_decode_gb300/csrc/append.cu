// Cache append ("reshape and cache") of one new token per sequence: the write
// that must precede the decode, since the paged-decode layout counts the new
// token in seq_lens ("Add Cuda Kernel" tutorial, include/kernels/attention.cuh,
// "Paged Attention - Decode").  For every sequence s with L = seq_lens[s] >= 1
// and every KV head g, the token t = L - 1 goes to
//
//     k_cache[block_tables[s, t / BS], g, t % BS, :] = k_new[s, g, :]   (v alike)
//
// One thread moves one 16-byte chunk (8 bf16) of one row of K or V.  The
// traffic is 4 * D bytes per (sequence, KV head) read and written, far below
// the decode's, so the kernel is only sized to fill the machine.
#include <cstdint>

#include <cuda_runtime.h>

#include "append.h"

namespace pagedattn {

__global__ void __launch_bounds__(256) paged_kv_append_kernel(const AppendParams a) {
  const int chunks_per_row = a.D / 8;                  // 16-byte chunks of one K or V row
  const long long per_seq = 2LL * a.H_kv * chunks_per_row;
  const long long total = (long long)a.num_seqs * per_seq;
  const int cap = a.maxb * a.BS;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(c / per_seq);
    const int r = (int)(c - (long long)s * per_seq);
    const int kv = r / (a.H_kv * chunks_per_row);      // 0: K, 1: V
    const int rr = r - kv * a.H_kv * chunks_per_row;
    const int g = rr / chunks_per_row;
    const int ch = rr - g * chunks_per_row;
    const int L = __ldg(a.seq_lens + s);
    if (L < 1 || L > cap) continue;  // no new token, or a length the caller got wrong
    const int t = L - 1;
    const int b = __ldg(a.block_tables + (size_t)s * a.maxb + t / a.BS);
    if (a.num_blocks > 0 && (b < 0 || (long long)b >= a.num_blocks)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(
        (kv ? a.v_new : a.k_new) + ((size_t)s * a.H_kv + g) * a.D) + ch;
    uint4* dst = reinterpret_cast<uint4*>(
        (kv ? a.v_cache : a.k_cache) + (((size_t)b * a.H_kv + g) * a.BS + t % a.BS) * a.D) + ch;
    *dst = __ldg(src);
  }
}

cudaError_t launch_append(const AppendParams& a, int sms, cudaStream_t stream) {
  const long long total = (long long)a.num_seqs * 2 * a.H_kv * (a.D / 8);
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int grid = (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
  paged_kv_append_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pagedattn
