// Cache append ("reshape and cache"): the write that must precede the decode,
// since the paged-decode layout counts the new tokens in seq_lens ("Add Cuda
// Kernel" tutorial, include/kernels/attention.cuh, "Paged Attention - Decode").
//
// One new token per sequence: for every sequence s with L = seq_lens[s] >= 1
// and every KV head g, the token t = L - 1 goes to
//
//     k_cache[block_tables[s, t / BS], g, t % BS, :] = k_new[s, g, :]   (v alike).
//
// Several per sequence (multi-token decode, rows through qo_indptr as on
// AstrAI's CUDA Kernels page, "Q Scheduling and KV Addressing"): row r =
// qo_indptr[s] + i of k_new / v_new is token t = L - q_len + i of sequence s
// (its last q_len tokens, q_len = qo_indptr[s+1] - qo_indptr[s]).
//
// FP8 caches (nvfp4-megamoe README, "FP8 KV Quantize/Dequant" and "Paged KV
// cache read/write"): each new row x is stored as e4m3 bytes
// e4m3_rn_satfinite(x[d] / f) with its dequant float f = max_d |x[d]| / 448
// (1 for an all-zero row), so that x[d] ~ e4m3(byte) * f.
//
// The traffic is a few bytes per (token, KV head), far below the decode's, so
// the kernels are only sized to fill the machine.
#include <cstdint>

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "append.h"

namespace pagedattn {
namespace {

constexpr float kE4m3Max = 448.f;

// Sequence owning row r (largest s with qo[s] <= r), or -1 when r is outside
// every sequence's rows.
__device__ int sequence_of_row(const int32_t* qo, int N, int r) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qo + mid) <= r)
      lo = mid;
    else
      hi = mid - 1;
  }
  return r >= __ldg(qo + lo) && r < __ldg(qo + lo + 1) ? lo : -1;
}

// Cache row (block * H_kv + g) * BS + slot that row r of the new tokens goes
// to for KV head g, or -1 when it is not written.
__device__ long long target_row(const AppendParams& a, int r, int g) {
  int s = r, ql = 1, i = 0;
  if (a.qo_indptr != nullptr) {
    s = sequence_of_row(a.qo_indptr, a.num_seqs, r);
    if (s < 0) return -1;
    const int q0 = __ldg(a.qo_indptr + s);
    ql = __ldg(a.qo_indptr + s + 1) - q0;
    i = r - q0;
  }
  const int L = __ldg(a.seq_lens + s);
  if (L < 1 || (long long)L > (long long)a.maxb * a.BS) return -1;  // no token / bad length
  const int t = L - ql + i;
  if (t < 0) return -1;  // more new rows than the sequence holds
  const int b = __ldg(a.block_tables + (size_t)s * a.maxb + t / a.BS);
  if (a.num_blocks > 0 && (b < 0 || (long long)b >= a.num_blocks)) {
    if (a.status != nullptr) atomicOr(a.status, 1);  // bad block id: nothing written
    return -1;
  }
  return ((long long)b * a.H_kv + g) * a.BS + t % a.BS;
}

// bf16: one thread moves one 16-byte chunk (8 values) of one K or V row.
__global__ void __launch_bounds__(256) paged_kv_append_kernel(const AppendParams a) {
  const int chunks_per_row = a.D / 8;
  const long long per_row = 2LL * a.H_kv * chunks_per_row;
  const int rows = a.qo_indptr != nullptr ? a.total_q : a.num_seqs;
  const long long total = (long long)rows * per_row;
  for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total;
       c += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(c / per_row);
    const int rem = (int)(c - (long long)r * per_row);
    const int kv = rem / (a.H_kv * chunks_per_row);  // 0: K, 1: V
    const int rr = rem - kv * a.H_kv * chunks_per_row;
    const int g = rr / chunks_per_row;
    const int ch = rr - g * chunks_per_row;
    const long long row = target_row(a, r, g);
    if (row < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(
                           (kv ? a.v_new : a.k_new) + ((size_t)r * a.H_kv + g) * a.D) + ch;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(kv ? a.v_cache : a.k_cache) +
                                          (size_t)row * a.D) + ch;
    *dst = __ldg(src);
  }
}

// FP8: one warp quantizes one new K or V row of D = 32 * E values.
template <int E>
__global__ void __launch_bounds__(256) paged_kv_append_fp8_kernel(const AppendParams a) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x / 32);
  const int rows = a.qo_indptr != nullptr ? a.total_q : a.num_seqs;
  const long long total = (long long)rows * a.H_kv * 2;
  for (long long w = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); w < total;
       w += warps) {
    const int r = (int)(w / (2 * a.H_kv));
    const int rem = (int)(w - (long long)r * 2 * a.H_kv);
    const int kv = rem / a.H_kv;
    const int g = rem - kv * a.H_kv;
    const long long row = target_row(a, r, g);  // uniform across the warp
    if (row < 0) continue;
    const __nv_bfloat16* src = (kv ? a.v_new : a.k_new) + ((size_t)r * a.H_kv + g) * a.D + lane * E;
    float x[E];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      x[e] = __bfloat162float(src[e]);
      amax = fmaxf(amax, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float f = amax > 0.f ? amax / kE4m3Max : 1.f;  // IEEE division (no fast math)
    uint8_t* dst = static_cast<uint8_t*>(kv ? a.v_cache : a.k_cache) + (size_t)row * a.D + lane * E;
    uint8_t b[E];
#pragma unroll
    for (int e = 0; e < E; ++e) b[e] = __nv_cvt_float_to_fp8(x[e] / f, __NV_SATFINITE, __NV_E4M3);
    uint32_t w4[E / 4];  // little-endian: value e in byte e
#pragma unroll
    for (int k = 0; k < E / 4; ++k)
      w4[k] = (uint32_t)b[4 * k] | ((uint32_t)b[4 * k + 1] << 8) | ((uint32_t)b[4 * k + 2] << 16) |
              ((uint32_t)b[4 * k + 3] << 24);
    if constexpr (E == 4)
      *reinterpret_cast<uint32_t*>(dst) = w4[0];
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(w4[0], w4[1]);
    if (lane == 0) (kv ? a.v_scale : a.k_scale)[row] = f;
  }
}

int grid_for(long long work_items, int per_block, int sms) {
  const long long want = (work_items + per_block - 1) / per_block;
  return (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
}

}  // namespace

cudaError_t launch_append(const AppendParams& a, int sms, cudaStream_t stream) {
  const int rows = a.qo_indptr != nullptr ? a.total_q : a.num_seqs;
  const long long total = (long long)rows * 2 * a.H_kv * (a.D / 8);
  if (total == 0) return cudaSuccess;
  paged_kv_append_kernel<<<grid_for(total, 256, sms), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append_fp8(const AppendParams& a, int sms, cudaStream_t stream) {
  const int rows = a.qo_indptr != nullptr ? a.total_q : a.num_seqs;
  const long long warps = (long long)rows * a.H_kv * 2;
  if (warps == 0) return cudaSuccess;
  const int grid = grid_for(warps, 8, sms);
  if (a.D == 128)
    paged_kv_append_fp8_kernel<4><<<grid, 256, 0, stream>>>(a);
  else if (a.D == 256)
    paged_kv_append_fp8_kernel<8><<<grid, 256, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pagedattn
