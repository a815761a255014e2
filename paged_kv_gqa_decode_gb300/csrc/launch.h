// Internal interface between the C-ABI layer and the per-head-dim kernel
// translation units (each instantiates the decode kernel for one head_dim).
#pragma once

#include <atomic>
#include <cstddef>

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_kernel.cuh"

namespace pagedattn {

// Launches the decode kernel for head_dim D (64, 128 or 256) with the given
// block size (16 or 32) and query-group class (g16: G > 8).
cudaError_t launch_decode_d64(int block_size, bool g16, const CUtensorMap& tk,
                              const CUtensorMap& tv, const DecodeParams& p, int grid,
                              size_t smem, cudaStream_t stream);
cudaError_t launch_decode_d128(int block_size, bool g16, const CUtensorMap& tk,
                               const CUtensorMap& tv, const DecodeParams& p, int grid,
                               size_t smem, cudaStream_t stream);
cudaError_t launch_decode_d256(int block_size, bool g16, const CUtensorMap& tk,
                               const CUtensorMap& tv, const DecodeParams& p, int grid,
                               size_t smem, cudaStream_t stream);
// The same over x-packed K / D-major V caches (bf16).
cudaError_t launch_decode_xp_d64(int block_size, bool g16, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const DecodeParams& p, int grid,
                                 size_t smem, cudaStream_t stream);
cudaError_t launch_decode_xp_d128(int block_size, bool g16, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const DecodeParams& p, int grid,
                                  size_t smem, cudaStream_t stream);
cudaError_t launch_decode_xp_d256(int block_size, bool g16, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const DecodeParams& p, int grid,
                                  size_t smem, cudaStream_t stream);
// Multi-token decode over bf16 caches.
cudaError_t launch_decode_multi_d64(int block_size, bool g16, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const DecodeParams& p, int grid,
                                    size_t smem, cudaStream_t stream);
cudaError_t launch_decode_multi_d128(int block_size, bool g16, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const DecodeParams& p, int grid,
                                     size_t smem, cudaStream_t stream);
cudaError_t launch_decode_multi_d256(int block_size, bool g16, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const DecodeParams& p, int grid,
                                     size_t smem, cudaStream_t stream);
// The same over FP8 caches (head_dim 128 or 256).
cudaError_t launch_decode_fp8_d128(int block_size, bool g16, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const DecodeParams& p, int grid,
                                   size_t smem, cudaStream_t stream);
cudaError_t launch_decode_fp8_d256(int block_size, bool g16, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const DecodeParams& p, int grid,
                                   size_t smem, cudaStream_t stream);

// Launches one instantiation, first raising its dynamic shared-memory limit on
// the current device when this launch needs more than was set before (the
// record is per instantiation and per device).
template <int D, int BS, bool G16, int KV, bool MULTI = false>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                       int grid, size_t smem, cudaStream_t stream) {
  // The first launch of this instantiation on a device raises its dynamic
  // shared-memory limit to all the device allows next to its static shared
  // memory; host threads may race here, and every racer sets the same value.
  static std::atomic<bool> limit_raised[64];
  auto kernel = paged_decode_kernel<D, BS, G16, KV, MULTI>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !limit_raised[dev].load(std::memory_order_acquire)) {
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) limit_raised[dev].store(true, std::memory_order_release);
  }
  // Programmatic stream serialization: this launch may begin while the previous
  // kernel in the stream finishes; the kernel waits for it (griddepcontrol.wait)
  // before reading any input, so results are those of plain stream order.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tk, tv, p);
}

template <int D, int KV = kKvBf16, bool MULTI = false>
cudaError_t launch_for_dim(int block_size, bool g16, const CUtensorMap& tk, const CUtensorMap& tv,
                           const DecodeParams& p, int grid, size_t smem, cudaStream_t stream) {
  if (block_size == 16)
    return g16 ? launch_one<D, 16, true, KV, MULTI>(tk, tv, p, grid, smem, stream)
               : launch_one<D, 16, false, KV, MULTI>(tk, tv, p, grid, smem, stream);
  return g16 ? launch_one<D, 32, true, KV, MULTI>(tk, tv, p, grid, smem, stream)
             : launch_one<D, 32, false, KV, MULTI>(tk, tv, p, grid, smem, stream);
}

}  // namespace pagedattn
