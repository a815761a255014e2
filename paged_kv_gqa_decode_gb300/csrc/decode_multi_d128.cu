// Multi-token decode kernel instantiations over bf16 caches for head_dim = 128
// (block sizes 16 and 32, pieces of 8 and 16 query rows).
#include "launch.h"

namespace pagedattn {

cudaError_t launch_decode_multi_d128(int block_size, bool g16, const CUtensorMap& tk,
                                     const CUtensorMap& tv, const DecodeParams& p, int grid,
                                     size_t smem, cudaStream_t stream) {
  return launch_for_dim<128, kKvBf16, true>(block_size, g16, tk, tv, p, grid, smem, stream);
}

}  // namespace pagedattn
