// Decode kernel instantiations over FP8 caches for head_dim = 128 (block sizes 16
// and 32, G <= 8 and G <= 16).
#include "launch.h"

namespace pagedattn {

cudaError_t launch_decode_fp8_d128(int block_size, bool g16, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const DecodeParams& p, int grid,
                                   size_t smem, cudaStream_t stream) {
  return launch_for_dim<128, kKvFp8>(block_size, g16, tk, tv, p, grid, smem, stream);
}

}  // namespace pagedattn
