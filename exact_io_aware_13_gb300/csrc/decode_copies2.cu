// The decode kernel with two copies of the rows in tensor memory (query groups of at
// most 32 rows), in a translation unit of its own so that it compiles in parallel.
#include "decode_tc.cuh"

namespace attn {
namespace dec {

cudaError_t launch_decode_copies2(const Args& a, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int grid, cudaStream_t st) {
  return launch_decode_copies<2>(a, tk, tv, grid, st);
}

}  // namespace dec
}  // namespace attn
