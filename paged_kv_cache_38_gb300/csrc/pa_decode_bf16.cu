// pa_decode_bf16.cu - decode kernel instantiations for bf16 KV blocks (one translation unit per
// KV dtype so the library builds in parallel).
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t launch_decode_bf16(int head_dim, int group, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const DecodeParams& p, dim3 grid,
                              size_t smem, cudaStream_t stream) {
  return launch_decode_kv<kKvBF16>(head_dim, group, kmap, vmap, p, grid, smem, stream);
}

}  // namespace pa
