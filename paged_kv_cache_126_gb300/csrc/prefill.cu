// Chunked-prefill kernels (fp16 and bf16 caches).
#include <type_traits>

#include "prefill_kernel.cuh"

namespace pa {

cudaError_t launch_prefill_f16(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, int grid, cudaStream_t stream) {
  return pk::launch<__half>(a, tq, tk, tv, grid, stream);
}

cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t stream) {
  return pk::launch<__nv_bfloat16>(a, tq, tk, tv, grid, stream);
}

size_t prefill_smem_bytes(int S, int unit_cap) { return pk::smem_bytes(S, unit_cap); }

}  // namespace pa
