// Decode kernels for float caches (one translation unit per element type so the
// build compiles them in parallel).
#include "decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_f32(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream, bool query_only, int* max_ctas) {
  return dk::launch_dtype<float>(a, c, tk, tv, stream, query_only, max_ctas);
}

}  // namespace pa
