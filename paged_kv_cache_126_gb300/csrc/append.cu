// Cache append (scatter of new K/V rows into their slots) and whole-frame copies
// for copy-on-write.
//
// "Solving the LLM Memory Wall" ("Implementation", PagedKVCache.update): a token's
// k and v rows are written at [frame, offset]; batched here over all new tokens
// of a step through a slot mapping (slot = frame * B + offset).
// "PagedAttention: Virtual Memory Guide for LLM Inference" ("2. Zero-Copy
// Branching via Copy-on-Write"): only the single shared frame being written is
// duplicated.
//
// Both are pure data movement: 16-byte vector loads and stores, one thread block
// per token row (append) or per slice of a frame (copy), 64-bit byte offsets.  An
// append is a few KB per row, so its time is latency: every thread issues all of
// its loads (K and V, up to kVecs each) before its first store, one DRAM round trip
// per row instead of one per vector.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kVecs = 4;  // 16-byte vectors per thread and cache held before storing

// Uncached loads from mapped host memory (the host rewrites it between launches).
__device__ __forceinline__ int32_t ld_host(const int32_t* p) {
  int32_t v;
  asm volatile("ld.global.cv.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_host(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cv.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p)
               : "memory");
  return v;
}

__global__ void __launch_bounds__(256) cache_append_kernel(const AppendArgs a) {
  // Launched with programmatic stream serialisation: let the next kernel start its
  // set-up now, and wait for the previous kernel's writes before reading inputs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The staging copy reads host memory the host wrote before this launch and writes a
  // buffer no running kernel reads (the caller's contract): it overlaps the wait.
  if (a.stage_vecs > 0) {
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < a.stage_vecs; i += step)
      a.stage_dst[i] = ld_host(a.stage_src + i);
  }
  // Slots in host memory were written before this launch: the block's first one is read
  // before the wait too, so its host round trip overlaps the previous kernel's tail.
  const int32_t first_slot = a.slots_host && blockIdx.x < a.T ? ld_host(a.slots + blockIdx.x) : 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t nvec = a.row_bytes >> 4;
  const int64_t stride = static_cast<int64_t>(blockDim.x);
  for (int t = blockIdx.x; t < a.T; t += gridDim.x) {
    const int32_t slot = a.slots_host ? (t == static_cast<int>(blockIdx.x) ? first_slot : ld_host(a.slots + t))
                                      : __ldg(a.slots + t);
    if (slot < 0) continue;  // padding
    if (slot >= a.num_slots) {
      if (threadIdx.x == 0) atomicOr(a.status, kDevBadSlot);
      continue;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(a.k_new + static_cast<int64_t>(t) * a.k_pitch);
    const uint4* vs = reinterpret_cast<const uint4*>(a.v_new + static_cast<int64_t>(t) * a.v_pitch);
    uint4* kd = reinterpret_cast<uint4*>(a.k_cache + static_cast<int64_t>(slot) * a.row_bytes);
    uint4* vd = reinterpret_cast<uint4*>(a.v_cache + static_cast<int64_t>(slot) * a.row_bytes);
    for (int64_t base = threadIdx.x; base < nvec; base += kVecs * stride) {
      uint4 kr[kVecs], vr[kVecs];
#pragma unroll
      for (int u = 0; u < kVecs; ++u) {
        const int64_t i = base + u * stride;
        if (i < nvec) {
          kr[u] = __ldg(ks + i);
          vr[u] = __ldg(vs + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kVecs; ++u) {
        const int64_t i = base + u * stride;
        if (i < nvec) {
          kd[i] = kr[u];
          vd[i] = vr[u];
        }
      }
    }
  }
}

// grid.x = pair, grid.y = slice of the frame, grid.z = 0 (K) / 1 (V)
__global__ void __launch_bounds__(256) copy_blocks_kernel(const CopyArgs a, const int64_t slice_vecs) {
  const int pair = blockIdx.x;
  const int32_t src = __ldg(a.pairs + 2 * pair);
  const int32_t dst = __ldg(a.pairs + 2 * pair + 1);
  if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(a.status, kDevBadCopy);
    return;
  }
  unsigned char* base = blockIdx.z == 0 ? a.k_cache : a.v_cache;
  const uint4* s = reinterpret_cast<const uint4*>(base + static_cast<int64_t>(src) * a.frame_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + static_cast<int64_t>(dst) * a.frame_bytes);
  const int64_t nvec = a.frame_bytes >> 4;
  const int64_t lo = static_cast<int64_t>(blockIdx.y) * slice_vecs;
  const int64_t hi = lo + slice_vecs < nvec ? lo + slice_vecs : nvec;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) d[i] = s[i];
}

// The decode step's frame copies: pairs in the parameters, launched with programmatic
// stream serialisation.  The next kernel (the step's append) may start now; its row
// writes still wait for this kernel to finish, so a copy lands before any row is
// written into its destination frame.
__global__ void __launch_bounds__(256) copy_blocks_inline_kernel(const __grid_constant__ InlineCopyArgs a,
                                                                 const int64_t slice_vecs) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int pair = blockIdx.x;
  const int32_t src = a.pairs[2 * pair];
  const int32_t dst = a.pairs[2 * pair + 1];
  if (src < 0 || src >= a.num_blocks || dst < 0 || dst >= a.num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(a.status, kDevBadCopy);
    return;
  }
  unsigned char* base = blockIdx.z == 0 ? a.k_cache : a.v_cache;
  const uint4* s = reinterpret_cast<const uint4*>(base + static_cast<int64_t>(src) * a.frame_bytes);
  uint4* d = reinterpret_cast<uint4*>(base + static_cast<int64_t>(dst) * a.frame_bytes);
  const int64_t nvec = a.frame_bytes >> 4;
  const int64_t lo = static_cast<int64_t>(blockIdx.y) * slice_vecs;
  const int64_t hi = lo + slice_vecs < nvec ? lo + slice_vecs : nvec;
  for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) d[i] = s[i];
}

}  // namespace

cudaError_t launch_copy_blocks_inline(const InlineCopyArgs& a, cudaStream_t stream) {
  if (a.n <= 0 || a.n > kInlineCopies) return a.n == 0 ? cudaSuccess : cudaErrorInvalidValue;
  const int64_t nvec = a.frame_bytes >> 4;
  const int64_t slice_vecs = 1024;  // 16 KiB per thread block
  const int64_t slices = (nvec + slice_vecs - 1) / slice_vecs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n, static_cast<unsigned>(slices), 2);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_blocks_inline_kernel, a, slice_vecs);
}

cudaError_t launch_cache_append(const AppendArgs& a, int num_sms, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int64_t nvec = a.row_bytes >> 4;
  const int threads = nvec >= 256 ? 256 : static_cast<int>(((nvec + 31) / 32) * 32);
  const int max_grid = num_sms * 16;
  const int grid = a.T < max_grid ? a.T : max_grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cache_append_kernel, a);
}

cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  const int64_t nvec = a.frame_bytes >> 4;
  const int64_t slice_vecs = 1024;  // 16 KiB per thread block
  const int64_t slices = (nvec + slice_vecs - 1) / slice_vecs;
  dim3 grid(a.n, static_cast<unsigned>(slices), 2);
  copy_blocks_kernel<<<grid, 256, 0, stream>>>(a, slice_vecs);
  return cudaGetLastError();
}

}  // namespace pa
