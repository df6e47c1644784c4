// Internal declarations shared by the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

namespace pa {

// Launch preparation of a kernel with dynamic shared memory, cached per (device,
// kernel, threads, bytes): raises the kernel's dynamic shared-memory limit to the
// largest size asked for so far and returns the resident blocks per SM.  Both CUDA
// calls cost microseconds of host time, which a decode step of tens of microseconds
// cannot afford on every launch.
inline cudaError_t kernel_prep(const void* fn, int threads, size_t smem, int* blocks_per_sm) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> occ;
  static std::map<std::pair<int, const void*>, size_t> limit;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  try {  // the caches allocate; no C++ exception crosses the C ABI
    const auto key = std::make_tuple(dev, fn, threads, smem);
    auto it = occ.find(key);
    if (it != occ.end()) {
      if (blocks_per_sm) *blocks_per_sm = it->second;
      return cudaSuccess;
    }
    size_t& lim = limit[{dev, fn}];
    if (smem > lim) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      lim = smem;
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
    if (e != cudaSuccess) return e;
    occ[key] = n;
    if (blocks_per_sm) *blocks_per_sm = n;
    return cudaSuccess;
  } catch (...) {
    return cudaErrorMemoryAllocation;
  }
}

// ---- cache append / frame copy ---------------------------------------------------------
struct AppendArgs {
  const unsigned char* k_new;   // [T, row_bytes] with row pitch k_pitch
  const unsigned char* v_new;
  int64_t k_pitch, v_pitch;     // bytes between token rows
  const int32_t* slots;         // [T]; device memory, or mapped pinned host memory (slots_host)
  unsigned char* k_cache;       // [num_slots, row_bytes]
  unsigned char* v_cache;
  int64_t row_bytes;            // H * D * elem (multiple of 16)
  int64_t num_slots;            // num_blocks * B
  int32_t T;
  int32_t slots_host;           // 1: slots are read from host memory, uncached
  int32_t* status;
  // Optional staging copy done by the same launch (stage_vecs > 0): stage_vecs 16-byte
  // vectors from mapped pinned host memory to device memory.  It runs before the wait
  // on the previous kernel, so stage_dst must not be read by any kernel that can still
  // be running when this one starts.
  const uint4* stage_src;
  uint4* stage_dst;
  int64_t stage_vecs;
};
cudaError_t launch_cache_append(const AppendArgs& a, int num_sms, cudaStream_t stream);

struct CopyArgs {
  unsigned char* k_cache;
  unsigned char* v_cache;
  const int32_t* pairs;         // [n, 2] in device memory
  int64_t frame_bytes;          // B * H * D * elem (multiple of 16)
  int32_t n;
  int32_t num_blocks;
  int32_t* status;
};
cudaError_t launch_copy_blocks(const CopyArgs& a, cudaStream_t stream);

// The same copies with the pairs passed in the kernel's parameters (no device buffer):
// the decode step's path, for up to kInlineCopies pairs.
constexpr int kInlineCopies = 256;
struct InlineCopyArgs {
  unsigned char* k_cache;
  unsigned char* v_cache;
  int64_t frame_bytes;
  int32_t n;
  int32_t num_blocks;
  int32_t* status;
  int32_t pairs[2 * kInlineCopies];  // (src, dst) frame ids
};
cudaError_t launch_copy_blocks_inline(const InlineCopyArgs& a, cudaStream_t stream);

// ---- decode ------------------------------------------------------------------------------
struct DecodeArgs {
  const void* q;                // [S, H, D], row stride q_row elements
  void* out;                    // [S, H, D], row stride out_row elements
  int64_t q_row, out_row;
  const int32_t* block_tables;  // [S, max_blocks], row stride bt_row
  int64_t bt_row;
  const int32_t* context_lens;  // [S]
  int32_t S, H, B, num_blocks, max_blocks;
  // tokens per staged unit: B, or R = 16 * warps_per_head when B divides R (R/B frames
  // share a stage) or R divides B (a frame is staged as B/R slices)
  int32_t R;
  int32_t G;                    // head groups per sequence = H / heads_per_cta
  float qk_scale_log2;          // scale * log2(e)
  // partitioning: fixed_part > 0 forces that many tokens per partition (multiple of
  // B); otherwise the partition length is chosen on the device from the lengths
  // (whole sequences if whole_first and they balance, else about target_items
  // items, never shorter than min_part).
  int32_t fixed_part;
  int32_t target_items;
  int32_t min_part;
  int32_t whole_first;          // automatic mode: keep whole sequences when they balance
  // workspace
  int32_t* sched;               // [3]: next item, retired blocks, next merge task (zero between launches)
  int32_t* ws_cnt;              // [S * H]: partitions finished per (sequence, head) (zero between launches)
  float* ws_ml;                 // [items][HG][2] = (running max in log2 units, sum); null if no split
  float* ws_o;                  // [items][HG][D] unnormalised partial outputs; null if no split
  int32_t* status;
  // shared-prefix decode only: lcp[s] = leading tokens s reads through the same frames as
  // s - 1 (written by its plan kernel); runs with lcp >= min_shared form chunks; the
  // workspace holds part_cap partial slots of [H][D] (ws_o) and [H][2] (ws_ml)
  int32_t* lcp;
  int32_t min_shared;
  int32_t part_cap;
};

struct DecodeCfg {
  int dtype;         // PA_F32 / PA_F16 / PA_BF16
  int D;
  int heads_per_cta;
  int warps_per_head;
  int stages;
  int grid;          // persistent thread blocks
  bool fast;         // allow the unrolled full-frame path (256-byte rows, B = 16 * warps_per_head)
};

// per-dtype launchers (one translation unit each).  query_only: set the kernel's
// shared-memory attribute and report resident blocks per SM in *max_ctas instead
// of launching.
cudaError_t launch_decode_f32(const DecodeArgs&, const DecodeCfg&, const CUtensorMap&, const CUtensorMap&,
                              cudaStream_t, bool query_only, int* max_ctas);
cudaError_t launch_decode_f16(const DecodeArgs&, const DecodeCfg&, const CUtensorMap&, const CUtensorMap&,
                              cudaStream_t, bool query_only, int* max_ctas);
cudaError_t launch_decode_bf16(const DecodeArgs&, const DecodeCfg&, const CUtensorMap&, const CUtensorMap&,
                               cudaStream_t, bool query_only, int* max_ctas);
// Dynamic shared memory of one decode thread block (mirrors the kernel's layout).
size_t decode_smem_bytes(const DecodeCfg& c, int elem_bytes, int R, int S);  // R: tokens per staged unit

// Shared-prefix decode (16-bit caches, D = 128): the plan kernel, then the decode over
// shared and private parts, which also merges split sequences.  query_only as for the launchers above.
cudaError_t launch_decode_shared(const DecodeArgs&, const DecodeCfg&, const CUtensorMap&, const CUtensorMap&,
                                 cudaStream_t, bool query_only, int* max_ctas);
size_t decode_shared_smem_bytes(const DecodeCfg& c, int R, int S);
bool decode_shared_combo(int heads_per_cta, int warps_per_head);

// ---- chunked prefill (tensor cores) ------------------------------------------------------------
struct PrefillArgs {
  const void* q;                // [T, H, 128], row stride q_row elements
  void* out;                    // [T, H, 128], row stride out_row elements
  int64_t q_row, out_row;
  const int32_t* block_tables;  // [S, max_blocks]
  int64_t bt_row;
  const int32_t* context_lens;  // [S] tokens in the cache, chunk included
  const int32_t* query_start;   // [S + 1] q rows of sequence s: query_start[s] .. query_start[s+1]-1
  int32_t S, H, B, num_blocks, max_blocks, T;
  int32_t unit_cap;             // room for (sequence, tile pair) units in shared memory
  float qk_scale_log2;
  int32_t* sched;               // [2] work counter, retired blocks (zero between launches)
  int32_t* status;
};
cudaError_t launch_prefill_f16(const PrefillArgs&, const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, int grid, cudaStream_t);
cudaError_t launch_prefill_bf16(const PrefillArgs&, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, int grid, cudaStream_t);
size_t prefill_smem_bytes(int S, int unit_cap);

// Decode over the split cache layout (k [nb, H, D/x, B, x], v [nb, H, D, B]).
struct SplitArgs {
  const void* q;                // [S, H, D], row stride q_row elements
  void* out;                    // [S, H, D], row stride out_row elements
  int64_t q_row, out_row;
  const void* k_cache;          // [num_blocks, H, D/x, B, x]
  const void* v_cache;          // [num_blocks, H, D, B]
  const int32_t* block_tables;  // [S, max_blocks]
  int64_t bt_row;
  const int32_t* context_lens;  // [S]
  int32_t S, H, num_blocks, max_blocks;
  int32_t P, NP;                // tokens per partition (multiple of B), partitions per sequence
  int32_t hg;                   // heads per work item and thread block: 4, or 2 when a frame of
                                //    4 heads would make a stage larger than 48 KB
  int32_t longest_first;        // 1: items of whole sequences in decreasing length (order kept in
                                //    shared memory after the kernel's own layout), 0: batch order
  float qk_scale_log2;
  int32_t* sched;               // [2] work counter, retired blocks (zero between launches)
  float* ws_ml;                 // [S * H/hg * NP][hg][2] partial (max, sum) when NP > 1
  float* ws_o;                  // [S * H/hg * NP][hg][D] partial unnormalised outputs
  int32_t* status;
};
cudaError_t launch_decode_split(int dtype, int D, int B, const SplitArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_append_split(int dtype, const void* k_new, const void* v_new, int64_t k_row, int64_t v_row,
                                const int32_t* slots, int32_t T, int32_t H, int32_t D, int32_t B,
                                int32_t num_blocks, void* k_cache, void* v_cache, int32_t* status,
                                int grid, cudaStream_t stream);

// status bits (mirror pa.h)
constexpr int32_t kDevBadSlot = 0x1;
constexpr int32_t kDevBadBlock = 0x2;
constexpr int32_t kDevBadLen = 0x4;
constexpr int32_t kDevBadCopy = 0x8;
constexpr int32_t kDevTimeout = 0x10;

}  // namespace pa
