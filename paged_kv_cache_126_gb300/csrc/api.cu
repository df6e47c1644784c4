// C ABI of libpa: argument validation, launch configuration, TMA descriptors,
// the library-owned split workspace and the sticky device status word.
// The operations themselves are specified in include/pa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "decode_kernel.cuh"
#include "pa.h"
#include "pa_internal.h"

#include <nvtx3/nvToolsExt.h>

namespace {

// NVTX range around a host entry point (phases show up in Nsight timelines; a push
// and a pop cost nanoseconds when no tool is attached).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};


// Sticky status word, one per device (each device holds its own copy of this
// module's globals).  Kernels in other translation units receive its address.
__device__ int32_t g_pa_status;

constexpr int kMaxDevices = 64;

// Self-test of the bounded wait that every kernel's mbarrier waits go through
// (dk::mbar_wait, budget kWaitCycles): warp 0 waits on an mbarrier that nothing ever
// arrives on, gives up when the budget runs out, raises PA_DEV_TIMEOUT and marks the
// block aborting; warp 1 then waits on the same barrier and must return at once.
// res[0], res[1]: the two waits' results (1 = completed, 0 = gave up); res[2], res[3]:
// the SM cycles each took.
__global__ void __launch_bounds__(64) selftest_wait_kernel(int32_t* status, long long* res) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  const uint32_t b = pa::dk::smem_u32(&bar);
  if (threadIdx.x == 0) {
    pa::dk::mbar_init(b, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t* ab = &abort_flag;
  if (warp == 0) {
    const long long t0 = clock64();
    const bool ok = __all_sync(pa::dk::kFull, pa::dk::mbar_wait(b, 0, ab, status));
    if (lane == 0) {
      res[0] = ok;
      res[2] = clock64() - t0;
    }
  }
  __syncthreads();
  if (warp == 1) {
    const long long t0 = clock64();
    const bool ok = __all_sync(pa::dk::kFull, pa::dk::mbar_wait(b, 0, ab, status));
    if (lane == 0) {
      res[1] = ok;
      res[3] = clock64() - t0;
    }
  }
}

std::atomic<int64_t> g_launches{0};

struct DeviceState {
  std::once_flag once;
  int32_t* status = nullptr;
  int num_sms = 0;
  cudaError_t err = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return PA_ERR_CUDA;
  DeviceState& d = g_dev[*dev];
  std::call_once(d.once, [&] {
    d.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_pa_status);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, *dev);
  });
  return d.err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---- TMA descriptor encoding (driver entry point, resolved once) -------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// 3-D view [num_blocks*B, H, D] of a cache, box {D, hg, box_rows}: box_rows rows (a
// frame, or a slice of one) of hg heads.
int make_cache_map(CUtensorMap* map, void* base, int dtype, int64_t nb, int64_t B, int64_t H, int64_t D, int hg,
                   int64_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  CUtensorMapDataType t = dtype == PA_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                          : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int64_t e = dtype == PA_F32 ? 4 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(nb * B)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * e), static_cast<cuuint64_t>(H * D * e)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(hg), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, t, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// 3-D view [rows, H, D] of a 16-bit tensor whose rows are `row_elems` apart, box {64, 1, box_rows},
// 128-byte swizzle (the layout tcgen05 reads as K-major or MN-major operands).
int make_sw128_map(CUtensorMap* map, void* base, int dtype, int64_t rows, int64_t H, int64_t D, int64_t row_elems,
                   int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  CUtensorMapDataType t = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(row_elems * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, t, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// A whole cache frame of one head in one copy, laid out in shared memory as
// [B/8 groups][2 column halves][8 rows][64 elements] with the 128-byte swizzle: the
// 5-D view splits the row index into (row mod 8, row / 8) and the head dimension
// into two 64-element halves, ordered so that the box lands half-major inside each
// 8-row group.  rows must be a multiple of 8; every coordinate of the view stays
// inside the cache, so the last frame's box never leaves the allocation.
int make_frame_map(CUtensorMap* map, void* base, int dtype, int64_t rows, int64_t H, int64_t D, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  if (rows % 8 != 0 || box_rows % 8 != 0 || D != 128) return PA_ERR_UNSUPPORTED;
  CUtensorMapDataType t = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(H * D * 2);
  cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(rows / 8), static_cast<cuuint64_t>(H)};
  cuuint64_t strides[4] = {row_bytes, 128, 8 * row_bytes, static_cast<cuuint64_t>(D * 2)};
  cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(box_rows / 8), 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(map, t, 5, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// 4-D view {64 elements, rows, 2 column halves, H} of a 16-bit cache with D = 128, box
// {64, box_rows, 2, hg}, 128-byte swizzle: a box lands in shared memory as
// [hg][2][box_rows][64] with every 128-byte line swizzled (the layout ldmatrix reads
// without bank conflicts).
int make_half_rows_map(CUtensorMap* map, void* base, int dtype, int64_t rows, int64_t H, int hg, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_CUDA;
  CUtensorMapDataType t = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), 2, static_cast<cuuint64_t>(H)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(H * 256), 128, 256};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 2, static_cast<cuuint32_t>(hg)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, t, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// ---- library-owned workspace, one per (device, stream) -------------------------------------
// Layout: [0, 256) scheduler counters | arrival counters, one per (sequence, head) |
// per-launch offsets and split partials.  Both counter regions must hold zeros
// when a launch starts; every decode launch leaves them zero.  They are zeroed when
// first allocated and whenever the arrival-counter region grows.
constexpr size_t kSchedBytes = 256;

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  size_t cnt_bytes = 0;  // arrival-counter region known to hold zeros
};
std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Returns the workspace base and the size of its arrival-counter region (>= cnt_need).
int workspace(int dev, cudaStream_t stream, size_t cnt_need, size_t rest_bytes, void** out, size_t* cnt_bytes) {
  std::lock_guard<std::mutex> lk(g_ws_mu);
  Workspace* wp = nullptr;
  try {  // no C++ exception crosses the C ABI
    wp = &g_ws[{dev, stream}];
  } catch (...) {
    return PA_ERR_HOST_MEMORY;
  }
  Workspace& w = *wp;
  const size_t cnt = std::max(round256(cnt_need), w.cnt_bytes);
  const size_t bytes = kSchedBytes + cnt + rest_bytes;
  if (w.bytes < bytes) {
    if (w.ptr) {
      // the old buffer may still be used by earlier launches on this stream
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
      w.cnt_bytes = 0;
    }
    const size_t grow = std::max(bytes, static_cast<size_t>(1) << 20);
    if (cudaMalloc(&w.ptr, grow) != cudaSuccess) return PA_ERR_CUDA;
    w.bytes = grow;
  }
  if (w.cnt_bytes < cnt || w.cnt_bytes == 0) {
    // zero the scheduler counters and any counter bytes not known to be zero
    if (w.cnt_bytes == 0) {
      if (cudaMemsetAsync(w.ptr, 0, kSchedBytes + cnt, stream) != cudaSuccess) return PA_ERR_CUDA;
    } else {
      unsigned char* base = static_cast<unsigned char*>(w.ptr) + kSchedBytes + w.cnt_bytes;
      if (cudaMemsetAsync(base, 0, cnt - w.cnt_bytes, stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    w.cnt_bytes = cnt;
  }
  *out = w.ptr;
  *cnt_bytes = cnt;
  return PA_OK;
}

// ---- validation helpers ---------------------------------------------------------------------
int elem_bytes(int dtype) { return dtype == PA_F32 || dtype == PA_I32 ? 4 : (dtype == PA_F16 || dtype == PA_BF16) ? 2 : 0; }
bool is_float(int dtype) { return dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Rows [s0, s0 + n) of a tensor whose first dimension is the sequence: a view with the
// same strides.
pa_tensor row_range(const pa_tensor* t, int64_t s0, int64_t n) {
  pa_tensor v = *t;
  v.data = static_cast<unsigned char*>(t->data) + s0 * t->stride[0] * elem_bytes(t->dtype);
  v.shape[0] = n;
  return v;
}

// [N, H, D] with the [H, D] part contiguous and a 16-byte-multiple row stride.
int check_rows(const pa_tensor* t, int dtype, int64_t H, int64_t D) {
  if (!t) return PA_ERR_INVALID;
  if (t->dtype != dtype) return PA_ERR_DTYPE;
  if (t->ndim != 3 || t->shape[1] != H || t->shape[2] != D || t->shape[0] < 0) return PA_ERR_SHAPE;
  if (t->shape[0] == 0) return PA_OK;
  if (!t->data) return PA_ERR_INVALID;
  if (t->stride[2] != 1 || t->stride[1] != D || (t->shape[0] > 1 && t->stride[0] < H * D)) return PA_ERR_STRIDE;
  if (!aligned16(t->data) || (t->stride[0] * elem_bytes(dtype)) % 16 != 0) return PA_ERR_ALIGN;
  return PA_OK;
}

int check_cache(const pa_tensor* c, const pa_tensor* other) {
  if (!c || !c->data) return PA_ERR_INVALID;
  if (!is_float(c->dtype)) return PA_ERR_DTYPE;
  if (c->ndim != 4) return PA_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (c->shape[i] <= 0) return PA_ERR_SHAPE;
  if (c->stride[3] != 1 || c->stride[2] != c->shape[3] || c->stride[1] != c->shape[2] * c->shape[3] ||
      c->stride[0] != c->shape[1] * c->shape[2] * c->shape[3])
    return PA_ERR_STRIDE;
  if (!aligned16(c->data) || (c->shape[3] * elem_bytes(c->dtype)) % 16 != 0) return PA_ERR_ALIGN;
  if (c->shape[0] * c->shape[1] > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (other) {
    if (other->dtype != c->dtype) return PA_ERR_DTYPE;
    for (int i = 0; i < 4; ++i)
      if (other->shape[i] != c->shape[i]) return PA_ERR_SHAPE;
  }
  return PA_OK;
}

int check_i32(const pa_tensor* t, int ndim) {
  if (!t || (!t->data && t->shape[0] > 0)) return PA_ERR_INVALID;
  if (t->dtype != PA_I32) return PA_ERR_DTYPE;
  if (t->ndim != ndim) return PA_ERR_SHAPE;
  if (t->stride[ndim - 1] != 1) return PA_ERR_STRIDE;
  return PA_OK;
}

#define PA_TRY(x)                  \
  do {                             \
    int _rc = (x);                 \
    if (_rc != PA_OK) return _rc;  \
  } while (0)

int round_up(int64_t x, int64_t m) { return static_cast<int>(((x + m - 1) / m) * m); }

cudaError_t dispatch_decode(const pa::DecodeArgs& a, const pa::DecodeCfg& c, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t st, bool query_only, int* max_ctas) {
  switch (c.dtype) {
    case PA_F32: return pa::launch_decode_f32(a, c, tk, tv, st, query_only, max_ctas);
    case PA_F16: return pa::launch_decode_f16(a, c, tk, tv, st, query_only, max_ctas);
    case PA_BF16: return pa::launch_decode_bf16(a, c, tk, tv, st, query_only, max_ctas);
    default: return cudaErrorInvalidValue;
  }
}

bool combo_built(int hg, int wph) {
  return (hg == 4 && (wph == 1 || wph == 2)) || (hg == 2 && (wph == 1 || wph == 2 || wph == 4)) ||
         (hg == 1 && (wph == 1 || wph == 2 || wph == 4 || wph == 8));
}

// Tokens per staged unit.  With 256-byte rows and B a power of two, the unrolled path
// takes units of R = 16 * warps_per_head tokens (1 or 2 warps per head): R/B frames
// share a stage when B < R, a frame is staged as B/R slices when B > R.  Otherwise a
// unit is one frame.
int64_t unit_rows(int64_t B, int wph, bool fast_rows) {
  const int64_t R = 16 * wph;
  if (fast_rows && (wph == 1 || wph == 2) && (R % B == 0 || B % R == 0)) return R;
  return B;
}

// pinned staging of pa_step_decode (defined with it, below)
void release_step_stages();

}  // namespace

size_t pa::decode_smem_bytes(const DecodeCfg& c, int elem, int R, int S) {
  const uint32_t stage_bytes = 2u * static_cast<uint32_t>(R) * c.heads_per_cta * c.D * elem;
  const dk::Layout lay(c.stages, stage_bytes, S, c.heads_per_cta * c.warps_per_head, c.D);
  return lay.total;
}

static int cache_append(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* slot_mapping,
                        const pa_tensor* k_cache, const pa_tensor* v_cache, pa_stream stream,
                        const pa::AppendArgs* stage);

extern "C" {

const char* pa_strerror(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_WARN_DOUBLE_FREE: return "sequence not live (free was a no-op)";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_DTYPE: return "unsupported or mismatched dtype";
    case PA_ERR_SHAPE: return "bad shape";
    case PA_ERR_STRIDE: return "bad stride (layout not supported)";
    case PA_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
    case PA_ERR_OUT_OF_BLOCKS: return "out of free blocks";
    case PA_ERR_UNKNOWN_SEQ: return "unknown sequence id";
    case PA_ERR_SEQ_EXISTS: return "sequence id already live";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_UNSUPPORTED: return "size or dtype outside the built kernels";
    case PA_ERR_HOST_MEMORY: return "host memory allocation failed";
    case PA_ERR_CAPACITY: return "output buffer too small";
    case PA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed 16 MiB array of pa_decode_static";
    default: return "unknown code";
  }
}

int64_t pa_launch_count(void) { return g_launches.load(); }

int pa_get_device_status(pa_stream stream, int32_t* status_out) {
  if (!status_out) return PA_ERR_INVALID;
  int dev;
  PA_TRY(current_device(&dev));
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, g_dev[dev].status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemset(g_dev[dev].status, 0, sizeof(v)) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  if (v & PA_DEV_TIMEOUT) {
    // A block that gave up a wait may have left scheduler or arrival counters
    // non-zero.  Nothing of this library runs on the device now (synchronised above):
    // mark every workspace of this device unknown, so its next use zeroes them.
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto& kv : g_ws)
      if (kv.first.first == dev) kv.second.cnt_bytes = 0;
  }
  *status_out = v;
  return PA_OK;
}

int pa_selftest_wait_timeout(int64_t* result_out, pa_stream stream) {
  if (!result_out) return PA_ERR_INVALID;
  int dev;
  PA_TRY(current_device(&dev));
  long long* d_res = nullptr;
  if (cudaMalloc(&d_res, 4 * sizeof(long long)) != cudaSuccess) return PA_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PA_OK;
  if (cudaMemsetAsync(d_res, 0xff, 4 * sizeof(long long), st) != cudaSuccess) rc = PA_ERR_CUDA;
  if (rc == PA_OK) {
    selftest_wait_kernel<<<1, 64, 0, st>>>(g_dev[dev].status, d_res);
    if (cudaGetLastError() != cudaSuccess) rc = PA_ERR_CUDA;
  }
  long long h[4] = {-1, -1, -1, -1};
  if (rc == PA_OK && (cudaMemcpyAsync(h, d_res, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
                      cudaStreamSynchronize(st) != cudaSuccess))
    rc = PA_ERR_CUDA;
  cudaFree(d_res);
  if (rc != PA_OK) return rc;
  for (int i = 0; i < 4; ++i) result_out[i] = h[i];
  g_launches.fetch_add(1);
  return PA_OK;
}

int pa_shutdown(void) {
  release_step_stages();
  std::lock_guard<std::mutex> lk(g_ws_mu);
  int prev = -1;
  cudaGetDevice(&prev);
  for (auto& kv : g_ws) {
    if (kv.second.ptr) {
      cudaSetDevice(kv.first.first);
      cudaFree(kv.second.ptr);
    }
  }
  g_ws.clear();
  if (prev >= 0) cudaSetDevice(prev);
  return PA_OK;
}

int pa_cache_append(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* slot_mapping,
                    const pa_tensor* k_cache, const pa_tensor* v_cache, pa_stream stream) {
  return cache_append(k_new, v_new, slot_mapping, k_cache, v_cache, stream, nullptr);
}

}  // extern "C"

// pa_cache_append, optionally with its slots in mapped host memory and a staging copy
// done by the same launch (stage != nullptr; the step path below).
static int cache_append(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* slot_mapping,
                        const pa_tensor* k_cache, const pa_tensor* v_cache, pa_stream stream,
                        const pa::AppendArgs* stage) {
  const Range range("pa_cache_append");
  PA_TRY(check_cache(k_cache, v_cache));
  const int dt = k_cache->dtype;
  const int64_t H = k_cache->shape[2], D = k_cache->shape[3];
  PA_TRY(check_rows(k_new, dt, H, D));
  PA_TRY(check_rows(v_new, dt, H, D));
  if (!slot_mapping) return PA_ERR_INVALID;
  PA_TRY(check_i32(slot_mapping, 1));
  const int64_t T = k_new->shape[0];
  if (v_new->shape[0] != T || slot_mapping->shape[0] != T) return PA_ERR_SHAPE;
  if (T > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (T == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  const int e = elem_bytes(dt);
  pa::AppendArgs a;
  a.k_new = static_cast<const unsigned char*>(k_new->data);
  a.v_new = static_cast<const unsigned char*>(v_new->data);
  a.k_pitch = k_new->stride[0] * e;
  a.v_pitch = v_new->stride[0] * e;
  a.slots = static_cast<const int32_t*>(slot_mapping->data);
  a.k_cache = static_cast<unsigned char*>(k_cache->data);
  a.v_cache = static_cast<unsigned char*>(v_cache->data);
  a.row_bytes = H * D * e;
  a.num_slots = k_cache->shape[0] * k_cache->shape[1];
  a.T = static_cast<int32_t>(T);
  a.slots_host = 0;
  a.status = g_dev[dev].status;
  a.stage_src = nullptr;
  a.stage_dst = nullptr;
  a.stage_vecs = 0;
  if (stage) {
    a.slots_host = stage->slots_host;
    a.stage_src = stage->stage_src;
    a.stage_dst = stage->stage_dst;
    a.stage_vecs = stage->stage_vecs;
  }
  if (pa::launch_cache_append(a, g_dev[dev].num_sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  g_launches.fetch_add(1);
  return PA_OK;
}

extern "C" {

// ---- the split cache layout ---------------------------------------------------------------
// k_cache viewed as [nb, H, D/x, B*x], v_cache as [nb, H, D, B], both contiguous, fp16/bf16.
static int check_split_caches(const pa_tensor* k, const pa_tensor* v, int64_t* nb, int64_t* H, int64_t* D,
                              int64_t* B) {
  if (!k || !v || !k->data || !v->data) return PA_ERR_INVALID;
  if (k->dtype != v->dtype || (k->dtype != PA_F16 && k->dtype != PA_BF16)) return PA_ERR_DTYPE;
  if (k->ndim != 4 || v->ndim != 4) return PA_ERR_SHAPE;
  const int64_t x = 8;
  *nb = v->shape[0];
  *H = v->shape[1];
  *D = v->shape[2];
  *B = v->shape[3];
  if (k->shape[0] != *nb || k->shape[1] != *H || k->shape[2] * x != *D || k->shape[3] != *B * x) return PA_ERR_SHAPE;
  for (const pa_tensor* t : {k, v}) {
    int64_t want = 1;
    for (int i = 3; i >= 0; --i) {
      if (t->shape[i] > 1 && t->stride[i] != want) return PA_ERR_STRIDE;
      want *= t->shape[i];
    }
    if (!aligned16(t->data)) return PA_ERR_ALIGN;
  }
  if (*nb <= 0 || *H <= 0) return PA_ERR_SHAPE;
  if (!(*D == 64 || *D == 128) || !(*B == 8 || *B == 16 || *B == 32) || *H % 4 != 0) return PA_ERR_UNSUPPORTED;
  if (*nb * *B > INT32_MAX) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

int pa_cache_append_split(const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* slot_mapping,
                          const pa_tensor* k_cache, const pa_tensor* v_cache, pa_stream stream) {
  int64_t nb, H, D, B;
  PA_TRY(check_split_caches(k_cache, v_cache, &nb, &H, &D, &B));
  const int dt = k_cache->dtype;
  PA_TRY(check_rows(k_new, dt, H, D));
  PA_TRY(check_rows(v_new, dt, H, D));
  if (!slot_mapping) return PA_ERR_INVALID;
  PA_TRY(check_i32(slot_mapping, 1));
  const int64_t T = k_new->shape[0];
  if (v_new->shape[0] != T || slot_mapping->shape[0] != T) return PA_ERR_SHAPE;
  if (T > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (T == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  const int64_t units = T * H * (D / 8);
  const int grid = static_cast<int>(std::min<int64_t>((units + 255) / 256, 16LL * g_dev[dev].num_sms));
  if (pa::launch_append_split(dt, k_new->data, v_new->data, k_new->stride[0], v_new->stride[0],
                              static_cast<const int32_t*>(slot_mapping->data), static_cast<int32_t>(T),
                              static_cast<int32_t>(H), static_cast<int32_t>(D), static_cast<int32_t>(B),
                              static_cast<int32_t>(nb), k_cache->data, v_cache->data, g_dev[dev].status, grid,
                              static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  g_launches.fetch_add(1);
  return PA_OK;
}

int pa_decode_split(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                    const pa_tensor* block_tables, const pa_tensor* context_lens, float scale, const pa_tensor* out,
                    pa_stream stream) {
  int64_t nb, H, D, B;
  PA_TRY(check_split_caches(k_cache, v_cache, &nb, &H, &D, &B));
  const int dt = k_cache->dtype;
  PA_TRY(check_rows(q, dt, H, D));
  PA_TRY(check_rows(out, dt, H, D));
  if (!block_tables || !context_lens) return PA_ERR_INVALID;
  PA_TRY(check_i32(block_tables, 2));
  PA_TRY(check_i32(context_lens, 1));
  const int64_t S = q->shape[0];
  if (out->shape[0] != S || block_tables->shape[0] != S || context_lens->shape[0] != S) return PA_ERR_SHAPE;
  const int64_t max_blocks = block_tables->shape[1];
  if (max_blocks < 0 || (S > 1 && block_tables->stride[0] < max_blocks)) return PA_ERR_STRIDE;
  if (max_blocks * B > INT32_MAX || S * H > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (S == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  const int sms = g_dev[dev].num_sms;
  // context partitions only when (sequence, head group) items cannot fill the GPU; then
  // about four per thread-block slot (two blocks per SM), so that the dynamic scheduler
  // ends the launch with short items on every block instead of a second wave of long
  // ones on a few
  // heads per work item: 4, or 2 where a stage of 4 heads' frame would pass 48 KB
  const int64_t hg = 2 * 4 * D * B * elem_bytes(dt) > 48 * 1024 ? 2 : 4;
  const int64_t groups = H / hg, cap = std::max<int64_t>(max_blocks * B, B);
  int64_t P = cap, NP = 1;
  if (S * groups < 2LL * sms) {
    const int64_t want = (8LL * sms + S * groups - 1) / (S * groups);
    P = std::max<int64_t>(256, ((cap + want - 1) / want + B - 1) / B * B);
    NP = (cap + P - 1) / P;
  }
  if (S * groups * NP > INT32_MAX / 4) return PA_ERR_UNSUPPORTED;
  pa::SplitArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q->data;
  a.out = out->data;
  a.q_row = q->stride[0];
  a.out_row = out->stride[0];
  a.k_cache = k_cache->data;
  a.v_cache = v_cache->data;
  a.block_tables = static_cast<const int32_t*>(block_tables->data);
  a.bt_row = block_tables->stride[0];
  a.context_lens = static_cast<const int32_t*>(context_lens->data);
  a.S = static_cast<int32_t>(S);
  a.H = static_cast<int32_t>(H);
  a.num_blocks = static_cast<int32_t>(nb);
  a.max_blocks = static_cast<int32_t>(max_blocks);
  a.P = static_cast<int32_t>(P);
  a.NP = static_cast<int32_t>(NP);
  a.hg = static_cast<int32_t>(hg);
  // whole sequences as items: hand them out longest first (the order costs 4 bytes of
  // shared memory per sequence, kept small enough to leave two blocks per SM)
  a.longest_first = NP == 1 && S <= 2048 ? 1 : 0;
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.status = g_dev[dev].status;
  const size_t items = static_cast<size_t>(S * groups * NP);
  const size_t rest = NP > 1 ? items * hg * (2 + static_cast<size_t>(D)) * sizeof(float) : 0;
  void* ws = nullptr;
  size_t cnt_bytes = 0;
  PA_TRY(workspace(dev, static_cast<cudaStream_t>(stream), 0, rest, &ws, &cnt_bytes));
  a.sched = static_cast<int32_t*>(ws);
  if (NP > 1) {
    float* base = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + kSchedBytes + cnt_bytes);
    a.ws_ml = base;
    a.ws_o = base + items * hg * 2;
  }
  if (pa::launch_decode_split(dt, static_cast<int>(D), static_cast<int>(B), a, sms,
                              static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  g_launches.fetch_add(NP > 1 ? 2 : 1);
  return PA_OK;
}

int pa_copy_blocks(const pa_tensor* k_cache, const pa_tensor* v_cache, const pa_tensor* pairs, pa_stream stream) {
  PA_TRY(check_cache(k_cache, v_cache));
  if (!pairs) return PA_ERR_INVALID;
  PA_TRY(check_i32(pairs, 2));
  if (pairs->shape[1] != 2 || (pairs->shape[0] > 1 && pairs->stride[0] != 2)) return PA_ERR_SHAPE;
  const int64_t n = pairs->shape[0];
  if (n < 0 || n > INT32_MAX) return PA_ERR_SHAPE;
  if (n == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  pa::CopyArgs a;
  a.k_cache = static_cast<unsigned char*>(k_cache->data);
  a.v_cache = static_cast<unsigned char*>(v_cache->data);
  a.pairs = static_cast<const int32_t*>(pairs->data);
  a.frame_bytes = k_cache->stride[0] * elem_bytes(k_cache->dtype);
  a.n = static_cast<int32_t>(n);
  a.num_blocks = static_cast<int32_t>(k_cache->shape[0]);
  a.status = g_dev[dev].status;
  if (pa::launch_copy_blocks(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  g_launches.fetch_add(1);
  return PA_OK;
}

}  // extern "C"

namespace {
// Shared-prefix decode (pa_decode_params.share_prefix).  Returns PA_OK after launching
// the plan kernel and the decode (which merges split sequences itself), kNotApplicable when the shapes fall outside what the
// shared-prefix kernel handles (the caller then runs the plain decode: same result),
// or an error code.
constexpr int kNotApplicable = 1;
// plan_decode: the batch needs more shared memory than one launch has (split it)
constexpr int kTooManySeqs = 2;

int decode_shared(int dev, const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                  const pa_tensor* block_tables, const pa_tensor* context_lens, float scale, const pa_tensor* out,
                  const pa_decode_params& p, pa_stream stream) {
  const int dt = k_cache->dtype;
  const int64_t nb = k_cache->shape[0], B = k_cache->shape[1], H = k_cache->shape[2], D = k_cache->shape[3];
  const int64_t S = q->shape[0];
  const int64_t max_blocks = block_tables->shape[1];
  if (!(dt == PA_F16 || dt == PA_BF16) || D != 128 || (B & (B - 1)) != 0 || B < 8 || S < 2 || S > 4096)
    return kNotApplicable;
  pa::DecodeCfg c;
  c.dtype = dt;
  c.D = 128;
  c.fast = true;
  c.heads_per_cta = p.heads_per_cta ? p.heads_per_cta : (H % 4 == 0 ? 4 : H % 2 == 0 ? 2 : 1);
  c.warps_per_head = p.warps_per_head ? p.warps_per_head : 1;
  if (!pa::decode_shared_combo(c.heads_per_cta, c.warps_per_head) || H % c.heads_per_cta != 0)
    return PA_ERR_INVALID;
  const int64_t R = 16;  // tokens per staged unit: one 16-key tensor-core tile
  const size_t smem_cap = 227 * 1024;
  auto smem_of = [&](int st) {
    pa::DecodeCfg t = c;
    t.stages = st;
    return pa::decode_shared_smem_bytes(t, static_cast<int>(R), static_cast<int>(S));
  };
  c.stages = 0;
  if (p.stages) {
    if (p.stages < 2 || p.stages > 8) return PA_ERR_INVALID;
    c.stages = p.stages;
  } else {
    for (int st = 8; st >= 3 && !c.stages; --st)
      if (smem_of(st) <= smem_cap / 2 - 1024) c.stages = st;
    for (int st = 8; st >= 2 && !c.stages; --st)
      if (smem_of(st) <= smem_cap) c.stages = st;
  }
  if (!c.stages || smem_of(c.stages) > smem_cap) return kNotApplicable;

  pa::DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q->data;
  a.out = out->data;
  a.q_row = q->stride[0];
  a.out_row = out->stride[0];
  a.block_tables = static_cast<const int32_t*>(block_tables->data);
  a.bt_row = block_tables->stride[0];
  a.context_lens = static_cast<const int32_t*>(context_lens->data);
  a.S = static_cast<int32_t>(S);
  a.H = static_cast<int32_t>(H);
  a.B = static_cast<int32_t>(B);
  a.R = static_cast<int32_t>(R);
  a.num_blocks = static_cast<int32_t>(nb);
  a.max_blocks = static_cast<int32_t>(max_blocks);
  a.G = static_cast<int32_t>(H / c.heads_per_cta);
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.status = g_dev[dev].status;
  a.min_shared = static_cast<int32_t>(std::max<int64_t>(p.share_prefix == 1 ? 256 : p.share_prefix, B));

  CUtensorMap tk, tv;
  PA_TRY(make_half_rows_map(&tk, k_cache->data, dt, nb * B, H, c.heads_per_cta, static_cast<int>(std::min(B, R))));
  PA_TRY(make_half_rows_map(&tv, v_cache->data, dt, nb * B, H, c.heads_per_cta, static_cast<int>(std::min(B, R))));
  int occ = 0;
  if (pa::launch_decode_shared(a, c, tk, tv, nullptr, true, &occ) != cudaSuccess || occ <= 0) return PA_ERR_CUDA;
  c.grid = g_dev[dev].num_sms * (p.ctas_per_sm ? std::min(p.ctas_per_sm, occ) : occ);

  // partition length and the number of partial slots the workspace holds (the kernel
  // falls back to whole segments, at most 2 per sequence, if its parts would not fit)
  const int64_t Lcap = max_blocks * B;
  int64_t part_cap;
  if (p.items_per_cta < 0) return PA_ERR_INVALID;
  if (p.partition_tokens == -1 || Lcap == 0) {
    a.fixed_part = static_cast<int32_t>(std::max<int64_t>(Lcap, B));
    part_cap = 2 * S;
  } else if (p.partition_tokens > 0) {
    a.fixed_part = round_up(p.partition_tokens, B);
    part_cap = S * ((Lcap + a.fixed_part - 1) / a.fixed_part + 2);
  } else if (p.partition_tokens == 0) {
    a.whole_first = p.items_per_cta == 0;
    a.target_items = p.items_per_cta ? p.items_per_cta * c.grid : (3 * c.grid) / 2;
    // parts of at least 512 tokens: an item carries up to 16 queries and pays their loads
    // and its epilogue once, so longer parts than the plain decode's amortise better
    a.min_part = round_up(512, B);
    // parts of the automatic choice: every member of a chunk holds its own partial of
    // each shared part, so up to 16 per shared part, plus the private parts
    part_cap = 3 * S + 2 * (16 + 1) * ((a.target_items + a.G - 1) / a.G) + 8;
  } else {
    return PA_ERR_INVALID;
  }
  const int64_t slot_bytes = H * (D + 2) * static_cast<int64_t>(sizeof(float));
  part_cap = std::max<int64_t>(2 * S, std::min<int64_t>(part_cap, (static_cast<int64_t>(1) << 32) / slot_bytes));
  a.part_cap = static_cast<int32_t>(part_cap);
  {
    const size_t o_bytes = static_cast<size_t>(part_cap * H * D) * sizeof(float);
    const size_t ml_bytes = static_cast<size_t>(part_cap * H * 2) * sizeof(float);
    const size_t lcp_bytes = static_cast<size_t>(S) * sizeof(int32_t);
    // arrival counters: parts finished per (sequence, head), for the in-kernel merges
    const size_t cnt_need = static_cast<size_t>(S * H) * sizeof(int32_t);
    void* ws = nullptr;
    size_t cnt_bytes = 0;
    PA_TRY(workspace(dev, static_cast<cudaStream_t>(stream), cnt_need, o_bytes + ml_bytes + lcp_bytes, &ws,
                     &cnt_bytes));
    unsigned char* w = static_cast<unsigned char*>(ws);
    unsigned char* rest = w + kSchedBytes + cnt_bytes;
    a.sched = reinterpret_cast<int32_t*>(w);
    a.ws_cnt = reinterpret_cast<int32_t*>(w + kSchedBytes);
    a.ws_o = reinterpret_cast<float*>(rest);
    a.ws_ml = reinterpret_cast<float*>(rest + o_bytes);
    a.lcp = reinterpret_cast<int32_t*>(rest + o_bytes + ml_bytes);
  }
  if (pa::launch_decode_shared(a, c, tk, tv, static_cast<cudaStream_t>(stream), false, nullptr) != cudaSuccess)
    return PA_ERR_CUDA;
  g_launches.fetch_add(2);
  return PA_OK;
}

// Argument checks of pa_decode and pa_decode_static; *S_out = number of sequences.
int check_decode(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* block_tables, const pa_tensor* context_lens, const pa_tensor* out,
                 int64_t* S_out) {
  PA_TRY(check_cache(k_cache, v_cache));
  const int dt = k_cache->dtype;
  const int64_t B = k_cache->shape[1], H = k_cache->shape[2], D = k_cache->shape[3];
  PA_TRY(check_rows(q, dt, H, D));
  PA_TRY(check_rows(out, dt, H, D));
  if (!block_tables || !context_lens) return PA_ERR_INVALID;
  PA_TRY(check_i32(block_tables, 2));
  PA_TRY(check_i32(context_lens, 1));
  const int64_t S = q->shape[0];
  if (out->shape[0] != S || block_tables->shape[0] != S || context_lens->shape[0] != S) return PA_ERR_SHAPE;
  const int64_t max_blocks = block_tables->shape[1];
  if (max_blocks < 0 || (S > 1 && block_tables->stride[0] < max_blocks)) return PA_ERR_STRIDE;
  if (B > 256) return PA_ERR_UNSUPPORTED;
  if (!(D == 64 || D == 128 || (D == 256 && dt != PA_F32))) return PA_ERR_UNSUPPORTED;
  if (max_blocks * B > INT32_MAX || S > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (S > 0 && max_blocks > 0 && !block_tables->data) return PA_ERR_INVALID;
  *S_out = S;
  return PA_OK;
}

// One decode launch, planned: configuration, kernel arguments (all but the scratch
// pointers), tensor maps, and the scratch it needs.  The scratch sizes follow the
// kernel's own partition rule (at most items_max partial results), so every caller
// that sizes its scratch from a plan gives the kernel enough.
struct DecodePlan {
  pa::DecodeCfg c;
  pa::DecodeArgs a;
  CUtensorMap tk, tv;
  int64_t items_max = 0;
  size_t o_bytes = 0;   // split partial outputs, fp32
  size_t ml_bytes = 0;  // split partial maxima and sums, fp32
  size_t cnt_need = 0;  // arrival counters, one int32 per (sequence, head), when a context may split
};

// Plans a checked decode with S > 0 sequences under launch options p (0 fields =
// automatic).
int plan_decode(int dev, const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                const pa_tensor* block_tables, const pa_tensor* context_lens, float scale, const pa_tensor* out,
                const pa_decode_params& p, DecodePlan* pl) {
  const int dt = k_cache->dtype;
  const int64_t nb = k_cache->shape[0], B = k_cache->shape[1], H = k_cache->shape[2], D = k_cache->shape[3];
  const int64_t S = q->shape[0];
  const int64_t max_blocks = block_tables->shape[1];
  const int e = elem_bytes(dt);
  pa::DecodeCfg& c = pl->c;
  c.dtype = dt;
  c.D = static_cast<int>(D);
  // Unrolled full-frame path: 256-byte rows, units of 16 * warps_per_head tokens.
  const bool fast_rows = D * e == 256 && (B & (B - 1)) == 0 && !p.generic_only;
  int wph = p.warps_per_head;
  if (!wph && fast_rows) wph = B >= 32 ? 2 : 1;
  const int64_t R = wph ? unit_rows(B, wph, fast_rows) : B;
  if (p.heads_per_cta) {
    if (!(p.heads_per_cta == 1 || p.heads_per_cta == 2 || p.heads_per_cta == 4) || H % p.heads_per_cta != 0)
      return PA_ERR_INVALID;
    c.heads_per_cta = p.heads_per_cta;
  } else {
    c.heads_per_cta = 1;
    for (int hg : {4, 2}) {
      if (H % hg == 0 && 2 * R * hg * D * e <= 32768) {
        c.heads_per_cta = hg;
        break;
      }
    }
  }
  c.warps_per_head = wph ? wph : 8 / c.heads_per_cta;
  c.fast = fast_rows && R == 16 * c.warps_per_head;
  if (!combo_built(c.heads_per_cta, c.warps_per_head)) return PA_ERR_INVALID;
  c.stages = 1;
  const size_t smem_cap = 227 * 1024;
  if (p.stages) {
    if (p.stages < 2 || p.stages > 8) return PA_ERR_INVALID;
    c.stages = p.stages;
  } else {
    // two resident blocks per SM when the staging ring still holds >= 3 frames
    for (int st = 8; st >= 2; --st) {
      c.stages = st;
      if (pa::decode_smem_bytes(c, e, static_cast<int>(R), static_cast<int>(S)) <= smem_cap / 2 - 1024 && st >= 3)
        break;
      c.stages = 0;
    }
    if (c.stages == 0) {
      for (int st = 8; st >= 2; --st) {
        c.stages = st;
        if (pa::decode_smem_bytes(c, e, static_cast<int>(R), static_cast<int>(S)) <= smem_cap) break;
        c.stages = 0;
      }
    }
  }
  if (c.stages == 0 || pa::decode_smem_bytes(c, e, static_cast<int>(R), static_cast<int>(S)) > smem_cap) {
    // every thread block keeps three int32 per sequence in shared memory beside its
    // staging ring: a batch too large for that is run as several launches
    pa::DecodeCfg one = c;
    one.stages = p.stages ? p.stages : 2;
    return pa::decode_smem_bytes(one, e, static_cast<int>(R), 1) <= smem_cap ? kTooManySeqs : PA_ERR_UNSUPPORTED;
  }

  pa::DecodeArgs& a = pl->a;
  std::memset(&a, 0, sizeof(a));
  a.q = q->data;
  a.out = out->data;
  a.q_row = q->stride[0];
  a.out_row = out->stride[0];
  a.block_tables = static_cast<const int32_t*>(block_tables->data);
  a.bt_row = block_tables->stride[0];
  a.context_lens = static_cast<const int32_t*>(context_lens->data);
  a.S = static_cast<int32_t>(S);
  a.H = static_cast<int32_t>(H);
  a.B = static_cast<int32_t>(B);
  a.R = static_cast<int32_t>(R);
  a.num_blocks = static_cast<int32_t>(nb);
  a.max_blocks = static_cast<int32_t>(max_blocks);
  a.G = static_cast<int32_t>(H / c.heads_per_cta);
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.status = g_dev[dev].status;

  PA_TRY(make_cache_map(&pl->tk, k_cache->data, dt, nb, B, H, D, c.heads_per_cta, std::min(B, R)));
  PA_TRY(make_cache_map(&pl->tv, v_cache->data, dt, nb, B, H, D, c.heads_per_cta, std::min(B, R)));

  int occ = 0;
  if (dispatch_decode(a, c, pl->tk, pl->tv, nullptr, true, &occ) != cudaSuccess || occ <= 0) return PA_ERR_CUDA;
  const int cps = p.ctas_per_sm ? std::min(p.ctas_per_sm, occ) : occ;
  c.grid = g_dev[dev].num_sms * cps;

  // ---- partitioning: the most partial results the kernel can write --------------------------
  const int64_t Lcap = max_blocks * B;
  int64_t items_max = 0;
  if (p.items_per_cta < 0 || p.generic_only < 0) return PA_ERR_INVALID;
  if (p.partition_tokens == -1 || Lcap == 0) {
    a.fixed_part = static_cast<int32_t>(std::max<int64_t>(Lcap, B));
  } else if (p.partition_tokens > 0) {
    a.fixed_part = round_up(p.partition_tokens, B);
    if (a.fixed_part < Lcap) items_max = S * a.G * ((Lcap + a.fixed_part - 1) / a.fixed_part);
  } else if (p.partition_tokens == 0) {
    a.fixed_part = 0;
    a.whole_first = p.items_per_cta == 0;
    a.target_items = p.items_per_cta ? p.items_per_cta * c.grid : (3 * c.grid) / 2;
    a.min_part = round_up(256, B);
    if (a.min_part < Lcap)  // the kernel may shorten its partitions down to half its first choice
      items_max = std::min<int64_t>(S * a.G * ((Lcap + a.min_part - 1) / a.min_part), 2 * a.target_items + S * a.G);
  } else {
    return PA_ERR_INVALID;
  }
  pl->items_max = items_max;
  pl->ml_bytes = static_cast<size_t>(items_max) * c.heads_per_cta * 2 * sizeof(float);
  pl->o_bytes = static_cast<size_t>(items_max) * c.heads_per_cta * D * sizeof(float);
  pl->cnt_need = items_max > 0 ? static_cast<size_t>(S * H) * sizeof(int32_t) : 0;
  return PA_OK;
}

// Scratch pointers of a planned decode: scheduler counters at `base`, arrival counters
// after kSchedBytes, partials after the cnt_bytes arrival-counter region.
void place_scratch(DecodePlan* pl, unsigned char* base, size_t cnt_bytes) {
  unsigned char* rest = base + kSchedBytes + cnt_bytes;
  pl->a.sched = reinterpret_cast<int32_t*>(base);
  pl->a.ws_cnt = reinterpret_cast<int32_t*>(base + kSchedBytes);
  if (pl->items_max > 0) {
    pl->a.ws_o = reinterpret_cast<float*>(rest);
    pl->a.ws_ml = reinterpret_cast<float*>(rest + pl->o_bytes);
  }
}
}  // namespace

extern "C" {

int pa_decode_ex(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                 const pa_tensor* block_tables, const pa_tensor* context_lens, float scale, const pa_tensor* out,
                 const pa_decode_params* params, pa_stream stream) {
  const Range range("pa_decode");
  int64_t S = 0;
  PA_TRY(check_decode(q, k_cache, v_cache, block_tables, context_lens, out, &S));
  if (S == 0) return PA_OK;
  pa_decode_params p;
  std::memset(&p, 0, sizeof(p));
  if (params) p = *params;
  if (p.heads_per_cta < 0 || p.warps_per_head < 0 || p.stages < 0 || p.ctas_per_sm < 0 || p.share_prefix < 0)
    return PA_ERR_INVALID;

  int dev;
  PA_TRY(current_device(&dev));
  if (p.share_prefix > 0) {
    const int rc = decode_shared(dev, q, k_cache, v_cache, block_tables, context_lens, scale, out, p, stream);
    if (rc != kNotApplicable) return rc;
  }
  // Sequences are independent: a batch too large for one launch's shared memory runs as
  // launches over consecutive ranges of sequences, the largest range that fits (found by
  // halving), one after another on the stream.
  int64_t chunk = S;
  for (int64_t s0 = 0; s0 < S;) {
    const int64_t n = std::min(chunk, S - s0);
    const pa_tensor qv = row_range(q, s0, n), ov = row_range(out, s0, n);
    const pa_tensor tv = row_range(block_tables, s0, n), lv = row_range(context_lens, s0, n);
    DecodePlan pl;
    const int rc = plan_decode(dev, &qv, k_cache, v_cache, &tv, &lv, scale, &ov, p, &pl);
    if (rc == kTooManySeqs && n > 1) {
      chunk = (n + 1) / 2;
      continue;
    }
    if (rc == kTooManySeqs) return PA_ERR_UNSUPPORTED;
    PA_TRY(rc);
    void* ws = nullptr;
    size_t cnt_bytes = 0;
    PA_TRY(workspace(dev, static_cast<cudaStream_t>(stream), pl.cnt_need, pl.o_bytes + pl.ml_bytes, &ws, &cnt_bytes));
    place_scratch(&pl, static_cast<unsigned char*>(ws), cnt_bytes);
    if (dispatch_decode(pl.a, pl.c, pl.tk, pl.tv, static_cast<cudaStream_t>(stream), false, nullptr) != cudaSuccess)
      return PA_ERR_CUDA;
    g_launches.fetch_add(1);
    s0 += n;
  }
  return PA_OK;
}

int pa_decode(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache, const pa_tensor* block_tables,
              const pa_tensor* context_lens, float scale, const pa_tensor* out, pa_stream stream) {
  return pa_decode_ex(q, k_cache, v_cache, block_tables, context_lens, scale, out, nullptr, stream);
}

int pa_prefill(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache, const pa_tensor* block_tables,
               const pa_tensor* context_lens, const pa_tensor* query_start, float scale, const pa_tensor* out,
               pa_stream stream) {
  const Range range("pa_prefill");
  PA_TRY(check_cache(k_cache, v_cache));
  const int dt = k_cache->dtype;
  if (dt != PA_F16 && dt != PA_BF16) return PA_ERR_UNSUPPORTED;
  const int64_t nb = k_cache->shape[0], B = k_cache->shape[1], H = k_cache->shape[2], D = k_cache->shape[3];
  if (D != 128 || !(B == 8 || B == 16 || B == 32 || B == 64 || B == 128)) return PA_ERR_UNSUPPORTED;
  PA_TRY(check_rows(q, dt, H, D));
  PA_TRY(check_rows(out, dt, H, D));
  if (!block_tables || !context_lens || !query_start) return PA_ERR_INVALID;
  PA_TRY(check_i32(block_tables, 2));
  PA_TRY(check_i32(context_lens, 1));
  PA_TRY(check_i32(query_start, 1));
  const int64_t T = q->shape[0], S = context_lens->shape[0];
  if (out->shape[0] != T || block_tables->shape[0] != S || query_start->shape[0] != S + 1) return PA_ERR_SHAPE;
  const int64_t max_blocks = block_tables->shape[1];
  if (max_blocks < 0 || (S > 1 && block_tables->stride[0] < max_blocks)) return PA_ERR_STRIDE;
  if (max_blocks * B > INT32_MAX || T > INT32_MAX || nb * B > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (S == 0 || T == 0) return PA_OK;
  // A sequence with n query rows forms ceil(ceil(n / 128) / 2) <= n / 256 + 1 units, so
  // n sequences of the batch form at most n + T / 256 + 1.  Every thread block keeps
  // their unit offsets and order in shared memory: a batch larger than that runs as
  // launches over consecutive ranges of sequences (q and out stay whole: query_start
  // entries index all of q).
  const int64_t tile_cap = (T + 255) / 256 + 1;
  auto fits = [&](int64_t n) {
    return n + tile_cap <= INT32_MAX &&
           pa::prefill_smem_bytes(static_cast<int>(n), static_cast<int>(n + tile_cap)) <= 227 * 1024;
  };
  if (!fits(1)) return PA_ERR_UNSUPPORTED;
  int64_t chunk = S;
  while (!fits(chunk)) chunk = (chunk + 1) / 2;
  int dev;
  PA_TRY(current_device(&dev));

  pa::PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q->data;
  a.out = out->data;
  a.q_row = q->stride[0];
  a.out_row = out->stride[0];
  a.block_tables = static_cast<const int32_t*>(block_tables->data);
  a.bt_row = block_tables->stride[0];
  a.context_lens = static_cast<const int32_t*>(context_lens->data);
  a.query_start = static_cast<const int32_t*>(query_start->data);
  a.S = static_cast<int32_t>(S);
  a.H = static_cast<int32_t>(H);
  a.B = static_cast<int32_t>(B);
  a.num_blocks = static_cast<int32_t>(nb);
  a.max_blocks = static_cast<int32_t>(max_blocks);
  a.T = static_cast<int32_t>(T);
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.status = g_dev[dev].status;

  CUtensorMap tq, tk, tv;
  PA_TRY(make_sw128_map(&tq, q->data, dt, T, H, D, q->stride[0], 128));
  PA_TRY(make_frame_map(&tk, k_cache->data, dt, nb * B, H, D, static_cast<int>(B)));
  PA_TRY(make_frame_map(&tv, v_cache->data, dt, nb * B, H, D, static_cast<int>(B)));
  void* ws = nullptr;
  size_t cnt_bytes = 0;
  PA_TRY(workspace(dev, static_cast<cudaStream_t>(stream), 0, 0, &ws, &cnt_bytes));
  a.sched = static_cast<int32_t*>(ws);
  const int grid = g_dev[dev].num_sms;
  for (int64_t s0 = 0; s0 < S; s0 += chunk) {
    const int64_t n = std::min(chunk, S - s0);
    pa::PrefillArgs r = a;
    r.block_tables = a.block_tables + s0 * a.bt_row;
    r.context_lens = a.context_lens + s0;
    r.query_start = a.query_start + s0;
    r.S = static_cast<int32_t>(n);
    r.unit_cap = static_cast<int32_t>(n + tile_cap);
    const cudaError_t e = dt == PA_F16 ? pa::launch_prefill_f16(r, tq, tk, tv, grid, static_cast<cudaStream_t>(stream))
                                       : pa::launch_prefill_bf16(r, tq, tk, tv, grid, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return PA_ERR_CUDA;
    g_launches.fetch_add(1);
  }
  return PA_OK;
}

}  // extern "C"

// ---- decode without any allocation ---------------------------------------------------------
// Some callers may not allocate device memory at all: a serving process that has
// handed the whole device to its own pool allocator (a cudaMalloc behind its back
// can fail or fragment the pool), or a latency-bound loop that cannot afford the
// device-wide synchronisation a first cudaMalloc brings.  For them
// pa_decode_static runs the same kernels with the scratch memory taken from this
// fixed array, which every device that loads the library holds until the process
// exits.  Host code must not use the array's name as a device address: it is a
// host-side stand-in.  The address is looked up once per device with
// cudaGetSymbolAddress, with that device current.
constexpr size_t kFixedScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_pa_fixed_scratch[kFixedScratchBytes];

namespace {
struct FixedScratch {
  std::once_flag once;
  unsigned char* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
FixedScratch g_fixed[kMaxDevices];

int fixed_scratch(int dev, unsigned char** out) {
  FixedScratch& f = g_fixed[dev];
  std::call_once(f.once, [&] { f.err = cudaGetSymbolAddress(reinterpret_cast<void**>(&f.ptr), g_pa_fixed_scratch); });
  if (f.err != cudaSuccess || f.ptr == nullptr) return PA_ERR_CUDA;
  *out = f.ptr;
  return PA_OK;
}
}  // namespace

extern "C" int pa_decode_static(const pa_tensor* q, const pa_tensor* k_cache, const pa_tensor* v_cache,
                                const pa_tensor* block_tables, const pa_tensor* context_lens, float scale,
                                const pa_tensor* out, pa_stream stream) {
  // The checks, automatic launch choices and scratch sizing of pa_decode (one plan).
  int64_t S = 0;
  PA_TRY(check_decode(q, k_cache, v_cache, block_tables, context_lens, out, &S));
  if (S == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  unsigned char* scratch = nullptr;
  PA_TRY(fixed_scratch(dev, &scratch));
  pa_decode_params p;
  std::memset(&p, 0, sizeof(p));
  DecodePlan pl;
  {
    const int rc = plan_decode(dev, q, k_cache, v_cache, block_tables, context_lens, scale, out, p, &pl);
    if (rc == kTooManySeqs) return PA_ERR_UNSUPPORTED;  // one launch only: no split into ranges
    PA_TRY(rc);
  }
  // Scratch layout inside the fixed array: counters | arrival counters | split partials.
  const size_t cnt_bytes = round256(pl.cnt_need);
  if (kSchedBytes + cnt_bytes + pl.o_bytes + pl.ml_bytes > kFixedScratchBytes) return PA_ERR_SCRATCH_LIMIT;
  place_scratch(&pl, scratch, cnt_bytes);
  // The counters must start at zero; the array keeps whatever the last call left.
  if (cudaMemsetAsync(scratch, 0, kSchedBytes + cnt_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  if (dispatch_decode(pl.a, pl.c, pl.tk, pl.tv, static_cast<cudaStream_t>(stream), false, nullptr) != cudaSuccess)
    return PA_ERR_CUDA;
  g_launches.fetch_add(1);
  return PA_OK;
}

// ---- one decode step in one call ------------------------------------------------------------
// The host side of a step (block-manager step, table export, one upload, three launches)
// costs tens of microseconds per call through a binding; a shared-prefix decode of a
// beam-search batch takes about as long on the GPU.  pa_step_decode does the whole host
// side natively.  Its staging buffers form a ring per (device, stream): pinned host
// memory the step writes, device memory one asynchronous copy fills, and an event per
// slot marking when the copy that last read it has run.
namespace {
constexpr int kStepRing = 4;

struct StepStage {
  int32_t* host[kStepRing] = {};
  int32_t* host_dev[kStepRing] = {};  // the same pinned memory, as the device addresses it
  int32_t* dev[kStepRing] = {};
  cudaEvent_t done[kStepRing] = {};
  bool recorded[kStepRing] = {};
  size_t cap = 0;  // int32 elements per slot
  int next = 0;
};
std::mutex g_step_mu;
std::map<std::pair<int, cudaStream_t>, StepStage> g_step;

void free_stage(StepStage& s) {
  for (int i = 0; i < kStepRing; ++i) {
    if (s.host[i]) cudaFreeHost(s.host[i]);
    if (s.dev[i]) cudaFree(s.dev[i]);
    if (s.done[i]) cudaEventDestroy(s.done[i]);
    s.host[i] = nullptr;
    s.host_dev[i] = nullptr;
    s.dev[i] = nullptr;
    s.done[i] = nullptr;
    s.recorded[i] = false;
  }
  s.cap = 0;
}

// A ring slot with room for `need` int32 values, free to overwrite; -1 on a CUDA error,
// -2 when host memory for the ring's bookkeeping cannot be had.
int stage_slot(int dev, cudaStream_t stream, size_t need, StepStage** out) {
  std::lock_guard<std::mutex> lk(g_step_mu);
  StepStage* sp = nullptr;
  try {  // no C++ exception crosses the C ABI
    sp = &g_step[{dev, stream}];
  } catch (...) {
    return -2;
  }
  StepStage& s = *sp;
  if (s.cap < need) {
    if (s.cap && cudaStreamSynchronize(stream) != cudaSuccess) return -1;
    free_stage(s);
    // whole 16-byte vectors: the append's staging copy moves the block in uint4 units
    const size_t cap = (std::max(need, static_cast<size_t>(1) << 14) + 3) & ~static_cast<size_t>(3);
    for (int i = 0; i < kStepRing; ++i) {
      if (cudaHostAlloc(reinterpret_cast<void**>(&s.host[i]), cap * sizeof(int32_t), cudaHostAllocMapped) !=
              cudaSuccess ||
          cudaHostGetDevicePointer(reinterpret_cast<void**>(&s.host_dev[i]), s.host[i], 0) != cudaSuccess ||
          cudaMalloc(reinterpret_cast<void**>(&s.dev[i]), cap * sizeof(int32_t)) != cudaSuccess ||
          cudaEventCreateWithFlags(&s.done[i], cudaEventDisableTiming) != cudaSuccess) {
        free_stage(s);
        return -1;
      }
    }
    s.cap = cap;
  }
  const int i = s.next;
  s.next = (s.next + 1) % kStepRing;
  if (s.recorded[i] && cudaEventSynchronize(s.done[i]) != cudaSuccess) return -1;
  *out = &s;
  return i;
}

void release_step_stages() {
  std::lock_guard<std::mutex> lk(g_step_mu);
  int prev = -1;
  cudaGetDevice(&prev);
  for (auto& kv : g_step) {
    cudaSetDevice(kv.first.first);
    free_stage(kv.second);
  }
  g_step.clear();
  if (prev >= 0) cudaSetDevice(prev);
}

pa_tensor i32_view(int32_t* p, int64_t d0, int64_t d1) {
  pa_tensor t;
  std::memset(&t, 0, sizeof(t));
  t.data = p;
  t.dtype = PA_I32;
  t.ndim = d1 > 0 ? 2 : 1;
  t.shape[0] = d0;
  t.stride[0] = d1 > 0 ? d1 : 1;
  if (d1 > 0) {
    t.shape[1] = d1;
    t.stride[1] = 1;
  }
  return t;
}
}  // namespace

extern "C" int pa_step_decode(pa_bm* bm, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                              const pa_tensor* k_new, const pa_tensor* v_new, const pa_tensor* q,
                              const pa_tensor* k_cache, const pa_tensor* v_cache, float scale, const pa_tensor* out,
                              const pa_decode_params* params, int32_t auto_share, pa_stream stream,
                              int32_t* n_copies_out, int32_t* lens_out) {
  const Range range("pa_step_decode");
  if (!bm || n < 0 || max_blocks <= 0 || (n > 0 && !seq_ids)) return PA_ERR_INVALID;
  if (n_copies_out) *n_copies_out = 0;
  if (n == 0) return PA_OK;
  int dev;
  PA_TRY(current_device(&dev));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // staging: slots [n] | copies [n][2] | lengths [n] | tables [n][max_blocks]
  const size_t need = static_cast<size_t>(n) * (4 + static_cast<size_t>(max_blocks));
  StepStage* s = nullptr;
  const int i = stage_slot(dev, st, need, &s);
  if (i < 0) return i == -2 ? PA_ERR_HOST_MEMORY : PA_ERR_CUDA;
  int32_t* h = s->host[i];
  int32_t* d = s->dev[i];
  int32_t nc = 0;
  {
    const Range bm_range("block manager step + tables");
    PA_TRY(pa_bm_step(bm, seq_ids, n, h, h + n, &nc));
    PA_TRY(pa_bm_block_tables(bm, seq_ids, n, max_blocks, h + 4 * n, h + 3 * n));
  }
  if (n_copies_out) *n_copies_out = nc;
  if (lens_out) std::memcpy(lens_out, h + 3 * n, sizeof(int32_t) * n);
  if (nc > pa::kInlineCopies) {
    // more copy-on-write copies than a launch's parameters carry: one upload of the
    // staged block, the copies, then the new rows with their slots from device memory
    if (cudaMemcpyAsync(d, h, need * sizeof(int32_t), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaEventRecord(s->done[i], st) != cudaSuccess)
      return PA_ERR_CUDA;
    s->recorded[i] = true;
    const pa_tensor pairs = i32_view(d + n, nc, 2);
    PA_TRY(pa_copy_blocks(k_cache, v_cache, &pairs, stream));
    const pa_tensor slots = i32_view(d, n, 0);
    PA_TRY(pa_cache_append(k_new, v_new, &slots, k_cache, v_cache, stream));
  } else {
    // Copy-on-write copies, if any, with their pairs in the kernel's parameters.  Then the
    // append: it reads its slots from the pinned block itself and copies the block
    // (lengths and tables for the decode) to device memory in the same launch, so no
    // copy-engine transfer sits between the previous step's decode and this step.  The
    // device slot it writes was last read by the decode three steps back, which has
    // finished once any kernel of the previous step runs (each step's kernels wait for
    // the one before them).
    if (nc) {
      PA_TRY(check_cache(k_cache, v_cache));
      pa::InlineCopyArgs c;
      std::memset(&c, 0, sizeof(c));
      c.k_cache = static_cast<unsigned char*>(k_cache->data);
      c.v_cache = static_cast<unsigned char*>(v_cache->data);
      c.frame_bytes = k_cache->stride[0] * elem_bytes(k_cache->dtype);
      c.n = nc;
      c.num_blocks = static_cast<int32_t>(k_cache->shape[0]);
      c.status = g_dev[dev].status;
      std::memcpy(c.pairs, h + n, sizeof(int32_t) * 2 * static_cast<size_t>(nc));
      if (pa::launch_copy_blocks_inline(c, st) != cudaSuccess) return PA_ERR_CUDA;
      g_launches.fetch_add(1);
    }
    pa::AppendArgs stage;
    std::memset(&stage, 0, sizeof(stage));
    stage.slots_host = 1;
    stage.stage_src = reinterpret_cast<const uint4*>(s->host_dev[i]);
    stage.stage_dst = reinterpret_cast<uint4*>(d);
    stage.stage_vecs = static_cast<int64_t>((need * sizeof(int32_t) + 15) / 16);
    const pa_tensor slots = i32_view(s->host_dev[i], n, 0);
    PA_TRY(cache_append(k_new, v_new, &slots, k_cache, v_cache, stream, &stage));
    if (cudaEventRecord(s->done[i], st) != cudaSuccess) return PA_ERR_CUDA;
    s->recorded[i] = true;
  }
  pa_decode_params p;
  const pa_decode_params* pp = params;
  if (!params && auto_share) {
    // the shared-prefix decode when two neighbouring sequences start on the same frame
    const int32_t* tb = h + 4 * n;
    for (int32_t j = 1; j < n; ++j) {
      if (tb[static_cast<int64_t>(j) * max_blocks] >= 0 &&
          tb[static_cast<int64_t>(j) * max_blocks] == tb[static_cast<int64_t>(j - 1) * max_blocks]) {
        std::memset(&p, 0, sizeof(p));
        p.share_prefix = 1;
        pp = &p;
        break;
      }
    }
  }
  const pa_tensor tables = i32_view(d + 4 * n, n, max_blocks);
  const pa_tensor lens = i32_view(d + 3 * n, n, 0);
  return pa_decode_ex(q, k_cache, v_cache, &tables, &lens, scale, out, pp, stream);
}
