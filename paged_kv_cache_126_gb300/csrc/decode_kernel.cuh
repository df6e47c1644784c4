// Paged single-query decode attention for sm_103a.
//
// What it computes ("Solving the LLM Memory Wall", "1. The Mathematical
// Foundation"): for every sequence s and head h, out = softmax(q.K^T * scale) V
// over the sequence's L_s tokens, where token i's K/V rows live in frame
// block_tables[s][i / B] at offset i % B of the caches [num_blocks, B, H, D].
// "PagedAttention: Virtual Memory Guide for LLM Inference" ("3. PagedAttention
// CUDA Kernel Execution"): the kernel reads the block table itself and stages the
// frames on chip; no gathered K/V copy is ever written to HBM.
//
// Design (GB300):
//   * Work item = (sequence, head group of HG heads, context partition).  A
//     persistent grid of thread blocks takes items from a global atomic counter
//     (dynamic scheduling), longest items first: every full partition of every
//     sequence, then the shorter last partitions.  The partition length is chosen
//     on the device from the actual context lengths so there are a few items per
//     thread block.  The counter resets itself: the last thread block to retire
//     zeroes it for the next launch on the stream.
//   * One producer warp: takes the next item, hands its id to the consumers
//     through a two-slot mbarrier ring, reads the item's block-table slice (one
//     coalesced load per 32 frames), bounds-checks every frame id, and for each
//     frame issues two 3-D TMA tile loads (K and V: box {D, HG, B} of the
//     [num_blocks*B, H, D] view) into a ring of `stages` shared-memory buffers.
//   * HG*WPH consumer warps: warp (h, w) owns head h and a share of the rows of
//     each staged frame.  A row (one token, one head) is read as 16-byte chunks by
//     LPR = D*elem/16 lanes (conflict-free shared-memory reads).  For 256-byte rows
//     and B = 16*WPH a fully unrolled path handles a whole frame: eight row steps
//     per warp, one transposed shuffle reduction for the eight dot products, one
//     block max, a rescale only when the max grows, and one shuffle per row step
//     to hand each lane its softmax weight.  Other shapes, and the partly filled
//     last frame of a sequence, take the generic path (xor reductions per step,
//     online update per chunk of steps).  Softmax runs in log2 units with
//     ex2.approx; all products and sums are fp32.
//   * Epilogue: row groups, then warps of a head (through shared memory, handed
//     over with mbarriers), are combined by the log-sum-exp rule.  A sequence that
//     fits in one partition is normalised and written directly; otherwise the
//     (m, l, o) partial goes to the workspace, an arrival counter per (sequence,
//     head) is bumped, and the warp that brings it to the partition count merges
//     all partials of that head and zeroes the counter -- no second kernel.
//   * Launched with programmatic stream serialisation: barrier set-up overlaps the
//     tail of the previous kernel; griddepcontrol.wait precedes every input read.
//   * Bad frame ids / context lengths: the affected output rows become zeros and a
//     sticky status bit is set.  Every wait is an mbarrier wait with a bound; a
//     wait that gives up sets PA_DEV_TIMEOUT, turns all later waits of the block
//     into no-ops, and the producer waits (again bounded) for its copies in
//     flight before the block retires.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa_internal.h"

namespace pa {
namespace dk {

constexpr unsigned kFull = 0xffffffffu;
// ~2 s at 2 GHz: far beyond any legitimate wait for one staged frame.
constexpr long long kWaitCycles = 4000000000LL;
constexpr long long kDrainCycles = 200000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Returns false when the block is aborting or the budget ran out
// (then the block is marked aborting and PA_DEV_TIMEOUT is raised).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(status, kDevTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- 16-byte chunk <-> fp32 ------------------------------------------------------------
template <typename T>
struct Chunk;

template <>
struct Chunk<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const void* p, float (&f)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ __forceinline__ static void store(void* p, const float (&f)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
  __device__ __forceinline__ static void store1(void* p, float f) { *reinterpret_cast<float*>(p) = f; }
};

template <>
struct Chunk<__half> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const void* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __half22float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ static void store(void* p, const float (&f)[8]) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
  __device__ __forceinline__ static void store1(void* p, float f) {
    *reinterpret_cast<__half*>(p) = __float2half_rn(f);
  }
};

template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const void* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static void store(void* p, const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
  __device__ __forceinline__ static void store1(void* p, float f) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(f);
  }
};

// ---- shared-memory layout (host and device agree) -------------------------------------------
struct Layout {
  uint32_t stage_pitch, bars, flags, offa, order, invpos, hist, comb, total;
  __host__ __device__ Layout(int stages, uint32_t stage_bytes, int S, int ncw, int D) {
    stage_pitch = (stage_bytes + 127u) & ~127u;
    // mbarriers: full[stages], empty[stages], item_full[2], item_empty[2], comb_full[4], comb_empty[4]
    bars = stages * stage_pitch;
    flags = bars + 16u * stages + 32u + 64u;          // poison[stages], abort, item_slot[2]
    offa = (flags + 4u * (stages + 3) + 15u) & ~15u;  // full-partition item offsets [S + 1]
    order = (offa + 4u * (S + 1) + 15u) & ~15u;       // sequences with a last partition, longest first [S]
    invpos = (order + 4u * S + 15u) & ~15u;           // position of a sequence in `order` [S]
    hist = (invpos + 4u * S + 15u) & ~15u;            // remainder buckets [32] + cursors [32]
    comb = hist + 256u;                               // combine scratch [ncw][D + 2]
    total = comb + 4u * ncw * (D + 2) + 128u;         // + slack for 128-byte base alignment
  }
};

// Validated context length, or -1.
__device__ __forceinline__ int valid_len(const DecodeArgs& a, int s) {
  const int L = a.context_lens[s];
  return (L < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks) * a.B) ? -1 : L;
}

// Number of partitions of a sequence: full ones, plus one shorter last partition
// when the length is not a multiple of P (an empty or invalid sequence has exactly
// one, empty, last partition).
__device__ __forceinline__ int full_parts(int Lv, int P) { return Lv / P; }
__device__ __forceinline__ int last_part(int Lv, int P) { return (Lv % P != 0 || Lv == 0) ? 1 : 0; }

// Largest s in [0, S) with off[s] <= x (off non-decreasing, off[0] = 0).
__device__ __forceinline__ int upper_seq(const int32_t* off, int S, int x) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct Item {
  int s, g, L;        // sequence, head group, validated length (-1 = invalid)
  int tok1, blk0, nblk;
  bool single;        // the sequence has one partition: write the output directly
};

__device__ __forceinline__ Item locate(const DecodeArgs& a, const int32_t* offa, const int32_t* order,
                                       int a_total, int P, int item) {
  Item it;
  int p;
  if (item < a_total) {
    it.s = upper_seq(offa, a.S, item);
    const int local = item - offa[it.s];
    p = local / a.G;
    it.g = local - p * a.G;
  } else {
    const int b = item - a_total;
    const int j = b / a.G;
    it.s = order[j];
    it.g = b - j * a.G;
    p = -1;  // the last partition
  }
  it.L = valid_len(a, it.s);
  const int Lv = it.L < 0 ? 0 : it.L;
  const int nf = full_parts(Lv, P);
  if (p < 0) p = nf;
  it.single = nf + last_part(Lv, P) == 1;
  const int tok0 = p * P;
  it.tok1 = min(Lv, tok0 + P);
  it.blk0 = tok0 / a.B;
  it.nblk = it.tok1 > tok0 ? (it.tok1 + a.B - 1) / a.B - it.blk0 : 0;
  return it;
}

// Online-softmax state of one consumer warp for one head: running max m (log2
// units, warp-uniform), l = sum of weights of this lane's row group, lf = weights
// gathered by the unrolled path (one row step per lane, folded into l at the end),
// o = weighted values of this lane's 16-byte chunk over its row group's tokens.
template <int VEC>
struct SoftState {
  float m, l, lf;
  float o[VEC];
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    l = 0.f;
    lf = 0.f;
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] = 0.f;
  }
  __device__ __forceinline__ void rescale(float m_new) {
    const float alpha = ex2(m - m_new);
    l *= alpha;
    lf *= alpha;
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] *= alpha;
    m = m_new;
  }
};

// Generic frame: any B, any valid-row count.  Rows are dealt to the WPH warps of a
// head in turn; online update once per CH row steps.
template <typename T, int D, int HG, int WPH>
__device__ __forceinline__ void frame_generic(SoftState<16 / sizeof(T)>& st, const float (&qv)[16 / sizeof(T)],
                                              const unsigned char* kst, const unsigned char* vst, int B,
                                              int n_valid, int w, int r) {
  constexpr int E = sizeof(T);
  constexpr int VEC = 16 / E;
  constexpr int LPR = D / VEC;
  constexpr int TPI = 32 / LPR;
  constexpr int CH = 8;
  constexpr uint32_t row_bytes = HG * D * E;
  const int NIT = (B + TPI - 1) / TPI;
  for (int it0 = w; it0 < NIT; it0 += WPH * CH) {
    float x[CH];
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const int it = it0 + u * WPH;
      const int t = it * TPI + r;
      float acc = 0.f;
      if (it < NIT) {
        if (t < n_valid) {
          float kv[VEC];
          Chunk<T>::load(kst + t * row_bytes, kv);
#pragma unroll
          for (int v = 0; v < VEC; ++v) acc = fmaf(qv[v], kv[v], acc);
        }
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
      }
      x[u] = (it < NIT && t < n_valid) ? acc : -INFINITY;
    }
    float cm = x[0];
#pragma unroll
    for (int u = 1; u < CH; ++u) cm = fmaxf(cm, x[u]);
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, off));
    if (cm > st.m) st.rescale(cm);   // warp-uniform
    if (st.m == -INFINITY) continue;  // nothing valid yet
#pragma unroll
    for (int u = 0; u < CH; ++u) {
      const int it = it0 + u * WPH;
      const int t = it * TPI + r;
      if (it < NIT && t < n_valid) {
        const float pw = ex2(x[u] - st.m);
        st.l += pw;
        float vv[VEC];
        Chunk<T>::load(vst + t * row_bytes, vv);
#pragma unroll
        for (int v = 0; v < VEC; ++v) st.o[v] = fmaf(pw, vv[v], st.o[v]);
      }
    }
  }
}

// Full frame of B = 16*WPH rows with 256-byte rows (16 lanes per row, 2 rows per
// warp step): warp w takes row steps 8w .. 8w+7, i.e. tokens 16w .. 16w+15.
template <typename T, int D, int HG>
__device__ __forceinline__ void frame_fast(SoftState<16 / sizeof(T)>& st, const float (&qv)[16 / sizeof(T)],
                                           const unsigned char* kst, const unsigned char* vst, int w, int r,
                                           int c) {
  constexpr int E = sizeof(T);
  constexpr int VEC = 16 / E;
  static_assert(D * E == 256, "fast path needs 256-byte rows");
  constexpr uint32_t row_bytes = HG * D * E;
  const unsigned char* kb = kst + (16 * w + r) * row_bytes;
  const unsigned char* vb = vst + (16 * w + r) * row_bytes;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float kv[VEC];
    Chunk<T>::load(kb + 2 * i * row_bytes, kv);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int v = 0; v < VEC; v += 2) {
      s0 = fmaf(qv[v], kv[v], s0);
      s1 = fmaf(qv[v + 1], kv[v + 1], s1);
    }
    acc[i] = s0 + s1;
  }
  // transposed reduction over the 16 lanes of the row group: afterwards lane c
  // holds the full dot product of row step (c >> 1) & 7.
  const bool b3 = (c & 8) != 0, b2 = (c & 4) != 0, b1 = (c & 2) != 0;
  float b[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = b3 ? acc[j] : acc[j + 4];
    const float keep = b3 ? acc[j + 4] : acc[j];
    b[j] = keep + __shfl_xor_sync(kFull, send, 8);
  }
  float d[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = b2 ? b[j] : b[j + 2];
    const float keep = b2 ? b[j + 2] : b[j];
    d[j] = keep + __shfl_xor_sync(kFull, send, 4);
  }
  float sc;
  {
    const float send = b1 ? d[0] : d[1];
    const float keep = b1 ? d[1] : d[0];
    sc = keep + __shfl_xor_sync(kFull, send, 2);
  }
  sc += __shfl_xor_sync(kFull, sc, 1);
  float bm = sc;
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, off));
  if (bm > st.m) st.rescale(bm);  // warp-uniform; rare once the running max settles
  const float p = ex2(sc - st.m);
  st.lf += p;
  const int src = (r << 4);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float pt = __shfl_sync(kFull, p, src | (2 * i));
    float vv[VEC];
    Chunk<T>::load(vb + 2 * i * row_bytes, vv);
#pragma unroll
    for (int v = 0; v < VEC; ++v) st.o[v] = fmaf(pt, vv[v], st.o[v]);
  }
}

// Log-sum-exp merge of the partitions of one (sequence, head), by one warp:
// out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p with M = max_p m_p (log2 units).
// Partition p of the sequence is item offa[s] + p*G + g (full partitions) or
// a_total + invpos[s]*G + g (the shorter last one).  Partials written by other
// thread blocks are read past L1.
template <typename T, int D, int HG>
__device__ __forceinline__ void merge_head(const DecodeArgs& a, const int32_t* offa, const int32_t* invpos,
                                           int a_total, int s, int g, int h, int head, int nf, int np, int lane,
                                           int c) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int LPR = D / VEC;
  auto item_of = [&](int p) { return p < nf ? offa[s] + p * a.G + g : a_total + invpos[s] * a.G + g; };
  // pass 1, lanes across partitions: M, bad flag
  float M = -INFINITY;
  bool bad = false;
  for (int p = lane; p < np; p += 32) {
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + (static_cast<int64_t>(item_of(p)) * HG + h) * 2));
    M = fmaxf(M, ml.x);
    bad |= ml.y < 0.f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  bad = __any_sync(kFull, bad);
  float num[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) num[v] = 0.f;
  float den = 0.f;
  if (!bad && M != -INFINITY) {
    // pass 2: weights computed lane-parallel, values accumulated by the chunk owners
    for (int p0 = 0; p0 < np; p0 += 32) {
      float wgt = 0.f, wl = 0.f;
      const int p = p0 + lane;
      if (p < np) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.ws_ml + (static_cast<int64_t>(item_of(p)) * HG + h) * 2));
        wgt = ex2(ml.x - M);
        wl = wgt * ml.y;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(kFull, wl, off);
      den += wl;
      const int n = min(32, np - p0);
      for (int j = 0; j < n; ++j) {
        const float sc = __shfl_sync(kFull, wgt, j);
        if (lane < LPR) {
          const float* src = a.ws_o + (static_cast<int64_t>(item_of(p0 + j)) * HG + h) * D + c * VEC;
#pragma unroll
          for (int v = 0; v < VEC; v += 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + v));
            num[v] = fmaf(sc, x.x, num[v]);
            num[v + 1] = fmaf(sc, x.y, num[v + 1]);
            num[v + 2] = fmaf(sc, x.z, num[v + 2]);
            num[v + 3] = fmaf(sc, x.w, num[v + 3]);
          }
        }
      }
    }
  }
  if (lane < LPR) {
    const bool zero = bad || !(den > 0.f);
    const float inv = zero ? 0.f : 1.f / den;
    float res[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) res[v] = zero ? 0.f : num[v] * inv;
    T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(s) * a.out_row + static_cast<int64_t>(head) * D + c * VEC;
    Chunk<T>::store(op, res);
  }
}

template <typename T, int D, int HG, int WPH, int BFAST>
__global__ void __launch_bounds__(32 * (HG * WPH + 1), (HG * WPH <= 4 ? 3 : 2))
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs a, const int stages) {
  constexpr int E = sizeof(T);
  constexpr int VEC = 16 / E;   // elements per 16-byte chunk
  constexpr int LPR = D / VEC;  // lanes per (token, head) row
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "unsupported head_dim");
  constexpr int NCW = HG * WPH;  // consumer warps
  static_assert(BFAST == 0 || (BFAST == 16 * WPH && D * E == 256), "fast path shape");

  const int B = a.B;
  const int R = a.R;                          // tokens per stage
  const int FPS = R > B ? R / B : 1;          // frames per stage
  const int SPF = B > R ? B / R : 1;          // stages per frame
  const uint32_t tile_bytes = static_cast<uint32_t>(R) * HG * D * E;
  const uint32_t stage_bytes = 2u * tile_bytes;
  const uint32_t box_bytes = static_cast<uint32_t>(R > B ? B : R) * HG * D * E;  // one copy (K or V)

  extern __shared__ unsigned char smem_raw[];
  const Layout lay(stages, stage_bytes, a.S, NCW, D);
  unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // 128-byte aligned
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + lay.bars;
  const uint32_t bar_empty = bar_full + 8u * stages;
  const uint32_t bar_ifull = bar_empty + 8u * stages;
  const uint32_t bar_iempty = bar_ifull + 16u;
  const uint32_t bar_cfull = bar_iempty + 16u;   // per head: warps 1.. of the head have written
  const uint32_t bar_cempty = bar_cfull + 32u;   // per head: warp 0 has read
  volatile int32_t* poison = reinterpret_cast<volatile int32_t*>(smem + lay.flags);
  volatile int32_t* abort_flag = poison + stages;
  volatile int32_t* item_slot = abort_flag + 1;
  int32_t* offa = reinterpret_cast<int32_t*>(smem + lay.offa);
  int32_t* order = reinterpret_cast<int32_t*>(smem + lay.order);
  int32_t* invpos = reinterpret_cast<int32_t*>(smem + lay.invpos);
  int32_t* hist = reinterpret_cast<int32_t*>(smem + lay.hist);
  float* comb = reinterpret_cast<float*>(smem + lay.comb);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- 0. shared-memory barriers, then wait for the previous kernel's writes -----------------
  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar_full + 8u * i, 1);
      mbar_init(bar_empty + 8u * i, NCW);
      poison[i] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_ifull + 8u * i, 1);
      mbar_init(bar_iempty + 8u * i, NCW);
    }
    for (int hh = 0; hh < HG; ++hh) {
      mbar_init(bar_cfull + 8u * hh, WPH > 1 ? WPH - 1 : 1);
      mbar_init(bar_cempty + 8u * hh, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == NCW && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- 1. partition length ------------------------------------------------------------------
  // Automatic: whole sequences when they already give every thread block work and
  // the longest is no longer than the average load per block (longest-first
  // scheduling then balances them); otherwise about target_items items of at least
  // min_part tokens, shortened so the longest sequence splits into equal parts.
  int P;
  {
    const int Lcap = a.max_blocks * B;
    if (a.fixed_part > 0) {
      P = a.fixed_part;
    } else {
      long long local = 0;
      int lmax = 0;
      for (int s = tid; s < a.S; s += blockDim.x) {
        const int L = valid_len(a, s);
        local += L > 0 ? L : 0;
        lmax = max(lmax, L);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        local += __shfl_xor_sync(kFull, local, o);
        lmax = max(lmax, __shfl_xor_sync(kFull, lmax, o));
      }
      long long* red = reinterpret_cast<long long*>(comb);
      int* redmax = reinterpret_cast<int*>(red + (blockDim.x >> 5));
      if (lane == 0) {
        red[warp] = local;
        redmax[warp] = lmax;
      }
      __syncthreads();
      long long total = 0;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        total += red[w];
        lmax = max(lmax, redmax[w]);
      }
      __syncthreads();
      const long long grid = gridDim.x;
      long long p;
      if (a.whole_first && static_cast<long long>(a.S) * a.G >= grid && lmax * grid <= total * a.G) {
        p = Lcap;
      } else {
        p = (total * a.G + a.target_items - 1) / (a.target_items > 0 ? a.target_items : 1);
        p = ((p + B - 1) / B) * B;
        if (p < a.min_part) p = a.min_part;
        if (p > Lcap) p = Lcap;
        if (lmax > p) {  // equal parts for the longest sequence
          const long long n = (lmax + p - 1) / p;
          const long long q = (((lmax + n - 1) / n + B - 1) / B) * B;
          if (q >= a.min_part) p = q;
        }
      }
      if (p < B) p = B;
      P = static_cast<int>(p);
    }
  }

  // ---- 2. work items: full partitions in sequence order, then the shorter last
  //      partitions ordered longest first (stable 32-bucket counting sort by length,
  //      identical in every thread block) ---------------------------------------------------
  for (int s = tid; s < a.S; s += blockDim.x) {
    const int L = valid_len(a, s);
    if (L < 0 && blockIdx.x == 0) atomicOr(a.status, kDevBadLen);
    const int Lv = L < 0 ? 0 : L;
    offa[s + 1] = full_parts(Lv, P) * a.G;
  }
  if (tid < 64) hist[tid] = 0;
  if (tid == 0) offa[0] = 0;
  __syncthreads();
  if (warp == 0) {  // prefix sum of the full-partition item counts
    int carry = 0;
    for (int base = 0; base < a.S; base += 32) {
      const int i = base + lane;
      int v = i < a.S ? offa[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      v += carry;
      if (i < a.S) offa[i + 1] = v;
      carry = __shfl_sync(kFull, v, 31);
    }
  } else if (warp == 1) {  // order of the last partitions
    auto bucket_of = [&](int s) {
      const int L = valid_len(a, s);
      const int Lv = L < 0 ? 0 : L;
      if (!last_part(Lv, P)) return -1;
      return min(31, static_cast<int>((static_cast<long long>(Lv % P) * 32) / P));
    };
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < a.S; base += 32) {
      const int s = base + lane;
      const int b = s < a.S ? bucket_of(s) : -1;
      const unsigned same = __match_any_sync(kFull, b);
      if (b >= 0 && (same & lt) == 0) hist[b] += __popc(same);
      __syncwarp();
    }
    // cursor[b] = number of entries in buckets above b (longest first)
    const int cnt = hist[31 - lane];
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += n;
    }
    hist[32 + (31 - lane)] = v - cnt;
    if (lane == 31) hist[31] = v;  // bucket 31's count is no longer needed: total entries
    __syncwarp();
    const int n_last = hist[31];
    __syncwarp();
    for (int base = 0; base < a.S; base += 32) {
      const int s = base + lane;
      const int b = s < a.S ? bucket_of(s) : -1;
      const unsigned same = __match_any_sync(kFull, b);
      if (b >= 0) {
        const int pos = hist[32 + b] + __popc(same & lt);
        order[pos] = s;
        invpos[s] = pos;
      }
      __syncwarp();
      if (b >= 0 && (same & lt) == 0) hist[32 + b] += __popc(same);
      __syncwarp();
    }
    if (lane == 0) hist[0] = n_last;
  }
  __syncthreads();
  const int a_total = offa[a.S];
  const int total_items = a_total + hist[0] * a.G;

  if (warp == NCW) {
    // ============================== producer warp ==============================
    int k = 0, ni = 0;
    uint32_t issued = 0;  // bit i: stage i holds copies not yet known complete
    while (true) {
      // An item is claimed only when the previous one is fully issued, so the
      // longest-first order is kept (claiming ahead would pin items to busy blocks).
      int item = 0;
      if (lane == 0) item = *abort_flag ? total_items : atomicAdd(a.sched, 1);
      item = __shfl_sync(kFull, item, 0);
      const bool done = item >= total_items;
      if (lane == 0) {
        const int sl = ni & 1;
        if (mbar_wait(bar_iempty + 8u * sl, static_cast<uint32_t>((ni >> 1) & 1) ^ 1u, abort_flag, a.status)) {
          item_slot[sl] = done ? -1 : item;
          mbar_arrive(bar_ifull + 8u * sl);
        }
      }
      ++ni;
      if (done) break;
      const Item it = locate(a, offa, order, a_total, P, item);
      const int32_t* row = a.block_tables + static_cast<int64_t>(it.s) * a.bt_row + it.blk0;
      // staged units of this item: R tokens each (FPS frames, or one slice of a frame)
      const int ntok = it.tok1 - it.blk0 * B;
      const int nvf = ntok > 0 ? (ntok + R - 1) / R : 0;
      int chunk = -1, frame = -1;  // lane-distributed block-table slice, 32 frames
      for (int vf = 0; vf < nvf; ++vf, ++k) {
        const int f0 = FPS > 1 ? vf * FPS : vf / SPF;  // first frame of the unit (item-relative)
        const int nf = FPS > 1 ? min(FPS, it.nblk - f0) : 1;
        if ((f0 >> 5) != chunk) {  // FPS divides 32: a unit never straddles two slices
          chunk = f0 >> 5;
          const int jj = chunk * 32 + lane;
          frame = jj < it.nblk ? row[jj] : 0;
          const bool bad = (jj < it.nblk) && (frame < 0 || frame >= a.num_blocks);
          if (__ballot_sync(kFull, bad) != 0u && lane == 0) atomicOr(a.status, kDevBadBlock);
        }
        const int fr = __shfl_sync(kFull, frame, (f0 & 31) + (lane < nf ? lane : 0));
        const bool poisoned = __ballot_sync(kFull, lane < nf && (fr < 0 || fr >= a.num_blocks)) != 0u;
        const int st = k % stages;
        const uint32_t ph = static_cast<uint32_t>(k / stages) & 1u;
        int go = 0;
        if (lane == 0) {
          if (mbar_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.status)) {
            if (poisoned) {
              poison[st] = 1;
              mbar_arrive(bar_full + 8u * st);
              issued &= ~(1u << st);
            } else {
              poison[st] = 0;
              mbar_arrive_expect_tx(bar_full + 8u * st, 2u * box_bytes * nf);
              issued |= 1u << st;
              go = 1;
            }
          } else {
            issued &= ~(1u << st);
          }
        }
        go = __shfl_sync(kFull, go, 0);
        if (go && lane < nf) {
          const uint32_t dst = sbase + st * lay.stage_pitch + lane * box_bytes;
          const int r0 = fr * B + (SPF > 1 ? (vf % SPF) * R : 0);
          tma_load_3d(dst, &tmap_k, 0, it.g * HG, r0, bar_full + 8u * st);
          tma_load_3d(dst + tile_bytes, &tmap_v, 0, it.g * HG, r0, bar_full + 8u * st);
        }
      }
    }
    if (lane == 0) {
      // An aborting block may still have copies landing in shared memory: wait for
      // them (bounded) before the block retires.
      if (*abort_flag) {
        for (int kk = (k > stages ? k - stages : 0); kk < k; ++kk) {
          const int st = kk % stages;
          if (!(issued & (1u << st))) continue;
          const uint32_t ph = static_cast<uint32_t>(kk / stages) & 1u;
          const long long t0 = clock64();
          while (!mbar_try_wait(bar_full + 8u * st, ph) && clock64() - t0 < kDrainCycles) {
          }
        }
      }
      // Retire: the last block to finish taking items resets the counters.
      __threadfence();
      if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        a.sched[0] = 0;
        a.sched[1] = 0;
        __threadfence();
      }
    }
    return;
  }

  // ============================== consumer warps ==============================
  const int h = warp / WPH;  // head within the group
  const int w = warp % WPH;  // share of rows within the head
  const int r = lane / LPR;  // row group within the warp
  const int c = lane % LPR;  // 16-byte chunk within the row
  const unsigned char* const stage0 = smem;
  int k = 0, ni = 0, nc = 0;
  SoftState<VEC> st;

  while (true) {
    const int sl = ni & 1;
    const bool got =
        __all_sync(kFull, mbar_wait(bar_ifull + 8u * sl, static_cast<uint32_t>((ni >> 1) & 1), abort_flag, a.status));
    const int item = got ? item_slot[sl] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_iempty + 8u * sl);
    ++ni;
    if (item < 0) break;
    const Item it = locate(a, offa, order, a_total, P, item);
    const int head = it.g * HG + h;

    float qv[VEC];
    {
      const T* qp = reinterpret_cast<const T*>(a.q) + static_cast<int64_t>(it.s) * a.q_row +
                    static_cast<int64_t>(head) * D + c * VEC;
      Chunk<T>::load(qp, qv);
#pragma unroll
      for (int v = 0; v < VEC; ++v) qv[v] *= a.qk_scale_log2;
    }
    st.reset();
    bool poisoned = it.L < 0;

    const int ntok = it.tok1 - it.blk0 * B;
    const int nvf = ntok > 0 ? (ntok + R - 1) / R : 0;
    for (int j = 0; j < nvf; ++j, ++k) {
      const int s_ = k % stages;
      const uint32_t ph = static_cast<uint32_t>(k / stages) & 1u;
      const bool ok = __all_sync(kFull, mbar_wait(bar_full + 8u * s_, ph, abort_flag, a.status));
      if (!ok || poison[s_]) poisoned = true;
      if (!poisoned) {
        const int n_valid = min(R, ntok - j * R);
        const unsigned char* kst = stage0 + s_ * lay.stage_pitch + (h * D + c * VEC) * E;
        const unsigned char* vst = kst + tile_bytes;
        if constexpr (BFAST > 0) {
          if (n_valid == BFAST) {
            frame_fast<T, D, HG>(st, qv, kst, vst, w, r, c);
          } else {
            frame_generic<T, D, HG, WPH>(st, qv, kst, vst, R, n_valid, w, r);
          }
        } else {
          frame_generic<T, D, HG, WPH>(st, qv, kst, vst, R, n_valid, w, r);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8u * s_);
    }

    // ---- epilogue: fold the unrolled path's weights, combine row groups, then warps ----
    if constexpr (BFAST > 0) {
      float lf = st.lf;
#pragma unroll
      for (int off = 2; off < LPR; off <<= 1) lf += __shfl_xor_sync(kFull, lf, off);
      st.l += lf;
    }
    float l = st.l, m = st.m;
    float o[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] = st.o[v];
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
      l += __shfl_xor_sync(kFull, l, off);
#pragma unroll
      for (int v = 0; v < VEC; ++v) o[v] += __shfl_xor_sync(kFull, o[v], off);
    }
    if constexpr (WPH > 1) {
      const uint32_t cph = static_cast<uint32_t>(nc & 1);
      float* mine = comb + (h * WPH + w) * (D + 2);
      if (w > 0) {
        // wait until warp 0 has read the previous item's states, then publish ours
        const bool free_ok =
            __all_sync(kFull, mbar_wait(bar_cempty + 8u * h, cph ^ 1u, abort_flag, a.status));
        if (free_ok && lane < LPR) {
#pragma unroll
          for (int v = 0; v < VEC; ++v) mine[c * VEC + v] = o[v];
          if (c == 0) {
            mine[D] = m;
            mine[D + 1] = l;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cfull + 8u * h);
      } else {
        const bool have = __all_sync(kFull, mbar_wait(bar_cfull + 8u * h, cph, abort_flag, a.status));
        if (!have) poisoned = true;
        float M = m;
#pragma unroll
        for (int ww = 1; ww < WPH; ++ww) M = fmaxf(M, comb[(h * WPH + ww) * (D + 2) + D]);
        if (M != -INFINITY) {
          const float s0 = ex2(m - M);
          l *= s0;
#pragma unroll
          for (int v = 0; v < VEC; ++v) o[v] *= s0;
#pragma unroll
          for (int ww = 1; ww < WPH; ++ww) {
            const float* src = comb + (h * WPH + ww) * (D + 2);
            const float sc = ex2(src[D] - M);
            l = fmaf(sc, src[D + 1], l);
#pragma unroll
            for (int v = 0; v < VEC; ++v) o[v] = fmaf(sc, src[c * VEC + v], o[v]);
          }
        }
        m = M;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_cempty + 8u * h);
      }
      ++nc;
    }
    if (w == 0) {
      if (it.single) {
        if (lane < LPR) {
          float res[VEC];
          const bool zero = poisoned || !(l > 0.f);
          const float inv = zero ? 0.f : 1.f / l;
#pragma unroll
          for (int v = 0; v < VEC; ++v) res[v] = zero ? 0.f : o[v] * inv;
          T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(it.s) * a.out_row +
                  static_cast<int64_t>(head) * D + c * VEC;
          Chunk<T>::store(op, res);
        }
      } else {
        if (lane < LPR) {
          float* wo = a.ws_o + (static_cast<int64_t>(item) * HG + h) * D + c * VEC;
#pragma unroll
          for (int v = 0; v < VEC; v += 4)
            *reinterpret_cast<float4*>(wo + v) = make_float4(o[v], o[v + 1], o[v + 2], o[v + 3]);
          if (c == 0)
            *reinterpret_cast<float2*>(a.ws_ml + (static_cast<int64_t>(item) * HG + h) * 2) =
                make_float2(m, poisoned ? -1.f : l);
        }
        // Publish the partial, count it; the last partition of (sequence, head) to
        // arrive merges all of them and resets the counter for the next launch.
        __threadfence();
        __syncwarp();
        const int Lv = it.L < 0 ? 0 : it.L;
        const int nf = full_parts(Lv, P);
        const int np = nf + last_part(Lv, P);
        int32_t* cnt = a.ws_cnt + static_cast<int64_t>(it.s) * a.H + head;
        int last = 0;
        if (lane == 0) last = atomicAdd(cnt, 1) == np - 1;
        if (__shfl_sync(kFull, last, 0)) {
          __threadfence();
          merge_head<T, D, HG>(a, offa, invpos, a_total, it.s, it.g, h, head, nf, np, lane, c);
          if (lane == 0) *cnt = 0;
        }
      }
    }
  }
}

// ---- host-side launcher for one element type ----------------------------------------------
template <typename T, int D, int HG, int WPH, int BFAST>
cudaError_t launch_one(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream, bool query_only, int* max_ctas) {
  constexpr int NCW = HG * WPH;
  const uint32_t stage_bytes = 2u * static_cast<uint32_t>(a.R) * HG * D * sizeof(T);
  const Layout lay(c.stages, stage_bytes, a.S, NCW, D);
  const size_t smem = lay.total;
  auto kern = decode_kernel<T, D, HG, WPH, BFAST>;
  int n = 0;
  cudaError_t e = kernel_prep(reinterpret_cast<const void*>(kern), 32 * (NCW + 1), smem, &n);
  if (e != cudaSuccess) return e;
  if (query_only) {
    if (max_ctas) *max_ctas = n;
    return e;
  }
  // Programmatic dependent launch: the grid may start while the previous kernel on
  // the stream drains; it waits (griddepcontrol.wait) before reading any input.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.grid);
  cfg.blockDim = dim3(32 * (NCW + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a, c.stages);
}

template <typename T, int D>
cudaError_t launch_d(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream, bool query_only, int* max_ctas) {
  constexpr bool kFastRows = D * sizeof(T) == 256;
  const bool fast = kFastRows && c.fast && (a.R == 16 * c.warps_per_head);
#define PA_DK_CASE(hg, wph)                                                                         \
  if (c.heads_per_cta == hg && c.warps_per_head == wph) {                                           \
    if constexpr (kFastRows && (wph == 1 || wph == 2))                                              \
      if (fast) return launch_one<T, D, hg, wph, 16 * wph>(a, c, tk, tv, stream, query_only, max_ctas); \
    return launch_one<T, D, hg, wph, 0>(a, c, tk, tv, stream, query_only, max_ctas);                \
  }
  PA_DK_CASE(1, 1) PA_DK_CASE(1, 2) PA_DK_CASE(1, 4) PA_DK_CASE(1, 8)
  PA_DK_CASE(2, 1) PA_DK_CASE(2, 2) PA_DK_CASE(2, 4)
  PA_DK_CASE(4, 1) PA_DK_CASE(4, 2)
#undef PA_DK_CASE
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_dtype(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                         cudaStream_t stream, bool query_only, int* max_ctas) {
  switch (c.D) {
    case 64: return launch_d<T, 64>(a, c, tk, tv, stream, query_only, max_ctas);
    case 128: return launch_d<T, 128>(a, c, tk, tv, stream, query_only, max_ctas);
    case 256:
      if constexpr (sizeof(T) == 2) return launch_d<T, 256>(a, c, tk, tv, stream, query_only, max_ctas);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dk
}  // namespace pa
