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
//     persistent grid of thread blocks walks the item list round-robin; the
//     partition length is chosen on the device from the actual context lengths
//     so that there are a few items per thread block.  Items of one sequence are
//     adjacent, so the K/V rows a thread block streams sit next to those of the
//     blocks working beside it.
//   * One producer warp: reads the item's block-table slice (one coalesced load
//     per 32 frames), bounds-checks every frame id, and for each frame issues two
//     3-D TMA tile loads (K and V: box {D, HG, B} of the [num_blocks*B, H, D] view)
//     into a ring of `stages` shared-memory buffers, completing on an mbarrier.
//   * HG*WPH consumer warps: warp (h, w) owns head h and every WPH-th group of
//     rows of each staged frame.  A row (one token, one head) is read as 16-byte
//     chunks by LPR = D*elem/16 lanes, so a warp covers TPI = 32/LPR tokens per
//     step with conflict-free shared-memory reads.  Dot products are reduced with
//     xor shuffles inside each row group; the softmax is online (running max m and
//     sum l in log2 units, ex2.approx) and the value accumulation is fp32.
//   * Epilogue: row groups, then warps of a head, are combined with the same
//     log-sum-exp rule.  A sequence that fits in one partition is normalised and
//     written directly; otherwise the (m, l, o) partial goes to the workspace and
//     merge_kernel combines the partitions.
//   * Bad frame ids / context lengths: the affected output rows become zeros and a
//     sticky status bit is set.  Every mbarrier wait is bounded; a wait that gives
//     up sets PA_DEV_TIMEOUT, turns all later waits of the block into no-ops and
//     the producer waits (again bounded) for its copies in flight before exiting.
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
  uint32_t stage_pitch, bars, flags, offs, comb, total;
  __host__ __device__ Layout(int stages, uint32_t stage_bytes, int S, int ncw, int D) {
    stage_pitch = (stage_bytes + 127u) & ~127u;
    bars = stages * stage_pitch;                    // full[stages], empty[stages]
    flags = bars + 16u * stages;                    // poison[stages], abort
    offs = (flags + 4u * (stages + 1) + 15u) & ~15u;  // item offsets [S + 1]
    comb = (offs + 4u * (S + 1) + 15u) & ~15u;      // combine scratch [ncw][D + 2]
    total = comb + 4u * ncw * (D + 2) + 128u;       // + slack for 128-byte base alignment
  }
};

// Partition count of one sequence (1 for an empty or invalid length).
__device__ __forceinline__ int parts_of(int L, int P) { return L <= P ? 1 : (L + P - 1) / P; }

// Validated context length, or -1.
__device__ __forceinline__ int valid_len(const DecodeArgs& a, int s) {
  const int L = a.context_lens[s];
  return (L < 0 || static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks) * a.B) ? -1 : L;
}

template <typename T, int D, int HG, int WPH>
__global__ void __launch_bounds__(32 * (HG * WPH + 1), 2)
    decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs a, const int stages) {
  constexpr int E = sizeof(T);
  constexpr int VEC = 16 / E;   // elements per 16-byte chunk
  constexpr int LPR = D / VEC;  // lanes per (token, head) row
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "unsupported head_dim");
  constexpr int TPI = 32 / LPR;  // rows per warp step
  constexpr int NCW = HG * WPH;  // consumer warps
  constexpr int CH = 8;          // row steps per online-softmax update

  const int B = a.B;
  const uint32_t tile_bytes = static_cast<uint32_t>(B) * HG * D * E;
  const uint32_t stage_bytes = 2u * tile_bytes;
  const uint32_t row_bytes = HG * D * E;  // one token's HG heads inside a staged tile

  extern __shared__ unsigned char smem_raw[];
  const Layout lay(stages, stage_bytes, a.S, NCW, D);
  unsigned char* smem =
      smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);  // 128-byte aligned base
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + lay.bars;
  const uint32_t bar_empty = bar_full + 8u * stages;
  volatile int32_t* poison = reinterpret_cast<volatile int32_t*>(smem + lay.flags);
  volatile int32_t* abort_flag = poison + stages;
  int32_t* item_off = reinterpret_cast<int32_t*>(smem + lay.offs);
  float* comb = reinterpret_cast<float*>(smem + lay.comb);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- 1. per-sequence item counts, partition length, prefix offsets ------------------------
  int P;
  {
    const int Lcap = a.max_blocks * B;
    if (a.fixed_part > 0) {
      P = a.fixed_part;
    } else {
      // total valid tokens (block-wide reduction through the combine scratch)
      long long local = 0;
      for (int s = tid; s < a.S; s += blockDim.x) {
        const int L = valid_len(a, s);
        local += L > 0 ? L : 0;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(kFull, local, o);
      long long* red = reinterpret_cast<long long*>(comb);
      if (lane == 0) red[warp] = local;
      __syncthreads();
      long long total = 0;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += red[w];
      __syncthreads();
      long long p = (total * a.G + a.target_items - 1) / (a.target_items > 0 ? a.target_items : 1);
      p = ((p + B - 1) / B) * B;
      if (p < a.min_part) p = a.min_part;
      if (p > Lcap) p = Lcap;
      if (p < B) p = B;
      P = static_cast<int>(p);
    }
  }
  for (int s = tid; s < a.S; s += blockDim.x) {
    const int L = valid_len(a, s);
    if (L < 0 && blockIdx.x == 0) atomicOr(a.status, kDevBadLen);
    item_off[s + 1] = parts_of(L < 0 ? 0 : L, P) * a.G;
  }
  if (tid == 0) {
    item_off[0] = 0;
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar_full + 8u * i, 1);
      mbar_init(bar_empty + 8u * i, NCW);
      poison[i] = 0;
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == NCW && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  __syncthreads();
  if (warp == 0) {  // inclusive scan of item counts
    int carry = 0;
    for (int base = 0; base < a.S; base += 32) {
      const int i = base + lane;
      int v = i < a.S ? item_off[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      v += carry;
      if (i < a.S) item_off[i + 1] = v;
      carry = __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
  const int total_items = item_off[a.S];
  if (blockIdx.x == 0 && a.ws_off != nullptr) {
    for (int i = tid; i <= a.S; i += blockDim.x) a.ws_off[i] = item_off[i];
    if (tid == 0) a.ws_off[a.S + 1] = P;
  }

  // item -> (s, p, g), token range and frame range
  auto locate = [&](int item, int& s, int& p, int& g, int& L, int& tok1, int& blk0, int& nblk, bool& single) {
    int lo = 0, hi = a.S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (item_off[mid] <= item) lo = mid; else hi = mid - 1;
    }
    s = lo;
    const int local = item - item_off[s];
    p = local / a.G;
    g = local - p * a.G;
    L = valid_len(a, s);
    const int Le = L < 0 ? 0 : L;
    single = parts_of(Le, P) == 1;
    const int tok0 = p * P;
    tok1 = min(Le, tok0 + P);
    blk0 = tok0 / B;
    nblk = tok1 > tok0 ? (tok1 + B - 1) / B - blk0 : 0;
  };

  if (warp == NCW) {
    // ============================== producer warp ==============================
    int k = 0;
    uint32_t issued = 0;  // bit i: stage i holds copies not yet known complete
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
      int s, p, g, L, tok1, blk0, nblk;
      bool single;
      locate(item, s, p, g, L, tok1, blk0, nblk, single);
      const int32_t* row = a.block_tables + static_cast<int64_t>(s) * a.bt_row + blk0;
      for (int j0 = 0; j0 < nblk; j0 += 32) {
        const int jj = j0 + lane;
        int frame = -1;
        if (jj < nblk) frame = row[jj];
        const bool bad = (jj < nblk) && (frame < 0 || frame >= a.num_blocks);
        if (__ballot_sync(kFull, bad) != 0u && lane == 0) atomicOr(a.status, kDevBadBlock);
        const int cnt = min(32, nblk - j0);
        for (int j = 0; j < cnt; ++j, ++k) {
          const int fr = __shfl_sync(kFull, frame, j);
          if (lane == 0) {
            const int st = k % stages;
            const uint32_t ph = static_cast<uint32_t>(k / stages) & 1u;
            if (mbar_wait(bar_empty + 8u * st, ph ^ 1u, abort_flag, a.status)) {
              if (fr < 0 || fr >= a.num_blocks) {
                poison[st] = 1;
                mbar_arrive(bar_full + 8u * st);
                issued &= ~(1u << st);
              } else {
                poison[st] = 0;
                const uint32_t dst = sbase + st * lay.stage_pitch;
                mbar_arrive_expect_tx(bar_full + 8u * st, stage_bytes);
                tma_load_3d(dst, &tmap_k, 0, g * HG, fr * B, bar_full + 8u * st);
                tma_load_3d(dst + tile_bytes, &tmap_v, 0, g * HG, fr * B, bar_full + 8u * st);
                issued |= 1u << st;
              }
            } else {
              issued &= ~(1u << st);
            }
          }
        }
      }
    }
    // If the block is aborting, copies may still be landing in shared memory:
    // wait for them (bounded) before the block retires.
    if (lane == 0 && *abort_flag) {
      for (int kk = (k > stages ? k - stages : 0); kk < k; ++kk) {
        const int st = kk % stages;
        if (!(issued & (1u << st))) continue;
        const uint32_t ph = static_cast<uint32_t>(kk / stages) & 1u;
        const long long t0 = clock64();
        while (!mbar_try_wait(bar_full + 8u * st, ph) && clock64() - t0 < kDrainCycles) {
        }
      }
    }
    return;
  }

  // ============================== consumer warps ==============================
  const int h = warp / WPH;  // head within the group
  const int w = warp % WPH;  // row-step slot within the head
  const int r = lane / LPR;  // row group within the warp
  const int c = lane % LPR;  // 16-byte chunk within the row
  const int NIT = (B + TPI - 1) / TPI;
  const unsigned char* const stage0 = smem;
  int k = 0;

  for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
    int s, p, g, L, tok1, blk0, nblk;
    bool single;
    locate(item, s, p, g, L, tok1, blk0, nblk, single);
    const int head = g * HG + h;

    float qv[VEC];
    {
      const T* qp = reinterpret_cast<const T*>(a.q) + static_cast<int64_t>(s) * a.q_row +
                    static_cast<int64_t>(head) * D + c * VEC;
      Chunk<T>::load(qp, qv);
#pragma unroll
      for (int v = 0; v < VEC; ++v) qv[v] *= a.qk_scale_log2;
    }
    float m = -INFINITY, l = 0.f;
    float o[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) o[v] = 0.f;
    bool poisoned = (L < 0);

    for (int j = 0; j < nblk; ++j, ++k) {
      const int st = k % stages;
      const uint32_t ph = static_cast<uint32_t>(k / stages) & 1u;
      const bool got = __all_sync(kFull, mbar_wait(bar_full + 8u * st, ph, abort_flag, a.status));
      if (!got) poisoned = true;
      if (got && poison[st]) poisoned = true;
      if (got && !poisoned) {
        const int n_valid = min(B, tok1 - (blk0 + j) * B);
        const unsigned char* kst = stage0 + st * lay.stage_pitch + (h * D + c * VEC) * E;
        const unsigned char* vst = kst + tile_bytes;
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
          const float m_new = fmaxf(m, cm);
          if (m_new == -INFINITY) continue;  // nothing valid yet (warp-uniform)
          const float alpha = ex2(m - m_new);
          l *= alpha;
#pragma unroll
          for (int v = 0; v < VEC; ++v) o[v] *= alpha;
          m = m_new;
#pragma unroll
          for (int u = 0; u < CH; ++u) {
            const int it = it0 + u * WPH;
            const int t = it * TPI + r;
            const float pw = ex2(x[u] - m);
            if (it < NIT && t < n_valid) {
              l += pw;
              float vv[VEC];
              Chunk<T>::load(vst + t * row_bytes, vv);
#pragma unroll
              for (int v = 0; v < VEC; ++v) o[v] = fmaf(pw, vv[v], o[v]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8u * st);
    }

    // ---- epilogue: combine row groups, then warps of the head -------------------------------
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
      l += __shfl_xor_sync(kFull, l, off);
#pragma unroll
      for (int v = 0; v < VEC; ++v) o[v] += __shfl_xor_sync(kFull, o[v], off);
    }
    if constexpr (WPH > 1) {
      named_bar(1, NCW * 32);  // previous item's readers are done with the scratch
      float* mine = comb + (h * WPH + w) * (D + 2);
      if (lane < LPR) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) mine[c * VEC + v] = o[v];
        if (c == 0) {
          mine[D] = m;
          mine[D + 1] = l;
        }
      }
      named_bar(1, NCW * 32);
      if (w == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < WPH; ++ww) M = fmaxf(M, comb[(h * WPH + ww) * (D + 2) + D]);
        l = 0.f;
#pragma unroll
        for (int v = 0; v < VEC; ++v) o[v] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int ww = 0; ww < WPH; ++ww) {
            const float* src = comb + (h * WPH + ww) * (D + 2);
            const float sc = ex2(src[D] - M);
            l = fmaf(sc, src[D + 1], l);
            if (lane < LPR) {
#pragma unroll
              for (int v = 0; v < VEC; ++v) o[v] = fmaf(sc, src[c * VEC + v], o[v]);
            }
          }
        }
        m = M;
      }
    }
    if (w == 0 && lane < LPR) {
      if (single) {
        float res[VEC];
        const bool zero = poisoned || !(l > 0.f);
        const float inv = zero ? 0.f : 1.f / l;
#pragma unroll
        for (int v = 0; v < VEC; ++v) res[v] = zero ? 0.f : o[v] * inv;
        T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(s) * a.out_row +
                static_cast<int64_t>(head) * D + c * VEC;
        Chunk<T>::store(op, res);
      } else {
        float* wo = a.ws_o + (static_cast<int64_t>(item) * HG + h) * D + c * VEC;
#pragma unroll
        for (int v = 0; v < VEC; ++v) wo[v] = o[v];
        if (c == 0) {
          float* wml = a.ws_ml + (static_cast<int64_t>(item) * HG + h) * 2;
          wml[0] = m;
          wml[1] = poisoned ? -1.f : l;
        }
      }
    }
  }
}

// Log-sum-exp merge of the partitions of every split (sequence, head).
// out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p, M = max_p m_p (log2 units).
template <typename T, int D>
__global__ void __launch_bounds__(D) merge_kernel(const DecodeArgs a, const int HG) {
  const int s = blockIdx.x / a.H;
  const int head = blockIdx.x - s * a.H;
  const int d = threadIdx.x;
  const int L = valid_len(a, s);
  if (L < 0) return;
  const int P = a.ws_off[a.S + 1];
  const int np = parts_of(L, P);
  if (np <= 1) return;
  const int g = head / HG;
  const int h = head - g * HG;
  const int base = a.ws_off[s] + g;
  float M = -INFINITY;
  bool bad = false;
  for (int p = 0; p < np; ++p) {
    const float* ml = a.ws_ml + (static_cast<int64_t>(base + p * a.G) * HG + h) * 2;
    M = fmaxf(M, ml[0]);
    bad |= ml[1] < 0.f;
  }
  float num = 0.f, den = 0.f;
  if (!bad && M != -INFINITY) {
    for (int p = 0; p < np; ++p) {
      const int64_t it = static_cast<int64_t>(base + p * a.G) * HG + h;
      const float sc = ex2(a.ws_ml[it * 2] - M);
      den = fmaf(sc, a.ws_ml[it * 2 + 1], den);
      num = fmaf(sc, a.ws_o[it * D + d], num);
    }
  }
  const float res = (bad || !(den > 0.f)) ? 0.f : num / den;
  T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(s) * a.out_row + static_cast<int64_t>(head) * D + d;
  Chunk<T>::store1(op, res);
}

// ---- host-side launcher for one element type ----------------------------------------------
template <typename T, int D, int HG, int WPH>
cudaError_t launch_one(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream, bool query_only, int* max_ctas) {
  constexpr int NCW = HG * WPH;
  const uint32_t stage_bytes = 2u * static_cast<uint32_t>(a.B) * HG * D * sizeof(T);
  const Layout lay(c.stages, stage_bytes, a.S, NCW, D);
  const size_t smem = lay.total;
  auto kern = decode_kernel<T, D, HG, WPH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (query_only) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * (NCW + 1), smem);
    if (max_ctas) *max_ctas = n;
    return e;
  }
  kern<<<c.grid, 32 * (NCW + 1), smem, stream>>>(tk, tv, a, c.stages);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.ws_off == nullptr) return e;
  merge_kernel<T, D><<<a.S * a.H, D, 0, stream>>>(a, HG);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_d(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream, bool query_only, int* max_ctas) {
#define PA_DK_CASE(hg, wph)                                                          \
  if (c.heads_per_cta == hg && c.warps_per_head == wph)                              \
    return launch_one<T, D, hg, wph>(a, c, tk, tv, stream, query_only, max_ctas);
  PA_DK_CASE(1, 4) PA_DK_CASE(1, 8)
  PA_DK_CASE(2, 2) PA_DK_CASE(2, 4)
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
