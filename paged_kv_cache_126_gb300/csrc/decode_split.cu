// Decode attention over the split cache layout of the kernel signature printed in
// "PagedAttention: Virtual Memory Guide for LLM Inference", "3. PagedAttention CUDA
// Kernel Execution": k_cache [num_blocks, H, D/x, B, x] and v_cache
// [num_blocks, H, D, B], x = elements per 16 bytes.  It computes what pa_decode
// computes ("Solving the LLM Memory Wall", "1. The Mathematical Foundation"):
// out = sum_j softmax(q . k_j * scale) v_j over the sequence's tokens.
//
// Design (one producer warp and HG consumer warps per block, persistent grid,
// dynamic work counter):
//   * Work item = (sequence, group of HG heads, context partition of P tokens); HG = 4,
//     or 2 where a frame of 4 heads would make a stage larger than 48 KB (D = 128,
//     B = 32), so that a block still holds three stages and two blocks fit an SM.  In
//     this layout the K (and the V) of one frame for HG consecutive heads is one
//     contiguous run of HG*D*B elements, so the producer stages a frame with two
//     bulk copies (cp.async.bulk) into a ring of stages completing on mbarriers.
//   * Consumer warp = one head.  Keys: lane (t, ph) = (lane mod B, lane / B) holds
//     q chunks ph, ph + 32/B, ... (16 bytes each) and reads the same chunks of token
//     t; one warp step reads 32 consecutive 16-byte chunks of shared memory (the
//     layout's purpose: consecutive lanes, consecutive addresses), then the chunk
//     phases are summed by shuffles.  Values: lane owns output elements
//     d = lane + 32 j and reads the B weights' rows v[d][0..B-1].  Online softmax in
//     log2 units with a rescale when the running max grows.
//   * NP > 1: unnormalised partials (max, sum, output) go to the workspace and a
//     second kernel combines them per (sequence, head) by log-sum-exp.
//   * Every wait is bounded (PA_DEV_TIMEOUT, then the block's later waits are
//     no-ops); frame ids outside [0, num_blocks) and lengths beyond the block table
//     set status bits and read as no tokens.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace sk {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;
constexpr long long kDrainCycles = 200000000LL;

template <typename T, int D, int B, int HG>
struct Geo {
  static constexpr int E = sizeof(T);
  static constexpr int X = 16 / E;                       // elements per 16-byte chunk
  static constexpr int NC = D / X;                       // chunks per head row
  static constexpr int PH = 32 / B;                      // lanes per token
  static constexpr int STEPS = NC / PH;                  // chunks per lane
  static constexpr int ND = D / 32;                      // output elements per lane (final rows)
  static constexpr int C = B / X;                        // 16-byte chunks per V row [D][B]
  static constexpr int RPI = 32 / C;                     // V rows one warp-wide read covers
  static constexpr int NR = D / RPI;                     // V rows each lane accumulates (part of)
  static constexpr uint32_t HEAD = D * B * E;            // one head of one frame (K or V)
  static constexpr uint32_t STAGE = 2 * HG * HEAD;       // K of HG heads, then V of HG heads
  static constexpr int NST = (96 * 1024 / STAGE) < 2 ? 2 : ((96 * 1024 / STAGE) > 6 ? 6 : 96 * 1024 / STAGE);
  static constexpr uint32_t BAR_OFF = NST * STAGE;       // [NST full][NST empty][2 item full][2 item empty]
  static constexpr uint32_t MISC_OFF = BAR_OFF + 8 * (2 * NST + 4);
  static constexpr uint32_t ORDER_OFF = (MISC_OFF + 4 * (4 + NST) + 15) & ~15u;  // [64] histogram, [1], [S] order
  static constexpr uint32_t SMEM = ORDER_OFF + 128;  // + 4 * (65 + S) when the items are ordered
  static_assert(PH * B == 32 && STEPS * PH == NC, "B must divide 32 and the chunk count");
  static_assert(C * RPI == 32 && NR * RPI == D, "V rows must tile the warp");
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (*abort_flag) return false;
    if (mbar_try(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(status, kDevTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}
// Contiguous global -> shared copy completing on an mbarrier (16-byte aligned, size
// a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__half>(const __half* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

struct Item {
  int s, g, p, t0, t1;  // tokens t0 .. t1-1 of sequence s, head group g, partition p
};
// order: sequence of each rank (longest first) when a.longest_first, else unused
template <int HG>
__device__ __forceinline__ Item locate(const SplitArgs& a, const int32_t* order, int item) {
  Item it;
  const int groups = a.H / HG;
  it.p = item % a.NP;
  const int sg = item / a.NP;
  it.g = sg % groups;
  it.s = a.longest_first ? order[sg / groups] : sg / groups;
  const int L = a.context_lens[it.s];  // lengths past the block table are cut by the callers
  it.t0 = it.p * a.P;
  it.t1 = min(max(L, 0), it.t0 + a.P);
  return it;
}

template <typename T, int D, int B, int HG>
__global__ void __launch_bounds__(32 * (HG + 1)) decode_split_kernel(const SplitArgs a) {
  using G = Geo<T, D, B, HG>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((128u - (su32(smem_raw) & 127u)) & 127u);
  const uint32_t sb = su32(smem);
  const uint32_t bars = sb + G::BAR_OFF;
  auto FULL = [&](int i) { return bars + 8u * i; };
  auto EMPTY = [&](int i) { return bars + 8u * (G::NST + i); };
  auto IFULL = [&](int i) { return bars + 8u * (2 * G::NST + i); };
  auto IEMPTY = [&](int i) { return bars + 8u * (2 * G::NST + 2 + i); };
  volatile int32_t* misc = reinterpret_cast<volatile int32_t*>(smem + G::MISC_OFF);
  volatile int32_t* abort_flag = misc;
  volatile int32_t* item_slot = misc + 1;  // [2]
  volatile int32_t* n_valid = misc + 4;    // [NST]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < G::NST; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), HG);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(IFULL(i), 1);
      mbar_init(IEMPTY(i), HG);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int64_t row_cap = static_cast<int64_t>(a.max_blocks) * B;
  int32_t* hist = reinterpret_cast<int32_t*>(smem + G::ORDER_OFF);  // [64]: counts, then cursors
  int32_t* longest = hist + 64;                                     // [1]
  int32_t* order = hist + 65;                                       // [S]
  if (a.longest_first) {
    // Whole-sequence items in decreasing length: a stable counting sort over 32 length
    // buckets, the same in every block, so item ids agree.  Lengths outside the table
    // count as empty.
    auto len_of = [&](int s) {
      const int L = a.context_lens[s];
      return (L < 0 || L > row_cap) ? 0 : L;
    };
    if (tid < 64) hist[tid] = 0;
    if (tid == 0) *longest = 0;
    __syncthreads();
    for (int s = tid; s < a.S; s += blockDim.x) atomicMax(longest, len_of(s));
    __syncthreads();
    const int lmax = *longest;
    if (warp == 0) {
      auto bucket_of = [&](int s) {
        return min(31, static_cast<int>((static_cast<long long>(len_of(s)) * 32) / (lmax + 1)));
      };
      const unsigned lt = (1u << lane) - 1u;
      for (int base = 0; base < a.S; base += 32) {
        const int s = base + lane;
        const int b = s < a.S ? bucket_of(s) : -1;
        const unsigned same = __match_any_sync(kFull, b);
        if (b >= 0 && (same & lt) == 0) hist[b] += __popc(same);
        __syncwarp();
      }
      // cursor of bucket b = sequences in buckets above b
      const int cnt = hist[31 - lane];
      int v = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      hist[32 + (31 - lane)] = v - cnt;
      __syncwarp();
      for (int base = 0; base < a.S; base += 32) {
        const int s = base + lane;
        const int b = s < a.S ? bucket_of(s) : -1;
        const unsigned same = __match_any_sync(kFull, b);
        if (b >= 0) order[hist[32 + b] + __popc(same & lt)] = s;
        __syncwarp();
        if (b >= 0 && (same & lt) == 0) hist[32 + b] += __popc(same);
        __syncwarp();
      }
    }
  }
  __syncthreads();
  const int total = a.S * (a.H / HG) * a.NP;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int ni = 0, kt = 0;
      while (true) {
        const int item = *abort_flag ? total : atomicAdd(a.sched, 1);
        const bool done = item >= total;
        const int sl = ni & 1;
        if (mbar_wait(IEMPTY(sl), ((ni >> 1) & 1) ^ 1, abort_flag, a.status)) {
          item_slot[sl] = done ? -1 : item;
          mbar_arrive(IFULL(sl));
        }
        ++ni;
        if (done) break;
        const Item it = locate<HG>(a, order, item);
        const int L = a.context_lens[it.s];
        if ((L < 0 || L > row_cap) && it.g == 0 && it.p == 0) atomicOr(a.status, kDevBadLen);
        const int t1 = (L < 0 || L > row_cap) ? 0 : it.t1;
        const int32_t* table = a.block_tables + static_cast<int64_t>(it.s) * a.bt_row;
        bool ok = true;
        for (int t = it.t0; t < t1 && ok; t += B, ++kt) {
          const int st = kt % G::NST;
          if (!mbar_wait(EMPTY(st), ((kt / G::NST) & 1) ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          int fr = table[t / B];
          int nv = min(B, t1 - t);
          if (fr < 0 || fr >= a.num_blocks) {
            atomicOr(a.status, kDevBadBlock);
            fr = 0;
            nv = 0;
          }
          n_valid[st] = nv;
          mbar_expect_tx(FULL(st), G::STAGE);
          const int64_t head0 = static_cast<int64_t>(fr) * a.H + it.g * HG;
          const uint32_t dst = sb + st * G::STAGE;
          bulk_load(dst, static_cast<const T*>(a.k_cache) + head0 * D * B, HG * G::HEAD, FULL(st));
          bulk_load(dst + HG * G::HEAD, static_cast<const T*>(a.v_cache) + head0 * D * B, HG * G::HEAD,
                    FULL(st));
        }
        if (!ok) break;
      }
      if (*abort_flag) {  // copies still landing must finish before the block retires
        const long long t0 = clock64();
        while (clock64() - t0 < kDrainCycles) {
        }
      }
      __threadfence();
      if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
        a.sched[0] = 0;
        a.sched[1] = 0;
        __threadfence();
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // Scores: lane (tok, ph) = (lane mod B, lane / B) dots token tok's chunks ph, ph + PH,
  // ... (one warp step reads 32 consecutive 16-byte chunks).  Values: V is [D][B] per
  // head; lane (r0, c) = (lane / C, lane mod C) reads chunk c (tokens cX .. cX+X-1) of
  // rows r0, r0 + RPI, ... -- again 32 consecutive chunks per warp step, conflict-free --
  // and keeps a partial sum per row over its chunk's tokens; the C lanes of a row add
  // their parts once per item.
  const int hh = warp - 1;
  const int tok = lane % B, ph = lane / B;
  const int vr0 = lane / G::C, vc = lane % G::C;
  int ni = 0, kt = 0;
  while (true) {
    const int sl = ni & 1;
    int item = -1;
    if (__all_sync(kFull, mbar_wait(IFULL(sl), (ni >> 1) & 1, abort_flag, a.status))) item = item_slot[sl];
    __syncwarp();
    if (lane == 0) mbar_arrive(IEMPTY(sl));
    ++ni;
    if (item < 0) break;
    const Item it = locate<HG>(a, order, item);
    const int L = a.context_lens[it.s];
    const int t1 = (L < 0 || L > row_cap) ? 0 : it.t1;
    const int h = it.g * HG + hh;
    // q chunks of this lane, in log2 units
    float qv[G::STEPS][8];
    {
      const T* qrow = static_cast<const T*>(a.q) + static_cast<int64_t>(it.s) * a.q_row + static_cast<int64_t>(h) * D;
#pragma unroll
      for (int k = 0; k < G::STEPS; ++k) {
        float v[8];
        load8<T>(qrow + (ph + k * G::PH) * G::X, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[k][i] = v[i] * a.qk_scale_log2;
      }
    }
    float m = -INFINITY, lsum = 0.f, o[G::NR];
#pragma unroll
    for (int j = 0; j < G::NR; ++j) o[j] = 0.f;
    bool ok = true;
    for (int t = it.t0; t < t1; t += B, ++kt) {
      const int st = kt % G::NST;
      if (!__all_sync(kFull, mbar_wait(FULL(st), (kt / G::NST) & 1, abort_flag, a.status))) {
        ok = false;
        break;
      }
      const int nv = n_valid[st];
      const T* kh = reinterpret_cast<const T*>(smem + st * G::STAGE + hh * G::HEAD);           // [NC][B][X]
      const T* vh = reinterpret_cast<const T*>(smem + st * G::STAGE + (HG + hh) * G::HEAD);    // [D][B]
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < G::STEPS; ++k) {
        float kv[8];
        load8<T>(kh + ((ph + k * G::PH) * B + tok) * G::X, kv);
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(qv[k][i], kv[i], dot);
      }
#pragma unroll
      for (int off = B; off < 32; off <<= 1) dot += __shfl_xor_sync(kFull, dot, off);
      const float x = tok < nv ? dot : -INFINITY;
      float fm = x;
#pragma unroll
      for (int off = 1; off < B; off <<= 1) fm = fmaxf(fm, __shfl_xor_sync(kFull, fm, off));
      if (fm > m) {  // warp-uniform
        const float alpha = ex2(m - fm);
        lsum *= alpha;
#pragma unroll
        for (int j = 0; j < G::NR; ++j) o[j] *= alpha;
        m = fm;
      }
      const float pw = tok < nv ? ex2(x - m) : 0.f;
      if (ph == 0) lsum += pw;
      // the weights of this lane's value chunk: tokens vc X .. vc X + X - 1
      float pt[G::X];
#pragma unroll
      for (int u = 0; u < G::X; ++u) pt[u] = __shfl_sync(kFull, pw, vc * G::X + u);
      // on a partly filled frame the slots past the context may hold anything (0 times a
      // non-finite value would poison the sum): take only the valid tokens' values
      const bool partial = nv < B;  // warp-uniform
#pragma unroll
      for (int j = 0; j < G::NR; ++j) {
        float vv[8];
        load8<T>(vh + (vr0 + G::RPI * j) * B + vc * G::X, vv);
        if (partial) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (vc * G::X + i >= nv) vv[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) o[j] = fmaf(pt[i], vv[i], o[j]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(st));
    }
    float l = lsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(kFull, l, off);
    // add the C lanes' parts of every row: lane (r0, 0) then holds rows r0 + RPI j
#pragma unroll
    for (int j = 0; j < G::NR; ++j)
#pragma unroll
      for (int off = 1; off < G::C; off <<= 1) o[j] += __shfl_xor_sync(kFull, o[j], off);
    if (a.NP == 1) {
      const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
      T* orow = static_cast<T*>(a.out) + static_cast<int64_t>(it.s) * a.out_row + static_cast<int64_t>(h) * D;
      if (vc == 0) {
#pragma unroll
        for (int j = 0; j < G::NR; ++j) orow[vr0 + G::RPI * j] = from_float<T>(o[j] * inv);
      }
    } else {
      // partial slots are keyed by (sequence, head group, partition), which the merge reads
      const int64_t slot = (static_cast<int64_t>(it.s * (a.H / HG) + it.g) * a.NP + it.p) * HG + hh;
      if (vc == 0) {
#pragma unroll
        for (int j = 0; j < G::NR; ++j) a.ws_o[slot * D + vr0 + G::RPI * j] = ok ? o[j] : 0.f;
      }
      if (lane == 0) {
        a.ws_ml[slot * 2] = ok ? m : -INFINITY;
        a.ws_ml[slot * 2 + 1] = ok ? l : 0.f;
      }
    }
    if (!ok) break;
  }
}

// Log-sum-exp combination of the NP partials of each (sequence, head): one warp each.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_split_kernel(const SplitArgs a) {
  constexpr int ND = D / 32;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= a.S * a.H) return;
  const int s = wid / a.H, h = wid % a.H;
  const int g = h / a.hg, hh = h % a.hg;
  const int groups = a.H / a.hg;
  auto slot = [&](int p) { return (static_cast<int64_t>((s * groups + g) * a.NP + p)) * a.hg + hh; };
  // 1. lane p holds part p's (max, sum), parts in chunks of 32: the largest max
  float M = -INFINITY;
  for (int p0 = 0; p0 < a.NP; p0 += 32)
    if (p0 + lane < a.NP) M = fmaxf(M, a.ws_ml[slot(p0 + lane) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  // 2. weights 2^(m_p - M) (lane-parallel), the denominator, and the weighted sum of the
  //    partial outputs with four parts' loads in flight
  float num[ND], den = 0.f;
#pragma unroll
  for (int j = 0; j < ND; ++j) num[j] = 0.f;
  if (M != -INFINITY) {
    for (int p0 = 0; p0 < a.NP; p0 += 32) {
      const bool have = p0 + lane < a.NP;
      const float mp = have ? a.ws_ml[slot(p0 + lane) * 2] : -INFINITY;
      const float w = mp == -INFINITY ? 0.f : ex2(mp - M);
      float wl = have ? w * a.ws_ml[slot(p0 + lane) * 2 + 1] : 0.f;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(kFull, wl, off);
      den += wl;
      const int n = min(32, a.NP - p0);
      for (int j0 = 0; j0 < n; j0 += 4) {
        float wj[4], x[4][ND];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          wj[u] = __shfl_sync(kFull, w, (j0 + u) & 31);
#pragma unroll
          for (int j = 0; j < ND; ++j)
            x[u][j] = j0 + u < n ? a.ws_o[slot(p0 + j0 + u) * D + lane + 32 * j] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int j = 0; j < ND; ++j) num[j] = fmaf(wj[u], x[u][j], num[j]);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T* orow = static_cast<T*>(a.out) + static_cast<int64_t>(s) * a.out_row + static_cast<int64_t>(h) * D;
#pragma unroll
  for (int j = 0; j < ND; ++j) orow[lane + 32 * j] = from_float<T>(num[j] * inv);
}

template <typename T, int D, int B, int HG>
cudaError_t launch(const SplitArgs& a, int num_sms, cudaStream_t stream) {
  using G = Geo<T, D, B, HG>;
  constexpr int kThreads = 32 * (HG + 1);
  auto kern = decode_split_kernel<T, D, B, HG>;
  int per_sm = 0;
  const size_t smem = G::SMEM + (a.longest_first ? 4u * (65u + static_cast<uint32_t>(a.S)) : 0u);
  cudaError_t e = kernel_prep(reinterpret_cast<const void*>(kern), kThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  const int total = a.S * (a.H / HG) * a.NP;
  const int grid = std::max(1, std::min(total, num_sms * std::max(per_sm, 1)));
  kern<<<grid, kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.NP == 1) return e;
  const int warps = a.S * a.H;
  merge_split_kernel<T, D><<<(warps + 3) / 4, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dt(int D, int B, const SplitArgs& a, int num_sms, cudaStream_t stream) {
  // heads per block: a.hg, chosen by the caller (4, or 2 for D = 128 and B = 32)
  if (D == 128) {
    if (B == 8 && a.hg == 4) return launch<T, 128, 8, 4>(a, num_sms, stream);
    if (B == 16 && a.hg == 4) return launch<T, 128, 16, 4>(a, num_sms, stream);
    if (B == 32 && a.hg == 2) return launch<T, 128, 32, 2>(a, num_sms, stream);
  } else if (D == 64 && a.hg == 4) {
    if (B == 8) return launch<T, 64, 8, 4>(a, num_sms, stream);
    if (B == 16) return launch<T, 64, 16, 4>(a, num_sms, stream);
    if (B == 32) return launch<T, 64, 32, 4>(a, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

// ---- append into the split layout ------------------------------------------------------
// One thread per (row, head, 16-byte chunk): the K chunk is one 16-byte store; the V
// chunk's x elements go to x rows of the [D][B] block, B elements apart.
template <typename T>
__global__ void append_split_kernel(const T* k_new, const T* v_new, int64_t k_row, int64_t v_row,
                                    const int32_t* slots, int32_t Tn, int32_t H, int32_t D, int32_t B,
                                    int32_t num_blocks, T* k_cache, T* v_cache, int32_t* status) {
  constexpr int X = 16 / sizeof(T);
  const int NC = D / X;
  const int64_t units = static_cast<int64_t>(Tn) * H * NC;
  for (int64_t u = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; u < units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(u % NC);
    const int h = static_cast<int>((u / NC) % H);
    const int t = static_cast<int>(u / (static_cast<int64_t>(NC) * H));
    const int32_t slot = slots[t];
    if (slot < 0) continue;
    if (static_cast<int64_t>(slot) >= static_cast<int64_t>(num_blocks) * B) {
      if (c == 0 && h == 0) atomicOr(status, kDevBadSlot);
      continue;
    }
    const int64_t frame = slot / B, b = slot % B;
    const int64_t fh = frame * H + h;
    const uint4 kk = *reinterpret_cast<const uint4*>(k_new + t * k_row + static_cast<int64_t>(h) * D + c * X);
    *reinterpret_cast<uint4*>(k_cache + ((fh * NC + c) * B + b) * X) = kk;
    const uint4 vv = *reinterpret_cast<const uint4*>(v_new + t * v_row + static_cast<int64_t>(h) * D + c * X);
    const T* ve = reinterpret_cast<const T*>(&vv);
#pragma unroll
    for (int i = 0; i < X; ++i) v_cache[(fh * D + c * X + i) * B + b] = ve[i];
  }
}

}  // namespace sk

cudaError_t launch_decode_split(int dtype, int D, int B, const SplitArgs& a, int num_sms, cudaStream_t stream) {
  if (dtype == PA_F16) return sk::launch_dt<__half>(D, B, a, num_sms, stream);
  if (dtype == PA_BF16) return sk::launch_dt<__nv_bfloat16>(D, B, a, num_sms, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_append_split(int dtype, const void* k_new, const void* v_new, int64_t k_row, int64_t v_row,
                                const int32_t* slots, int32_t T, int32_t H, int32_t D, int32_t B,
                                int32_t num_blocks, void* k_cache, void* v_cache, int32_t* status, int grid,
                                cudaStream_t stream) {
  if (dtype == PA_F16)
    sk::append_split_kernel<__half><<<grid, 256, 0, stream>>>(
        static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), k_row, v_row, slots, T, H, D, B,
        num_blocks, static_cast<__half*>(k_cache), static_cast<__half*>(v_cache), status);
  else if (dtype == PA_BF16)
    sk::append_split_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), k_row, v_row, slots,
        T, H, D, B, num_blocks, static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
        status);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pa
