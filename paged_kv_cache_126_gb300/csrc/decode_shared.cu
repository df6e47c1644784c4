// Shared-prefix paged decode for sm_103a: frames that consecutive sequences share
// are read once for all of them.
//
// What it computes is pa_decode's result ("Solving the LLM Memory Wall", "1. The
// Mathematical Foundation"): for every sequence s and head h, out = softmax(q.K^T *
// scale) V over the sequence's own L_s tokens.  Only the number of times a shared
// frame is read changes.  A fork copies the block table and raises reference counts
// ("PagedAttention: Virtual Memory Guide for LLM Inference", "Key Architectural
// Mechanics"), so sibling sequences hold block tables that begin with the same
// physical frames, and for the tokens in those frames the siblings' keys and values
// are the same bytes.  Softmax attention over a sequence splits over any partition
// of its tokens and recombines exactly by the log-sum-exp rule, so the shared tokens
// can be attended by all siblings' queries in one pass: one read of a shared frame
// serves up to NQ queries.
//
// Design (GB300):
//   * plan kernel: lcp[s] = the number of leading tokens that sequence s reads through
//     the same frame ids as sequence s-1 (equal leading table entries, capped by both
//     lengths).  One warp per sequence, coalesced 32-entry compares.
//   * main kernel: the persistent producer / consumer structure of decode_kernel (one
//     TMA producer warp, HG consumer warps, a ring of staged units of R = 16 tokens,
//     bounded mbarrier waits, dynamic work counter that resets itself).
//     - Setup, identical in every thread block: runs of consecutive sequences whose
//       lcp is at least min_shared are cut into chunks of at most NQ sequences; a
//       chunk's shared length sh is the smallest lcp inside it, rounded down to whole
//       frames.  Every sequence's tokens are the shared segment [0, sh) (empty for a
//       chunk of one) and its private segment [sh, L).  Segments are cut into parts of
//       P tokens (P chosen from the unique work, as in decode_kernel).
//     - Work items, in this order: shared parts (chunk leader's table, all members'
//       queries), full private parts, then the shorter last private parts longest
//       first.  Item = (part, head group).
//     - Consumers, one warp per head, put the item's queries (1 .. NQ = 16 members)
//       in the rows of a 16-row tensor-core tile and take every staged unit of 16 keys
//       through mma.sync m16n8k16: S = Q K^T, online softmax in fp32, O += P V with P
//       carried as a high and a low 16-bit part (fp32-accurate weights).  One read
//       of a shared frame serves all members; K/V rows reach the tensor cores
//       through conflict-free ldmatrix loads from a 128-byte-swizzled layout.
//     - Every part's (m, l, o) goes to slot pbase[s] + part of the workspace, or
//       straight to the output when the sequence has one part.
//     - A part of a sequence with more than one part raises that (sequence, head)'s
//       arrival counter once its stores are visible; a consumer warp publishes its
//       parts in one batch when its block has no items left (a fence per item stalled
//       the staging ring).  Warps whose block has no items left take merge tasks
//       (sequence, head) from a second counter, in the order the sequences' parts
//       finish, wait (bounded) for the task's parts, and merge them by the log-sum-exp
//       rule.  This replaces a separate merge launch after the whole kernel; merging in
//       the consumer that brings the last part (up to 16 members' merges by one warp)
//       stalled its block's staging ring.
//   * Bad frame ids / lengths: as in decode_kernel (rows of the affected sequences
//     become zeros, sticky status bits).  A bad length ends a run (its lcp is 0).
#include <climits>
#include <type_traits>

#include "decode_kernel.cuh"
#include "pa.h"

namespace pa {
namespace ds {

using dk::kFull;
using dk::mbar_arrive;
using dk::mbar_arrive_expect_tx;
using dk::mbar_init;
using dk::mbar_try_wait;
using dk::mbar_wait;
using dk::smem_u32;
using dk::prefetch_tmap;
using dk::ex2;
using dk::valid_len;
using dk::upper_seq;

constexpr int NQ = 16;  // queries served by one read of a shared frame (rows of one mma tile)
constexpr long long kDrainCycles = dk::kDrainCycles;

// ---- tensor-core helpers (mma.sync m16n8k16, fp32 accumulate) -------------------------------
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Two fp32 values as one 16-bit pair (x0 in the low half), round to nearest even,
// and the pair of what rounding left over (x - round(x), rounded the same way): the
// two pairs together carry x to about 16 more bits.
template <typename T>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  if constexpr (std::is_same<T, __half>::value) {
    const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
    const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
    hi = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
    lo = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
  } else {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
    hi = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
    lo = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) | (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
  }
}

// ---- shared-memory layout (host and device agree) ---------------------------------------------
// A staged unit holds R = 16 tokens of HG heads for K, then for V, as TMA boxes of Rb =
// min(B, 16) rows laid out [HG][2 column halves][Rb][64 elements] with the 128-byte
// swizzle (16-byte chunk c of a 128-byte line stored at c ^ (line mod 8)): eight
// consecutive rows of one half fall in eight different bank groups, so ldmatrix reads
// them without conflicts.  Stages start on 1024-byte boundaries.
struct SLayout {
  uint32_t stage_pitch, bars, flags, lv, lc, cinfo, shl, pbase, sbase, offa, order, hist, comb, total;
  __host__ __device__ SLayout(int stages, uint32_t stage_bytes, int S) {
    stage_pitch = (stage_bytes + 1023u) & ~1023u;
    // mbarriers: full[stages], empty[stages], item_full[2], item_empty[2]
    bars = stages * stage_pitch;
    flags = bars + 16u * stages + 32u;  // poison[stages], abort, item_slot[2]
    const uint32_t arr = 4u * static_cast<uint32_t>(S + 1);
    lv = (flags + 4u * (stages + 3) + 15u) & ~15u;     // validated context lengths (-1: bad) [S]
    lc = (lv + arr + 15u) & ~15u;                      // tokens shared with the previous sequence, then merge order [S]
    cinfo = (lc + arr + 15u) & ~15u;                   // chunk leader | chunk size << 24 [S]
    shl = (cinfo + arr + 15u) & ~15u;                  // shared tokens of the sequence's chunk [S]
    pbase = (shl + arr + 15u) & ~15u;                  // first partial slot of each sequence [S + 1]
    sbase = (pbase + arr + 15u) & ~15u;                // shared-part item offsets [S + 1]
    offa = (sbase + arr + 15u) & ~15u;                 // full private-part item offsets [S + 1]
    order = (offa + arr + 15u) & ~15u;                 // run starts, then last private parts [S]
    hist = (order + arr + 15u) & ~15u;                 // remainder buckets [32] + cursors [32]
    comb = hist + 256u;                                // reduction scratch
    total = comb + 256u + 1024u;                       // + slack for 1024-byte base alignment
  }
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

struct SItem {
  int s, n, g, L;      // first sequence, queries (members s .. s+n-1), head group, validated length of s
  int tok0, tok1;      // token range of the part
  int blk0, nblk;      // frames holding it
  int part;            // partial slot index within each member's slots
};

struct Plan {
  const int32_t* lv;
  const int32_t* cinfo;
  const int32_t* shl;
  const int32_t* pbase;
  const int32_t* sbase;
  const int32_t* offa;
  const int32_t* order;
  int a_sh, a_pf, P;
};

__device__ __forceinline__ SItem locate(const DecodeArgs& a, const Plan& pl, int item) {
  SItem it;
  int p;
  if (item < pl.a_sh) {
    it.s = upper_seq(pl.sbase, a.S, item);
    const int local = item - pl.sbase[it.s];
    p = local / a.G;
    it.g = local - p * a.G;
    it.n = pl.cinfo[it.s] >> 24;
    const int sh = pl.shl[it.s];
    it.tok0 = p * pl.P;
    it.tok1 = min(sh, it.tok0 + pl.P);
    it.part = p;
    it.L = pl.lv[it.s];
  } else {
    int s;
    if (item < pl.a_sh + pl.a_pf) {
      const int b = item - pl.a_sh;
      s = upper_seq(pl.offa, a.S, b);
      const int local = b - pl.offa[s];
      p = local / a.G;
      it.g = local - p * a.G;
    } else {
      const int b = item - pl.a_sh - pl.a_pf;
      const int j = b / a.G;
      s = pl.order[j];
      it.g = b - j * a.G;
      p = -1;
    }
    it.s = s;
    it.n = 1;
    it.L = pl.lv[s];
    const int Lv = it.L < 0 ? 0 : it.L;
    const int shs = pl.shl[s];
    const int nsh = ceil_div(shs, pl.P);
    const int Lp = Lv - shs;
    if (p < 0) p = Lp / pl.P;  // the last private part
    it.tok0 = shs + p * pl.P;
    it.tok1 = min(Lv, it.tok0 + pl.P);
    it.part = nsh + p;
  }
  it.blk0 = it.tok0 / a.B;
  it.nblk = it.tok1 > it.tok0 ? (it.tok1 + a.B - 1) / a.B - it.blk0 : 0;
  return it;
}

// One work item of a consumer warp (head h of the item's head group): the n <= 16
// queries of sequences s .. s+n-1 as the rows of a 16-row tensor-core tile (rows >= n
// zero), every staged unit of 16 keys as
//   S = Q K^T        (16 mma: 8 steps of 16 dimensions x 2 blocks of 8 keys)
//   online softmax   (rows spread over 4 lanes; running max raised lazily, by at
//                     least 8 in log2 units, so rescaling the outputs is rare)
//   O += P V         (32 mma: P as a 16-bit pair of high and low parts, 16 blocks of 8
//                     dimensions)
// then outputs or partials for each member.  Lane (g, t) = (lane / 4, lane % 4) holds
// rows g and g + 8, columns 2t, 2t + 1 of every 16 x 8 block.
template <typename T, int HG, int RB>
__device__ __forceinline__ void run_item(const DecodeArgs& a, const Plan& pl, const SItem& it, const SLayout& lay,
                                         uint32_t stage0, uint32_t bar_full, uint32_t bar_empty,
                                         volatile int32_t* poison, volatile int32_t* abort_flag, int stages, int& k,
                                         int h, int lane) {
  constexpr int D = 128;
  constexpr int R = 16;
  constexpr uint32_t tile_bytes = static_cast<uint32_t>(R) * HG * D * 2;
  constexpr uint32_t box_bytes = static_cast<uint32_t>(RB) * HG * D * 2;
  constexpr uint32_t half_bytes = RB * 128u;  // one column half of one head in a box
  const int head = it.g * HG + h;
  const int g = lane >> 2, t = lane & 3;

  // queries as A fragments, unscaled storage values (the scale goes on the fp32 scores)
  uint32_t qa[8][4];
  {
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                                            static_cast<int64_t>(it.s + g) * a.q_row +
                                                            static_cast<int64_t>(head) * D);
    const uint32_t* q1 = reinterpret_cast<const uint32_t*>(reinterpret_cast<const T*>(a.q) +
                                                            static_cast<int64_t>(it.s + g + 8) * a.q_row +
                                                            static_cast<int64_t>(head) * D);
    const bool v0 = g < it.n, v1 = g + 8 < it.n;
#pragma unroll
    for (int kd = 0; kd < 8; ++kd) {
      qa[kd][0] = v0 ? q0[kd * 8 + t] : 0u;
      qa[kd][1] = v1 ? q1[kd * 8 + t] : 0u;
      qa[kd][2] = v0 ? q0[kd * 8 + 4 + t] : 0u;
      qa[kd][3] = v1 ? q1[kd * 8 + 4 + t] : 0u;
    }
  }
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  bool poisoned = it.L < 0;

  // per-lane ldmatrix addresses.  K (no transpose): lanes 8i..8i+7 give the rows of
  // matrix i = (keys 0-7 | 8-15) x (chunk 2kd | 2kd+1); V (transpose): matrix i = (keys
  // 0-7 | 8-15) x (chunk 2jj | 2jj+1).  Chunk c of row r sits at 16 * (c ^ (r mod 8))
  // in its 128-byte line; with the chunk pair's even index a compile-time constant the
  // lane-dependent part folds into one XOR term per lane.
  const int kr = (lane & 7) + ((lane >> 4) << 3), kc = (lane >> 3) & 1;
  const int vr = (lane & 7) + (((lane >> 3) & 1) << 3), vc = lane >> 4;
  const uint32_t krow = (kr / RB) * box_bytes + (h * 2 * RB + kr % RB) * 128u;
  const uint32_t vrow = (vr / RB) * box_bytes + (h * 2 * RB + vr % RB) * 128u;
  const uint32_t kx = static_cast<uint32_t>(kc ^ (kr & 7)) << 4;
  const uint32_t vx = static_cast<uint32_t>(vc ^ (vr & 7)) << 4;

  const int ntok = it.tok1 - it.blk0 * a.B;
  const int nvf = ntok > 0 ? (ntok + R - 1) / R : 0;
  for (int j = 0; j < nvf; ++j, ++k) {
    const int s_ = k % stages;
    const uint32_t ph = static_cast<uint32_t>(k / stages) & 1u;
    const bool ok = __all_sync(kFull, mbar_wait(bar_full + 8u * s_, ph, abort_flag, a.status));
    if (!ok || poison[s_]) poisoned = true;
    if (!poisoned) {
      const int n_valid = min(R, ntok - j * R);
      const uint32_t kb = stage0 + s_ * lay.stage_pitch;
      const uint32_t vb = kb + tile_bytes;
      if (n_valid < R) {
        // rows past the context: zero this head's V rows (0 * non-finite would poison the
        // product); its K rows are masked in the scores.  Then order these writes before
        // the next TMA write into the stage.
        for (int r = n_valid + (lane >> 4); r < R; r += 2) {
          const int half = (lane >> 3) & 1, c8 = lane & 7;
          const uint32_t ad = vb + static_cast<uint32_t>(r / RB) * box_bytes +
                              static_cast<uint32_t>(((h * 2 + half) * RB + (r % RB)) * 128 + (c8 << 4));
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(ad), "r"(0u) : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      // ---- S = Q K^T ----
      float sc[2][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[0][e] = sc[1][e] = 0.f;
      const uint32_t kaddr = kb + krow;
#pragma unroll
      for (int kd = 0; kd < 8; ++kd) {
        uint32_t b[4];
        ldsm_x4(kaddr + (kd >> 2) * half_bytes + ((static_cast<uint32_t>((2 * kd) & 7) << 4) ^ kx), b);
        mma16816<T>(sc[0], qa[kd], b[0], b[1]);
        mma16816<T>(sc[1], qa[kd], b[2], b[3]);
      }
      // ---- online softmax (log2 units) ----
      float x[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = nb * 8 + 2 * t + (e & 1);
          x[nb][e] = key < n_valid ? sc[nb][e] * a.qk_scale_log2 : -INFINITY;
        }
      float tm[2];
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        tm[ri] = fmaxf(fmaxf(x[0][2 * ri], x[0][2 * ri + 1]), fmaxf(x[1][2 * ri], x[1][2 * ri + 1]));
        tm[ri] = fmaxf(tm[ri], __shfl_xor_sync(kFull, tm[ri], 1));
        tm[ri] = fmaxf(tm[ri], __shfl_xor_sync(kFull, tm[ri], 2));
      }
      const bool raise0 = tm[0] > m[0] + 8.f || (m[0] == -INFINITY && tm[0] != -INFINITY);
      const bool raise1 = tm[1] > m[1] + 8.f || (m[1] == -INFINITY && tm[1] != -INFINITY);
      if (__any_sync(kFull, raise0 || raise1)) {
        float al[2] = {1.f, 1.f};
        if (raise0) {
          const float mn = fmaxf(m[0], tm[0]);
          al[0] = ex2(m[0] - mn);
          m[0] = mn;
        }
        if (raise1) {
          const float mn = fmaxf(m[1], tm[1]);
          al[1] = ex2(m[1] - mn);
          m[1] = mn;
        }
        l[0] *= al[0];
        l[1] *= al[1];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          o[jj][0] *= al[0];
          o[jj][1] *= al[0];
          o[jj][2] *= al[1];
          o[jj][3] *= al[1];
        }
      }
      float p[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mm = m[e >> 1];
          p[nb][e] = mm == -INFINITY ? 0.f : ex2(x[nb][e] - mm);
        }
      l[0] += (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
      l[1] += (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
      uint32_t ph_[4], pl_[4];
      split2<T>(p[0][0], p[0][1], ph_[0], pl_[0]);
      split2<T>(p[0][2], p[0][3], ph_[1], pl_[1]);
      split2<T>(p[1][0], p[1][1], ph_[2], pl_[2]);
      split2<T>(p[1][2], p[1][3], ph_[3], pl_[3]);
      // ---- O += P V ----
      const uint32_t vaddr = vb + vrow;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t b[4];
        ldsm_x4_t(vaddr + (jj >> 2) * half_bytes + ((static_cast<uint32_t>((2 * jj) & 7) << 4) ^ vx), b);
        mma16816<T>(o[2 * jj], ph_, b[0], b[1]);
        mma16816<T>(o[2 * jj], pl_, b[0], b[1]);
        mma16816<T>(o[2 * jj + 1], ph_, b[2], b[3]);
        mma16816<T>(o[2 * jj + 1], pl_, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8u * s_);
  }

  // ---- outputs or partials, per member row ----
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    l[ri] += __shfl_xor_sync(kFull, l[ri], 1);
    l[ri] += __shfl_xor_sync(kFull, l[ri], 2);
  }
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int row = g + 8 * ri;
    if (row >= it.n) continue;
    const int sj = it.s + row;
    const int base = pl.pbase[sj];
    const int np = pl.pbase[sj + 1] - base;
    if (np == 1) {
      const bool zero = poisoned || !(l[ri] > 0.f);
      const float inv = zero ? 0.f : 1.f / l[ri];
      T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(sj) * a.out_row + static_cast<int64_t>(head) * D;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const float v0 = zero ? 0.f : o[jj][2 * ri] * inv, v1 = zero ? 0.f : o[jj][2 * ri + 1] * inv;
        if constexpr (std::is_same<T, __half>::value) {
          *reinterpret_cast<__half2*>(op + jj * 8 + 2 * t) = __floats2half2_rn(v0, v1);
        } else {
          *reinterpret_cast<__nv_bfloat162*>(op + jj * 8 + 2 * t) = __floats2bfloat162_rn(v0, v1);
        }
      }
    } else {
      const int64_t slot = static_cast<int64_t>(base + it.part) * a.H + head;
      float* wo = a.ws_o + slot * D;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        *reinterpret_cast<float2*>(wo + jj * 8 + 2 * t) = make_float2(o[jj][2 * ri], o[jj][2 * ri + 1]);
      if (t == 0) *reinterpret_cast<float2*>(a.ws_ml + slot * 2) = make_float2(m[ri], poisoned ? -1.f : l[ri]);
    }
  }
  // partials of sequences with more than one part are published by the caller
}

// Inclusive scan of arr[1 .. n] in place by one warp (arr[0] = 0 is left alone).
__device__ __forceinline__ void warp_scan(int32_t* arr, int n, int lane) {
  int carry = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    int v = i < n ? arr[i + 1] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += t;
    }
    v += carry;
    if (i < n) arr[i + 1] = v;
    carry = __shfl_sync(kFull, v, 31);
  }
}

// Log-sum-exp merge of one split (sequence, head) by one warp, once its parts have
// arrived.  Lane p holds part p's (max, sum) -- parts in chunks of 32 -- and lane l
// accumulates output dimensions 4l .. 4l+3 over the parts, with the loads of four parts
// in flight at a time.  ready = false (the wait gave up): the row becomes zeros.
template <typename T>
__device__ __forceinline__ void merge_one(const DecodeArgs& a, int s, int head, int base, int np, bool ready,
                                          int lane) {
  constexpr int D = 128;
  auto ml_at = [&](int p) {
    return __ldcg(reinterpret_cast<const float2*>(a.ws_ml + (static_cast<int64_t>(base + p) * a.H + head) * 2));
  };
  const float* ob = a.ws_o + (static_cast<int64_t>(base) * a.H + head) * D + 4 * lane;
  const int64_t pstride = static_cast<int64_t>(a.H) * D;
  // up to four parts: their outputs are loaded with their (max, sum), one round trip
  float4 pre[4];
  if (ready && np <= 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      pre[u] = u < np ? __ldcg(reinterpret_cast<const float4*>(ob + u * pstride)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // 1. the largest running max, and whether any part was poisoned
  float M = -INFINITY;
  bool bad = !ready;
  float2 first = make_float2(-INFINITY, 0.f);
  if (ready) {
    for (int p0 = 0; p0 < np; p0 += 32) {
      const float2 ml = p0 + lane < np ? ml_at(p0 + lane) : make_float2(-INFINITY, 0.f);
      if (p0 == 0) first = ml;
      M = fmaxf(M, ml.x);
      bad |= p0 + lane < np && ml.y < 0.f;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
  bad = __any_sync(kFull, bad);
  // 2. weights 2^(m_p - M), the denominator, and the weighted sum of the partial outputs
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (!bad && M != -INFINITY && np <= 4) {
    const float wgt = lane < np ? ex2(first.x - M) : 0.f;
    float wl = wgt * first.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(kFull, wl, off);
    den = wl;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = __shfl_sync(kFull, wgt, u);
      if (u >= np) break;
      num.x = fmaf(w, pre[u].x, num.x);
      num.y = fmaf(w, pre[u].y, num.y);
      num.z = fmaf(w, pre[u].z, num.z);
      num.w = fmaf(w, pre[u].w, num.w);
    }
  } else if (!bad && M != -INFINITY) {
    for (int p0 = 0; p0 < np; p0 += 32) {
      const float2 ml = p0 == 0 ? first : (p0 + lane < np ? ml_at(p0 + lane) : make_float2(-INFINITY, 0.f));
      const float wgt = p0 + lane < np ? ex2(ml.x - M) : 0.f;
      float wl = wgt * ml.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(kFull, wl, off);
      den += wl;
      const int n = min(32, np - p0);
      for (int j = 0; j < n; j += 4) {
        float4 x[4];
        float w4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w4[u] = __shfl_sync(kFull, wgt, (j + u) & 31);
          x[u] = j + u < n ? __ldcg(reinterpret_cast<const float4*>(ob + (p0 + j + u) * pstride))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (j + u >= n) break;
          num.x = fmaf(w4[u], x[u].x, num.x);
          num.y = fmaf(w4[u], x[u].y, num.y);
          num.z = fmaf(w4[u], x[u].z, num.z);
          num.w = fmaf(w4[u], x[u].w, num.w);
        }
      }
    }
  }
  const bool zero = bad || !(den > 0.f);
  const float inv = zero ? 0.f : 1.f / den;
  T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(s) * a.out_row + static_cast<int64_t>(head) * D + 4 * lane;
  if constexpr (std::is_same<T, __half>::value) {
    const __half2 lo = __floats2half2_rn(num.x * inv, num.y * inv), hi = __floats2half2_rn(num.z * inv, num.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(op) = u;
  } else {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(num.x * inv, num.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(num.z * inv, num.w * inv);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&lo);
    u.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(op) = u;
  }
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The merges, taken from a task counter by every warp once its block has no items left:
// task t is head t mod H of sequence morder[t / H], in the order the sequences' parts
// finish.  Every item was claimed before any warp gets here, by a
// block that is running and finishes it without waiting on a merge, so the waits end;
// each is bounded all the same and gives up early once a timeout is on record.
template <typename T>
__device__ __forceinline__ void merge_phase(const DecodeArgs& a, const int32_t* pbase, const int32_t* morder,
                                            int lane) {
  const int ntask = a.S * a.H;
  while (true) {
    int t = 0;
    if (lane == 0) t = atomicAdd(a.sched + 2, 1);
    t = __shfl_sync(kFull, t, 0);
    if (t >= ntask) break;
    const int i = t / a.H, head = t - i * a.H;
    const int s = morder[i];
    const int task = s * a.H + head;
    const int base = pbase[s];
    const int np = pbase[s + 1] - base;
    if (np <= 1) continue;  // written directly by its item
    const int32_t* cnt = a.ws_cnt + task;
    bool ready = __all_sync(kFull, ld_acquire(cnt) >= np);
    if (!ready) {
      const long long t0 = clock64();
      while (true) {
        __nanosleep(200);
        if (__all_sync(kFull, ld_acquire(cnt) >= np)) {
          ready = true;
          break;
        }
        if (*reinterpret_cast<volatile int32_t*>(a.status) & kDevTimeout) break;
        if (clock64() - t0 > dk::kWaitCycles) {
          if (lane == 0) atomicOr(a.status, kDevTimeout);
          break;
        }
      }
    }
    merge_one<T>(a, s, head, base, np, ready, lane);
    if (lane == 0 && ready) a.ws_cnt[task] = 0;  // zero between launches
  }
}

template <typename T, int HG>
__global__ void __launch_bounds__(32 * (HG + 1), 2)
    decode_shared_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                         const DecodeArgs a, const int stages) {
  constexpr int D = 128;
  constexpr int E = sizeof(T);
  constexpr int NCW = HG;  // one consumer warp per head
  static_assert(D * E == 256, "shared-prefix decode needs 256-byte rows");

  const int B = a.B;
  const int R = a.R;
  const int FPS = R > B ? R / B : 1;
  const int SPF = B > R ? B / R : 1;
  const uint32_t tile_bytes = static_cast<uint32_t>(R) * HG * D * E;
  const uint32_t stage_bytes = 2u * tile_bytes;
  const uint32_t box_bytes = static_cast<uint32_t>(R > B ? B : R) * HG * D * E;

  extern __shared__ unsigned char smem_raw[];
  const SLayout lay(stages, stage_bytes, a.S);
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned
  const uint32_t sbase_u = smem_u32(smem);
  const uint32_t bar_full = sbase_u + lay.bars;
  const uint32_t bar_empty = bar_full + 8u * stages;
  const uint32_t bar_ifull = bar_empty + 8u * stages;
  const uint32_t bar_iempty = bar_ifull + 16u;
  volatile int32_t* poison = reinterpret_cast<volatile int32_t*>(smem + lay.flags);
  volatile int32_t* abort_flag = poison + stages;
  volatile int32_t* item_slot = abort_flag + 1;
  int32_t* lv = reinterpret_cast<int32_t*>(smem + lay.lv);
  int32_t* lc = reinterpret_cast<int32_t*>(smem + lay.lc);
  int32_t* cinfo = reinterpret_cast<int32_t*>(smem + lay.cinfo);
  int32_t* shl = reinterpret_cast<int32_t*>(smem + lay.shl);
  int32_t* pbase = reinterpret_cast<int32_t*>(smem + lay.pbase);
  int32_t* sbase = reinterpret_cast<int32_t*>(smem + lay.sbase);
  int32_t* offa = reinterpret_cast<int32_t*>(smem + lay.offa);
  int32_t* order = reinterpret_cast<int32_t*>(smem + lay.order);
  int32_t* hist = reinterpret_cast<int32_t*>(smem + lay.hist);
  float* comb = reinterpret_cast<float*>(smem + lay.comb);  // setup reductions

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- 0. barriers, then wait for the plan kernel's writes ---------------------------------
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

  // ---- 1. lengths and shared-token counts into shared memory (one coalesced pass) ---------
  for (int s = tid; s < a.S; s += blockDim.x) {
    lv[s] = valid_len(a, s);
    lc[s] = a.lcp[s];
  }
  __syncthreads();
  // chunks: run starts (warp 0, max-scan of break positions, kept in `order`)
  if (warp == 0) {
    int carry = -1;
    for (int base = 0; base < a.S; base += 32) {
      const int s = base + lane;
      int v = -1;
      if (s < a.S) v = (s == 0 || lc[s] < a.min_shared) ? s : -1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v = max(v, t);
      }
      v = max(v, carry);
      if (s < a.S) order[s] = v;
      carry = __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
  // leader, chunk size and shared length of every sequence (each member derives the
  // same values from the same run starts)
  for (int s = tid; s < a.S; s += blockDim.x) {
    const int r0 = order[s];
    int lead = s - ((s - r0) % NQ);
    int n = 1;
    while (n < NQ && lead + n < a.S && order[lead + n] == r0) ++n;
    int sh = 0;
    if (n > 1) {
      int mn = INT_MAX;
      for (int j = 1; j < n; ++j) mn = min(mn, lc[lead + j]);
      sh = (mn / B) * B;
    }
    if (sh <= 0) {
      lead = s;
      n = 1;
      sh = 0;
    }
    cinfo[s] = lead | (n << 24);
    shl[s] = sh;
  }
  __syncthreads();

  // ---- 2. partition length from the unique work ------------------------------------------
  const int Lcap = a.max_blocks * B;
  int P;
  {
    long long local = 0;
    int lmax = 0, segs = 0;
    for (int s = tid; s < a.S; s += blockDim.x) {
      const int L = lv[s];
      const int Lv = L < 0 ? 0 : L;
      const int sh = shl[s];
      const bool leader = (cinfo[s] & 0xffffff) == s && sh > 0;
      local += (Lv - sh) + (leader ? sh : 0);
      lmax = max(lmax, max(Lv - sh, leader ? sh : 0));
      segs += 1 + (leader ? 1 : 0);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      local += __shfl_xor_sync(kFull, local, o);
      lmax = max(lmax, __shfl_xor_sync(kFull, lmax, o));
      segs += __shfl_xor_sync(kFull, segs, o);
    }
    long long* red = reinterpret_cast<long long*>(comb);
    int* redmax = reinterpret_cast<int*>(red + (blockDim.x >> 5));
    int* redseg = redmax + (blockDim.x >> 5);
    if (lane == 0) {
      red[warp] = local;
      redmax[warp] = lmax;
      redseg[warp] = segs;
    }
    __syncthreads();
    long long total = 0;
    segs = 0;
    for (int ww = 0; ww < static_cast<int>(blockDim.x >> 5); ++ww) {
      total += red[ww];
      lmax = max(lmax, redmax[ww]);
      segs += redseg[ww];
    }
    __syncthreads();
    long long p;
    if (a.fixed_part > 0) {
      p = a.fixed_part;
    } else if (a.whole_first && static_cast<long long>(segs) * a.G >= gridDim.x &&
               static_cast<long long>(lmax) * gridDim.x <= total * a.G) {
      p = Lcap;
    } else {
      p = (total * a.G + a.target_items - 1) / (a.target_items > 0 ? a.target_items : 1);
      p = ((p + B - 1) / B) * B;
      if (p < a.min_part) p = a.min_part;
      if (p > Lcap) p = Lcap;
      if (lmax > p) {  // equal parts for the longest segment
        const long long n = (lmax + p - 1) / p;
        const long long q = (((lmax + n - 1) / n + B - 1) / B) * B;
        if (q >= a.min_part) p = q;
      }
    }
    if (p < B) p = B;
    P = static_cast<int>(p);
  }

  // ---- 3. parts per sequence, item offsets, last private parts longest first --------------
  auto parts_of = [&](int s, int Pp, int* nsh, int* nf, int* last) {
    const int L = lv[s];
    const int Lv = L < 0 ? 0 : L;
    const int sh = shl[s];
    const int Lp = Lv - sh;
    *nsh = ceil_div(sh, Pp);
    *nf = Lp / Pp;
    *last = (Lp % Pp != 0 || (Lp == 0 && sh == 0)) ? 1 : 0;
    return *nsh + *nf + *last;
  };
  {
    // the workspace holds part_cap partial slots; whole segments always fit (2 per sequence)
    int cnt = 0;
    for (int s = tid; s < a.S; s += blockDim.x) {
      int x, y, z;
      cnt += parts_of(s, P, &x, &y, &z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    int* redc = reinterpret_cast<int*>(comb);
    if (lane == 0) redc[warp] = cnt;
    __syncthreads();
    cnt = 0;
    for (int ww = 0; ww < static_cast<int>(blockDim.x >> 5); ++ww) cnt += redc[ww];
    __syncthreads();
    // too many parts for the workspace: double P until they fit (whole segments, at most
    // two parts per sequence, always do)
    for (int guard = 0; cnt > a.part_cap && P < Lcap && guard < 32; ++guard) {
      P = min(Lcap, 2 * P);
      int c2 = 0;
      for (int s = tid; s < a.S; s += blockDim.x) {
        int x, y, z;
        c2 += parts_of(s, P, &x, &y, &z);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c2 += __shfl_xor_sync(kFull, c2, o);
      if (lane == 0) redc[warp] = c2;
      __syncthreads();
      cnt = 0;
      for (int ww = 0; ww < static_cast<int>(blockDim.x >> 5); ++ww) cnt += redc[ww];
      __syncthreads();
    }
    if (cnt > a.part_cap) P = Lcap > B ? Lcap : B;
  }
  for (int s = tid; s < a.S; s += blockDim.x) {
    if (blockIdx.x == 0 && lv[s] < 0) atomicOr(a.status, kDevBadLen);
    int nsh, nf, last;
    pbase[s + 1] = parts_of(s, P, &nsh, &nf, &last);
    const bool leader = (cinfo[s] & 0xffffff) == s && shl[s] > 0;
    sbase[s + 1] = leader ? nsh * a.G : 0;
    offa[s + 1] = nf * a.G;
  }
  if (tid < 64) hist[tid] = 0;
  if (tid == 0) {
    pbase[0] = 0;
    sbase[0] = 0;
    offa[0] = 0;
  }
  __syncthreads();
  if (warp == 0) {
    warp_scan(pbase, a.S, lane);
    warp_scan(sbase, a.S, lane);
    warp_scan(offa, a.S, lane);
  } else if (warp == 1) {
    auto bucket_of = [&](int s) {
      int nsh, nf, last;
      parts_of(s, P, &nsh, &nf, &last);
      if (!last) return -1;
      const int L = lv[s];
      const int Lp = (L < 0 ? 0 : L) - shl[s];
      return min(31, static_cast<int>((static_cast<long long>(Lp % P) * 32) / P));
    };
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < a.S; base += 32) {
      const int s = base + lane;
      const int b = s < a.S ? bucket_of(s) : -1;
      const unsigned same = __match_any_sync(kFull, b);
      if (b >= 0 && (same & lt) == 0) hist[b] += __popc(same);
      __syncwarp();
    }
    const int cntb = hist[31 - lane];
    int v = cntb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += t;
    }
    hist[32 + (31 - lane)] = v - cntb;
    if (lane == 31) hist[31] = v;
    __syncwarp();
    const int n_last = hist[31];
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
    if (lane == 0) hist[0] = n_last;
    // merge order (over the shared-token counts, which nothing reads any more): sequences
    // without a last private part first (their parts finish earlier), then the others in
    // the order their last parts are scheduled
    __syncwarp();
    int n0 = 0;
    for (int base = 0; base < a.S; base += 32) {
      const int s = base + lane;
      const bool none = s < a.S && bucket_of(s) < 0;
      const unsigned m = __ballot_sync(kFull, none);
      if (none) lc[n0 + __popc(m & lt)] = s;
      n0 += __popc(m);
    }
    for (int i = lane; i < n_last; i += 32) lc[n0 + i] = order[i];
  }
  __syncthreads();
  // `order` held the run starts until the sort above overwrote it; nothing reads them after
  // the chunk pass.
  Plan pl;
  pl.lv = lv;
  pl.cinfo = cinfo;
  pl.shl = shl;
  pl.pbase = pbase;
  pl.sbase = sbase;
  pl.offa = offa;
  pl.order = order;
  pl.a_sh = sbase[a.S];
  pl.a_pf = offa[a.S];
  pl.P = P;
  const int total_items = pl.a_sh + pl.a_pf + hist[0] * a.G;

  if (warp == NCW) {
    // ============================== producer warp ==============================
    int k = 0, ni = 0;
    uint32_t issued = 0;
    while (true) {
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
      const SItem it = locate(a, pl, item);
      const int32_t* row = a.block_tables + static_cast<int64_t>(it.s) * a.bt_row + it.blk0;
      const int ntok = it.tok1 - it.blk0 * B;
      const int nvf = ntok > 0 ? (ntok + R - 1) / R : 0;
      int chunk = -1, frame = -1;
      for (int vf = 0; vf < nvf; ++vf, ++k) {
        const int f0 = FPS > 1 ? vf * FPS : vf / SPF;
        const int nf = FPS > 1 ? min(FPS, it.nblk - f0) : 1;
        if ((f0 >> 5) != chunk) {
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
          const uint32_t dst = sbase_u + st * lay.stage_pitch + lane * box_bytes;
          const int r0 = fr * B + (SPF > 1 ? (vf % SPF) * R : 0);
          tma_load_4d(dst, &tmap_k, 0, r0, 0, it.g * HG, bar_full + 8u * st);
          tma_load_4d(dst + tile_bytes, &tmap_v, 0, r0, 0, it.g * HG, bar_full + 8u * st);
        }
      }
    }
    if (lane == 0) {
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
    }
  } else {
  // ============================== consumer warps ==============================
  const int h = warp;
  int k = 0, ni = 0;
  // Partials of split sequences are published in batches, not per item: a GPU-scope
  // fence after every item stalled the warp (and with it the staging ring).  The ids of
  // the items whose partials await publication sit in the setup scratch (free by now).
  constexpr int kPubCap = 64 / HG - 1;  // entry kPubCap holds the count
  int32_t* plist = reinterpret_cast<int32_t*>(comb) + h * (kPubCap + 1);
  volatile int32_t* npub_s = plist + kPubCap;
  if (lane == 0) *npub_s = 0;
  __syncwarp();
  auto publish = [&]() {
    // after a timeout nothing is published: the merges see the status bit and give up
    const int npub = *abort_flag ? 0 : *npub_s;
    if (npub == 0) return;
    __threadfence();  // every lane's partial stores, visible at GPU scope
    __syncwarp();
    for (int j = 0; j < npub; ++j) {
      const SItem pit = locate(a, pl, plist[j]);
      if (lane < pit.n) {
        const int sj = pit.s + lane;
        if (pl.pbase[sj + 1] - pl.pbase[sj] > 1)
          atomicAdd(a.ws_cnt + static_cast<int64_t>(sj) * a.H + pit.g * HG + h, 1);
      }
    }
    __syncwarp();
    if (lane == 0) *npub_s = 0;
    __syncwarp();
  };
  while (true) {
    const int sl = ni & 1;
    const bool got =
        __all_sync(kFull, mbar_wait(bar_ifull + 8u * sl, static_cast<uint32_t>((ni >> 1) & 1), abort_flag, a.status));
    const int item = got ? item_slot[sl] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_iempty + 8u * sl);
    ++ni;
    if (item < 0) break;
    const SItem it = locate(a, pl, item);
    // listed now, published after this item's stores at the next batch
    const bool split = lane < it.n && pl.pbase[it.s + lane + 1] - pl.pbase[it.s + lane] > 1;
    if (__any_sync(kFull, split)) {
      if (*npub_s == kPubCap) publish();
      if (lane == 0) {
        const int n = *npub_s;
        plist[n] = item;
        *npub_s = n + 1;
      }
      __syncwarp();
    }
    if (B >= 16) {
      run_item<T, HG, 16>(a, pl, it, lay, sbase_u, bar_full, bar_empty, poison, abort_flag, stages, k, h, lane);
    } else {
      run_item<T, HG, 8>(a, pl, it, lay, sbase_u, bar_full, bar_empty, poison, abort_flag, stages, k, h, lane);
    }
  }
  publish();
  }

  // ---- 4. merges of split sequences, then the block retires ----------------------------
  merge_phase<T>(a, pbase, lc, lane);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      // the last block: every item and merge task has been claimed
      a.sched[0] = 0;
      a.sched[1] = 0;
      a.sched[2] = 0;
      __threadfence();
    }
  }
}

// lcp[s]: leading tokens sequence s reads through the same frame ids as s - 1.
__global__ void __launch_bounds__(256) share_plan_kernel(const DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x * 8 + warp;
  if (s >= a.S) return;
  int res = 0;
  if (s > 0) {
    const int L1 = valid_len(a, s), L0 = valid_len(a, s - 1);
    if (L1 > 0 && L0 > 0) {
      const int m = min(L1, L0);
      const int nb = (m + a.B - 1) / a.B;
      const int32_t* t1 = a.block_tables + static_cast<int64_t>(s) * a.bt_row;
      const int32_t* t0 = t1 - a.bt_row;
      int nf = nb;
      for (int f0 = 0; f0 < nb; f0 += 32) {
        const int f = f0 + lane;
        const bool diff = f < nb && t1[f] != t0[f];
        const unsigned msk = __ballot_sync(kFull, diff);
        if (msk) {
          nf = f0 + __ffs(msk) - 1;
          break;
        }
      }
      res = min(nf * a.B, m);
    }
  }
  if (lane == 0) a.lcp[s] = res;
}

template <typename T, int HG>
cudaError_t launch_one(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                       cudaStream_t stream, bool query_only, int* max_ctas) {
  constexpr int NCW = HG;
  const uint32_t stage_bytes = 2u * static_cast<uint32_t>(a.R) * HG * 128 * sizeof(T);
  const SLayout lay(c.stages, stage_bytes, a.S);
  const size_t smem = lay.total;
  auto kern = decode_shared_kernel<T, HG>;
  int n = 0;
  cudaError_t e = kernel_prep(reinterpret_cast<const void*>(kern), 32 * (NCW + 1), smem, &n);
  if (e != cudaSuccess) return e;
  if (query_only) {
    if (max_ctas) *max_ctas = n;
    return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.S + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, share_plan_kernel, a);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.grid);
  cfg.blockDim = dim3(32 * (NCW + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, a, c.stages);
}

template <typename T>
cudaError_t launch_t(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk, const CUtensorMap& tv,
                     cudaStream_t stream, bool query_only, int* max_ctas) {
  if (c.warps_per_head != 1) return cudaErrorInvalidValue;
  switch (c.heads_per_cta) {
    case 1: return launch_one<T, 1>(a, c, tk, tv, stream, query_only, max_ctas);
    case 2: return launch_one<T, 2>(a, c, tk, tv, stream, query_only, max_ctas);
    case 4: return launch_one<T, 4>(a, c, tk, tv, stream, query_only, max_ctas);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ds

bool decode_shared_combo(int hg, int wph) { return (hg == 1 || hg == 2 || hg == 4) && wph == 1; }

size_t decode_shared_smem_bytes(const DecodeCfg& c, int R, int S) {
  const uint32_t stage_bytes = 2u * static_cast<uint32_t>(R) * c.heads_per_cta * 128 * 2;
  const ds::SLayout lay(c.stages, stage_bytes, S);
  return lay.total;
}

cudaError_t launch_decode_shared(const DecodeArgs& a, const DecodeCfg& c, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t stream, bool query_only, int* max_ctas) {
  switch (c.dtype) {
    case PA_F16: return ds::launch_t<__half>(a, c, tk, tv, stream, query_only, max_ctas);
    case PA_BF16: return ds::launch_t<__nv_bfloat16>(a, c, tk, tv, stream, query_only, max_ctas);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
