// Causal multi-query attention over the paged cache (prefill / chunked prefill)
// on the 5th-generation tensor cores of sm_103a.
//
// What it computes ("Solving the LLM Memory Wall", "1. The Mathematical
// Foundation", general causal form): for a chunk of n_s queries that are the last
// n_s positions of sequence s (its keys already appended to the cache), query i
// at position p attends keys 0..p:  o_i = sum_{j<=p} softmax(q_i.k_j * scale) v_j.
// Keys and values are read through the block table from the caches
// [num_blocks, B, H, D] ("PagedAttention: Virtual Memory Guide for LLM
// Inference", "The Mathematics of Block Translation").
//
// Design (one thread block per SM, persistent, dynamic work counter):
//   * Work item = (sequence, head, pair of consecutive 128-query tiles); pairs are
//     taken longest first (stable 32-bucket counting sort on their key-tile count).  Both tiles of a pair share every K/V
//     tile, which halves the copies and the L2 traffic per FLOP.  K/V are walked in
//     tiles of 128 keys, each assembled from 128/B frames, one TMA copy per frame
//     through a 5-D view of the cache that lands the frame as [B/8 row groups]
//     [2 column halves][8 rows][64] (128-byte swizzle; the MMA descriptors stride
//     2048 bytes per 8 keys); frames past the sequence end are read at an
//     out-of-range group, i.e. zero-filled.  Q tiles are [2 halves][128 rows][64].
//   * warp 0: TMA producer (Q tiles, then K_t, V_t into two-stage rings; the frame
//     copies of a tile are issued by the warp's lanes).  warp 1 (one lane):
//     tcgen05.mma issuer, fp32 accumulators in TMEM (512 columns: S_0 S_1 O_0 O_1).
//     S_q = Q_q K_t^T from shared memory; O_q (+)= P_q V_t with P_q read from TMEM,
//     where the softmax left it over S_q's columns (each half of the keys over its own
//     scores; bf16: the weights' high parts and their remainders, two products).
//     warps 2-9: softmax of both slots, tile by tile (thread = query row = TMEM
//     lane; warps w and w + 4 share a lane quadrant and split each tile's keys and
//     the output dimensions in halves, exchanging row maxima and sums through shared
//     memory): causal mask, online softmax in log2 units (ex2.approx, fp32) with a
//     lazily raised reference max, P (operand type; bf16 as high part + remainder)
//     back to TMEM, O rescaled in TMEM
//     when the reference max moves; normalised rows are written to `out`.
//   * Every wait is a bounded mbarrier wait; one that gives up sets PA_DEV_TIMEOUT
//     and makes the block's later waits no-ops; before the TMEM is freed the MMA
//     lane waits (bounded) for its own MMAs and the producer for its copies.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pa_internal.h"

namespace pa {
namespace pk {

constexpr unsigned kFull = 0xffffffffu;
constexpr long long kWaitCycles = 4000000000LL;
constexpr long long kDrainCycles = 200000000LL;
constexpr int kD = 128;           // head_dim
constexpr int kBM = 128;          // queries per tile
constexpr int kBN = 128;          // keys per tile
constexpr int kThreads = 320;     // 10 warps
constexpr int kSmxWarp0 = 2;      // softmax warps 2 .. 9; half h: warps 2 + 4h .. 5 + 4h
constexpr uint32_t kTile = 32768; // bytes of one 128 x 128 16-bit tile
constexpr uint32_t kHalf = 16384; // one 64-column half of a Q tile

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kSmQ = 0;                  // [2 slots] Q tiles: [2 halves][128 rows][64]
constexpr uint32_t kSmK = kSmQ + 2 * kTile;   // [2 stages] K tiles: [16 groups][2 halves][8 rows][64]
constexpr uint32_t kSmV = kSmK + 2 * kTile;   // [2 stages] V tiles, same layout
constexpr uint32_t kSmBar = kSmV + 2 * kTile; // mbarriers
constexpr uint32_t kSmMisc = kSmBar + 32 * 8; // flags, TMEM address, item ring
constexpr uint32_t kSmX = kSmMisc + 64;       // row-max / row-sum exchange [2 phases][2 halves][128 rows] fp32
constexpr uint32_t kSmOff = kSmX + 2048;      // unit offsets [S + 1] | histogram [64] | unit order [unit_cap]
__host__ __device__ constexpr uint32_t smem_bytes(int S, int unit_cap) {
  return kSmOff + 4u * (S + 1) + 4u * 64u + 4u * unit_cap + 1024u;
}

// TMEM (512 columns): S_q at column 128 q, O_q at 256 + 128 q (fp32, lane = query row);
// P_q (16-bit, two per column) overwrites S_q: keys 0-63 in columns 0-31, keys 64-127 in
// columns 64-95 (bf16 remainders in columns 32-63 and 96-127).
constexpr uint32_t kTmemS = 0, kTmemO = 256;

// mbarrier indices
enum : int {
  BQ_FULL = 0, BQ_EMPTY = 1,
  BK_FULL = 2, BK_EMPTY = 4, BV_FULL = 6, BV_EMPTY = 8,  // [2 stages] each
  BS_FULL = 10, BP_FULL = 12, BO_FULL = 14,              // [2 slots] each
  BI_FULL = 16, BI_EMPTY = 18,                           // item ring [2]
  BDRAIN = 20,
  BX = 21,                                               // [4 TMEM lane quadrants] half exchange
  NBARS = 25
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// Whole frame of one head: coordinates (0, 0, 0, first 8-row group, head) of the 5-D
// frame view of a cache.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int group, int head,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %2, %2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(group), "r"(head), "r"(bar)
      : "memory");
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input max and packed two-lane fp32 arithmetic (one instruction per pair).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// tcgen05 shared-memory matrix descriptor: 128-byte swizzle, SM100 version field.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// kind::f16 instruction descriptor, fp32 accumulate, M = N = 128, A K-major.
template <typename T>
__host__ __device__ constexpr uint32_t idesc(bool b_mn_major) {
  constexpr uint32_t fmt = sizeof(T) == 2 && !std::is_same<T, __half>::value ? 1u : 0u;  // bf16 = 1
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(b_mn_major) << 16) | ((128u >> 3) << 17) |
         ((128u >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
// A operand from TMEM (M = 128 lanes, 16-bit elements two per column), B from shared memory.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// tcgen05.ld of 32 columns without waiting; pair with tmem_wait_ld() and tie32().
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tie16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Empty statement that claims to rewrite the registers: every later use depends on it,
// and it is ordered after the (volatile) wait that precedes it.
__device__ __forceinline__ void tie32(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
      "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ int upper_seq(const int32_t* off, int S, int x) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// A unit is a pair of consecutive 128-query tiles of one sequence: slot 1 holds the
// later tile, slot 0 the one before it (absent when the chunk has an odd tile count
// and this is its first pair).  A work item is (unit, head); both tiles share every
// K/V tile.
struct PItem {
  int s, h;
  int nkv;       // key tiles the item walks (those of slot 1)
  int qrow0[2];  // first q row of the slot's tile (global row index)
  int nrows[2];  // valid rows of the slot's tile, 0 when the slot is unused
  int pos0[2];   // position of the slot's first row
  int nkv_q[2];  // key tiles the slot visits, 0 when unused
};

// A sequence is skipped (and flagged) unless 0 <= qs <= qe <= T, n = qe - qs <= L and
// L fits its block table.
__device__ __forceinline__ bool seq_bad(int qs, int qe, int L, const PrefillArgs& a) {
  return qs < 0 || qe < qs || qe > a.T || L < qe - qs ||
         static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks) * a.B;
}

// Tiles of pair p (counted from the end of the chunk) of a sequence.
__device__ __forceinline__ void pair_tiles(const PrefillArgs& a, int s, int p, PItem& it) {
  const int qs = a.query_start[s], qe = a.query_start[s + 1];
  const int n = qe - qs;
  const int L = a.context_lens[s];
  const bool bad = seq_bad(qs, qe, L, a);
  const int ntiles = n > 0 ? (n + kBM - 1) / kBM : 0;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int qt = ntiles - 1 - 2 * p - (1 - q);
    if (bad || qt < 0) {
      it.qrow0[q] = qs;
      it.nrows[q] = 0;
      it.pos0[q] = 0;
      it.nkv_q[q] = 0;
    } else {
      it.qrow0[q] = qs + qt * kBM;
      it.nrows[q] = min(kBM, n - qt * kBM);
      it.pos0[q] = L - n + qt * kBM;
      it.nkv_q[q] = (it.pos0[q] + it.nrows[q] - 1 + kBN) / kBN;
    }
  }
  it.nkv = it.nkv_q[1];
}

// Item -> (unit of rank item / H in the longest-first order, head item % H).
__device__ __forceinline__ PItem locate(const PrefillArgs& a, const int32_t* offu, const int32_t* order,
                                        int item) {
  PItem it;
  const int r = item / a.H;
  it.h = item - r * a.H;
  const int u = order[r];
  it.s = upper_seq(offu, a.S, u);
  pair_tiles(a, it.s, u - offu[it.s], it);
  return it;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
  // bf16 weights keep 8 significant bits: each weight goes to the value product as a
  // high part and the remainder (two products into the same accumulator), which
  // leaves 2^-16 of it; fp16 weights (11 bits) go once.
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + kSmBar;
  auto BAR = [&](int i) { return bars + 8u * i; };
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + kSmMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmMisc + 4);
  volatile int32_t* item_slot = reinterpret_cast<volatile int32_t*>(smem + kSmMisc + 8);  // [2]
  int32_t* offu = reinterpret_cast<int32_t*>(smem + kSmOff);  // [S + 1] units per sequence, prefix
  int32_t* hist = offu + (a.S + 1);                            // [64] bucket counts, cursors
  int32_t* order = hist + 64;                                  // [unit_cap] units, longest first
  int32_t* max_nkv = reinterpret_cast<int32_t*>(smem + kSmMisc + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B;
  const int fpt = kBN / B;  // frames per key tile

  if (tid == 0) {
    for (int i = 0; i < NBARS; ++i) {
      uint32_t cnt = 1;
      if (i == BP_FULL || i == BP_FULL + 1) cnt = 8;        // all eight softmax warps
      if (i == BI_EMPTY || i == BI_EMPTY + 1) cnt = 9;      // MMA warp + eight softmax warps
      if (i >= BX && i < BX + 4) cnt = 2;                   // the two warps of a lane quadrant
      mbar_init(BAR(i), cnt);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // TMEM: S0 S1 O0 O1, 128 columns each
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_v)) : "memory");
  }
  // ---- work list: units (sequence, tile pair) ordered longest first by a stable
  //      32-bucket counting sort on their key-tile count (identical in every block);
  //      item = (unit rank, head) -------------------------------------------------------
  if (tid == 0) *max_nkv = 0;
  if (tid < 64) hist[tid] = 0;
  if (tid == 0) offu[0] = 0;
  __syncthreads();
  for (int s = tid; s < a.S; s += blockDim.x) {
    const int qs = a.query_start[s], qe = a.query_start[s + 1];
    const int L = a.context_lens[s];
    const bool bad = seq_bad(qs, qe, L, a);
    if (bad && blockIdx.x == 0) atomicOr(a.status, kDevBadLen);
    const int n = bad ? 0 : qe - qs;
    const int ntiles = (n + kBM - 1) / kBM;
    offu[s + 1] = (ntiles + 1) / 2;
    if (n > 0) atomicMax(max_nkv, (L + kBN - 1) / kBN);  // the last tile sees the whole context
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < a.S; base += 32) {
      const int i = base + lane;
      int v = i < a.S ? offu[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
      }
      v += carry;
      if (i < a.S) offu[i + 1] = v;
      carry = __shfl_sync(kFull, v, 31);
    }
  }
  __syncthreads();
  const int n_units = offu[a.S];
  if (n_units > a.unit_cap) {  // query ranges overlap beyond the rows given: no work
    if (tid == 0 && blockIdx.x == 0) atomicOr(a.status, kDevBadLen);
  } else if (warp == 1) {
    const int mx = *max_nkv;
    auto bucket_of = [&](int u) {
      if (u >= n_units) return -1;
      PItem t;
      const int s = upper_seq(offu, a.S, u);
      pair_tiles(a, s, u - offu[s], t);
      return min(31, static_cast<int>((static_cast<long long>(t.nkv) * 32) / (mx + 1)));
    };
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < n_units; base += 32) {
      const int b = bucket_of(base + lane);
      const unsigned same = __match_any_sync(kFull, b);
      if (b >= 0 && (same & lt) == 0) hist[b] += __popc(same);
      __syncwarp();
    }
    // cursor[b] = units in buckets above b (longest first)
    const int cnt = hist[31 - lane];
    int v = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += n;
    }
    hist[32 + (31 - lane)] = v - cnt;
    __syncwarp();
    for (int base = 0; base < n_units; base += 32) {
      const int u = base + lane;
      const int b = bucket_of(u);
      const unsigned same = __match_any_sync(kFull, b);
      if (b >= 0) order[hist[32 + b] + __popc(same & lt)] = u;
      __syncwarp();
      if (b >= 0 && (same & lt) == 0) hist[32 + b] += __popc(same);
      __syncwarp();
    }
  }
  __syncthreads();
  const int total = n_units > a.unit_cap ? 0 : n_units * a.H;
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ====================================== producer ======================================
    // Lane 0 takes work items and arms the barriers; lane f issues the copy of frame
    // f of a key tile (one 5-D box holds a whole frame of one head, both column
    // halves), after reading its own block-table entry: a tile costs one table-load
    // latency, and the entries of the next tile are read before its ring slot is
    // waited for.
    int ni = 0, kt = 0, qi = 0;
    while (true) {
      int item = 0;
      if (lane == 0) item = *abort_flag ? total : atomicAdd(a.sched, 1);
      item = __shfl_sync(kFull, item, 0);
      const bool done = item >= total;
      const int sl = ni & 1;
      if (lane == 0 && mbar_wait(BAR(BI_EMPTY + sl), ((ni >> 1) & 1) ^ 1, abort_flag, a.status)) {
        item_slot[sl] = done ? -1 : item;
        mbar_arrive(BAR(BI_FULL + sl));
      }
      ++ni;
      if (done) break;
      const PItem it = locate(a, offu, order, item);
      if (it.nkv == 0) continue;
      // Q tiles of the used slots (two 64-column halves each)
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait(BAR(BQ_EMPTY), (qi & 1) ^ 1, abort_flag, a.status);
        if (ok) {
          mbar_expect_tx(BAR(BQ_FULL), kTile * ((it.nrows[0] > 0) + (it.nrows[1] > 0)));
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (it.nrows[q] > 0) {
              tma_load_3d(sb + kSmQ + q * kTile, &tmap_q, 0, it.h, it.qrow0[q], BAR(BQ_FULL));
              tma_load_3d(sb + kSmQ + q * kTile + kHalf, &tmap_q, 64, it.h, it.qrow0[q], BAR(BQ_FULL));
            }
          }
        }
      }
      ok = __shfl_sync(kFull, ok, 0);
      if (!ok) break;
      ++qi;
      const int32_t* table = a.block_tables + static_cast<int64_t>(it.s) * a.bt_row;
      const int Lv = a.context_lens[it.s];
      const int oob_group = a.num_blocks * (B / 8);  // any frame past the cache: zero fill
      // first 8-row group (in the frame view) of the frame lane f copies in tile j
      auto frame_group = [&](int j) -> int {
        const int lb = j * fpt + lane;
        int g = oob_group;
        if (lane < fpt && lb * B < Lv) {
          const int fr = __ldg(table + lb);
          if (fr >= 0 && fr < a.num_blocks) g = fr * (B / 8);
          else atomicOr(a.status, kDevBadBlock);
        }
        return g;
      };
      auto issue = [&](const CUtensorMap* map, uint32_t ring, int empty_bar, int full_bar, int t, int g) -> bool {
        const int st = t & 1;
        int w = 1;
        if (lane == 0) {
          w = mbar_wait(BAR(empty_bar + st), ((t >> 1) & 1) ^ 1, abort_flag, a.status);
          if (w) mbar_expect_tx(BAR(full_bar + st), kTile);
        }
        w = __shfl_sync(kFull, w, 0);
        if (!w) return false;
        if (lane < fpt) tma_load_5d(sb + ring + st * kTile + lane * B * 256, map, g, it.h, BAR(full_bar + st));
        return true;
      };
      int g = frame_group(0);
      for (int j = 0; j < it.nkv && ok; ++j) {
        ok = issue(&tmap_k, kSmK, BK_EMPTY, BK_FULL, kt + j, g);
        if (ok) ok = issue(&tmap_v, kSmV, BV_EMPTY, BV_FULL, kt + j, g);
        if (j + 1 < it.nkv) g = frame_group(j + 1);
      }
      kt += it.nkv;
      if (!ok) break;
    }
    if (lane == 0) {
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
  } else if (warp == 1) {
    // ====================================== MMA issuer ======================================
    // Per key tile t of an item:  S_0 = Q_0 K_t^T, S_1 = Q_1 K_t^T, then for each slot
    // in turn O_q (+)= P_q V_t followed by S_q = Q_q K_{t+1}^T, so that one slot's
    // products run while the other slot's softmax works.  P_q lives in S_q's columns:
    // the next S_q is issued after the P V that reads it (the tensor core keeps issue
    // order), and the commit that publishes S_q also covers that P V, so the softmax
    // may rescale O_q once it sees S_q.
    int ni = 0, kt = 0, qi = 0;
    uint32_t pc0 = 0, pc1 = 0;  // P V products issued per slot (P_FULL phases)
    const uint32_t id_qk = idesc<T>(false);
    const uint32_t id_pv = idesc<T>(true);
    auto qk = [&](int q, int t) {
      const int st = t & 1;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t ad = sdesc(sb + kSmQ + q * kTile + (ks >> 2) * kHalf + (ks & 3) * 32, 0, 1024);
        const uint64_t bd = sdesc(sb + kSmK + st * kTile + (ks >> 2) * 1024 + (ks & 3) * 32, 0, 2048);
        mma(tmem + kTmemS + q * 128, ad, bd, id_qk, ks > 0 ? 1u : 0u);
      }
      commit(BAR(BS_FULL + q));
    };
    // weights of keys 16 ks .. 16 ks + 15 (16-bit pairs): columns 64 (ks / 4) + 8 (ks mod 4)
    // of S_q, over the scores of the half of the tile they belong to
    auto pcol_of = [](int ks) { return static_cast<uint32_t>((ks >> 2) * 64 + (ks & 3) * 8); };
    auto pv = [&](int q, int t, bool first) {
      const int st = t & 1;
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks) {
        const uint64_t bd = sdesc(sb + kSmV + st * kTile + ks * 2 * 2048, 1024, 2048);
        mma_ts(tmem + kTmemO + q * 128, tmem + kTmemS + q * 128 + pcol_of(ks), bd, id_pv,
               (!first || ks > 0) ? 1u : 0u);
      }
      if constexpr (kSplitP) {  // the weights' low parts, 32 columns after the high parts
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t bd = sdesc(sb + kSmV + st * kTile + ks * 2 * 2048, 1024, 2048);
          mma_ts(tmem + kTmemO + q * 128, tmem + kTmemS + q * 128 + pcol_of(ks) + 32, bd, id_pv, 1u);
        }
      }
    };
    auto wait = [&](int bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(BAR(bar), parity, abort_flag, a.status);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      return w;
    };
    if (lane == 0) {
      while (true) {
        const int sl = ni & 1;
        int item = -1;
        if (mbar_wait(BAR(BI_FULL + sl), (ni >> 1) & 1, abort_flag, a.status)) item = item_slot[sl];
        mbar_arrive(BAR(BI_EMPTY + sl));
        ++ni;
        if (item < 0) break;
        const PItem it = locate(a, offu, order, item);
        if (it.nkv == 0) continue;
        const int n0 = it.nkv_q[0], n1 = it.nkv_q[1];
        bool ok = wait(BQ_FULL, qi & 1);
        ++qi;
        ok = ok && wait(BK_FULL + (kt & 1), (kt >> 1) & 1);
        if (ok) {
          if (n0 > 0) qk(0, kt);
          qk(1, kt);
          commit(BAR(BK_EMPTY + (kt & 1)));
          if (n1 == 1) commit(BAR(BQ_EMPTY));
        }
        for (int j = 0; j < n1 && ok; ++j) {
          const int t = kt + j;
          bool have_v = false, have_k = false;
          if (j < n0) {
            ok = wait(BP_FULL + 0, pc0 & 1) && wait(BV_FULL + (t & 1), (t >> 1) & 1);
            if (!ok) break;
            have_v = true;
            pv(0, t, j == 0);
            ++pc0;
            if (j == n0 - 1) commit(BAR(BO_FULL + 0));
            if (j + 1 < n0) {
              ok = wait(BK_FULL + ((t + 1) & 1), ((t + 1) >> 1) & 1);
              if (!ok) break;
              have_k = true;
              qk(0, t + 1);
            }
          }
          ok = wait(BP_FULL + 1, pc1 & 1) && (have_v || wait(BV_FULL + (t & 1), (t >> 1) & 1));
          if (!ok) break;
          pv(1, t, j == 0);
          ++pc1;
          commit(BAR(BV_EMPTY + (t & 1)));
          if (j == n1 - 1) commit(BAR(BO_FULL + 1));
          if (j + 1 < n1) {
            ok = have_k || wait(BK_FULL + ((t + 1) & 1), ((t + 1) >> 1) & 1);
            if (!ok) break;
            qk(1, t + 1);
            commit(BAR(BK_EMPTY + ((t + 1) & 1)));
            if (j + 1 == n1 - 1) commit(BAR(BQ_EMPTY));
          }
        }
        kt += n1;
        if (!ok) break;
      }
      // all MMAs of this lane complete before the TMEM can be freed
      commit(BAR(BDRAIN));
      const long long t0 = clock64();
      while (!mbar_try(BAR(BDRAIN), 0) && clock64() - t0 < kDrainCycles) {
      }
    }
  } else {
    // ====================================== softmax / epilogue ======================================
    // All eight warps work on every tile of both slots, in the order the MMA warp
    // publishes them (slot 0 tile j, then slot 1 tile j).  Warps w and w + 4 share TMEM
    // lane quadrant w mod 4 (query rows 32 (w mod 4) ..): the first takes keys 0-63 of
    // a tile and output dimensions 0-63, the second keys 64-127 and dimensions 64-127.
    // Thread = query row = TMEM lane.  Per tile each half finds its row max, the two
    // halves exchange it through shared memory (one mbarrier per quadrant, bounded
    // wait), and both take the same decision: the reference max m_ref the weights are
    // taken against moves only when the tile's row max passed it by more than 8 (log2
    // units), so weights stay <= 2^8 and O is rescaled rarely.  For bf16 a half posts its
    // max, computes and stores its weights against the current m_ref, and only then reads
    // the partner's max; when m_ref moves (every row's first tile, rarely afterwards) the
    // weights are computed again.  Each half keeps a partial row sum; the halves add
    // them at the epilogue.  P goes back to TMEM over the half's own 64 score columns
    // (keys 64h + 2k, 64h + 2k + 1 in column 64h + k; bf16 remainders 32 columns on).
    const int half = (warp - kSmxWarp0) >> 2;
    const int quad = warp & 3;        // TMEM lane quadrant a warp may access
    const int row = quad * 32 + lane; // query row in the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    float* xbuf = reinterpret_cast<float*>(smem + kSmX);  // [2 phases][2 halves][128 rows]
    const uint32_t xbar = BAR(BX + quad);
    const float sl2 = a.qk_scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    int ni = 0;
    uint32_t sc[2] = {0u, 0u}, oc[2] = {0u, 0u};  // S_FULL and O_FULL phases per slot
    uint32_t xk = 0;                              // exchanges done (phase of xbar)
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = __all_sync(kFull, mbar_wait(bar, parity, abort_flag, a.status));
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      return w;
    };
    // Give the partner half this row's value and take its one (false: the block aborts).
    auto exchange = [&](float mine, float& theirs) -> bool {
      float* xb = xbuf + (xk & 1u) * 256;
      xb[half * 128 + row] = mine;
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      const bool w = wait_all(xbar, xk & 1u);
      ++xk;
      theirs = xb[(half ^ 1) * 128 + row];
      return w;
    };
    auto row_sum = [](const uint64_t (&v)[2]) {
      float a0, a1, b0, b1;
      unf2(v[0], a0, a1);
      unf2(v[1], b0, b1);
      return (a0 + a1) + (b0 + b1);
    };
    while (true) {
      const int sl = ni & 1;
      int item = -1;
      if (__all_sync(kFull, mbar_wait(BAR(BI_FULL + sl), (ni >> 1) & 1, abort_flag, a.status)))
        item = item_slot[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(BI_EMPTY + sl));
      ++ni;
      if (item < 0) break;
      const PItem it = locate(a, offu, order, item);
      const int n0 = it.nkv_q[0], n1 = it.nkv_q[1];
      if (n1 == 0) continue;
      // rows past the chunk end attend everything they are shown (not stored)
      int pos[2];
      float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 2; ++q) pos[q] = row < it.nrows[q] ? it.pos0[q] + row : 0x3fffffff;
      bool ok = true;
      // per tile of slot q (slot 0 tile j, then slot 1 tile j): scores of this half's 64
      // keys -> weights, O rescaled if the reference moved
      for (int j = 0; j < n1 && ok; ++j) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if ((q == 0 && j >= n0) || !ok) continue;
        if (!wait_all(BAR(BS_FULL + q), sc[q] & 1u)) { ok = false; continue; }
        ++sc[q];
        const uint32_t s_tmem = tmem + lane_base + kTmemS + q * 128;
        // keys of this half a row may see: 64 half + (0 .. nv-1).  Rows of a warp are
        // consecutive positions, so a 32-key chunk is (warp-uniformly) fully visible,
        // fully masked (weight 0, not loaded) or split by the diagonal.
        const int nvalid = max(0, min(kBN, pos[q] - j * kBN + 1));
        const int nv = max(0, min(64, nvalid - 64 * half));
        const int wmin = __reduce_min_sync(kFull, nv), wmax = __reduce_max_sync(kFull, nv);
        uint32_t sr[2][32];
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (wmax > 0) {
          tmem_ld32_async(s_tmem + 64 * half, sr[0]);
          if (wmax > 32) tmem_ld32_async(s_tmem + 64 * half + 32, sr[1]);
          tmem_wait_ld();
          tie32(sr[0]);
          if (wmax > 32) tie32(sr[1]);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            if (wmax <= cc * 32) break;
            uint32_t(&cur)[32] = sr[cc];
            if (wmin < (cc + 1) * 32) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (cc * 32 + i >= nv) cur[i] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], __uint_as_float(cur[i]), __uint_as_float(cur[i + 1]));
          }
        }
        // Give the partner half this row's max now.  bf16 (two 16-bit parts per weight):
        // read the partner's max only after the weights, computed against the current
        // reference; they are final unless the tile's max passes it by more than 8, which
        // after a row's first tile is rare, and then computed again from the scores, still
        // in registers (fp16, with half the weight work, measured faster without this:
        // 991 against 939 TF/s; bf16 755 against 735).  Each half writes its weights over
        // its own score columns only, so it may store them before the partner has read
        // its scores.
        const float mine = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        float* xb = xbuf + (xk & 1u) * 256;
        xb[half * 128 + row] = mine;
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar);
        const bool spec = kSplitP && __all_sync(kFull, m_ref[q] > -INFINITY && mine * sl2 <= m_ref[q] + 8.f);
        uint64_t sum2[2];  // packed fp32 pairs of partial row sums
        auto weights = [&](float mref) {
          const uint64_t nm2 = f2(-mref, -mref);
          sum2[0] = sum2[1] = 0ull;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t pcol = s_tmem + 64 * half + 16 * cc;
            uint32_t w[16];
            uint32_t wl[kSplitP ? 16 : 1];  // low parts (bf16 only)
            if (wmax <= cc * 32) {
#pragma unroll
              for (int k = 0; k < 16; ++k) w[k] = 0u;
              if constexpr (kSplitP) {
#pragma unroll
                for (int k = 0; k < 16; ++k) wl[k] = 0u;
              }
            } else {
              const uint32_t(&cur)[32] = sr[cc];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float x0, x1;
                unf2(ffma2(f2(__uint_as_float(cur[i]), __uint_as_float(cur[i + 1])), sl2x2, nm2), x0, x1);
                const float p0 = ex2(x0), p1 = ex2(x1);
                sum2[(i >> 1) & 1] = fadd2(sum2[(i >> 1) & 1], f2(p0, p1));
                const uint32_t hi = pack2<T>(p0, p1);
                w[i >> 1] = hi;
                if constexpr (kSplitP) {
                  // p - bf16(p) is exact in fp32; its own bf16 rounding leaves 2^-16 p
                  float r0, r1;
                  unf2(ffma2(f2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)), f2(-1.f, -1.f),
                             f2(p0, p1)),
                       r0, r1);
                  wl[i >> 1] = pack2<T>(r0, r1);
                }
              }
            }
            tmem_st16(pcol, w);
            if constexpr (kSplitP) tmem_st16(pcol + 32, wl);
          }
        };
        if (spec) weights(m_ref[q]);
        if (!wait_all(xbar, xk & 1u)) { ok = false; continue; }
        ++xk;
        const float other = xb[(half ^ 1) * 128 + row];
        const float m_t = fmaxf(mine, other) * sl2;
        // one decision per tile, the same in both halves (always on a row's first tile)
        float alpha = 1.f;
        if (m_t > m_ref[q] + 8.f) {
          alpha = ex2(m_ref[q] - m_t);
          m_ref[q] = m_t;
        }
        if (!spec || __any_sync(kFull, alpha != 1.f)) {
          if (spec) tmem_wait_st();  // the stores above land before these
          weights(m_ref[q]);
        }
        if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
          // O_q holds the previous tiles (the S commit covered their P V); this half's
          // dimensions, rows whose reference did not move scale by 1
          const uint32_t o_tmem = tmem + lane_base + kTmemO + q * 128 + 64 * half;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            tmem_ld32_async(o_tmem + c * 32, r);
            tmem_wait_ld();
            tie32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(o_tmem + c * 32, r);
          }
        }
        l[q] = l[q] * alpha + row_sum(sum2);
        tmem_wait_st();
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(BP_FULL + q));
      }
      }
      // epilogues, slot 0 then slot 1: wait for the slot's last P V, add the halves'
      // row sums, normalise this half's 64 dimensions, store
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if ((q ? n1 : n0) == 0) continue;
        if (ok && !wait_all(BAR(BO_FULL + q), oc[q] & 1u)) ok = false;
        ++oc[q];
        float other = 0.f;
        if (ok && !exchange(l[q], other)) ok = false;
        const float lt = l[q] + other;
        const bool zero = !ok || !(lt > 0.f);
        const float inv = zero ? 0.f : 1.f / lt;
        const bool valid = row < it.nrows[q];
        const uint32_t o_tmem = tmem + lane_base + kTmemO + q * 128 + 64 * half;
        T* op = reinterpret_cast<T*>(a.out) + static_cast<int64_t>(it.qrow0[q] + row) * a.out_row +
                static_cast<int64_t>(it.h) * kD + 64 * half;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32_async(o_tmem + c * 32, r);
          tmem_wait_ld();
          tie32(r);
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 w4;
              w4.x = pack2<T>(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv);
              w4.y = pack2<T>(__uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
              w4.z = pack2<T>(__uint_as_float(r[i + 4]) * inv, __uint_as_float(r[i + 5]) * inv);
              w4.w = pack2<T>(__uint_as_float(r[i + 6]) * inv, __uint_as_float(r[i + 7]) * inv);
              if (zero) w4 = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(op + c * 32 + i) = w4;
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      if (!ok) break;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

template <typename T>
cudaError_t launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   int grid, cudaStream_t stream) {
  const size_t smem = smem_bytes(a.S, a.unit_cap);
  auto kern = prefill_kernel<T>;
  cudaError_t e = kernel_prep(reinterpret_cast<const void*>(kern), kThreads, smem, nullptr);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace pk
}  // namespace pa
