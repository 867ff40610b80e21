// decode_tc.cuh -- paged decode attention on the tensor cores (tcgen05 + TMEM):
// the kernel template, included by the translation units that instantiate it
// (16-bit caches, 8-bit caches), so they compile in parallel.
//
// Same computation as the CUDA-core kernel ("vLLM" page, section "PageAttention":
// softmax(q K^T / sqrt(d)) V per sequence and query head, keys and values found
// through the block table; FlashDecoding partitions merged by log-sum-exp), for
// head_size 128 and up to 16 query heads per kv head.
//
// The cache layout stores every (block, kv head) chunk as 128-byte-swizzled
// 8-token groups [K dims 0-63 | K dims 64-127 | V dims 0-63 | V dims 64-127],
// so a tile of 128 tokens staged by one bulk copy per block is directly
//   * the K-major A operand of S^T = K Q^T   (M = 128 tokens, N = 16 heads,
//     K = 128 dims; 8-token groups 4 KiB apart), and
//   * the MN-major A operand of O^T = V^T P^T (M = 128 dims, N = 16 heads,
//     K = 128 tokens).
// Q^T (K-major, swizzled, written by the planner warp) and P^T (MN-major, no
// swizzle, written by the softmax warps) are the B operands; S^T and O^T
// accumulate in fp32 in tensor memory (TMEM), double-buffered.
//
// One persistent CTA per SM walks a static share of the work items (sequence,
// kv head, partition): every CTA builds the same list in shared memory -- full
// partitions first, then the remainder partitions from the most tiles down --
// and takes one item per round in snake order, so the CTAs get about the same
// number of tiles and none is spent on empty partitions.  Roles:
//   planner     (16-bit caches: the warp before the PV issuer; 8-bit caches:
//               warp 0) orders the items and works out each one in turn: its
//               place, context, first 32 block ids and query rows, written as
//               the Q^T operand of the item's slot.  16-bit caches hand the
//               item to the streamer through a two-slot record ring.
//   warp 0      16-bit caches: streamer -- per item, one bulk copy per (block,
//               kv head) chunk into a ring of NS 64 KiB stages, block ids
//               checked per tile; per-stage metadata travels with the stage's
//               mbarrier.  With the set-up in the planner, the next item's
//               first copies leave as soon as a stage is free.
//   warp 1      MMA issue (one lane): QK(t) as soon as tile t is staged and its
//               S buffer is free, PV(t) as soon as P(t) is written and its O
//               buffer is free.  16-bit caches give PV its own issuer (the last
//               warp), since one lane issuing all 16 MMAs of a tile is the limit.
//   warps 2-5   softmax (thread = TMEM lane = token row): tile max across the
//               128 rows, p = 2^(s - m) in fp32, written in the cache type as
//               p_hi = round(p) and p_lo = round(p - p_hi) side by side in one
//               P^T operand (N = 16, or 32 at 16 heads), so one PV product gives
//               O_hi and O_lo and the weights reach the tensor core with ~16
//               significant bits even for bf16.  For 16-bit caches (up to 8
//               heads per kv head) a second softmax warpgroup (warps 10-13)
//               takes the odd tiles, each group with its own running maximum
//               and sums; the tile metadata reaches each group through the QK
//               issuer, one buffer per S buffer.
//   warps 6-9   output (thread = TMEM lane = head dim): once per item, read
//               each softmax group's O^T = O_hi + O_lo, accumulated in TMEM over
//               the group's tiles of the item (the softmax warps rescale it when
//               their running maximum moves), merge the groups by log-sum-exp
//               and write the item's result (or the partition's partial results).
// 8-bit caches (codes + one fp32 scale per token and kv head) change the
// staging: warp 0 only plans (items, Q, block ids per tile into a descriptor
// ring); one copy warp bulk-copies each tile's 8-bit chunks into two rings of
// 64-token raw half tiles; converter warps turn the codes into exact fp16
// operands -- K rows straight into TMEM (the A operand of QK is then read from
// TMEM), V rows into a V-only stage in shared memory -- and pass the token
// scales on; the softmax warps fold the scales into scores and weights.
// Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT and ends the CTA.
#pragma once

#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 128;                         // tokens per tile
// Remainder-partition classes (tiles in the remainder): 1 .. P / kTile, and P is
// at most 8192 tokens; a larger class (only a larger P) shares the top slot.
constexpr int kClasses = 8192 / kTile + 1;
constexpr int kTileBytes = kTile * 2 * kD * 2;     // K + V of 128 tokens: 64 KiB
constexpr int kGroupBytes = 8 * 2 * kD * 2;        // one 8-token group: 4 KiB
constexpr int kN = 16;                             // MMA N: query heads, zero-padded
constexpr int kQBytes = kN * kD * 2;               // 4 KiB
constexpr int kPBytes = kTile * 32 * 2;            // P^T operand: 128 tokens x up to 32 columns (8 KiB)
// Q^T slots, by item index: 16-bit caches keep four items' queries staged (the
// planner runs up to that far ahead of the tensor core); 8-bit caches two.
// 16-bit caches write each tile's P^T into the K atoms of the tile's own stage
// (dead once QK(t) has completed: 512 B of each 8-token group's 2 KiB), so
// they need no P^T buffers; 8-bit stages hold V only and keep two.
__host__ __device__ constexpr int q_slots(bool i8) { return i8 ? 2 : 4; }
// Items in flight between the softmax and output warps (hand-off slots and O
// accumulators in TMEM, by item index mod this): 16-bit caches four, so the
// output warps can fall behind a run of short items without holding up the
// tensor core; 8-bit caches two.
__host__ __device__ constexpr int item_slots(bool i8) { return i8 ? 2 : 4; }
__host__ __device__ constexpr int p_buffers(bool i8) { return i8 ? 2 : 0; }
constexpr int kThreads = 320;                      // warp 0, MMA issue, 4 softmax warps, 4 output warps
// 8-bit caches add converter warps: 8 when the registers allow it (group <= 4), else 4
__host__ __device__ constexpr int converter_warps(int G) { return G <= 4 ? 8 : 4; }
// 8-bit caches also add one copy warp (after the converters) that only issues
// the bulk copies: a bulk copy instruction holds its warp for ~100 cycles per
// active lane, so nothing else waits behind it.
// Two softmax warpgroups take alternate tiles (warps 2-5 the even ones, four
// warps after all other roles the odd ones), so one tile's softmax overlaps the
// next -- for every 16-bit cache (8-bit caches: their registers are spent on
// the converter warps).
__host__ __device__ constexpr bool ping_pong(bool i8, int G) { return !i8; }
// Lazy running maximum: a softmax group raises its running maximum m (and
// rescales what it has summed) only when some score of a tile exceeds m by
// more than kLazyMax (base-2 units).  Weights 2^(s - m) then stay <= 2^8, exact
// relative to the m they are taken against, and most tiles skip the maximum
// reduction across the 128 rows.
constexpr float kLazyMax = 8.f;

// Reduce K columns (K a power of two <= 32) over the 32 lanes of a warp with
// log2(32) exchanges that halve the columns each lane holds: afterwards lane l
// holds, in v[0], the reduction of column l >> (5 - log2 K) (K + ... shuffles
// instead of 5 K for K separate butterflies).
template <int K, typename Op>
__device__ __forceinline__ void transpose_reduce(float (&v)[K], int lane, Op op) {
  int k = K;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (k > 1) {
      const int half = k >> 1;
      const bool hi = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < K / 2; ++j) {
        if (j < half) {
          const float keep = hi ? v[half + j] : v[j];
          const float send = hi ? v[j] : v[half + j];
          v[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
      }
      k = half;
    } else {
      v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
    }
  }
}
__host__ __device__ constexpr int log2_of(int k) { return k <= 1 ? 0 : 1 + log2_of(k >> 1); }

// The maximum of v over the warp, in every lane (NaN inputs are ignored, as
// by fmaxf).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// 2^x on the MUFU unit (relative error about 2^-22; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 16-bit caches issue QK and PV from two warps (one lane each); 8-bit caches,
// whose tiles are paced by the converter warps, keep one event-driven issuer
// (measured faster there).
__host__ __device__ constexpr bool split_issue(bool i8) { return !i8; }
// 16-bit caches: a planner warp works out each item (its place in the order,
// block ids, query rows) ahead of the streaming warp, which then only issues
// copies; 8-bit caches plan in warp 0, whose copies the copy warp issues.
__host__ __device__ constexpr bool split_plan(bool i8) { return !i8; }
__host__ __device__ constexpr int threads_of(bool i8, int G) {
  return kThreads + (i8 ? 32 * (converter_warps(G) + 1) : 0) + (ping_pong(i8, G) ? 128 : 0) +
         (split_issue(i8) ? 32 : 0) + (split_plan(i8) ? 32 : 0);
}
constexpr int kND = 4;                             // 8-bit: tile descriptors in flight (planner -> copy warp)
constexpr int kRawBytes = 64 * (2 * kD + 32);      // one 64-token half tile of 8-bit chunks (bs 1: 288 B/token)
// TMEM columns: S0 S1 (16 each) | the O accumulators, 32 columns each, one per
// (item slot, softmax group): O^T of an item accumulates across its tiles,
// so the output warps read it once per item; 8-bit caches (one softmax group)
// add the fp16 K operand of each stage (128 tokens x 128 dims, two per column:
// 64 columns) from column kKCol.
constexpr uint32_t kKCol = 128;
constexpr uint32_t kOCol = 32;
__host__ __device__ constexpr uint32_t tmem_cols(bool i8, int ns) {
  return !i8 ? 512u : (kKCol + 64u * ns <= 256u ? 256u : 512u);   // 16-bit: 8 O slots from kOCol
}
// A stage holds the tile's K and V operands (16-bit caches) or, for 8-bit
// caches, only the converted V operand (K lives in TMEM).
__host__ __device__ constexpr int stage_bytes(bool i8) { return i8 ? kTile * kD * 2 : kTileBytes; }
constexpr uint32_t kFull = 0xffffffffu;

struct TileMeta {
  int s, kvh, part, valid;       // sequence (< 0: no more work), kv head, partition, rows < valid hold tokens
  int last, qslot, n_parts, lo;  // last tile of the item, Q buffer, partitions, rows < lo precede the window
  int tail;                      // tiles of the item after this one
  float qinv;                    // 8-bit caches with bf16 q: 2^-e undoing the exact prescale of Q to fp16
  int seq0, ncol, pbase;         // column n: sequence seq0 + n / G, head kvh * G + n % G (ncol real columns);
                                 // the workspace partition of partition `part` is pbase + part
  int head, item;                // tiles of the item before this one; the item's index in this CTA
  int bad;                       // 16-bit caches: a block id of the item so far was out of range (block 0 read
                                 // instead); the item's last tile has the item's verdict
};

// One item as the planner hands it to the streaming warp (16-bit caches).
struct ItemRec {
  int s, kvh, part, n_parts, t_first, t0, t1, jb;   // table row, kv head, partition; its token range
  int seq0, ncol, pbase, qslot, item;               // columns, Q slot, item index (-1: no more work)
  int ids[32];                                      // its first 32 block ids
};

template <int NS, bool I8, int NRH>
struct Shared {
  uint64_t full[NS], empty[NS];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], q_free[4];
  // O accumulator slot o = item slot * groups + group: the PV of the group's
  // last tile of an item completed (ofin), the output warps read it (ofree)
  uint64_t ofin[8], ofree[8];
  uint64_t m_full[2];             // MMA issuer -> softmax: tile t's metadata in smeta[t & 1]
  uint64_t mma_drain[2];          // each MMA-issuing lane's own MMAs, waited for before TMEM is freed
  TileMeta smeta[2];
  uint64_t max_bar[2];            // softmax-warp exchange (bounded waits, unlike bar.sync)
  uint64_t c_full[4], c_free[4];  // softmax -> output warps: per-item hand-off, by item slot
  TileMeta meta[NS];
  struct ItemHand {                // an item's metadata for the output warps (by item slot)
    TileMeta meta;                // its last tile's
    int ntiles, first_grp;        // its tiles, and the softmax group of its first tile
  } ihand[4];
  struct Final {                  // a softmax group's maximum and sums per TMEM lane quarter
    float m[kN];                  // at the end of an item: [item slot][group]
    float Lq[4][kN];
  } fin[4][2];
  // the maximum exchange of a softmax group (ring slot t & 1), double-buffered
  // by the group's tile parity: a warp may write tile t + 2's values only after
  // every warp of its group arrived for tile t + 1... which follows its reads of t
  float red_max[2][2][4][kN];
  int red_up[2][2][4];
  // more than 8 columns: each softmax warp's copy of its group's running
  // maxima (double-buffered) and of the corrections of its latest rescale
  alignas(16) float mrun[2][4][2][kN];
  alignas(16) float mcorr[2][4][kN];
  // each output warp's per-column factors of the two groups' O for the item
  // it is writing
  float2 colout[4][kN];
  uint32_t tmem_base;
  volatile int abort_flag;
  volatile int end_tile;          // QK issuer -> PV issuer: tiles in this CTA (set at the end)
  int sp_ok;                      // shared prefix: the group starts are ordered and in range
  // item ordering (set-up only): remainder partitions per class, cursors;
  // afterwards (16-bit caches) the planner -> streamer records, by item parity
  union {
    struct {
      int cnt[kClasses], cur[kClasses];
    } ord;
    ItemRec rec[2];
  } u;
  uint64_t rec_full[2], rec_empty[2];
  // 8-bit caches: copy warp -> converter ring of raw half tiles, and the token
  // scales of each converted stage
  // (two rings of NRH slots, one per 64-token half: slot h * NRH + k % NRH)
  uint64_t raw_full[I8 ? 2 * NRH : 1], raw_empty[I8 ? 2 * NRH : 1];
  TileMeta raw_meta[I8 ? 2 * NRH : 1];
  // planner -> copy warp: per tile its metadata and block ids
  struct TileDesc {
    TileMeta meta;
    int ids[I8 ? kTile : 1];
  } desc[I8 ? kND : 1];
  uint64_t desc_full[I8 ? kND : 1], desc_empty[I8 ? kND : 1];
  float sk[I8 ? NS : 1][I8 ? kTile : 1];
  float sv[I8 ? NS : 1][I8 ? kTile : 1];
};

// 16 8-bit codes -> 16 exact 16-bit values (8 words, two per word, in order).
// fp16: the byte goes into the mantissa of 1024 (0x64XX = 1024 + byte), then
// 1152 is taken off; bf16: the byte goes into the mantissa of 2^23 in fp32,
// 2^23 + 128 is taken off, and the (exact) high halves are packed.
template <typename T>
__device__ __forceinline__ void codes_to_16bit(const uint4 w4, uint32_t (&o)[8]) {
  const uint32_t w[4] = {w4.x ^ 0x80808080u, w4.y ^ 0x80808080u, w4.z ^ 0x80808080u, w4.w ^ 0x80808080u};
  if constexpr (std::is_same<T, __half>::value) {
    const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t a = __byte_perm(w[k], 0x64646464u, 0x4140), b = __byte_perm(w[k], 0x64646464u, 0x4342);
      __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), off), hb = __hsub2(*reinterpret_cast<__half2*>(&b), off);
      o[2 * k] = *reinterpret_cast<uint32_t*>(&ha);
      o[2 * k + 1] = *reinterpret_cast<uint32_t*>(&hb);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int b = 0; b < 4; b += 2) {
        const float f0 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7540 + b)) - 8388736.0f;
        const float f1 = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7540 + b + 1)) - 8388736.0f;
        o[2 * k + (b >> 1)] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
      }
  }
}

__device__ __forceinline__ bool ctx_invalid(const DecodeParams& p, int ctx) { return !context_ok(p, ctx); }

// Byte offsets, inside the dynamic shared memory after the operand buffers, of
// the item-ordering tables (per virtual sequence: full partitions prefix sum,
// remainder order, remainder class) and, for shared-prefix launches, the
// per-sequence and per-prefix tables.  NV = virtual sequences at most: the
// sequences, plus (shared prefix) one prefix per group chunk (<= S).
struct ItemTables {
  size_t pre, rseq, rcls, eff, tot, npre, pv_seq0, pv_n, pv_eff, gch, ctx, end;
  __host__ __device__ ItemTables(int S, bool sp) {
    const size_t nv = sp ? 2 * (size_t)S : (size_t)S;
    auto a4 = [](size_t x) { return (x + 3) & ~(size_t)3; };
    pre = 0;
    rseq = pre + (nv + 1) * 4;
    rcls = rseq + nv * 2;
    eff = a4(rcls + nv);
    tot = eff + (sp ? (size_t)S * 4 : 0);
    npre = tot + (sp ? (size_t)S * 2 : 0);
    pv_seq0 = npre + (sp ? (size_t)S * 2 : 0);
    pv_n = pv_seq0 + (sp ? (size_t)S * 2 : 0);
    pv_eff = a4(pv_n + (sp ? (size_t)S : 0));
    gch = pv_eff + (sp ? (size_t)S * 4 : 0);
    ctx = gch + (sp ? ((size_t)S + 1) * 4 : 0);
    end = ctx + (sp ? (size_t)S * 4 : 0);
  }
};

// Work items of one sequence: its partitions, or one item that only writes zeros.
// A sequence's work: F full partitions (P / 128 tiles each) and, if the
// attended length is not a multiple of P, one remainder partition of
// ceil(rem / 128) tiles (its "class", 1 .. P / 128: a remainder of P - 1 tokens
// has P / 128 tiles).  A sequence with no (or an invalid) context is one
// remainder item of class 1 that writes zeros.
__device__ __forceinline__ void work_of(const DecodeParams& p, int ctx, int& full, int& cls) {
  if (ctx <= 0 || ctx_invalid(p, ctx)) {
    full = 0;
    cls = 1;
    return;
  }
  const int len = ctx - attended_from(p, ctx);
  full = len / p.partition_size;
  const int rem = len - full * p.partition_size;
  cls = min((rem + kTile - 1) / kTile, kClasses - 1);
}

// Work of a virtual sequence of `len` tokens (len > 0): full partitions and the
// remainder's class (0: no remainder).
__device__ __forceinline__ void work_of_len(int len, int P, int& full, int& cls) {
  full = len / P;
  const int rem = len - full * P;
  cls = min((rem + kTile - 1) / kTile, kClasses - 1);
}

template <typename T, int G>
__device__ void warp_zero_rows(const DecodeParams& p, int s, int kvh, int lane) {
  T* out = static_cast<T*>(p.out) + ((int64_t)s * p.num_q_heads + kvh * G) * kD;
  for (int i = lane * 8; i < G * kD; i += 32 * 8) *reinterpret_cast<uint4*>(out + i) = make_uint4(0, 0, 0, 0);
}

// SP (shared prefix): items are virtual sequences -- each sequence's own tail
// after its group's shared prefix, and one prefix per group chunk whose
// columns are the query heads of up to 16 / G member sequences (kN columns).
template <typename T, int G, int NS, bool I8, int NRH, bool SP>
__global__ void __launch_bounds__(threads_of(I8, SP ? kN : G), 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(!(SP && I8), "shared-prefix decode is for 16-bit caches");
  // columns of an item: the G query heads of one sequence, or (shared prefix)
  // up to kN heads of several sequences
  constexpr int CN = SP ? kN : G;
  // P^T holds p_hi for the CN columns in [0, HG) and p_lo in [HG, 2 HG):
  // one PV product (N = 2 HG) yields both halves of O^T.
  constexpr int HG = CN < 8 ? 8 : CN;
  constexpr int NPV = 2 * HG;
  __shared__ Shared<NS, I8, NRH> sh;
  constexpr int kStage = stage_bytes(I8);
  constexpr uint32_t kCols = tmem_cols(I8, NS);
  extern __shared__ __align__(1024) uint8_t dyn_raw[];
  const uint32_t raw_s = smem_u32(dyn_raw);
  uint8_t* dyn = dyn_raw + (((raw_s + 1023u) & ~1023u) - raw_s);   // 1024-aligned in the shared window
  uint8_t* stages = dyn;
  uint8_t* qbuf = dyn + NS * kStage;
  uint8_t* pbuf = qbuf + q_slots(I8) * kQBytes;               // 8-bit: 2 buffers of [p_hi | p_lo]
  uint8_t* raw = pbuf + p_buffers(I8) * kPBytes;
  uint8_t* tables = raw + (I8 ? 2 * NRH * kRawBytes : 0);
  const ItemTables tl(p.num_seqs, SP);
  int* pre = reinterpret_cast<int*>(tables + tl.pre);            // [NV + 1] full partitions, prefix sum
  int16_t* rseq = reinterpret_cast<int16_t*>(tables + tl.rseq);  // [NV] remainder order
  uint8_t* rcls = tables + tl.rcls;                               // [NV] remainder class
  // shared prefix: per sequence its group's effective prefix, its partitions in
  // all and its group's prefix partitions; per prefix (group chunk) its first
  // member, members and length; per group its first prefix (exclusive scan)
  int* sp_eff = reinterpret_cast<int*>(tables + tl.eff);
  int16_t* sp_tot = reinterpret_cast<int16_t*>(tables + tl.tot);
  int16_t* sp_npre = reinterpret_cast<int16_t*>(tables + tl.npre);
  int16_t* pv_seq0 = reinterpret_cast<int16_t*>(tables + tl.pv_seq0);
  uint8_t* pv_n = tables + tl.pv_n;
  int* pv_eff = reinterpret_cast<int*>(tables + tl.pv_eff);
  int* gch = reinterpret_cast<int*>(tables + tl.gch);
  int* sctx = reinterpret_cast<int*>(tables + tl.ctx);              // context lengths, staged once

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_seqs, Hkv = p.num_kv_heads, bs = p.block_size;
  const int64_t chunk_bytes = I8 ? I8Layout{bs, Hkv}.chunk_bytes() : (int64_t)bs * 2 * kD * 2;
  // Operand type of the MMAs.  8-bit caches always use fp16 operands: codes
  // (|c| <= 127) are exact in fp16, and bf16 queries are brought into fp16 by
  // an exact power-of-two prescale per item (undone on the scores).
  using OpT = std::conditional_t<I8, __half, T>;
  constexpr bool kBF16 = std::is_same<OpT, __nv_bfloat16>::value;
  constexpr bool kQConvert = I8 && std::is_same<T, __nv_bfloat16>::value;
  constexpr int NCW = I8 ? converter_warps(G) : 0;
  constexpr int kSoftB = kThreads / 32 + (I8 ? NCW + 1 : 0);   // first warp of softmax group 1
  constexpr bool kSplitIssue = split_issue(I8);
  static_assert(!ping_pong(I8, CN) || kSplitIssue, "two softmax groups take their tile metadata from the QK issuer");
  constexpr int kPVWarp = threads_of(I8, CN) / 32 - 1;          // with split issue, the PV issuer: the last warp
  constexpr bool kSplitPlan = split_plan(I8);
  constexpr int kPlanWarp = kSplitPlan ? kPVWarp - 1 : 0;       // the planner: before the PV issuer, else warp 0

  // ---- set-up: barriers, zeroed Q buffers (padding heads stay zero), TMEM
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.full[i], I8 ? NCW : 1);   // 8-bit: the converter warps arrive
      mbar_init(&sh.empty[i], 1);
    }
    if (I8) {
      for (int i = 0; i < 2 * NRH; ++i) {
        mbar_init(&sh.raw_full[i], 1);
        mbar_init(&sh.raw_empty[i], NCW / 2);   // the converter warps of the half's TMEM lane quarters
      }
      for (int i = 0; i < kND; ++i) {
        mbar_init(&sh.desc_full[i], 1);
        mbar_init(&sh.desc_empty[i], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.m_full[i], 1);
      mbar_init(&sh.s_free[i], 4);
      mbar_init(&sh.p_full[i], 4);
      mbar_init(&sh.pv_done[i], 1);
      mbar_init(&sh.max_bar[i], 4);
      mbar_init(&sh.mma_drain[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      // every warp of each softmax group that had a tile in the item (the group
      // of a one-tile item arrives for both)
      mbar_init(&sh.c_full[i], ping_pong(I8, CN) ? 8 : 4);
      mbar_init(&sh.c_free[i], 4);
      mbar_init(&sh.q_free[i], 1);
    }
    for (int i = 0; i < 8; ++i) {
      mbar_init(&sh.ofin[i], 1);
      mbar_init(&sh.ofree[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.rec_full[i], 1);
      mbar_init(&sh.rec_empty[i], 1);
    }
    sh.abort_flag = 0;
    sh.end_tile = 0x7fffffff;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < q_slots(I8) * kQBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  // Shared prefix: per group (consecutive sequences group_start[g] ..
  // group_start[g + 1] - 1) the effective prefix -- the caller's prefix_lens[g]
  // cut to whole blocks and to the shortest member context, so every member
  // attends all of it -- and one prefix item per chunk of kN / G members.  Any
  // group start out of order disables sharing for the call (each sequence then
  // reads its own table row: the same result) and reports PA_DEVERR_PREFIX.
  // CTA 0 also records, per sequence, its partitions in all, its prefix and
  // its prefix item's first member for the merge kernel.
  int NV = S;   // virtual sequences: the sequences (their tails), then the prefixes
  if constexpr (SP) {
    constexpr int MB = kN / G;
    const int NGr = p.num_groups, P = p.partition_size;
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
      sctx[i] = p.context_lens[i];
      sp_eff[i] = 0;
      sp_npre[i] = 0;
      if (blockIdx.x == 0) p.ws_seq[2 * S + i] = i;
    }
    for (int i = threadIdx.x; i <= NGr; i += blockDim.x) gch[i] = 0;
    if (threadIdx.x == 0) sh.sp_ok = 1;
    __syncthreads();
    for (int g = threadIdx.x; g < NGr; g += blockDim.x) {
      const int a = p.group_start[g], b = p.group_start[g + 1];
      if (a < 0 || b < a || b > S) sh.sp_ok = 0;
    }
    __syncthreads();
    if (sh.sp_ok) {
      for (int g = threadIdx.x; g < NGr; g += blockDim.x) {
        const int a = p.group_start[g], b = p.group_start[g + 1];
        int m = p.prefix_lens[g];
        for (int i = a; i < b && m > 0; ++i) {
          const int c = sctx[i];
          m = (c <= 0 || ctx_invalid(p, c)) ? 0 : min(m, c);
        }
        const int eff = b - a >= 2 ? max(0, m / bs * bs) : 0;   // a group of one shares nothing
        if (eff > 0) {
          for (int i = a; i < b; ++i) {
            sp_eff[i] = eff;
            sp_npre[i] = (int16_t)((eff + P - 1) / P);
            if (blockIdx.x == 0) p.ws_seq[2 * S + i] = a + (i - a) / MB * MB;
          }
          gch[g] = (b - a + MB - 1) / MB;
        }
      }
    } else if (threadIdx.x == 0 && blockIdx.x == 0) {
      report(p.dev_err, PA_DEVERR_PREFIX);
    }
    __syncthreads();
    if (warp == 0) {   // exclusive scan: the first prefix item of each group, the total at gch[NGr]
      int carry = 0;
      for (int base = 0; base < NGr; base += 32) {
        const int i = base + lane;
        const int own = i < NGr ? gch[i] : 0;
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFull, x, o);
          if (lane >= o) x += y;
        }
        if (i < NGr) gch[i] = carry + x - own;
        carry += __shfl_sync(kFull, x, 31);
      }
      if (lane == 0) gch[NGr] = carry;
    }
    __syncthreads();
    NV = S + gch[NGr];
    for (int g = threadIdx.x; g < NGr; g += blockDim.x) {
      const int c0 = gch[g], nc = gch[g + 1] - c0;
      const int a = p.group_start[g], b = p.group_start[g + 1];
      for (int k = 0; k < nc; ++k) {
        pv_seq0[c0 + k] = (int16_t)(a + k * MB);
        pv_n[c0 + k] = (uint8_t)min(MB, b - a - k * MB);
        pv_eff[c0 + k] = sp_eff[a];
      }
    }
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
      const int c = sctx[i];
      const int tot = (c <= 0 || ctx_invalid(p, c)) ? 0 : sp_npre[i] + (c - sp_eff[i] + P - 1) / P;
      sp_tot[i] = (int16_t)tot;
      if (blockIdx.x == 0) {
        p.ws_seq[i] = tot;
        p.ws_seq[S + i] = sp_eff[i];
      }
    }
    __syncthreads();
  }
  // per virtual sequence its full partitions and its remainder's class, all
  // loaded at once (the planner orders the items below)
  for (int i = threadIdx.x; i < NV; i += blockDim.x) {
    int full, cls;
    if (SP && i >= S) {
      work_of_len(pv_eff[i - S], p.partition_size, full, cls);
    } else if (SP) {
      const int c = sctx[i];
      if (c <= 0 || ctx_invalid(p, c)) {
        full = 0;
        cls = 1;
      } else {
        work_of_len(c - sp_eff[i], p.partition_size, full, cls);
      }
    } else {
      work_of(p, p.context_lens[i], full, cls);
    }
    pre[i + 1] = full;
    rcls[i] = (uint8_t)cls;
  }
  for (int i = threadIdx.x; i < kClasses; i += blockDim.x) sh.u.ord.cnt[i] = 0;
  if (warp == 1) {
    tc::tmem_alloc(&sh.tmem_base, kCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (kSplitPlan && warp == 0) {
    // =================================================================== streamer (16-bit caches)
    // Takes the planner's items in order and streams each one's tiles: a free
    // stage, the tile's metadata, its block copies.
    int tile_seq = 0, item_seq = 0;
    bool aborted = false;
    for (;; ++item_seq) {
      const int rs = item_seq & 1;
      if (!__all_sync(kFull, mbar_wait(&sh.rec_full[rs], (item_seq >> 1) & 1)) || sh.abort_flag) {
        aborted = true;
        break;
      }
      const ItemRec& R = sh.u.rec[rs];
      if (R.item < 0) break;   // no more work
      const int s = R.s, kvh = R.kvh, part = R.part, n_parts = R.n_parts, t_first = R.t_first;
      const int t0 = R.t0, t1 = R.t1, jb = R.jb;
      const int seq0 = R.seq0, ncol = R.ncol, pbase = R.pbase, qslot = R.qslot;
      const int id_lane = R.ids[lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.rec_empty[rs]);
      const int32_t* row = p.block_tables + (int64_t)s * p.bt_stride;   // entry table_index(j) holds block j
      const int ntiles = (t1 - t0 + kTile - 1) / kTile;
      // 16-bit: the block id of this lane's chunk of tile k.  The item's first 32
      // come from the prefetched id_lane; a later one is loaded a tile ahead, so
      // the load overlaps the wait for a free stage instead of delaying the copy.
      auto tile_id = [&](int k) {
        const int bi = k * (kTile / bs) + lane;
        const int nbk = (min(kTile, t1 - (t0 + k * kTile)) + bs - 1) / bs;
        const int id_sh = __shfl_sync(kFull, id_lane, bi & 31);
        return lane < nbk ? (bi < 32 ? id_sh : row[table_index(jb + bi, p.ring_blocks)]) : 0;
      };
      int id_k = ntiles > 0 ? tile_id(0) : 0;
      bool item_bad = false;
      for (int k = 0; k < ntiles; ++k) {
        const int slot = tile_seq % NS;
        if (tile_seq >= NS && !mbar_wait(&sh.empty[slot], ((tile_seq / NS) - 1) & 1)) {
          aborted = true;
          break;
        }
        const int valid = min(kTile, t1 - (t0 + k * kTile));
        const int nb = (valid + bs - 1) / bs;
        // an id out of range is never read: block 0 stands in, the item's
        // result is discarded (zero rows) and the error reported once per item
        const bool id_bad = lane < nb && (id_k < 0 || id_k >= p.num_blocks);
        if (__any_sync(kFull, id_bad)) {
          if (lane == 0 && !item_bad) report(p.dev_err, PA_DEVERR_BLOCK_ID);
          item_bad = true;
        }
        if (id_bad) id_k = 0;
        if (lane == 0) {
          TileMeta m;
          m.s = s; m.kvh = kvh; m.part = part; m.valid = valid;
          m.last = (k == ntiles - 1); m.qslot = qslot; m.n_parts = n_parts;
          m.lo = max(0, t_first - (t0 + k * kTile));
          m.tail = ntiles - 1 - k;
          m.qinv = 1.f;
          m.seq0 = seq0; m.ncol = ncol; m.pbase = pbase;
          m.head = k; m.item = item_seq; m.bad = item_bad ? 1 : 0;
          sh.meta[slot] = m;
          mbar_arrive_expect_tx(&sh.full[slot], (uint32_t)(nb * chunk_bytes));
        }
        __syncwarp();
        if (lane < nb)
          bulk_g2s(stages + slot * kStage + lane * chunk_bytes,
                   p.cache + ((int64_t)id_k * Hkv + kvh) * chunk_bytes, (uint32_t)chunk_bytes, &sh.full[slot]);
        if (k + 1 < ntiles) id_k = tile_id(k + 1);
        ++tile_seq;
      }
      if (aborted) break;
    }
    // ---- no more work: a stage whose metadata says so
    const int slot = tile_seq % NS;
    if (!aborted && tile_seq >= NS && !mbar_wait(&sh.empty[slot], ((tile_seq / NS) - 1) & 1)) aborted = true;
    if (lane == 0) {
      // never leave copies in flight, whether or not another role gave up:
      // wait (bounded) for the latest phase of every stage.  Normally they
      // have landed or are about to, and the end mark below is only read
      // after the last tile anyway.
      for (int t = max(0, tile_seq - NS); t < tile_seq; ++t)
        if (!mbar_wait(&sh.full[t % NS], (t / NS) & 1)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    if (lane == 0) {
      if (aborted) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      sh.meta[slot].s = -1;
      sh.meta[slot].item = item_seq;     // the index the next item would have
      mbar_arrive(&sh.full[slot]);
    }
    __syncwarp();
  } else if (warp == kPlanWarp) {
    // =================================================================== planner
    int carry = 0;
    for (int base = 0; base < NV; base += 32) {
      int x = (base + lane < NV) ? pre[base + lane + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (base + lane < NV) pre[base + lane + 1] = carry + x;
      carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) pre[0] = 0;
    __syncwarp();
    // Item order (identical in every CTA): all full partitions in (sequence,
    // partition) order, then the remainder partitions from the most tiles down,
    // stably by sequence; kv heads innermost.  CTAs take the items round by
    // round in snake order (c, then 151 - c, ...), so every CTA gets about the
    // same number of tiles (longest first).
    const int n_full = carry;
    // remainder partitions per class: one shared-memory atomic per distinct
    // class per 32 virtual sequences (most share a class)
    for (int base = 0; base < NV; base += 32) {
      const int i = base + lane;
      const int cls = i < NV ? rcls[i] : -1;
      const uint32_t same = __match_any_sync(kFull, cls);
      if (cls >= 0 && (same & ((1u << lane) - 1u)) == 0) atomicAdd(&sh.u.ord.cnt[cls], __popc(same));
    }
    __syncwarp();
    // each class's first slot: an exclusive scan over the classes from the
    // most tiles down (class c at index kClasses - 1 - c), 32 at a time
    {
      int at = 0;
      for (int base = 0; base < kClasses - 1; base += 32) {
        const int c = kClasses - 1 - (base + lane);   // classes kClasses-1 .. 1
        const int own = c >= 1 ? sh.u.ord.cnt[c] : 0;
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kFull, x, o);
          if (lane >= o) x += y;
        }
        if (c >= 1) sh.u.ord.cur[c] = at + x - own;
        at += __shfl_sync(kFull, x, 31);
      }
      __syncwarp();
      if (lane == 0) sh.u.ord.cnt[0] = at;   // remainder partitions in all
    }
    __syncwarp();
    for (int base = 0; base < NV; base += 32) {
      const int i = base + lane;
      const int cls = i < NV ? rcls[i] : 0;
      const uint32_t same = __match_any_sync(kFull, cls);
      const int slot_in = __popc(same & ((1u << lane) - 1u));
      if (cls > 0) rseq[sh.u.ord.cur[cls] + slot_in] = (int16_t)i;
      __syncwarp();
      if (cls > 0 && slot_in == 0) sh.u.ord.cur[cls] += __popc(same);
      __syncwarp();
    }
    const int total = (n_full + sh.u.ord.cnt[0]) * Hkv;
    const int P = p.partition_size;
    // the item a CTA takes in round k (snake order); >= total: none
    auto item_of_round = [&](int k) {
      return k * (int)gridDim.x + ((k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
    };
    const bool windowed = p.window > 0 || p.ring_blocks > 0;
    constexpr int kQChunks = (CN * 16 + 31) / 32;
    // What an item is (virtual sequence, kv head, partition, table row, columns,
    // context and first block) is worked out 32 rounds at a time, lane l for
    // round rbase + l, and handed to the item by shuffles: the set-up of an item
    // never walks the shared-memory tables or waits for its context length.
    struct Desc {
      int v, kvh, part, row, ctx;   // virtual sequence, kv head, partition, table row, its end
      int t0, seq0, ncol, pbase;    // shared prefix: first position, column map, partition base
      int fb;                       // the partition's first logical block
    };
    auto describe = [&](int k) {   // per lane; a round past the last item gets v = -1
      Desc d;
      const int it = item_of_round(k);
      d.v = -1;
      d.kvh = d.part = d.row = d.ctx = d.t0 = d.seq0 = d.ncol = d.pbase = d.fb = 0;
      if (it < total) {
        const int j = it / Hkv;
        d.kvh = it - j * Hkv;
        if (j < n_full) {
          int lo = 0, hi = NV - 1;   // last virtual sequence whose first full partition is <= j
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= j) lo = mid;
            else hi = mid - 1;
          }
          d.v = lo;
          d.part = j - pre[lo];
        } else {
          d.v = rseq[j - n_full];
          d.part = pre[d.v + 1] - pre[d.v];   // the remainder follows the full partitions
        }
        if (SP && d.v >= S) {   // a group's shared prefix, read through its first member's row
          const int k2 = d.v - S;
          d.row = d.seq0 = pv_seq0[k2];
          d.ncol = pv_n[k2] * G;
          d.ctx = pv_eff[k2];
        } else {                // a sequence (shared prefix: its tail after the prefix)
          d.row = d.seq0 = d.v;
          d.ncol = G;
          d.ctx = SP ? sctx[d.v] : p.context_lens[d.v];
          d.t0 = SP ? sp_eff[d.v] : 0;
          d.pbase = SP ? sp_npre[d.v] : 0;
        }
        d.fb = windowed ? (attended_from(p, d.ctx) + d.part * P) / bs
                        : d.t0 / bs + d.part * (P / bs);   // P is a multiple of 128, bs divides it
      }
      return d;
    };
    int rbase = 0;
    Desc dl = describe(lane);
    // round k's description; every lane calls it, k never decreases, and a
    // call for k never follows one for k + 3 or later (the window keeps the
    // two rounds before the one that moves it)
    auto desc_of = [&](int k) {
      if (k >= rbase + 32) {
        rbase = k - 2;
        dl = describe(rbase + lane);
      }
      const int l = k - rbase;
      Desc d;
      d.v = __shfl_sync(kFull, dl.v, l);
      d.kvh = __shfl_sync(kFull, dl.kvh, l);
      d.part = __shfl_sync(kFull, dl.part, l);
      d.row = __shfl_sync(kFull, dl.row, l);
      d.ctx = __shfl_sync(kFull, dl.ctx, l);
      d.t0 = __shfl_sync(kFull, dl.t0, l);
      d.seq0 = __shfl_sync(kFull, dl.seq0, l);
      d.ncol = __shfl_sync(kFull, dl.ncol, l);
      d.pbase = __shfl_sync(kFull, dl.pbase, l);
      d.fb = __shfl_sync(kFull, dl.fb, l);
      return d;
    };
    // An item's loads (its first 32 block ids, the query rows) are issued a
    // round ahead, while the item before it streams, and the lines they read
    // are brought into L2 a round before that (prefetch_item), so that they
    // have arrived when the item starts even if the item before it is short.
    auto prefetch_item = [&](const Desc& d) {
      // the query rows: lane l takes 128-byte line l (column l / 2, half l % 2)
      const int n = lane >> 1;
      if (n < d.ncol && n < CN)
        prefetch_l2(static_cast<const T*>(p.q) + (int64_t)(d.seq0 + n / G) * p.q_seq_stride +
                    (int64_t)(d.kvh * G + n % G) * kD + (lane & 1) * 64);
      if (lane == 0) {
        const int ti = windowed ? table_index(d.fb, p.ring_blocks) : d.fb;
        if (ti >= 0 && ti < p.bt_stride) prefetch_l2(p.block_tables + (int64_t)d.row * p.bt_stride + ti);
      }
    };
    struct Item {
      int id_lane;
      uint4 qv[kQChunks];
    };
    auto fetch = [&](const Desc& d) {
      Item r;
      const int ti = windowed ? table_index(d.fb + lane, p.ring_blocks) : d.fb + lane;
      if (!windowed) {
        // the partition's later block ids, checked when the item starts: into L2
        // now, a whole item ahead, so that check waits for L2, not HBM (lane i
        // covers ids 32 (i + 1) .. 32 (i + 1) + 31; P / bs <= 1024)
        const int row_end = min(p.bt_stride, d.fb + P / bs);
        const int t = d.fb + 32 * (lane + 1);
        if (t < row_end) {
          const int32_t* rp = p.block_tables + (int64_t)d.row * p.bt_stride;
          prefetch_l2(rp + t);
          prefetch_l2(rp + min(t + 31, row_end - 1));
        }
      }
      r.id_lane =
          (lane < P / bs && ti < p.bt_stride && ti >= 0) ? p.block_tables[(int64_t)d.row * p.bt_stride + ti] : 0;
      // query rows: column n is head kvh * G + n % G of sequence seq0 + n / G
#pragma unroll
      for (int k = 0; k < kQChunks; ++k) {
        const int c = lane + 32 * k, n = c >> 4;
        const T* qsrc = static_cast<const T*>(p.q) + (int64_t)(d.seq0 + n / G) * p.q_seq_stride +
                        (int64_t)(d.kvh * G + n % G) * kD;
        r.qv[k] = (c < CN * 16 && n < d.ncol) ? *reinterpret_cast<const uint4*>(qsrc + (c & 15) * 8)
                                               : make_uint4(0, 0, 0, 0);
      }
      return r;
    };
    int tile_seq = 0, item_seq = 0;
    bool aborted = false;
    Item nxt;
    if (item_of_round(0) < total) nxt = fetch(desc_of(0));
    if (item_of_round(1) < total) prefetch_item(desc_of(1));
    for (int round = 0; item_of_round(round) < total && !aborted; ++round) {
      const Desc cd = desc_of(round);
      const Item cur = nxt;
      const bool more = item_of_round(round + 1) < total;
      if (more) nxt = fetch(desc_of(round + 1));
      if (item_of_round(round + 2) < total) prefetch_item(desc_of(round + 2));
      const int s = cd.row, kvh = cd.kvh, part = cd.part, ctx = cd.ctx, id_lane = cur.id_lane;
      const int32_t* row = p.block_tables + (int64_t)s * p.bt_stride;   // entry table_index(j) holds block j
      const bool is_prefix = SP && cd.v >= S;                          // valid by construction
      if (!is_prefix && ctx_invalid(p, ctx)) {
        warp_zero_rows<T, G>(p, s, kvh, lane);
        if (lane == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
        continue;
      }
      if (!is_prefix && ctx <= 0) {
        warp_zero_rows<T, G>(p, s, kvh, lane);
        continue;
      }
      const int t_first = SP ? cd.t0 : window_start(ctx, bs, p.window, p.ring_blocks);
      const int t_base = (t_first / bs) * bs;
      const int n_parts = (ctx - t_base + P - 1) / P;
      const int t0 = t_base + part * P, t1 = min(ctx, t0 + P);
      const int jb = t0 / bs;
      const int nblk = (t1 - t0 + bs - 1) / bs;
      // 8-bit caches check the item's block ids before it starts; 16-bit
      // caches check each tile's ids as they are issued (no round trip before
      // the item's first copy) and mark the item bad instead
      bool bad = false;
      if constexpr (I8) {
        bad = lane < nblk && (id_lane < 0 || id_lane >= p.num_blocks);
#pragma unroll 4
        for (int b = lane + 32; b < nblk; b += 32) {   // unrolled: several loads in flight
          const int id = row[table_index(jb + b, p.ring_blocks)];
          bad |= (id < 0 || id >= p.num_blocks);
        }
      }
      if (__any_sync(kFull, bad)) {
        if (lane == 0) report(p.dev_err, PA_DEVERR_BLOCK_ID);
        if constexpr (SP) {
          // per column: a row written directly is zeroed, else the partition is
          // marked invalid and the merge writes zeros
          for (int n = 0; n < cd.ncol; ++n) {
            const int sq = cd.seq0 + n / G;
            const int64_t hrow = (int64_t)sq * p.num_q_heads + kvh * G + n % G;
            if (sp_eff[sq] == 0 && sp_tot[sq] == 1) {
              if (lane < kD / 8) *reinterpret_cast<uint4*>(static_cast<T*>(p.out) + hrow * kD + lane * 8) =
                  make_uint4(0, 0, 0, 0);
            } else if (lane == 0) {
              const int64_t r = hrow * p.max_parts + cd.pbase + part;
              p.ws_ml[r * 2 + 0] = 0.f;
              p.ws_ml[r * 2 + 1] = -1.f;
            }
          }
        } else if (n_parts == 1) {
          warp_zero_rows<T, G>(p, s, kvh, lane);
        } else if (lane < G) {
          const int64_t r = ((int64_t)s * p.num_q_heads + kvh * G + lane) * p.max_parts + part;
          p.ws_ml[r * 2 + 0] = 0.f;
          p.ws_ml[r * 2 + 1] = -1.f;   // invalid partition: the merge writes zeros
        }
        continue;
      }
      // ---- Q^T of this item into a K-major 128B-swizzled buffer
      constexpr int QS = q_slots(I8);
      const int qslot = item_seq % QS;
      if (item_seq >= QS && !mbar_wait(&sh.q_free[qslot], ((item_seq / QS) - 1) & 1)) {
        aborted = true;
        break;
      }
      float qinv = 1.f;
      {
        uint8_t* qb = qbuf + qslot * kQBytes;
        uint4 qw[kQChunks];
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) qw[k] = cur.qv[k];
        if constexpr (kQConvert) {
          // bf16 -> fp16 times 2^e, e chosen so the item's max |q| lands in
          // [2^14, 2^15): exact for every element within 2^28 of the max
          float mx = 0.f;
#pragma unroll
          for (int k = 0; k < kQChunks; ++k) {
            const uint32_t w[4] = {qw[k].x, qw[k].y, qw[k].z, qw[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = Elem<T>::to_float2(w[i]);
              mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o2));
          int e = 0;
          if (mx > 0.f) e = min(100, max(-100, 14 - ilogbf(mx)));
          const float up = ldexpf(1.f, e);
          qinv = ldexpf(1.f, -e);
#pragma unroll
          for (int k = 0; k < kQChunks; ++k) {
            uint32_t w[4] = {qw[k].x, qw[k].y, qw[k].z, qw[k].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = Elem<T>::to_float2(w[i]);
              w[i] = Elem<__half>::pack2(f.x * up, f.y * up);
            }
            qw[k] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = lane + 32 * k;
          if (c < CN * 16) {
            const int n = c >> 4, cc = c & 15, atom = cc >> 3, piece = cc & 7;
            *reinterpret_cast<uint4*>(qb + (atom * 2 + (n >> 3)) * 1024 + (n & 7) * 128 + ((piece ^ (n & 7)) << 4)) =
                qw[k];
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      // ---- 8-bit: the tiles, as descriptors for the copy warp; 16-bit: the
      // item, as a record for the streaming warp
      const int ntiles = (t1 - t0 + kTile - 1) / kTile;
      for (int k = 0; k < ntiles && I8; ++k) {
        // 8-bit: each tile goes to the copy warp as a descriptor (metadata and
        // block ids); it stages the tile as two 64-token half tiles
        const int valid = min(kTile, t1 - (t0 + k * kTile));
        TileMeta m;
        m.s = s; m.kvh = kvh; m.part = part; m.valid = valid;
        m.last = (k == ntiles - 1); m.qslot = qslot; m.n_parts = n_parts;
        m.lo = max(0, t_first - (t0 + k * kTile));
        m.tail = ntiles - 1 - k;
        m.qinv = qinv;
        m.seq0 = cd.seq0; m.ncol = cd.ncol; m.pbase = cd.pbase;
        m.head = k; m.item = item_seq; m.bad = 0;
        // the tile's block ids, lane i holding blocks i + 32 c of the tile: the
        // item's first 32 come from the prefetched id_lane, the rest are loaded
        // here, all in flight together
        const int nbt = (valid + bs - 1) / bs;
        int idr[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int b = lane + 32 * c, bi = k * (kTile / bs) + b;
          const int id_sh = __shfl_sync(kFull, id_lane, bi & 31);
          idr[c] = b < nbt ? (bi < 32 ? id_sh : row[table_index(jb + bi, p.ring_blocks)]) : 0;
        }
        // hand the tile to the copy warp
        const int d = tile_seq % kND;
        if (tile_seq >= kND && !mbar_wait(&sh.desc_empty[d], ((tile_seq / kND) - 1) & 1)) {
          aborted = true;
          break;
        }
        if (lane == 0) sh.desc[d].meta = m;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (lane + 32 * c < nbt) sh.desc[d].ids[lane + 32 * c] = idr[c];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.desc_full[d]);
        if (aborted) break;
        ++tile_seq;
      }
      if constexpr (!I8) {
        // hand the item to the streaming warp, in the record slot of its
        // parity once the streamer has taken the item two before it
        const int rs = item_seq & 1;
        if (item_seq >= 2 && !__all_sync(kFull, mbar_wait(&sh.rec_empty[rs], ((item_seq >> 1) - 1) & 1))) {
          aborted = true;
          break;
        }
        ItemRec& R = sh.u.rec[rs];
        if (lane == 0) {
          R.s = s; R.kvh = kvh; R.part = part; R.n_parts = n_parts; R.t_first = t_first;
          R.t0 = t0; R.t1 = t1; R.jb = jb;
          R.seq0 = cd.seq0; R.ncol = cd.ncol; R.pbase = cd.pbase; R.qslot = qslot; R.item = item_seq;
        }
        R.ids[lane] = id_lane;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.rec_full[rs]);
      }
      ++item_seq;
    }
    // ---- no more work: a stage (8-bit: a raw half tile) whose metadata says so
    if (I8) {
      // a descriptor that says so; the copy warp passes it on to both halves
      const int d = tile_seq % kND;
      if (!aborted && tile_seq >= kND && !mbar_wait(&sh.desc_empty[d], ((tile_seq / kND) - 1) & 1)) aborted = true;
      if (lane == 0) {
        if (aborted) {
          report(p.dev_err, PA_DEVERR_TIMEOUT);
          sh.abort_flag = 1;
        }
        sh.desc[d].meta.s = -1;
        sh.desc[d].meta.item = item_seq;   // the index the next item would have
        mbar_arrive(&sh.desc_full[d]);
      }
    } else {
      // a record that says so (once the streamer has taken the item two before)
      const int rs = item_seq & 1;
      if (!aborted && item_seq >= 2 && !__all_sync(kFull, mbar_wait(&sh.rec_empty[rs], ((item_seq >> 1) - 1) & 1)))
        aborted = true;
      if (lane == 0) {
        if (aborted) {
          report(p.dev_err, PA_DEVERR_TIMEOUT);
          sh.abort_flag = 1;
        }
        sh.u.rec[rs].item = -1;
        mbar_arrive(&sh.rec_full[rs]);
      }
    }
    __syncwarp();
  } else if (warp == 1 && !kSplitIssue) {
    // =================================================================== MMA issuer (8-bit caches)
    // Event-driven: QK(t) as soon as tile t has landed (converted) and its S
    // buffer is free, PV(t) as soon as P(t) is written and its O buffer is free
    // -- neither waits for the other stream, so a stage is released right after
    // its own PV.  The barriers are tested without blocking.
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16(128, kN, kBF16, false, false);
      const uint32_t id_pv = tc::idesc_f16(128, NPV, kBF16, true, true);
      uint32_t used = 0, par = 0;   // per O slot: used by an item yet, parity of its uses
      int qk = 0, pv = 0, end = 0x7fffffff;
      uint32_t idle = 0;
      bool ok = true;
      while (pv < end) {
        bool progressed = false;
        if (qk < end) {
          const int slot = qk % NS;
          if (mbar_test_wait(&sh.full[slot], (qk / NS) & 1)) {
            const TileMeta m = sh.meta[slot];
            if (m.s < 0) {
              end = qk;
              progressed = true;
            } else if (qk < 2 || mbar_test_wait(&sh.s_free[qk & 1], ((qk >> 1) - 1) & 1)) {
              tc::fence_after_sync();
              const uint32_t st = smem_u32(stages + slot * kStage), qa = smem_u32(qbuf + m.qslot * kQBytes);
  #pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t qd = tc::smem_desc(qa + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B);
                if constexpr (I8)   // K (fp16, token = TMEM lane) converted into TMEM: 16 dims = 8 columns
                  tc::mma_f16_ta(tmem + (qk & 1) * 16, tmem + kKCol + slot * 64 + kk * 8, qd, id_qk, kk > 0);
                else
                  tc::mma_f16(tmem + (qk & 1) * 16,
                              tc::smem_desc(st + (kk >> 2) * 1024 + (kk & 3) * 32, 16, kGroupBytes, tc::kSwizzle128B),
                              qd, id_qk, kk > 0);
              }
              tc::commit(&sh.s_full[qk & 1]);
              if (m.last) tc::commit(&sh.q_free[m.qslot]);
              ++qk;
              progressed = true;
            }
          }
        }
        if (pv < qk) {
          // PV(pv) accumulates into the O slot of its item (one softmax group):
          // the item's first tile overwrites it once the output warps have read
          // the slot's previous item; its last tile signals the output warps
          const int pb = pv & 1;
          if (mbar_test_wait(&sh.p_full[pb], (pv >> 1) & 1)) {
            const int slot = pv % NS;
            const TileMeta& mr = sh.meta[slot];     // the stage is not refilled before this PV completes
            const int valid = mr.valid, os = mr.item % item_slots(I8);
            const bool first = mr.head == 0, lastg = mr.tail == 0;
            if (!first || !((used >> os) & 1) || mbar_test_wait(&sh.ofree[os], ((par >> os) & 1) ^ 1)) {
              tc::fence_after_sync();
              const uint32_t st = smem_u32(stages + slot * kStage), pa = smem_u32(pbuf + pb * kPBytes);
              const int nsteps = (valid + 15) >> 4;
              // V of 8-token group g: at g * 4 KiB + 2 KiB among the K atoms (16-bit
              // caches), at g * 2 KiB in a V-only stage (8-bit caches)
              constexpr uint32_t kVGroup = I8 ? 2048 : kGroupBytes, kVOff = I8 ? 0 : 2048;
              for (int kk = 0; kk < nsteps; ++kk)
                tc::mma_f16(tmem + kOCol + os * 32,
                            tc::smem_desc(st + kk * 2 * kVGroup + kVOff, 1024, kVGroup, tc::kSwizzle128B),
                            tc::smem_desc(pa + kk * (NPV / 8) * 256, (NPV / 8) * 128, 128, tc::kSwizzleNone), id_pv,
                            (kk > 0 || !first) ? 1u : 0u);
              tc::commit(&sh.pv_done[pb]);
              tc::commit(&sh.empty[slot]);
              if (lastg) tc::commit(&sh.ofin[os]);
              if (first) {
                used |= 1u << os;
                par ^= 1u << os;
              }
              ++pv;
              progressed = true;
            }
          }
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > kSpinLimit || sh.abort_flag) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      // every MMA this lane issued completes before TMEM can be freed
      tc::commit(&sh.mma_drain[0]);
      if (!mbar_wait(&sh.mma_drain[0], 0)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =================================================================== QK issuer (16-bit caches)
    // One lane: QK(t) as soon as tile t has landed and its S buffer is free.
    // The PV products have their own issuer warp, so neither stream waits for
    // the other's issue.  Descriptors are built once per tile and advanced by
    // constant offsets (16-byte units in the start-address field).
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16(128, kN, kBF16, false, false);
      int qk = 0;
      bool ok = true;
      while (true) {
        const int slot = qk % NS;
        if (!mbar_spin(&sh.full[slot], (qk / NS) & 1) || sh.abort_flag) { ok = false; break; }
        const TileMeta m = sh.meta[slot];
        if (m.s < 0) break;
        if (qk >= 2 && !mbar_spin(&sh.s_free[qk & 1], ((qk >> 1) - 1) & 1)) { ok = false; break; }
        // the softmax warps take the tile's metadata from here (smeta[b] was
        // last read for tile qk - 2, before its S buffer was freed)
        sh.smeta[qk & 1] = m;
        mbar_arrive(&sh.m_full[qk & 1]);
        tc::fence_after_sync();
        const uint64_t qd = tc::smem_desc(smem_u32(qbuf + m.qslot * kQBytes), 16, 1024, tc::kSwizzle128B);
        const uint64_t kd = tc::smem_desc(smem_u32(stages + slot * kStage), 16, kGroupBytes, tc::kSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t q_k = qd + (uint64_t)((((kk >> 2) * 2048) + (kk & 3) * 32) >> 4);
          if constexpr (I8)   // K (fp16, token = TMEM lane) converted into TMEM: 16 dims = 8 columns
            tc::mma_f16_ta(tmem + (qk & 1) * 16, tmem + kKCol + slot * 64 + kk * 8, q_k, id_qk, kk > 0);
          else
            tc::mma_f16(tmem + (qk & 1) * 16, kd + (uint64_t)((((kk >> 2) * 1024) + (kk & 3) * 32) >> 4), q_k, id_qk,
                        kk > 0);
        }
        tc::commit(&sh.s_full[qk & 1]);
        if (m.last) tc::commit(&sh.q_free[m.qslot]);
        ++qk;
      }
      sh.end_tile = qk;   // the PV issuer stops there
      const int end_item = sh.meta[qk % NS].item;   // the end mark's (valid when ok)
      if (ok) {
        // no more work: both metadata buffers say so (marked with the end tile,
        // so only the softmax warps waiting for tile `end` pass it on), once
        // the softmax warps have read the last metadata of each buffer (they
        // release S(t) after reading smeta for tile t)
        const int end = qk;
        for (int u = max(0, end - 2); u < end && ok; ++u)
          ok = mbar_wait(&sh.s_free[u & 1], (u >> 1) & 1);
        if (ok) {
          for (int b2 = 0; b2 < 2; ++b2) {
            sh.smeta[b2].s = -1;
            sh.smeta[b2].valid = end;
            sh.smeta[b2].item = end_item;
            mbar_arrive(&sh.m_full[b2]);
          }
        }
      }
      if (!ok) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      // every MMA this lane issued completes before TMEM can be freed
      tc::commit(&sh.mma_drain[0]);
      if (!mbar_wait(&sh.mma_drain[0], 0)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (kSplitIssue && warp == kPVWarp) {
    // =================================================================== PV issuer (16-bit caches)
    // One lane: PV(t) as soon as P(t) is written and its O buffer is free; the
    // commit after it releases the stage (QK(t) completed before the softmax of
    // tile t began).
    if (lane == 0) {
      const uint32_t id_pv = tc::idesc_f16(128, NPV, kBF16, true, true);
      // V of 8-token group g: at g * 4 KiB + 2 KiB among the K atoms (16-bit
      // caches), at g * 2 KiB in a V-only stage (8-bit caches)
      constexpr uint32_t kVGroup = I8 ? 2048 : kGroupBytes, kVOff = I8 ? 0 : 2048;
      constexpr bool PP = ping_pong(I8, CN);
      // PV(pv) accumulates into the O slot of (its item's slot, its softmax
      // group): a group's first tile of an item overwrites the slot once the
      // output warps have read the slot's previous item; its last tile
      // signals the output warps
      uint32_t used = 0, par = 0;   // per O slot: used by an item yet, parity of its uses
      int pv = 0;
      uint32_t idle = 0;
      bool ok = true;
      while (pv < sh.end_tile) {
        const int pb = pv & 1;
        bool issued = false;
        if (mbar_test_wait(&sh.p_full[pb], (pv >> 1) & 1)) {
          const int slot = pv % NS;
          const TileMeta& mr = sh.meta[slot];   // the stage is not refilled before this PV completes
          const int valid = mr.valid;
          const int os = (mr.item % item_slots(I8)) * (PP ? 2 : 1) + (PP ? pb : 0);
          const bool first = PP ? mr.head < 2 : mr.head == 0, lastg = PP ? mr.tail < 2 : mr.tail == 0;
          if (!first || !((used >> os) & 1) || mbar_test_wait(&sh.ofree[os], ((par >> os) & 1) ^ 1)) {
            tc::fence_after_sync();
            const uint64_t vd =
                tc::smem_desc(smem_u32(stages + slot * kStage) + kVOff, 1024, kVGroup, tc::kSwizzle128B);
            // P^T: 8-token groups at the start of the stage's groups (I8: in a P^T buffer)
            const uint64_t pd = I8 ? tc::smem_desc(smem_u32(pbuf + pb * kPBytes), (NPV / 8) * 128, 128, tc::kSwizzleNone)
                                   : tc::smem_desc(smem_u32(stages + slot * kStage), kGroupBytes, 128, tc::kSwizzleNone);
            constexpr uint32_t kPStep = I8 ? (NPV / 8) * 256 : 2 * kGroupBytes;   // 16 tokens
            const int nsteps = (valid + 15) >> 4;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              if (kk < nsteps)
                tc::mma_f16(tmem + kOCol + os * 32, vd + (uint64_t)((kk * 2 * kVGroup) >> 4),
                            pd + (uint64_t)((kk * kPStep) >> 4), id_pv, (kk > 0 || !first) ? 1u : 0u);
            tc::commit(&sh.pv_done[pb]);
            tc::commit(&sh.empty[slot]);
            if (lastg) tc::commit(&sh.ofin[os]);
            if (first) {
              used |= 1u << os;
              par ^= 1u << os;
            }
            ++pv;
            issued = true;
          }
        }
        if (issued) {
          idle = 0;
        } else if (++idle > kSpinLimit || sh.abort_flag) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      tc::commit(&sh.mma_drain[1]);
      if (!mbar_wait(&sh.mma_drain[1], 0)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if ((warp >= 2 && warp < 6) || (ping_pong(I8, CN) && warp >= kSoftB && warp < kSoftB + 4)) {
    // =================================================================== softmax warps (2-5, group 1)
    // (wait results are made warp-uniform in the softmax and output warps: the
    // TMEM loads after them are warp-collective and must never run diverged)
    // Tile t: S^T -> tile maxima -> P^T (hi, lo) for the PV product; at the end
    // of an item, the normaliser.  Hands per-tile factors to the output warps.
    // With two warpgroups, group g takes tiles t = g mod 2 and keeps its own
    // running maximum and sums for the item; the output warps merge the two.
    constexpr bool PP = ping_pong(I8, CN);
    const int grp = (PP && warp >= kSoftB) ? 1 : 0;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // TMEM lane = token row of S^T
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    // The running maxima are the same in every thread of the group.  With
    // more than 8 columns each warp keeps them in shared memory (row mb of its
    // double-buffered copy) and reads them back with broadcast vector loads
    // where they are needed, which keeps the per-thread state small enough
    // that nothing spills.
    constexpr bool kSM = CN > 8;
    float m[kSM ? 1 : CN], lp[CN];
    float* mrow = sh.mrun[grp][quarter][0];
    float* crow = sh.mcorr[grp][quarter];
    int mb = 0;
#pragma unroll
    for (int n = 0; n < CN; ++n) lp[n] = 0.f;
    if constexpr (kSM) {
      if (lane < kN) mrow[lane] = -INFINITY;
      __syncwarp();
    } else {
#pragma unroll
      for (int n = 0; n < CN; ++n) m[n] = -INFINITY;
    }
    auto load_m = [&](float (&mv)[CN]) {   // the running maxima of the CN columns
      if constexpr (kSM) {
#pragma unroll
        for (int n = 0; n < CN; n += 4) {
          const float4 v = *reinterpret_cast<const float4*>(mrow + mb * kN + n);
          mv[n] = v.x;
          mv[n + 1] = v.y;
          mv[n + 2] = v.z;
          mv[n + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int n = 0; n < CN; ++n) mv[n] = m[n];
      }
    };
    int tile_seq = grp;
    bool ok = true;
    while (true) {
      const int slot = tile_seq % NS;
      const int hb = tile_seq & 1;
      // the tile's metadata: with one group straight from the stage (it comes
      // with the stage's barrier); with two, forwarded by the QK issuer per S
      // buffer, so each group only ever waits on its own buffer's phases
      TileMeta mt;
      if constexpr (PP) {
        if (!__all_sync(kFull, mbar_wait(&sh.m_full[hb], (tile_seq >> 1) & 1))) { ok = false; break; }
        mt = sh.smeta[hb];
      } else {
        if (!__all_sync(kFull, mbar_wait(&sh.full[slot], (tile_seq / NS) & 1))) { ok = false; break; }
        mt = sh.meta[slot];
      }
      if (__any_sync(kFull, mt.s < 0 || sh.abort_flag)) {
        // tell the output warps there is no more work (the group whose turn
        // the end tile is; the forwarded end mark carries the end tile in valid
        // and the index the next item would have in item), in the hand-off slot
        // of that item index once its previous user is done
        if (mt.s < 0 && (!PP || mt.valid == tile_seq)) {
          constexpr int IS = item_slots(I8);
          const int k = mt.item, q = k % IS;
          if (k >= IS && !__all_sync(kFull, mbar_wait(&sh.c_free[q], ((k / IS) - 1) & 1))) { ok = false; break; }
          if (lane == 0 && quarter == 0) sh.ihand[q].meta.s = -1;
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sh.c_full[q]);
            if (PP) mbar_arrive(&sh.c_full[q]);
          }
        }
        break;
      }
      // this group's first and last tiles of the item: the first starts its O
      // accumulator afresh, the last hands over its maximum and sums
      const bool first = PP ? mt.head < 2 : mt.head == 0;
      const bool fin = PP ? mt.tail < 2 : mt.tail == 0;
      const int os = (mt.item % item_slots(I8)) * (PP ? 2 : 1) + grp;   // this group's O slot for the item
      const int sb = tile_seq & 1;
      if (!__all_sync(kFull, mbar_wait(&sh.s_full[sb], (tile_seq >> 1) & 1))) { ok = false; break; }
      tc::fence_after_sync();
      float sv[16];
      tc::tmem_ld16(lane_addr + sb * 16, sv);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_free[sb]);
      const bool rv = row >= mt.lo && row < mt.valid;
      // 8-bit: K_t = sk_t * codes and V_t = sv_t * codes; sk_t scales this row's
      // scores and sv_t its P^T row (the normaliser keeps the unscaled p)
      const float kscale = I8 ? sh.sk[slot][row] * (p.scale_log2 * mt.qinv) : p.scale_log2;
      const float vscale = I8 ? sh.sv[slot][row] : 1.f;
      // scores; does any exceed the running maximum by more than kLazyMax?  (On
      // the group's first tile of an item m = -inf, so every valid row does.)
      float x[CN];
      bool up = false;
      {
        float mv[CN];
        load_m(mv);
#pragma unroll
        for (int n = 0; n < CN; ++n) {
          x[n] = rv ? sv[n] * kscale : -INFINITY;
          up |= x[n] > mv[n] + (I8 ? 0.f : kLazyMax);   // 8-bit: the V scales ride on P, keep p <= 1
        }
      }
      const bool wup = __any_sync(kFull, up);
      const int par = (tile_seq >> 1) & 1;   // exchange buffer of this tile (the group's tile parity)
      if (wup) {   // this warp's column maxima over its 32 rows (one warp reduction per column)
#pragma unroll
        for (int n = 0; n < CN; ++n) {
          const float v = warp_max(x[n]);
          if (lane == 0) sh.red_max[hb][par][quarter][n] = v;
        }
      }
      if (lane == 0) sh.red_up[hb][par][quarter] = wup ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.max_bar[hb]);
      if (!__all_sync(kFull, mbar_wait(&sh.max_bar[hb], (tile_seq >> 1) & 1))) { ok = false; break; }
      const int* ups = sh.red_up[hb][par];
      const bool rescale = (ups[0] | ups[1] | ups[2] | ups[3]) != 0;   // the same in all four warps
      if (rescale) {
        // new maximum: the old one, or the maxima of the warps that saw a score
        // above it (the other warps' scores are within kLazyMax of it); what
        // was summed against the old one -- the row sums, and (after the
        // group's first tile of the item) the O accumulator in TMEM -- is
        // rescaled, the latter once the group's previous PV has completed and
        // before this tile's PV is issued
        float corr[CN];
        if constexpr (kSM) {
          // lane n (< CN) works out column n into the other row, then every
          // lane reads the corrections back
          const int n = lane & (CN - 1);
          const float mo = mrow[mb * kN + n];
          float mx = mo;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (ups[w]) mx = fmaxf(mx, sh.red_max[hb][par][w][n]);
          if (lane < CN) {
            mrow[(mb ^ 1) * kN + n] = mx;
            crow[n] = (mo == -INFINITY) ? 0.f : exp2f(mo - mx);
          }
          __syncwarp();
          mb ^= 1;
#pragma unroll
          for (int k = 0; k < CN; k += 4) {
            const float4 v = *reinterpret_cast<const float4*>(crow + k);
            corr[k] = v.x;
            corr[k + 1] = v.y;
            corr[k + 2] = v.z;
            corr[k + 3] = v.w;
          }
#pragma unroll
          for (int k = 0; k < CN; ++k) lp[k] *= corr[k];
        } else {
#pragma unroll
          for (int n = 0; n < CN; ++n) {
            float mx = m[n];
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (ups[w]) mx = fmaxf(mx, sh.red_max[hb][par][w][n]);
            corr[n] = (m[n] == -INFINITY) ? 0.f : exp2f(m[n] - mx);
            lp[n] *= corr[n];
            m[n] = mx;
          }
        }
        if (!first) {
          // thread = TMEM lane = head dim 32 quarter + lane of O^T; columns: p_hi
          // products of the CN columns, then p_lo products at HG + n
          const int prev = tile_seq - (PP ? 2 : 1);   // the group's previous tile (same item)
          if (!__all_sync(kFull, mbar_wait(&sh.pv_done[prev & 1], (prev >> 1) & 1))) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t oaddr = lane_addr + kOCol + os * 32;
#pragma unroll
          for (int c16 = 0; c16 < NPV / 16; ++c16) {
            float o[16];
            tc::tmem_ld16(oaddr + c16 * 16, o);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = (c16 * 16 + j) % HG;   // the column this product belongs to
              if (n < CN) o[j] *= corr[n];
            }
            tc::tmem_st16(oaddr + c16 * 16, o);
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
        }
      }
      float (&pr)[CN] = x;   // the weights replace the scores
      {
        float mv[CN];
        load_m(mv);
#pragma unroll
        for (int n = 0; n < CN; ++n) {
          pr[n] = rv ? ex2_approx(x[n] - mv[n]) : 0.f;
          lp[n] += pr[n];
        }
      }
      uint32_t pk[NPV / 2];   // [p_hi of heads 0..HG-1 | p_lo of heads 0..HG-1], two per word
#pragma unroll
      for (int n2 = 0; n2 < HG; n2 += 2) {
        const float a = (n2 < CN) ? pr[n2] * vscale : 0.f, b = (n2 + 1 < CN) ? pr[n2 + 1] * vscale : 0.f;
        pk[n2 >> 1] = Elem<OpT>::pack2(a, b);
        const float2 r = Elem<OpT>::to_float2(pk[n2 >> 1]);
        pk[(HG + n2) >> 1] = Elem<OpT>::pack2(a - r.x, b - r.y);
      }
      // 8-bit: P^T buffer hb was last read by PV(t - 2): wait for it to complete.
      // (16-bit caches write P^T into this tile's own stage, over K atoms that
      // QK(t) has finished reading; the stage is refilled only after PV(t); they
      // wait for PV(t - 2) only before completing p_full, below.)
      if (I8 && tile_seq >= 2 && !__all_sync(kFull, mbar_wait(&sh.pv_done[hb], ((tile_seq - 2) >> 1) & 1))) {
        ok = false;
        break;
      }
      // MN-major without swizzle: core matrix = 8 tokens x 8 columns (128 B);
      // column chunks 128 B apart, 8-token groups (NPV / 8) * 128 B apart in a
      // P^T buffer, one stage group (4 KiB) apart in a stage
      uint8_t* prow = I8 ? pbuf + hb * kPBytes + (row >> 3) * (NPV / 8) * 128 + (row & 7) * 16
                         : stages + slot * kStage + (row >> 3) * kGroupBytes + (row & 7) * 16;
#pragma unroll
      for (int c = 0; c < NPV / 8; ++c)
        *reinterpret_cast<uint4*>(prow + c * 128) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      // V rows of tokens past the context inside the last 16-token MMA step
      // must not hold NaN/Inf (0 * NaN = NaN): zero them.
      // (8-bit caches: the converter warps write zero rows there.)
      if (!I8 && !rv && row < ((mt.valid + 15) & ~15)) {
        uint8_t* vrow = stages + slot * kStage + (row >> 3) * kGroupBytes + 2048 + (row & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + 1024 + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // p_full[hb] may complete tile t's phase only once the PV issuer has
      // taken tile t - 2's: it tells the phases apart by parity, and while
      // PV(t - 2) waits for its O slot this group could otherwise finish tile t
      // and make that phase look pending again.  (8-bit caches waited above.)
      if (!I8 && tile_seq >= 2 && !__all_sync(kFull, mbar_wait(&sh.pv_done[hb], ((tile_seq - 2) >> 1) & 1))) {
        ok = false;
        break;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[hb]);
      // hand-off to the output warps at the group's last tile of the item:
      // its maximum and sums (and, with the item's last tile, the item's
      // metadata) into the item's hand-off slot, once the output warps have
      // taken the slot's previous item.  The maximum is stored first, so it is
      // dead while the sums are reduced.
      if (fin) {
        constexpr int IS = item_slots(I8);
        const int k = mt.item, q = k % IS;
        if (k >= IS && !__all_sync(kFull, mbar_wait(&sh.c_free[q], ((k / IS) - 1) & 1))) { ok = false; break; }
        if constexpr (kSM) {
          if (quarter == 0 && lane < CN) sh.fin[q][grp].m[lane] = mrow[mb * kN + lane];
        }
        if (lane == 0 && quarter == 0) {
          if constexpr (!kSM) {
#pragma unroll
            for (int n = 0; n < CN; ++n) sh.fin[q][grp].m[n] = m[n];
          }
          if (mt.tail == 0) {
            sh.ihand[q].meta = mt;
            sh.ihand[q].ntiles = mt.head + 1;
            sh.ihand[q].first_grp = PP ? ((tile_seq - mt.head) & 1) : 0;
          }
        }
        // this group's part of the normaliser from this quarter's 32 rows (the
        // output warps add the quarters and the groups), reduced in place:
        // lp[0] becomes the sum over the quarter's rows of column
        // lane >> (5 - log2 CN), and the sums start afresh with the next item
        transpose_reduce<CN>(lp, lane, [](float a, float b) { return a + b; });
        constexpr int sh_ = 5 - log2_of(CN);
        if ((lane & ((1 << sh_) - 1)) == 0) sh.fin[q][grp].Lq[quarter][lane >> sh_] = lp[0];
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.c_full[q]);
          if (PP && mt.head == 0 && mt.tail == 0) mbar_arrive(&sh.c_full[q]);   // a one-tile item: for both groups
        }
#pragma unroll
        for (int n = 0; n < CN; ++n) lp[n] = 0.f;
        if constexpr (kSM) {
          __syncwarp();
          if (lane < CN) mrow[mb * kN + lane] = -INFINITY;
          __syncwarp();
        } else {
#pragma unroll
          for (int n = 0; n < CN; ++n) m[n] = -INFINITY;
        }
      }
      tile_seq += PP ? 2 : 1;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, PA_DEVERR_TIMEOUT);
      sh.abort_flag = 1;
    }
  } else if (warp < 10) {
    // =================================================================== output warps (6-9)
    // Once per item: each softmax group's O^T, accumulated in its TMEM slot
    // over the item's tiles (thread = TMEM lane = head dim), merged with the
    // other group's exactly (log-sum-exp) into out = O / L, or into the
    // partition's partial results.
    constexpr bool PP = ping_pong(I8, CN);
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t used = 0;   // per O slot: parity of the items read from it so far
    bool ok = true;
    for (int k = 0;; ++k) {
      constexpr int IS = item_slots(I8);
      const int q = k % IS;
      if (!__all_sync(kFull, mbar_wait(&sh.c_full[q], (k / IS) & 1))) { ok = false; break; }
      const TileMeta mt = sh.ihand[q].meta;
      if (mt.s < 0) break;
      // the groups that had a tile in this item: the group of its first tile,
      // and (two groups) the other one when it has more than one tile
      const int ntiles = sh.ihand[q].ntiles, g_first = sh.ihand[q].first_grp;
      const bool has0 = !PP || g_first == 0 || ntiles >= 2, has1 = PP && (g_first == 1 || ntiles >= 2);
      // lane n (< CN): column n's maximum and sum from each group
      float mg0 = -INFINITY, mg1 = -INFINITY, Lg0 = 0.f, Lg1 = 0.f;
      if (lane < CN) {
        const typename Shared<NS, I8, NRH>::Final& F0 = sh.fin[q][0];
        const typename Shared<NS, I8, NRH>::Final& F1 = sh.fin[q][1];
        if (has0) {
          mg0 = F0.m[lane];
          Lg0 = (F0.Lq[0][lane] + F0.Lq[1][lane]) + (F0.Lq[2][lane] + F0.Lq[3][lane]);
        }
        if (has1) {
          mg1 = F1.m[lane];
          Lg1 = (F1.Lq[0][lane] + F1.Lq[1][lane]) + (F1.Lq[2][lane] + F1.Lq[3][lane]);
        }
      }
      // with that read, fin[q] and ihand[q] are free for the item IS later:
      // the softmax warps need not wait for this item's rows
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.c_free[q]);
      // O of each group: p_hi products + p_lo products of every column
      float x0[CN], x1[CN];
#pragma unroll
      for (int g = 0; g < (PP ? 2 : 1); ++g) {
        const bool has = g == 0 ? has0 : has1;
        const int os = q * (PP ? 2 : 1) + g;
        if (has) {
          if (!__all_sync(kFull, mbar_wait(&sh.ofin[os], (used >> os) & 1))) { ok = false; break; }
          used ^= 1u << os;
          tc::fence_after_sync();
          float o[2][16];
          tc::tmem_ld16(lane_addr + kOCol + os * 32, o[0]);
          if (NPV > 16) tc::tmem_ld16(lane_addr + kOCol + os * 32 + 16, o[1]);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.ofree[os]);
#pragma unroll
          for (int n = 0; n < CN; ++n) {
            const float v = o[n >> 4][n & 15] + o[(HG + n) >> 4][(HG + n) & 15];   // O_hi + O_lo
            if (g == 0) x0[n] = v;
            else x1[n] = v;
          }
        } else {
#pragma unroll
          for (int n = 0; n < CN; ++n) {
            if (g == 0) x0[n] = 0.f;
            else x1[n] = 0.f;
          }
        }
      }
      if (!ok) break;
      {
        T* out = static_cast<T*>(p.out);
        // Where the item's rows go is the same for all its columns: straight to
        // the output when this item is their only partition (for a shared
        // prefix: a sequence with no prefix and one partition -- a prefix item
        // never), else to the workspace's partial results.  Column n is head
        // kvh * G + n % G of sequence seq0 + n / G.
        const bool direct = SP ? (sp_eff[mt.seq0] == 0 && sp_tot[mt.seq0] == 1) : mt.n_parts == 1;
        const int64_t hbase = (int64_t)mt.seq0 * p.num_q_heads + mt.kvh * G;
        const int nc = SP ? mt.ncol : CN;   // the item's columns that have a row
        // Per column, the groups' exact log-sum-exp merge -- M = max(m0, m1),
        // f_g = 2^(m_g - M), L = f0 L0 + f1 L1 -- is the same for every thread:
        // lane n works it out for column n into this warp's table, as the
        // factors of the groups' O (f_g, or f_g / L for a row written directly),
        // and every thread reads them back.
        float2* tab = sh.colout[quarter];
        if (lane < CN) {
          const int n = lane;
          const float M = fmaxf(mg0, mg1);
          const float cf0 = (mg0 == -INFINITY) ? 0.f : exp2f(mg0 - M);
          const float cf1 = (mg1 == -INFINITY) ? 0.f : exp2f(mg1 - M);
          const float cL = PP ? fmaf(Lg0, cf0, Lg1 * cf1) : Lg0;
          if (direct) {
            const float inv = 1.f / cL;   // L >= 1: the maximum's own weight is 1
            tab[n] = make_float2(cf0 * inv, cf1 * inv);
          } else {
            tab[n] = make_float2(cf0, cf1);
            if (quarter == 0 && n < nc) {
              const int64_t r = (hbase + (n / G) * p.num_q_heads + n % G) * p.max_parts + mt.pbase + mt.part;
              p.ws_ml[r * 2 + 0] = mt.bad ? 0.f : M;
              p.ws_ml[r * 2 + 1] = mt.bad ? -1.f : cL;   // an invalid partition: the merge writes zeros
            }
          }
        }
        __syncwarp();
        // the rows: a bad item (it read block 0 for an id out of range) writes
        // zero rows directly and nothing to the workspace
        if (direct) {
#pragma unroll
          for (int n = 0; n < CN; ++n) {
            if (n < nc) {   // the same in every lane
              const float2 g = tab[n];
              const float O = PP ? fmaf(x0[n], g.x, x1[n] * g.y) : x0[n] * g.x;
              const int64_t hrow = hbase + (n / G) * p.num_q_heads + n % G;
              out[hrow * kD + row] = Elem<T>::from_float(mt.bad ? 0.f : O);
            }
          }
        } else if (!mt.bad) {
#pragma unroll
          for (int n = 0; n < CN; ++n) {
            if (n < nc) {
              const float2 g = tab[n];
              const float O = PP ? fmaf(x0[n], g.x, x1[n] * g.y) : x0[n] * g.x;
              const int64_t r = (hbase + (n / G) * p.num_q_heads + n % G) * p.max_parts + mt.pbase + mt.part;
              p.ws_o[r * kD + row] = O;
            }
          }
        }
        __syncwarp();   // every lane has read the table before the next item rewrites it
      }
    }
    if (!ok && lane == 0) {
      report(p.dev_err, PA_DEVERR_TIMEOUT);
      sh.abort_flag = 1;
    }
  } else if (I8 && warp >= kThreads / 32 && warp < kThreads / 32 + NCW) {
    // =================================================================== converter warps (8-bit)
    // A warp may access TMEM lanes 32 (warp % 4) .. + 31, so thread `lane` owns
    // token row t = 32 (warp % 4) + lane of every tile (in half tile t / 64).
    // With 8 warps the two warps of a lane quarter split the 128 dims into
    // halves; with 4, one warp converts all of them.  For its row a thread turns
    // the K codes into fp16 pairs stored to TMEM (row t = lane t: the A operand
    // of S^T = K Q^T), the V codes into the stage's V atoms (swizzled 128-byte
    // rows: the MN-major A operand of O^T = V^T P^T), and copies the token's
    // scales.  Rows past the tile's last token become zeros (scale 0).
    constexpr int kSplit = NCW == 8 ? 2 : 1;
    constexpr int kPc = 8 / kSplit;                       // 16-code pieces per row and thread
    const int quarter = warp & 3;
    const int t = quarter * 32 + lane, h = t >> 6, u = t & 63;
    const int dh = kSplit == 2 ? ((warp - kThreads / 32) >> 2) : 0;
    const uint32_t k_lane = tmem + ((uint32_t)(quarter * 32) << 16) + kKCol + dh * (kPc * 8);
    const I8Layout L8{bs, Hkv};
    const int64_t sbytes = L8.scale_bytes();
    int tile_seq = 0;
    bool ok = true;
    while (true) {
      const int slot = tile_seq % NS;
      const int r = h * NRH + tile_seq % NRH;
      if (!__all_sync(kFull, mbar_wait(&sh.raw_full[r], (tile_seq / NRH) & 1))) { ok = false; break; }
      const TileMeta mt = sh.raw_meta[r];
      const bool end = mt.s < 0;                             // "no more work"
      if (__any_sync(kFull, !end && sh.abort_flag)) { ok = false; break; }
      // the stage and its TMEM K operand were last read by PV(t - NS)
      if (tile_seq >= NS && !__all_sync(kFull, mbar_wait(&sh.empty[slot], ((tile_seq / NS) - 1) & 1))) {
        ok = false;
        break;
      }
      if (!end) {
        uint4 kin[kPc], vin[kPc];
        float skv = 0.f, svv = 0.f;
#pragma unroll
        for (int j = 0; j < kPc; ++j) kin[j] = vin[j] = make_uint4(0, 0, 0, 0);   // zero codes -> +0
        if (t < mt.valid) {
          const int b = u / bs, tb = u - b * bs;
          const uint8_t* chunk = raw + r * kRawBytes + b * chunk_bytes;
          const uint8_t* ks = chunk + (int64_t)tb * kD;
          const uint8_t* vs = chunk + (int64_t)(bs + tb) * kD;
#pragma unroll
          for (int j = 0; j < kPc; ++j) {
            const int off = ((dh * kPc + j) ^ (tb & 7)) << 4;
            kin[j] = *reinterpret_cast<const uint4*>(ks + off);
            vin[j] = *reinterpret_cast<const uint4*>(vs + off);
          }
          skv = *reinterpret_cast<const float*>(chunk + 2LL * bs * kD + 4 * tb);
          svv = *reinterpret_cast<const float*>(chunk + 2LL * bs * kD + sbytes + 4 * tb);
        }
        // V -> the stage's V atoms (8-token group t / 8 at 2 KiB per group)
        uint8_t* vrow = stages + slot * kStage + (t >> 3) * 2048 + (t & 7) * 128;
#pragma unroll
        for (int j = 0; j < kPc; ++j) {
          uint32_t o[8];
          codes_to_16bit<__half>(vin[j], o);
          const int pg = dh * kPc + j;                       // 16 dims: two 16-byte pieces of atom pg / 4
          uint8_t* atom = vrow + (pg >> 2) * 1024;
          const int p0 = (2 * pg) & 7;
          *reinterpret_cast<uint4*>(atom + ((p0 ^ (t & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(atom + (((p0 + 1) ^ (t & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        // K -> TMEM, 32 columns (64 dims) per store
#pragma unroll
        for (int g = 0; g < kPc / 4; ++g) {
          uint32_t kr[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t o[8];
            codes_to_16bit<__half>(kin[4 * g + j], o);
#pragma unroll
            for (int e = 0; e < 8; ++e) kr[8 * j + e] = o[e];
          }
          tc::tmem_st32u(k_lane + slot * 64 + g * 32, kr);
        }
        if (dh == 0) sh.sk[slot][t] = skv;
        if (dh == kSplit - 1) sh.sv[slot][t] = svv;
        tc::tmem_wait_st();
      }
      if (warp == kThreads / 32 && lane == 0) sh.meta[slot] = mt;   // a real tile, or "no more work"
      tc::fence_before_sync();
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.raw_empty[r]);
        mbar_arrive(&sh.full[slot]);
      }
      if (end) break;
      ++tile_seq;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, PA_DEVERR_TIMEOUT);
      sh.abort_flag = 1;
    }
  } else if (I8 && warp == kThreads / 32 + NCW) {
    // =================================================================== copy warp (8-bit)
    // Tile t: wait for its descriptor and for both halves' raw slots, then one
    // instruction issues the bulk copies of all its (block, kv head) chunks
    // (lanes i + 32 c; blocks past the first half go to the half-1 slot).
    const int bph = 64 / bs;                      // blocks per half tile
    int tile = 0;
    bool ok = true;
    while (true) {
      const int d = tile % kND;
      if (!__all_sync(kFull, mbar_wait(&sh.desc_full[d], (tile / kND) & 1))) { ok = false; break; }
      TileMeta m = sh.desc[d].meta;
      const int r0 = tile % NRH, r1 = NRH + r0;
      if (tile >= NRH && !__all_sync(kFull, mbar_wait(&sh.raw_empty[r0], ((tile / NRH) - 1) & 1) &&
                                                mbar_wait(&sh.raw_empty[r1], ((tile / NRH) - 1) & 1))) {
        ok = false;
        break;
      }
      if (__any_sync(kFull, sh.abort_flag)) {
        ok = false;
        break;
      }
      if (m.s < 0) {
        // no more work: the mark goes into both halves' slots (each converter
        // warp watches its own half's ring) -- after the drain below, whose
        // waits on a slot's latest phase would otherwise alias the mark's
        if (lane == 0) {
          for (int h = 0; h < 2; ++h)
            for (int t = max(0, tile - NRH); t < tile; ++t)
              if (!mbar_wait(&sh.raw_full[h * NRH + t % NRH], (t / NRH) & 1)) report(p.dev_err, PA_DEVERR_TIMEOUT);
          sh.raw_meta[r0] = m;
          sh.raw_meta[r1] = m;
          mbar_arrive(&sh.raw_full[r0]);
          mbar_arrive(&sh.raw_full[r1]);
        }
        break;
      }
      const int nbt = (m.valid + bs - 1) / bs;
      const int nb0 = min(nbt, bph);
      if (lane == 0) {
        sh.raw_meta[r0] = m;
        sh.raw_meta[r1] = m;
        mbar_arrive_expect_tx(&sh.raw_full[r0], (uint32_t)(nb0 * chunk_bytes));
        mbar_arrive_expect_tx(&sh.raw_full[r1], (uint32_t)((nbt - nb0) * chunk_bytes));
      }
      __syncwarp();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int b = lane + 32 * c;
        if (b < nbt) {
          const int h = b >= bph, r = h ? r1 : r0;
          bulk_g2s(raw + r * kRawBytes + (b - h * bph) * chunk_bytes,
                   p.cache + ((int64_t)sh.desc[d].ids[b] * Hkv + m.kvh) * chunk_bytes, (uint32_t)chunk_bytes,
                   &sh.raw_full[r]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.desc_empty[d]);
      ++tile;
    }
    if (!ok && lane == 0) {
      // never leave copies in flight: wait (bounded) for the latest phase of
      // every raw slot (the normal end drained them before posting its mark)
      for (int h = 0; h < 2; ++h)
        for (int t = max(0, tile - NRH); t < tile; ++t) mbar_wait(&sh.raw_full[h * NRH + t % NRH], (t / NRH) & 1);
      report(p.dev_err, PA_DEVERR_TIMEOUT);
      sh.abort_flag = 1;   // the other roles see it and leave their (bounded) loops
    }
  }

  // ---- tear-down: release TMEM once every role is done
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kCols);
  }
}

// Dynamic shared memory of one CTA: stages, Q slots, P^T buffers (8-bit), 8-bit raw rings,
// the item tables (1024 bytes of slack align the stages to 1024).
__host__ __device__ inline size_t decode_tc_smem(int NS, bool I8, int NRH, bool SP, int S) {
  return 1024 + (size_t)NS * stage_bytes(I8) + (size_t)q_slots(I8) * kQBytes + (size_t)p_buffers(I8) * kPBytes +
         (I8 ? (size_t)2 * NRH * kRawBytes : 0) +
         ItemTables(S, SP).end;
}

template <typename T, int G, int NS, bool I8, int NRH, bool SP = false>
cudaError_t launch_typed(const DecodeParams& p, int num_sms, cudaStream_t stream) {
  const size_t smem = decode_tc_smem(NS, I8, NRH, SP, p.num_seqs);
  auto kern = decode_tc_kernel<T, G, NS, I8, NRH, SP>;
  cudaError_t e = set_smem_attribute_once<decode_tc_kernel<T, G, NS, I8, NRH, SP>>(smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, threads_of(I8, SP ? kN : G), smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int NS, bool I8, int NRH>
cudaError_t launch_group(const DecodeParams& p, int group, int num_sms, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_typed<T, 1, NS, I8, NRH>(p, num_sms, stream);
    case 2: return launch_typed<T, 2, NS, I8, NRH>(p, num_sms, stream);
    case 4: return launch_typed<T, 4, NS, I8, NRH>(p, num_sms, stream);
    case 8: return launch_typed<T, 8, NS, I8, NRH>(p, num_sms, stream);
    case 16:
      if constexpr (I8) return cudaErrorInvalidValue;   // 8-bit caches serve groups up to 8
      else return launch_typed<T, 16, NS, false, 1>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

// 8-bit caches: 3 converted stages (V in shared memory, K in TMEM) and 2 raw
// 64-token half tiles of 8-bit chunks per half in flight (~74 KB)
constexpr int kI8Stages = 3, kI8Raw = 2;

}  // namespace
}  // namespace pkv
