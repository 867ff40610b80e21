// decode_tc.cu -- paged decode attention on the tensor cores (tcgen05 + TMEM).
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
// Q^T (K-major, swizzled, written by the producer warp) and P^T (MN-major, no
// swizzle, written by the softmax warps) are the B operands; S^T and O^T
// accumulate in fp32 in tensor memory (TMEM), double-buffered.
//
// One persistent CTA per SM walks a static round-robin share of the work items
// (sequence, kv head, partition); the list of items is built in shared memory
// from a prefix sum of partitions per sequence, so no CTA is spent on empty
// partitions.  Roles:
//   warp 0      producer: item walk, block-id validation, Q staging, one bulk
//               copy per (block, kv head) chunk into a ring of NS 64 KiB stages;
//               per-stage metadata travels with the stage's mbarrier.
//   warp 1      MMA issuer (one lane): QK(t) and PV(t) each issued as soon as
//               their inputs are ready (polled, bounded).
//   warps 2-5   softmax (thread = TMEM lane): tile max across the 128 rows,
//               p = 2^(s - m) in fp32, written as two operands in the cache type,
//               p_hi = round(p) and p_lo = round(p - p_hi); the PV product is
//               issued for both into the same accumulator, so the weights reach
//               the tensor core with ~16 significant bits even for bf16.  Then
//               O^T of the previous tile is folded into registers with the
//               online-softmax correction.
// Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT and ends the CTA.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 128;                         // tokens per tile
constexpr int kTileBytes = kTile * 2 * kD * 2;     // K + V of 128 tokens: 64 KiB
constexpr int kGroupBytes = 8 * 2 * kD * 2;        // one 8-token group: 4 KiB
constexpr int kN = 16;                             // MMA N: query heads, zero-padded
constexpr int kQBytes = kN * kD * 2;               // 4 KiB
constexpr int kPBytes = kTile * kN * 2;            // 4 KiB per P^T operand (hi or lo)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 64;                 // S0 S1 | O0 O1, 16 columns each
constexpr uint32_t kFull = 0xffffffffu;

struct TileMeta {
  int s, kvh, part, valid;       // sequence (< 0: no more work), kv head, partition, valid tokens
  int last, qslot, n_parts, pad;
};

template <int NS>
struct Shared {
  uint64_t full[NS], empty[NS];
  uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2], q_free[2];
  uint64_t max_bar[2], sum_bar;   // softmax-warp exchanges (bounded waits, unlike bar.sync)
  TileMeta meta[NS];
  float red_max[2][4][kN];
  float red_sum[4][kN];
  uint32_t tmem_base;
  volatile int abort_flag;
};

__device__ __forceinline__ bool ctx_invalid(const DecodeParams& p, int ctx) {
  return (int64_t)ctx > (int64_t)p.bt_stride * p.block_size || ctx > p.max_context_len;
}

// Work items of one sequence: its partitions, or one item that only writes zeros.
__device__ __forceinline__ int items_of(const DecodeParams& p, int ctx) {
  if (ctx <= 0 || ctx_invalid(p, ctx)) return 1;
  return (ctx + p.partition_size - 1) / p.partition_size;
}

template <typename T, int G>
__device__ void warp_zero_rows(const DecodeParams& p, int s, int kvh, int lane) {
  T* out = static_cast<T*>(p.out) + ((int64_t)s * p.num_q_heads + kvh * G) * kD;
  for (int i = lane * 8; i < G * kD; i += 32 * 8) *reinterpret_cast<uint4*>(out + i) = make_uint4(0, 0, 0, 0);
}

template <typename T, int G, int NS>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ Shared<NS> sh;
  extern __shared__ __align__(1024) uint8_t dyn_raw[];
  const uint32_t raw_s = smem_u32(dyn_raw);
  uint8_t* dyn = dyn_raw + (((raw_s + 1023u) & ~1023u) - raw_s);   // 1024-aligned in the shared window
  uint8_t* stages = dyn;
  uint8_t* qbuf = dyn + NS * kTileBytes;
  uint8_t* pbuf = qbuf + 2 * kQBytes;
  int* pre = reinterpret_cast<int*>(pbuf + 4 * kPBytes);   // pbuf: 2 x (p_hi, p_lo)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.num_seqs, Hkv = p.num_kv_heads, bs = p.block_size;
  const int64_t chunk_bytes = (int64_t)bs * 2 * kD * 2;
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;

  // ---- set-up: barriers, zeroed Q buffers (padding heads stay zero), TMEM
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_free[i], 4);
      mbar_init(&sh.p_full[i], 4);
      mbar_init(&sh.o_full[i], 1);
      mbar_init(&sh.o_free[i], 4);
      mbar_init(&sh.q_free[i], 1);
      mbar_init(&sh.max_bar[i], 4);
    }
    mbar_init(&sh.sum_bar, 4);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 2 * kQBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 1) {
    tc::tmem_alloc(&sh.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // =================================================================== producer
    int carry = 0;
    for (int base = 0; base < S; base += 32) {
      int x = (base + lane < S) ? items_of(p, p.context_lens[base + lane]) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (base + lane < S) pre[base + lane + 1] = carry + x;
      carry += __shfl_sync(kFull, x, 31);
    }
    if (lane == 0) pre[0] = 0;
    __syncwarp();
    const int total = carry * Hkv;
    int tile_seq = 0, item_seq = 0;
    bool aborted = false;
    for (int it = blockIdx.x; it < total && !aborted; it += gridDim.x) {
      const int j = it / Hkv, kvh = it - (it / Hkv) * Hkv;
      int lo = 0, hi = S - 1;   // last sequence whose first item index is <= j
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= j) lo = mid;
        else hi = mid - 1;
      }
      const int s = lo, part = j - pre[s];
      const int P = p.partition_size;
      const int jb = part * (P / bs);                      // first logical block of the partition
      const int32_t* row = p.block_tables + (int64_t)s * p.bt_stride + jb;
      // issue the item's independent loads together: context length, the first
      // 32 block ids of the partition, and the query rows
      const int ctx = p.context_lens[s];
      const int id_lane = (lane < P / bs && jb + lane < p.bt_stride) ? row[lane] : 0;
      constexpr int kQChunks = (G * 16 + 31) / 32;
      const T* qsrc = static_cast<const T*>(p.q) + (int64_t)s * p.q_seq_stride + (int64_t)kvh * G * kD;
      uint4 qv[kQChunks];
#pragma unroll
      for (int k = 0; k < kQChunks; ++k) {
        const int c = lane + 32 * k;
        if (c < G * 16) qv[k] = *reinterpret_cast<const uint4*>(qsrc + (c >> 4) * kD + (c & 15) * 8);
      }
      if (ctx_invalid(p, ctx)) {
        warp_zero_rows<T, G>(p, s, kvh, lane);
        if (lane == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
        continue;
      }
      if (ctx <= 0) {
        warp_zero_rows<T, G>(p, s, kvh, lane);
        continue;
      }
      const int n_parts = (ctx + P - 1) / P;
      const int t0 = part * P, t1 = min(ctx, t0 + P);
      const int nblk = (t1 - t0 + bs - 1) / bs;
      bool bad = lane < nblk && (id_lane < 0 || id_lane >= p.num_blocks);
      for (int b = lane + 32; b < nblk; b += 32) {
        const int id = row[b];
        bad |= (id < 0 || id >= p.num_blocks);
      }
      if (__any_sync(kFull, bad)) {
        if (lane == 0) report(p.dev_err, PA_DEVERR_BLOCK_ID);
        if (n_parts == 1) {
          warp_zero_rows<T, G>(p, s, kvh, lane);
        } else if (lane < G) {
          const int64_t r = ((int64_t)s * p.num_q_heads + kvh * G + lane) * p.max_parts + part;
          p.ws_ml[r * 2 + 0] = 0.f;
          p.ws_ml[r * 2 + 1] = -1.f;   // invalid partition: the merge writes zeros
        }
        continue;
      }
      // ---- Q^T of this item into a K-major 128B-swizzled buffer
      const int qslot = item_seq & 1;
      if (item_seq >= 2 && !mbar_wait(&sh.q_free[qslot], ((item_seq >> 1) - 1) & 1)) {
        aborted = true;
        break;
      }
      {
        uint8_t* qb = qbuf + qslot * kQBytes;
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = lane + 32 * k;
          if (c < G * 16) {
            const int n = c >> 4, cc = c & 15, atom = cc >> 3, piece = cc & 7;
            *reinterpret_cast<uint4*>(qb + (atom * 2 + (n >> 3)) * 1024 + (n & 7) * 128 + ((piece ^ (n & 7)) << 4)) =
                qv[k];
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
      }
      // ---- stream the tiles
      const int ntiles = (t1 - t0 + kTile - 1) / kTile;
      for (int k = 0; k < ntiles; ++k) {
        const int slot = tile_seq % NS;
        if (tile_seq >= NS && !mbar_wait(&sh.empty[slot], ((tile_seq / NS) - 1) & 1)) {
          aborted = true;
          break;
        }
        const int valid = min(kTile, t1 - (t0 + k * kTile));
        const int nb = (valid + bs - 1) / bs;
        if (lane == 0) {
          TileMeta m;
          m.s = s; m.kvh = kvh; m.part = part; m.valid = valid;
          m.last = (k == ntiles - 1); m.qslot = qslot; m.n_parts = n_parts; m.pad = 0;
          sh.meta[slot] = m;
          mbar_arrive_expect_tx(&sh.full[slot], (uint32_t)(nb * chunk_bytes));
        }
        __syncwarp();
        const int bi = k * (kTile / bs) + lane;             // block of this lane's copy
        const int id_sh = __shfl_sync(kFull, id_lane, bi & 31);
        if (lane < nb) {
          const int id = bi < 32 ? id_sh : row[bi];
          bulk_g2s(stages + slot * kTileBytes + lane * chunk_bytes,
                   p.cache + ((int64_t)id * Hkv + kvh) * chunk_bytes, (uint32_t)chunk_bytes, &sh.full[slot]);
        }
        ++tile_seq;
      }
      ++item_seq;
    }
    // ---- no more work: a stage whose metadata says so
    const int slot = tile_seq % NS;
    if (!aborted && tile_seq >= NS && !mbar_wait(&sh.empty[slot], ((tile_seq / NS) - 1) & 1)) aborted = true;
    if (aborted && lane == 0) {
      // never leave copies in flight: wait (bounded) for the latest phase of every stage
      for (int t = max(0, tile_seq - NS); t < tile_seq; ++t) mbar_wait(&sh.full[t % NS], (t / NS) & 1);
    }
    if (lane == 0) {
      if (aborted) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      sh.meta[slot].s = -1;
      mbar_arrive(&sh.full[slot]);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =================================================================== MMA issuer
    // Event-driven: QK(t) as soon as tile t has landed and its S buffer is free,
    // PV(t) as soon as P(t) is written and its O buffer is free -- neither waits
    // for the other stream, so a stage is released right after its own PV.
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16(128, kN, kBF16, false, false);
      const uint32_t id_pv = tc::idesc_f16(128, kN, kBF16, true, true);
      int qk = 0, pv = 0, end = 0x7fffffff;
      uint32_t idle = 0;
      bool ok = true;
      while (pv < end) {
        bool progressed = false;
        if (qk < end) {
          const int slot = qk % NS;
          if (mbar_try_wait(&sh.full[slot], (qk / NS) & 1)) {
            const TileMeta m = sh.meta[slot];
            if (m.s < 0) {
              end = qk;
              progressed = true;
            } else if (qk < 2 || mbar_try_wait(&sh.s_free[qk & 1], ((qk >> 1) - 1) & 1)) {
              tc::fence_after_sync();
              const uint32_t st = smem_u32(stages + slot * kTileBytes), qa = smem_u32(qbuf + m.qslot * kQBytes);
#pragma unroll
              for (int kk = 0; kk < kD / 16; ++kk)
                tc::mma_f16(tmem + (qk & 1) * 16,
                            tc::smem_desc(st + (kk >> 2) * 1024 + (kk & 3) * 32, 16, kGroupBytes, tc::kSwizzle128B),
                            tc::smem_desc(qa + (kk >> 2) * 2048 + (kk & 3) * 32, 16, 1024, tc::kSwizzle128B), id_qk,
                            kk > 0);
              tc::commit(&sh.s_full[qk & 1]);
              if (m.last) tc::commit(&sh.q_free[m.qslot]);
              ++qk;
              progressed = true;
            }
          }
        }
        if (pv < qk) {
          const int pb = pv & 1;
          if (mbar_try_wait(&sh.p_full[pb], (pv >> 1) & 1) &&
              (pv < 2 || mbar_try_wait(&sh.o_free[pb], ((pv >> 1) - 1) & 1))) {
            tc::fence_after_sync();
            const int slot = pv % NS;
            const int valid = sh.meta[slot].valid;   // the stage is not refilled before this PV completes
            const uint32_t st = smem_u32(stages + slot * kTileBytes), pa = smem_u32(pbuf + pb * 2 * kPBytes);
            const int nsteps = (valid + 15) >> 4;
            for (int half = 0; half < 2; ++half)      // p_hi, then p_lo into the same accumulator
              for (int kk = 0; kk < nsteps; ++kk)
                tc::mma_f16(tmem + 32 + pb * 16,
                            tc::smem_desc(st + kk * 8192 + 2048, 1024, kGroupBytes, tc::kSwizzle128B),
                            tc::smem_desc(pa + half * kPBytes + kk * 512, 256, 128, tc::kSwizzleNone), id_pv,
                            (half | kk) > 0);
            tc::commit(&sh.o_full[pb]);
            tc::commit(&sh.empty[slot]);
            ++pv;
            progressed = true;
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
    }
    __syncwarp();
  } else {
    // =================================================================== softmax warps
    // Iteration t: probabilities of tile t first (so the tensor core can run
    // PV(t-1) meanwhile), then fold O^T of tile t-1 into the accumulators and,
    // if t-1 ended its item, write that item's result.
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;   // TMEM lane: token row of S^T, dim row of O^T
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    float m[G], lp[G], acc[G], corr[G], corr_prev[G], m_fin[G], lp_fin[G];
#pragma unroll
    for (int n = 0; n < G; ++n) {
      m[n] = -INFINITY;
      lp[n] = 0.f;
      acc[n] = 0.f;
      corr[n] = 0.f;
      corr_prev[n] = 0.f;
      m_fin[n] = -INFINITY;
      lp_fin[n] = 0.f;
    }
    TileMeta prev;
    prev.s = -1;
    int tile_seq = 0, sum_uses = 0;
    bool ok = true;
    while (true) {
      const int slot = tile_seq % NS;
      if (!mbar_wait(&sh.full[slot], (tile_seq / NS) & 1)) { ok = false; break; }
      const TileMeta mt = sh.meta[slot];
      // state of the item that tile t-1 finishes (if it does)
#pragma unroll
      for (int n = 0; n < G; ++n) corr_prev[n] = corr[n];
      if (prev.s >= 0 && (prev.last || mt.s < 0)) {
#pragma unroll
        for (int n = 0; n < G; ++n) {
          m_fin[n] = m[n];
          lp_fin[n] = lp[n];
          m[n] = -INFINITY;
          lp[n] = 0.f;
        }
      }

      // ---- 1. S^T of tile t -> probabilities P^T (hi and lo parts)
      if (mt.s >= 0) {
        const int sb = tile_seq & 1;
        if (!mbar_wait(&sh.s_full[sb], (tile_seq >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        float sv[16];
        tc::tmem_ld16(lane_addr + sb * 16, sv);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_free[sb]);
        const bool rv = row < mt.valid;
        float x[G];
#pragma unroll
        for (int n = 0; n < G; ++n) {
          x[n] = rv ? sv[n] * p.scale_log2 : -INFINITY;
          float v = x[n];
#pragma unroll
          for (int o2 = 16; o2 > 0; o2 >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o2));
          if (lane == 0) sh.red_max[tile_seq & 1][quarter][n] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.max_bar[tile_seq & 1]);
        if (!mbar_wait(&sh.max_bar[tile_seq & 1], (tile_seq >> 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int n = 0; n < G; ++n) {
          const float (*rm)[kN] = sh.red_max[tile_seq & 1];
          const float mx = fmaxf(fmaxf(rm[0][n], rm[1][n]), fmaxf(rm[2][n], rm[3][n]));
          const float mn = fmaxf(m[n], mx);
          corr[n] = (m[n] == -INFINITY) ? 0.f : exp2f(m[n] - mn);
          m[n] = mn;
        }
        float pr[G];
#pragma unroll
        for (int n = 0; n < G; ++n) {
          pr[n] = rv ? exp2f(x[n] - m[n]) : 0.f;
          lp[n] = fmaf(lp[n], corr[n], pr[n]);
        }
        uint32_t hi[kN / 2], lo[kN / 2];
#pragma unroll
        for (int n2 = 0; n2 < kN; n2 += 2) {
          const float a = (n2 < G) ? pr[n2] : 0.f, b = (n2 + 1 < G) ? pr[n2 + 1] : 0.f;
          hi[n2 >> 1] = Elem<T>::pack2(a, b);
          const float2 r = Elem<T>::to_float2(hi[n2 >> 1]);
          lo[n2 >> 1] = Elem<T>::pack2(a - r.x, b - r.y);
        }
        uint8_t* prow = pbuf + (tile_seq & 1) * 2 * kPBytes + (row >> 3) * 256 + (row & 7) * 16;
        *reinterpret_cast<uint4*>(prow) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(prow + 128) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        *reinterpret_cast<uint4*>(prow + kPBytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(prow + kPBytes + 128) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        // V rows of tokens past the context inside the last 16-token MMA step
        // must not hold NaN/Inf (0 * NaN = NaN): zero them.
        if (!rv && row < ((mt.valid + 15) & ~15)) {
          uint8_t* vrow = stages + slot * kTileBytes + (row >> 3) * kGroupBytes + 2048 + (row & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + 1024 + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.p_full[tile_seq & 1]);
      }

      // ---- 2. O^T of tile t-1: online-softmax correction; finish its item
      if (prev.s >= 0) {
        const int seq = tile_seq - 1, pb = seq & 1;
        if (!mbar_wait(&sh.o_full[pb], (seq >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        float o[16];
        tc::tmem_ld16(lane_addr + 32 + pb * 16, o);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.o_free[pb]);
#pragma unroll
        for (int n = 0; n < G; ++n) acc[n] = fmaf(acc[n], corr_prev[n], o[n]);
        if (prev.last) {
          float L[G];
#pragma unroll
          for (int n = 0; n < G; ++n) {
            float v = lp_fin[n];
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(kFull, v, o2);
            if (lane == 0) sh.red_sum[quarter][n] = v;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.sum_bar);
          if (!mbar_wait(&sh.sum_bar, sum_uses & 1)) { ok = false; break; }
          ++sum_uses;
#pragma unroll
          for (int n = 0; n < G; ++n)
            L[n] = sh.red_sum[0][n] + sh.red_sum[1][n] + sh.red_sum[2][n] + sh.red_sum[3][n];
          const int64_t h0 = (int64_t)prev.s * p.num_q_heads + prev.kvh * G;
          if (prev.n_parts == 1) {
            T* out = static_cast<T*>(p.out);
#pragma unroll
            for (int n = 0; n < G; ++n) out[(h0 + n) * kD + row] = Elem<T>::from_float(acc[n] / L[n]);
          } else {
#pragma unroll
            for (int n = 0; n < G; ++n) {
              const int64_t r = (h0 + n) * p.max_parts + prev.part;
              p.ws_o[r * kD + row] = acc[n];
              if (row == 0) {
                p.ws_ml[r * 2 + 0] = m_fin[n];
                p.ws_ml[r * 2 + 1] = L[n];
              }
            }
          }
#pragma unroll
          for (int n = 0; n < G; ++n) acc[n] = 0.f;
        }
      }
      if (mt.s < 0 || sh.abort_flag) break;
      prev = mt;
      ++tile_seq;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, PA_DEVERR_TIMEOUT);
      sh.abort_flag = 1;
    }
  }

  // ---- tear-down: release TMEM once every role is done
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int G, int NS>
cudaError_t launch_typed(const DecodeParams& p, int num_sms, cudaStream_t stream) {
  const size_t smem = 1024 + (size_t)NS * kTileBytes + 2 * kQBytes + 4 * kPBytes + (size_t)(p.num_seqs + 1) * 4;
  auto kern = decode_tc_kernel<T, G, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int NS>
cudaError_t launch_group(const DecodeParams& p, int group, int num_sms, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_typed<T, 1, NS>(p, num_sms, stream);
    case 2: return launch_typed<T, 2, NS>(p, num_sms, stream);
    case 4: return launch_typed<T, 4, NS>(p, num_sms, stream);
    case 8: return launch_typed<T, 8, NS>(p, num_sms, stream);
    case 16: return launch_typed<T, 16, NS>(p, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams& p, int dtype, int group, int num_sms, cudaStream_t stream) {
  if (p.num_seqs > kTcMaxSeqs) return cudaErrorInvalidValue;
  const bool three = p.num_seqs <= 1024;   // shared memory: 3 stages + prefix of <= 1025 ints
  cudaError_t e;
  if (dtype == PA_F16)
    e = three ? launch_group<__half, 3>(p, group, num_sms, stream) : launch_group<__half, 2>(p, group, num_sms, stream);
  else if (dtype == PA_BF16)
    e = three ? launch_group<__nv_bfloat16, 3>(p, group, num_sms, stream)
              : launch_group<__nv_bfloat16, 2>(p, group, num_sms, stream);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  return launch_merge(p, dtype, kD, stream);
}

}  // namespace pkv
