// prefill_tc.cu -- causal prefill / extend attention over the paged cache on the
// tensor cores (tcgen05 + TMEM).
//
// What is computed: the prefill of the "vLLM" page (the whole prompt, or under
// chunked prefill one chunk of it, attends over the KV cache with a causal
// mask; the chunk's own K/V were written by reshape_and_cache first).  Sequence
// s owns the packed query tokens query_start_loc[s] .. [s+1]; query j of its
// q_len sits at position ctx - q_len + j and attends positions 0 .. that
// position, found through the block table as in decode.
//
// One CTA per (query tile, kv head, sequence).  A tile is M = 128 rows: 128/G
// consecutive query positions x the G query heads of the kv head (row =
// position * G + head), so one pass over the KV serves all G heads.  Per
// 64-token KV tile t:
//     S_t = Q K_t^T        (M = 128 rows, N = 64 tokens, K = D)   -> TMEM (fp32)
//     O  += P_t V_t        (M = 128 rows, N = D, K = 64 tokens)   -> TMEM (fp32)
// (64-token tiles keep a CTA at ~100 KB of shared memory and 256 TMEM columns,
// so two CTAs share an SM and hide each other's softmax and set-up latency.)
// Q (written once, 128B-swizzled K-major, shared memory) is the A operand of
// S; the cache's 8-token groups staged by bulk copies are directly the K-major
// B operand (K) and the MN-major B operand (V).  P is written by the softmax
// threads into TMEM over the S columns they have just read and is the A
// operand of PV straight from TMEM, so P double-buffers with S: the softmax
// of tile t+1 runs while PV of tile t executes.  (This relies on the tcgen05
// operations of the issuing thread executing in issue order: S_{t+2} is
// issued after PV_t has been, and overwrites P_t only after PV_t read it.)
// For bf16, P goes to the tensor core as p_hi = round(p) and p_lo =
// round(p - p_hi) (two products, ~16 significant bits); fp16 weights (11
// bits) need no p_lo.
// Roles:
//   warp 0      bulk copies of each KV tile's (block, kv head) chunks into a
//               2-stage ring (mbarrier transaction counts).
//   warp 1      one lane, event-driven: S_t as soon as tile t has landed (and
//               PV_{t-2} has been issued), O += P_t V_t as soon as P_t is written.
// TMEM columns: S/P buffer 0 [0, 64), S/P buffer 1 [64, 128), O [128, 128 + D);
// within a buffer P occupies p_hi [0, 32) and p_lo [32, 64) (tokens packed two
// per column).
//   warps 2-9   thread = TMEM lane = query row, in two warpgroups that own
//               half of the tile's 64 columns (and half of O's columns)
//               each: causal mask, online softmax in base 2 with the row
//               maxima exchanged through shared memory.  The running max is
//               raised only when a tile's max exceeds it by more than 8 (a
//               factor 256), and only then is the row of O rescaled in TMEM;
//               otherwise the stale max is kept for both p and the sum, which
//               is the same arithmetic.  They also zero V rows past the tile's
//               last token (0 * NaN = NaN) and write the output rows.
// Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT and the CTA drains
// its own copies and MMAs before releasing TMEM.
#include <math.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;                // MMA M: (position, head) rows of one query tile
constexpr int kKv = 64;                   // tokens per KV tile (two CTAs fit an SM)
constexpr int kThreads = 320;             // producer, MMA, 8 softmax warps (two column halves)
constexpr int kSoftmaxWarps = 8;
constexpr uint32_t kTmemCols = 256;       // S0 [0,64) S1 [64,128) O [128, 128 + D): two CTAs per SM
constexpr uint32_t kOCol = 2 * kKv;
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kRescaleThreshold = 8.f;  // base-2 units

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;                      // 128-byte rows per K (or V) vector
  static constexpr int kGroupBytes = 8 * 2 * D * 2;          // one 8-token group: K atoms, then V atoms
  static constexpr int kStageBytes = kKv * 2 * D * 2;        // K + V of one KV tile
  static constexpr int kQAtomBytes = kRows * 128;            // one 64-dim column block of Q (or P)
  static constexpr int kQBytes = kRows * D * 2;
  static constexpr int kStages = 2;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kQBytes;
};

struct Shared {
  // pv_done[b]: PV of the tiles using S/P buffer b (j & 1 == b) completed.  A
  // barrier that a waiter may trail by a tile is kept per buffer, so a waiter is
  // never two phases behind (the parity it waits for would then alias).
  uint64_t full[2], empty[2], s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t xbar;                  // the two softmax warpgroups' per-row exchanges
  uint64_t mma_drain;             // the issuer's own MMAs, waited for before TMEM is freed
  float red[2][2][kRows];         // [exchange parity][warpgroup][row]
  uint32_t tmem_base;
  int bad;
  volatile int abort_flag;
};

// 2^x by the MUFU instruction (relative error about 2^-22; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Offset of the 16-byte piece `piece` (8 elements) of row r in a 128B-swizzled
// K-major operand of 128 rows whose 64-element column blocks are kQAtomBytes apart.
__device__ __forceinline__ uint32_t op_offset(int r, int piece) {
  return (uint32_t)((piece >> 3) * (kRows * 128) + (r >> 3) * 1024 + (r & 7) * 128 + (((piece & 7) ^ (r & 7)) << 4));
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads, 2) prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using C = Cfg<D>;
  constexpr int PT = kRows / G;                      // query positions per tile
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
  __shared__ Shared sh;
  extern __shared__ __align__(1024) uint8_t dyn_raw[];
  const uint32_t raw_s = smem_u32(dyn_raw);
  uint8_t* dyn = dyn_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint8_t* stages = dyn;
  uint8_t* qbuf = stages + C::kStages * C::kStageBytes;
  constexpr bool kLo = kBF16;                        // fp16 weights keep 11 bits: no p_lo

  const int tile = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = p.query_start_loc[s];
  const int q_len = p.query_start_loc[s + 1] - first;
  const int ctx = p.context_lens[s];
  const int bs = p.block_size;
  T* out = static_cast<T*>(p.out);
  auto zero_rows = [&](int q0, int npos) {
    const int n = npos * G * (D / 8);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int r = i / (D / 8), c = i % (D / 8);
      const int64_t tok = first + q0 + r / G;
      *reinterpret_cast<uint4*>(out + (tok * p.num_q_heads + kvh * G + r % G) * D + c * 8) = make_uint4(0, 0, 0, 0);
    }
  };
  if (q_len > p.max_query_len) {
    // the grid does not cover this sequence: tile 0 clears all its rows
    if (tile == 0) {
      for (int q0 = 0; q0 < q_len; q0 += PT) zero_rows(q0, min(PT, q_len - q0));
      if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
    }
    return;
  }
  const int q0 = tile * PT;
  if (q0 >= q_len) return;
  const int npos = min(PT, q_len - q0);
  if (q_len > ctx || (int64_t)ctx > (int64_t)p.bt_stride * bs) {
    zero_rows(q0, npos);
    if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
    return;
  }
  const int pos0 = ctx - q_len + q0;        // position of the tile's first query
  const int kv_len = pos0 + npos;           // the tile attends positions [0, kv_len)
  const int nblk = (kv_len + bs - 1) / bs;
  const int32_t* row_ids = p.block_tables + (int64_t)s * p.bt_stride;
  if (threadIdx.x == 0) sh.bad = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
    const int b = row_ids[i];
    if (b < 0 || b >= p.num_blocks) sh.bad = 1;
  }
  __syncthreads();
  if (sh.bad) {
    zero_rows(q0, npos);
    if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_BLOCK_ID);
    return;
  }

  // ---- set-up: barriers, Q tile (rows past the tile's queries are zero), TMEM
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.s_free[i], kSoftmaxWarps);
    }
    mbar_init(&sh.p_full[0], kSoftmaxWarps);
    mbar_init(&sh.p_full[1], kSoftmaxWarps);
    mbar_init(&sh.pv_done[0], 1);
    mbar_init(&sh.pv_done[1], 1);
    mbar_init(&sh.xbar, kSoftmaxWarps);
    mbar_init(&sh.mma_drain, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  {
    const T* qsrc = static_cast<const T*>(p.q);
    for (int i = threadIdx.x; i < kRows * (D / 8); i += kThreads) {
      const int r = i / (D / 8), c = i % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < npos * G)
        v = *reinterpret_cast<const uint4*>(qsrc + (int64_t)(first + q0 + r / G) * p.q_token_stride +
                                            (int64_t)(kvh * G + r % G) * D + c * 8);
      *reinterpret_cast<uint4*>(qbuf + op_offset(r, c)) = v;
    }
    tc::fence_proxy_async_smem();
  }
  if (warp == 1) {
    tc::tmem_alloc(&sh.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sh.tmem_base;
  const int n_kv = (kv_len + kKv - 1) / kKv;
  const int64_t chunk_bytes = (int64_t)bs * 2 * D * 2;

  if (warp == 0) {
    // =================================================================== producer
    int issued = 0;
    bool aborted = false;
    for (int j = 0; j < n_kv; ++j) {
      const int slot = j & 1;
      if (j >= 2 && !mbar_wait(&sh.empty[slot], ((j >> 1) - 1) & 1)) {
        aborted = true;
        break;
      }
      if (sh.abort_flag) {
        aborted = true;
        break;
      }
      const int valid = min(kKv, kv_len - j * kKv);
      const int nb = (valid + bs - 1) / bs;
      if (lane == 0) mbar_arrive_expect_tx(&sh.full[slot], (uint32_t)(nb * chunk_bytes));
      __syncwarp();
      for (int b = lane; b < nb; b += 32) {
        const int id = row_ids[j * (kKv / bs) + b];
        bulk_g2s(stages + slot * C::kStageBytes + b * chunk_bytes, p.cache + ((int64_t)id * p.num_kv_heads + kvh) * chunk_bytes,
                 (uint32_t)chunk_bytes, &sh.full[slot]);
      }
      issued = j + 1;
    }
    if (lane == 0) {
      if (aborted) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      // never leave copies in flight, whether or not another role gave up
      for (int j = max(0, issued - 2); j < issued; ++j)
        if (!mbar_wait(&sh.full[j & 1], (j >> 1) & 1)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // =================================================================== MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_f16(kRows, kKv, kBF16, false, false);
      const uint32_t id_pv = tc::idesc_f16(kRows, D, kBF16, false, true);
      const uint32_t qa = smem_u32(qbuf);
      // Event-driven: QK(j) as soon as tile j has landed (and P(j - 2), which it
      // overwrites in TMEM, has gone to PV(j - 2)); PV(j) as soon as P(j) is
      // written -- so PV(j), and with it the release of tile j's stage, never
      // waits for the next tile's data.  Barriers are tested without blocking.
      // (tcgen05 operations of this thread execute in issue order, so S(j + 2)
      // overwrites P(j) only after PV(j) has read it.)
      const uint64_t qd0 = tc::smem_desc(qa, 16, 1024, tc::kSwizzle128B);
      int qk = 0, pv = 0;
      uint32_t idle = 0;
      bool ok = true;
      while (pv < n_kv) {
        bool progressed = false;
        if (qk < n_kv && pv >= qk - 1) {
          const int slot = qk & 1;
          if (mbar_test_wait(&sh.full[slot], (qk >> 1) & 1) &&
              (qk < 2 || mbar_test_wait(&sh.s_free[slot], ((qk >> 1) - 1) & 1))) {
            tc::fence_after_sync();
            const uint64_t kd0 = tc::smem_desc(smem_u32(stages + slot * C::kStageBytes), 16, C::kGroupBytes,
                                               tc::kSwizzle128B);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              tc::mma_f16(tmem + slot * kKv, qd0 + (uint64_t)((((kk >> 2) * C::kQAtomBytes) + (kk & 3) * 32) >> 4),
                          kd0 + (uint64_t)((((kk >> 2) * 1024) + (kk & 3) * 32) >> 4), id_qk, kk > 0);
            tc::commit(&sh.s_full[slot]);
            ++qk;
            progressed = true;
          }
        }
        if (pv < qk) {
          const int slot = pv & 1;
          if (mbar_test_wait(&sh.p_full[slot], (pv >> 1) & 1)) {
            tc::fence_after_sync();
            const uint64_t vd0 = tc::smem_desc(smem_u32(stages + slot * C::kStageBytes) + C::kAtoms * 1024, 1024,
                                               C::kGroupBytes, tc::kSwizzle128B);
            const int valid = min(kKv, kv_len - pv * kKv);
            const int nsteps = (valid + 15) >> 4;
#pragma unroll
            for (int kk = 0; kk < kKv / 16; ++kk) {
              if (kk < nsteps) {
                const uint64_t vdesc = vd0 + (uint64_t)((kk * 2 * C::kGroupBytes) >> 4);
                const uint32_t pa = tmem + slot * kKv + kk * 8;      // 16 tokens = 8 packed columns
                tc::mma_f16_ta(tmem + kOCol, pa, vdesc, id_pv, (pv > 0 || kk > 0) ? 1u : 0u);
                if (kLo) tc::mma_f16_ta(tmem + kOCol, pa + kKv / 2, vdesc, id_pv, 1u);
              }
            }
            tc::commit(&sh.pv_done[slot]);
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
      // every MMA this lane issued completes before TMEM can be freed
      tc::commit(&sh.mma_drain);
      if (!mbar_wait(&sh.mma_drain, 0)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // =================================================================== softmax warps (2-9)
    // Warpgroup wg = 0 / 1 owns S columns [64 wg, 64 wg + 64) (tokens) and O
    // columns [D/2 wg, D/2 wg + D/2) of the same 128 rows; per tile the two
    // exchange their row maxima (and at the end their row sums) through shared
    // memory under a bounded mbarrier.
    constexpr int kCols = kKv / 2;
    constexpr int kOC = D / 2;
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;               // TMEM lane = query row = (position, head)
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const int ipos = row / G;
    const bool row_ok = ipos < npos;
    const int pos = pos0 + ipos;                       // attends tokens t <= pos
    float m = -INFINITY, l = 0.f;                      // l: this half's share of the row sum
    bool ok = true;
    auto exchange = [&](int k, float v) -> float {     // k-th exchange: returns the other half's v
      sh.red[k & 1][wg][row] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.xbar);
      if (!__all_sync(kFull, mbar_wait(&sh.xbar, k & 1))) {
        ok = false;
        return 0.f;
      }
      return sh.red[k & 1][wg ^ 1][row];
    };
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      // wait results are made warp-uniform: the TMEM loads and stores below are
      // warp-collective (.sync.aligned) and must never run in a diverged warp
      if (!__all_sync(kFull, mbar_wait(&sh.s_full[sb], (j >> 1) & 1) && !sh.abort_flag)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float x[kCols / 16][16];
#pragma unroll
      for (int c = 0; c < kCols / 16; ++c) tc::tmem_ld16(lane_addr + sb * kKv + wg * kCols + c * 16, x[c]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_free[sb]);
      const int lim = (row_ok ? min(kKv, pos + 1 - j * kKv) : 0) - wg * kCols;   // columns of this half attended
      // x stays in raw score units (the scale, > 0, is folded into the exponent
      // below); masked columns become -inf.  Tiles wholly below the diagonal
      // skip the mask.
      float mt = -INFINITY;
      if (lim >= kCols) {
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c)
#pragma unroll
          for (int e = 0; e < 16; ++e) mt = fmaxf(mt, x[c][e]);
      } else {
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            x[c][e] = (c * 16 + e < lim) ? x[c][e] : -INFINITY;
            mt = fmaxf(mt, x[c][e]);
          }
      }
      mt *= p.scale_log2;   // base-2 units
      // after the exchange both halves have read their S columns, so P may be
      // written over them
      mt = fmaxf(mt, exchange(j, mt));
      if (!ok) break;
      // both halves see the same m and mt, so they take the same decisions
      const float m_new = fmaxf(m, mt);
      const bool need = m != -INFINITY && m_new > m + kRescaleThreshold;
      if (m == -INFINITY) m = m_new;
      if (__any_sync(kFull, need)) {
        // O holds exactly tiles < j once PV_{j-1} has completed (PV_j waits for
        // this warp's P).  The whole warp takes the O round trip; rows that keep
        // their max scale by 1.
        if (!__all_sync(kFull, mbar_wait(&sh.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float alpha = need ? exp2f(m - m_new) : 1.f;
        if (need) {
          l *= alpha;
          m = m_new;
        }
#pragma unroll
        for (int c = 0; c < kOC / 16; ++c) {
          float o[16];
          tc::tmem_ld16(lane_addr + kOCol + wg * kOC + c * 16, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= alpha;
          tc::tmem_st16(lane_addr + kOCol + wg * kOC + c * 16, o);
        }
      }
      // p = 2^(x - m) in fp32; P (in TMEM, two tokens per column) gets round(p)
      // and, for bf16, round(p - round(p))
      // (a row with every column so far masked has m = -inf: its x are all -inf
      // and with nm = 0 its p come out 0)
      const float nm = (m == -INFINITY) ? 0.f : -m;
#pragma unroll
      for (int h = 0; h < kCols / 32; ++h) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = h * 32 + 2 * e;
          const float a = ex2_approx(fmaf(x[c >> 4][c & 15], p.scale_log2, nm));
          const float b = ex2_approx(fmaf(x[c >> 4][(c & 15) + 1], p.scale_log2, nm));
          l += a + b;
          hi[e] = Elem<T>::pack2(a, b);
          if (kLo) {
            const float2 r = Elem<T>::to_float2(hi[e]);
            lo[e] = Elem<T>::pack2(a - r.x, b - r.y);
          }
        }
        const uint32_t col = lane_addr + sb * kKv + wg * (kCols / 2) + h * 16;
        tc::tmem_st16u(col, hi);
        if (kLo) tc::tmem_st16u(col + kKv / 2, lo);
      }
      // V rows of tokens past the tile's last token must not hold NaN/Inf
      // (0 * NaN = NaN): zero them, after the stage's bulk copy is complete
      const int valid = min(kKv, kv_len - j * kKv);
      if (valid & 15) {
        if (!__all_sync(kFull, mbar_wait(&sh.full[sb], (j >> 1) & 1))) {
          ok = false;
          break;
        }
      }
      uint8_t* stage = stages + sb * C::kStageBytes;
      // V rows of tokens past the tile's last token (thread = token row here):
      // zero, half of the 64-dim atoms per warpgroup
      if (row >= valid && row < ((valid + 15) & ~15)) {
        uint8_t* vrow = stage + (row >> 3) * C::kGroupBytes + C::kAtoms * 1024 + (row & 7) * 128;
#pragma unroll
        for (int a = 0; a < C::kAtoms; ++a)
          if ((a & 1) == wg)
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + a * 1024 + c * 16) = make_uint4(0, 0, 0, 0);
      }
      tc::tmem_wait_st();
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[sb]);
    }
    if (ok && n_kv > 0) ok = __all_sync(kFull, mbar_wait(&sh.pv_done[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1));
    float l_tot = 0.f;
    if (ok) l_tot = l + exchange(n_kv, l);
    if (ok) {
      tc::fence_after_sync();
      const float inv = row_ok && l_tot > 0.f ? 1.f / l_tot : 0.f;
      T* orow = out + ((int64_t)(first + q0 + ipos) * p.num_q_heads + kvh * G + row % G) * D + wg * kOC;
#pragma unroll
      for (int c = 0; c < kOC / 16; ++c) {
        float o[16];
        tc::tmem_ld16(lane_addr + kOCol + wg * kOC + c * 16, o);
        if (row_ok) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = Elem<T>::pack2(o[2 * e] * inv, o[2 * e + 1] * inv);
          *reinterpret_cast<uint4*>(orow + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(orow + c * 16 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    } else {
      if (lane == 0) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        sh.abort_flag = 1;
      }
      if (row_ok) {
        T* orow = out + ((int64_t)(first + q0 + ipos) * p.num_q_heads + kvh * G + row % G) * D + wg * kOC;
        for (int c = 0; c < kOC / 8; ++c) *reinterpret_cast<uint4*>(orow + c * 8) = make_uint4(0, 0, 0, 0);
      }
    }
  }

  // ---- tear-down: every MMA this CTA issued has completed (pv_done / s_full
  // waited above, or abandoned after a timeout), then TMEM is released
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D, int G>
cudaError_t launch_typed(const PrefillParams& p, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = set_smem_attribute_once<prefill_tc_kernel<T, D, G>>(C::kSmem);
  if (e != cudaSuccess) return e;
  constexpr int PT = kRows / G;
  const dim3 grid((unsigned)((p.max_query_len + PT - 1) / PT), (unsigned)p.num_kv_heads, (unsigned)p.num_seqs);
  prefill_tc_kernel<T, D, G><<<grid, kThreads, C::kSmem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_group(const PrefillParams& p, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_typed<T, D, 1>(p, stream);
    case 2: return launch_typed<T, D, 2>(p, stream);
    case 4: return launch_typed<T, D, 4>(p, stream);
    case 8: return launch_typed<T, D, 8>(p, stream);
    case 16: return launch_typed<T, D, 16>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, int head_size, int group, cudaStream_t stream) {
  if (dtype == PA_F16 && head_size == 128) return launch_group<__half, 128>(p, group, stream);
  if (dtype == PA_F16 && head_size == 64) return launch_group<__half, 64>(p, group, stream);
  if (dtype == PA_BF16 && head_size == 128) return launch_group<__nv_bfloat16, 128>(p, group, stream);
  if (dtype == PA_BF16 && head_size == 64) return launch_group<__nv_bfloat16, 64>(p, group, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
