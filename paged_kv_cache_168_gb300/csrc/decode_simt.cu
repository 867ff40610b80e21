// decode_simt.cu -- paged decode attention on CUDA cores.
//
// What is computed ("vLLM" page, section "PageAttention"): for each sequence s
// and query head h, softmax(scale * q . K_t) over the sequence's ctx tokens,
// applied to V_t, where token t is found through the block table (two-level
// addressing: logical block t / bs -> physical block, slot t % bs).  GQA: query
// head h reads kv head h / G.  Long contexts are cut into partitions of P
// tokens (FlashDecoding, "vLLM" page "Prefill vs decoding" item 5); each
// partition yields (m, l, o~) and a second kernel merges them by log-sum-exp.
//
// Structure of one CTA = (partition, kv head, sequence):
//   * warp 4 (producer): one lane issues a 1-D bulk copy (cp.async.bulk) per
//     block of the partition -- a (block, kv head) chunk is one contiguous
//     2*bs*D*2-byte piece of the cache -- into a 4-stage ring of 16 KiB stages,
//     completion tracked by mbarriers (full / empty per stage).
//   * warps 0-3 (consumers): lanes form groups of 8; a group owns one token at a
//     time and each lane owns one 16-byte piece of every 128-byte K/V row, so a
//     warp-wide 16-byte shared load touches four rows with no bank conflict.
//     Scores are reduced over the 8 lanes with three xor-shuffles; each group
//     keeps its own running max / sum / accumulator (online softmax), combined
//     across groups and warps once per partition.
//   * all G query heads of the kv head are handled by the CTA, so each KV byte
//     is read from HBM once.  For G > 2 the heads are split over warps
//     ("head teams", 2 heads per warp) which then all read the staged chunk.
// Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT and abandons the item.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

template <int D, int G>
struct SimtCfg {
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int HPW = G == 1 ? 1 : 2;                    // query heads per warp
  static constexpr int NT = G / HPW;                            // head teams
  static constexpr int TW = kConsumerWarps / NT;                // token warps per team
  static constexpr int kAtoms = D / 64;                         // 128-byte rows per K (or V) vector
  static constexpr int kTokBytes = 2 * D * 2;                   // K + V bytes per token per kv head
  static constexpr int kStageBytes = 16384;
  static constexpr int kStageTokens = kStageBytes / kTokBytes;  // 32 (D=128) or 64 (D=64)
  static constexpr int kStages = 4;
  static constexpr int kTokPerGroup = kStageTokens / (4 * TW);  // tokens per lane group per stage
  static constexpr int kRedFloats = TW * G * (D + 2);           // cross-warp reduction area
  static_assert(NT * TW == kConsumerWarps, "head teams must tile the consumer warps");
};

template <typename T>
__device__ __forceinline__ void load_row8(const uint8_t* p, float (&f)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const float2 a = Elem<T>::to_float2(u.x), b = Elem<T>::to_float2(u.y);
  const float2 c = Elem<T>::to_float2(u.z), d = Elem<T>::to_float2(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

// Zero the output rows of the CTA's query heads (context <= 0 or invalid item).
template <typename T, int D, int G>
__device__ void write_zero_rows(const DecodeParams& p, int s, int kvh) {
  T* out = static_cast<T*>(p.out);
  for (int i = threadIdx.x; i < G * D; i += blockDim.x)
    out[((int64_t)s * p.num_q_heads + kvh * G + i / D) * D + i % D] = Elem<T>::from_float(0.f);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(SimtCfg<D, G>::kThreads, 3)
    decode_simt_kernel(const __grid_constant__ DecodeParams p) {
  using C = SimtCfg<D, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes);
  int32_t* ids = reinterpret_cast<int32_t*>(red + C::kRedFloats);
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int flag_bad;
  __shared__ volatile int flag_abort;

  const int part = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.block_size, P = p.partition_size;
  const int ctx = p.context_lens[s];

  if (!context_ok(p, ctx)) {
    if (part == 0) {
      write_zero_rows<T, D, G>(p, s, kvh);
      if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
    }
    return;
  }
  if (ctx <= 0) {
    if (part == 0) write_zero_rows<T, D, G>(p, s, kvh);
    return;
  }
  const int t_first = window_start(ctx, bs, p.window, p.ring_blocks);   // first attended position
  const int t_base = (t_first / bs) * bs;                              // partitions start here
  const int t0 = t_base + part * P;
  if (t0 >= ctx) return;
  const int t1 = min(ctx, t0 + P);
  const int n_parts = (ctx - t_base + P - 1) / P;
  const int j0 = t0 / bs;
  const int nblk = (t1 - t0 + bs - 1) / bs;
  const int64_t chunk_bytes = 2LL * bs * D * 2;
  const int blocks_per_stage = C::kStageTokens / bs;
  const int R = bs < 8 ? bs : 8;              // token rows per atom (8, or the whole block)
  const int atom_bytes = R * 128;
  const int n_stages = (t1 - t0 + C::kStageTokens - 1) / C::kStageTokens;

  if (threadIdx.x == 0) {
    flag_bad = 0;
    flag_abort = 0;
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], C::kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
    const int b = p.block_tables[(int64_t)s * p.bt_stride + table_index(j0 + i, p.ring_blocks)];
    ids[i] = b;
    if (b < 0 || b >= p.num_blocks) flag_bad = 1;
  }
  __syncthreads();

  const int64_t ws_row = ((int64_t)s * p.num_q_heads + kvh * G) * p.max_parts + part;  // head 0 of the CTA
  if (flag_bad) {
    if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_BLOCK_ID);
    if (n_parts == 1) {
      write_zero_rows<T, D, G>(p, s, kvh);
    } else if (threadIdx.x < G) {
      // mark this partition invalid for the merge (sum < 0 never occurs otherwise)
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 0] = 0.f;
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 1] = -1.f;
    }
    return;
  }

  if (warp == C::kConsumerWarps) {
    // ---------------- producer: lane 0 arms each stage, all lanes issue its copies
    int issued = 0;
    bool aborted = false;
    for (int st = 0; st < n_stages && !aborted; ++st) {
      const int slot = st % C::kStages;
      if (st >= C::kStages && !mbar_wait_polls(&empty_bar[slot], ((st / C::kStages) - 1) & 1, p.wait_polls)) {
        aborted = true;
        break;
      }
      if (flag_abort) {
        aborted = true;
        break;
      }
      const int jb = st * blocks_per_stage;
      const int je = min(nblk, jb + blocks_per_stage);
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)((je - jb) * chunk_bytes));
      __syncwarp();
      uint8_t* dst = stages + slot * C::kStageBytes;
      for (int j = jb + lane; j < je; j += 32)
        bulk_g2s(dst + (j - jb) * chunk_bytes, p.cache + ((int64_t)ids[j] * p.num_kv_heads + kvh) * chunk_bytes,
                 (uint32_t)chunk_bytes, &full_bar[slot]);
      issued = st + 1;
    }
    if (lane == 0) {
      if (aborted) {
        report(p.dev_err, PA_DEVERR_TIMEOUT);
        flag_abort = 1;
      }
      // never leave the CTA with copies in flight: wait (bounded) for the last
      // phase issued on every stage
      for (int st = max(0, issued - C::kStages); st < issued; ++st)
        if (!mbar_wait(&full_bar[st % C::kStages], (st / C::kStages) & 1)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    return;   // the CTA's shared memory lives until every thread has exited
  }

  // ---------------- consumers
  const int team = warp / C::TW, tw = warp % C::TW;
  const int gi = lane >> 3, j = lane & 7;
  constexpr int HPW = C::HPW, A = C::kAtoms, TPG = C::kTokPerGroup;

  float q[HPW][A][8];
  {
    const T* qp = static_cast<const T*>(p.q) + (int64_t)s * p.q_seq_stride;
#pragma unroll
    for (int i = 0; i < HPW; ++i)
#pragma unroll
      for (int a = 0; a < A; ++a) {
        load_row8<T>(reinterpret_cast<const uint8_t*>(qp + (kvh * G + team * HPW + i) * D + a * 64 + j * 8),
                     q[i][a]);
#pragma unroll
        for (int e = 0; e < 8; ++e) q[i][a][e] *= p.scale_log2;
      }
  }
  float m[HPW], l[HPW], acc[HPW][A][8];
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int a = 0; a < A; ++a)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][a][e] = 0.f;
  }

  bool aborted = false;
  for (int st = 0; st < n_stages; ++st) {
    const int slot = st % C::kStages;
    if (!mbar_wait_polls(&full_bar[slot], (st / C::kStages) & 1, p.wait_polls)) {
      if (lane == 0) report(p.dev_err, PA_DEVERR_TIMEOUT);
      flag_abort = 1;
      aborted = true;
      break;
    }
    const uint8_t* buf = stages + slot * C::kStageBytes;
    const int valid = min(C::kStageTokens, t1 - (t0 + st * C::kStageTokens));
    const int lo = t_first - (t0 + st * C::kStageTokens);   // positions before the window (first stage only)

    float sc[TPG][HPW];
#pragma unroll
    for (int k = 0; k < TPG; ++k) {
      const int pos = tw * 4 + gi + k * 4 * C::TW;
      float part_dot[HPW];
#pragma unroll
      for (int i = 0; i < HPW; ++i) part_dot[i] = 0.f;
      if (pos >= lo && pos < valid) {
        const int blk = pos / bs, tb = pos % bs, g8 = tb / R, r = tb % R;
        const uint8_t* kb = buf + blk * chunk_bytes + (g8 * 2 * A) * atom_bytes + r * 128 + ((j ^ r) << 4);
#pragma unroll
        for (int a = 0; a < A; ++a) {
          float kf[8];
          load_row8<T>(kb + a * atom_bytes, kf);
#pragma unroll
          for (int i = 0; i < HPW; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) part_dot[i] = fmaf(q[i][a][e], kf[e], part_dot[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        float v = part_dot[i];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        sc[k][i] = (pos >= lo && pos < valid) ? v : -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      float mt = sc[0][i];
#pragma unroll
      for (int k = 1; k < TPG; ++k) mt = fmaxf(mt, sc[k][i]);
      const float mn = fmaxf(m[i], mt);
      if (mn != -INFINITY) {
        const float alpha = exp2f(m[i] - mn);   // 0 when m was -inf
        l[i] *= alpha;
#pragma unroll
        for (int a = 0; a < A; ++a)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][a][e] *= alpha;
        m[i] = mn;
      }
    }
#pragma unroll
    for (int k = 0; k < TPG; ++k) {
      const int pos = tw * 4 + gi + k * 4 * C::TW;
      if (pos >= lo && pos < valid) {
        const int blk = pos / bs, tb = pos % bs, g8 = tb / R, r = tb % R;
        const uint8_t* vb = buf + blk * chunk_bytes + ((g8 * 2 + 1) * A) * atom_bytes + r * 128 + ((j ^ r) << 4);
        float w[HPW];
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
          w[i] = exp2f(sc[k][i] - m[i]);
          l[i] += w[i];
        }
#pragma unroll
        for (int a = 0; a < A; ++a) {
          float vf[8];
          load_row8<T>(vb + a * atom_bytes, vf);
#pragma unroll
          for (int i = 0; i < HPW; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][a][e] = fmaf(w[i], vf[e], acc[i][a][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }

  // combine the four lane groups of the warp (lanes differing in bits 3 and 4)
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    float mw = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 8));
    mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
    const float f = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mw);
    l[i] *= f;
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 8);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 16);
#pragma unroll
    for (int a = 0; a < A; ++a)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = acc[i][a][e] * f;
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        acc[i][a][e] = v;
      }
    m[i] = mw;
  }
  // cross-warp combine through shared memory: red = [TW][G][D] acc, then [TW][G] m, [TW][G] l
  float* red_acc = red;
  float* red_m = red + C::TW * G * D;
  float* red_l = red_m + C::TW * G;
  if (gi == 0) {
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      const int g = team * HPW + i;
#pragma unroll
      for (int a = 0; a < A; ++a)
#pragma unroll
        for (int e = 0; e < 8; ++e) red_acc[(tw * G + g) * D + a * 64 + j * 8 + e] = acc[i][a][e];
      if (j == 0) {
        red_m[tw * G + g] = m[i];
        red_l[tw * G + g] = l[i];
      }
    }
  }
  named_bar_sync(1, C::kConsumerWarps * 32);
  constexpr int kCT = C::kConsumerWarps * 32;
  if (aborted || flag_abort) {
    if (n_parts == 1) {
      T* out = static_cast<T*>(p.out);
      for (int i = threadIdx.x; i < G * D; i += kCT)
        out[((int64_t)s * p.num_q_heads + kvh * G + i / D) * D + i % D] = Elem<T>::from_float(0.f);
    } else if (threadIdx.x < G) {
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 0] = 0.f;
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 1] = -1.f;
    }
    return;
  }
  T* out = static_cast<T*>(p.out);
  for (int idx = threadIdx.x; idx < G * D; idx += kCT) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::TW; ++w) M = fmaxf(M, red_m[w * G + g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < C::TW; ++w) {
      const float mw = red_m[w * G + g];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      L = fmaf(f, red_l[w * G + g], L);
      O = fmaf(f, red_acc[(w * G + g) * D + d], O);
    }
    if (n_parts == 1) {
      out[((int64_t)s * p.num_q_heads + kvh * G + g) * D + d] = Elem<T>::from_float(O / L);
    } else {
      const int64_t row = ws_row + (int64_t)g * p.max_parts;
      p.ws_o[row * D + d] = O;
      if (d == 0) {
        p.ws_ml[row * 2 + 0] = M;
        p.ws_ml[row * 2 + 1] = L;
      }
    }
  }
}

// Log-sum-exp merge of partition results: M = max_p m_p,
// out = sum_p 2^(m_p - M) o~_p / sum_p 2^(m_p - M) l_p  (scores in base-2 units).
// grid = (num_q_heads / GB, sequences), block = GB x D threads: GB query
// heads of one kv head per CTA.  Rows with a single partition were written by the
// decode kernel and are skipped here; a row with an invalid partition (l < 0)
// gets zeros.
// Shared prefix (SP): the partitions of a row are its group's prefix
// partitions, then its own; the decode kernel recorded their number, the
// effective prefix and the first member of the sequence's prefix item, whose
// table row the prefix was read through.  A member whose block ids differ from
// that row inside the prefix gets zero rows and PA_DEVERR_PREFIX.
constexpr int kMergeRegs = 8;   // rows with up to this many partitions merge from registers

template <typename T, int D, bool SP, int GB>
__global__ void __launch_bounds__(D * GB) merge_partitions_kernel(const __grid_constant__ DecodeParams p) {
  const int s = blockIdx.y, d = threadIdx.x % D, sub = threadIdx.x / D;
  const int h = blockIdx.x * GB + sub;             // this thread's query head
  T* out_s = static_cast<T*>(p.out) + (int64_t)s * p.num_q_heads * D;
  int n;
  bool differ = false, check = false;
  if constexpr (SP) {
    n = p.ws_seq[s];                               // 0 for an empty or invalid context
    const int eff = p.ws_seq[p.num_seqs + s], lead = p.ws_seq[2 * p.num_seqs + s];
    if (n == 0 || (eff == 0 && n <= 1)) return;   // zero rows, or written by the decode kernel
    // the member's prefix block ids against its leader's: loaded now, decided
    // (one barrier) after the merge's own loads
    check = eff > 0 && lead != s;
    if (check) {
      const int32_t* mine = p.block_tables + (int64_t)s * p.bt_stride;
      const int32_t* theirs = p.block_tables + (int64_t)lead * p.bt_stride;
      for (int j = threadIdx.x; j < eff / p.block_size; j += D * GB) differ |= mine[j] != theirs[j];
    }
  } else {
    const int ctx = p.context_lens[s];
    if (ctx <= 0 || !context_ok(p, ctx)) return;
    n = (ctx - attended_from(p, ctx) + p.partition_size - 1) / p.partition_size;
    if (n <= 1) return;
  }
  const int64_t row0 = ((int64_t)s * p.num_q_heads + h) * p.max_parts;
  float res;
  if (n <= kMergeRegs) {
    // the usual case: every partition's (m, l) and o loaded at once
    float mv[kMergeRegs], lv[kMergeRegs], ov[kMergeRegs];
#pragma unroll
    for (int i = 0; i < kMergeRegs; ++i) {
      if (i < n) {
        mv[i] = p.ws_ml[(row0 + i) * 2 + 0];
        lv[i] = p.ws_ml[(row0 + i) * 2 + 1];
        ov[i] = p.ws_o[(row0 + i) * D + d];
      }
    }
    float M = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kMergeRegs; ++i)
      if (i < n) {
        bad |= lv[i] < 0.f;
        M = fmaxf(M, mv[i]);
      }
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int i = 0; i < kMergeRegs; ++i)
      if (i < n) {
        const float w = exp2f(mv[i] - M);
        L = fmaf(w, lv[i], L);
        O = fmaf(w, ov[i], O);
      }
    res = bad ? 0.f : O / L;
  } else {
    // every thread runs the same iterations (the same n), so the barriers
    // below are reached uniformly
    __shared__ float sm_w[GB][256];
    float M = -INFINITY;
    bool bad = false;
    for (int i = 0; i < n; ++i) {
      bad |= p.ws_ml[(row0 + i) * 2 + 1] < 0.f;
      M = fmaxf(M, p.ws_ml[(row0 + i) * 2 + 0]);
    }
    float L = 0.f, O = 0.f;
    for (int i0 = 0; i0 < n; i0 += 256) {
      const int cnt = min(256, n - i0);
      __syncthreads();
      for (int i = d; i < cnt; i += D) sm_w[sub][i] = exp2f(p.ws_ml[(row0 + i0 + i) * 2 + 0] - M);
      __syncthreads();
      for (int i = 0; i < cnt; ++i) {
        const float w = sm_w[sub][i];
        L = fmaf(w, p.ws_ml[(row0 + i0 + i) * 2 + 1], L);
        O = fmaf(w, p.ws_o[(row0 + i0 + i) * D + d], O);
      }
    }
    res = bad ? 0.f : O / L;
  }
  if (SP && check && __syncthreads_or(differ)) {   // check is the same in every thread of the CTA
    res = 0.f;
    if (threadIdx.x == 0 && blockIdx.x == 0) report(p.dev_err, PA_DEVERR_PREFIX);
  }
  out_s[h * D + d] = Elem<T>::from_float(res);
}

// Launches the merge over every sequence, GB query heads of one kv head per
// CTA: the most (up to 4) that still leave two CTAs per SM of a 152-SM GPU.
template <typename T, int D, bool SP>
static cudaError_t launch_merge_typed(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.num_q_heads / p.num_kv_heads;
  const int64_t rows = (int64_t)p.num_seqs * p.num_q_heads;
  int gb = 1;
  while (gb < 4 && G % (2 * gb) == 0 && rows / (2 * gb) >= 2 * 152) gb *= 2;
  const dim3 grid((unsigned)(p.num_q_heads / gb), (unsigned)p.num_seqs);
  if (gb == 1) merge_partitions_kernel<T, D, SP, 1><<<grid, D, 0, stream>>>(p);
  else if (gb == 2) merge_partitions_kernel<T, D, SP, 2><<<grid, 2 * D, 0, stream>>>(p);
  else merge_partitions_kernel<T, D, SP, 4><<<grid, 4 * D, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int D, int G>
static cudaError_t launch_typed(const DecodeParams& p, cudaStream_t stream) {
  using C = SimtCfg<D, G>;
  const int max_blk = (p.partition_size + p.block_size - 1) / p.block_size + 1;
  const size_t smem = (size_t)C::kStages * C::kStageBytes + (size_t)C::kRedFloats * 4 + (size_t)max_blk * 4;
  auto kern = decode_simt_kernel<T, D, G>;
  cudaError_t e = set_smem_attribute_once<decode_simt_kernel<T, D, G>>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.max_parts, (unsigned)p.num_kv_heads, (unsigned)p.num_seqs);
  kern<<<grid, C::kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.max_parts <= 1) return e;
  return launch_merge_typed<T, D, false>(p, stream);
}

cudaError_t launch_merge(const DecodeParams& p, int dtype, int head_size, cudaStream_t stream) {
  if (p.max_parts <= 1) return cudaSuccess;
  if (dtype == PA_F16 && head_size == 128) return launch_merge_typed<__half, 128, false>(p, stream);
  if (dtype == PA_F16 && head_size == 64) return launch_merge_typed<__half, 64, false>(p, stream);
  if (dtype == PA_BF16 && head_size == 128) return launch_merge_typed<__nv_bfloat16, 128, false>(p, stream);
  if (dtype == PA_BF16 && head_size == 64) return launch_merge_typed<__nv_bfloat16, 64, false>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_merge_sp(const DecodeParams& p, int dtype, int head_size, cudaStream_t stream) {
  if (dtype == PA_F16 && head_size == 128) return launch_merge_typed<__half, 128, true>(p, stream);
  if (dtype == PA_BF16 && head_size == 128) return launch_merge_typed<__nv_bfloat16, 128, true>(p, stream);
  return cudaErrorInvalidValue;
}

template <typename T, int D>
static cudaError_t launch_group(const DecodeParams& p, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_typed<T, D, 1>(p, stream);
    case 2: return launch_typed<T, D, 2>(p, stream);
    case 4: return launch_typed<T, D, 4>(p, stream);
    case 8: return launch_typed<T, D, 8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, int head_size, int group,
                               cudaStream_t stream) {
  if (dtype == PA_F16) {
    if (head_size == 64) return launch_group<__half, 64>(p, group, stream);
    if (head_size == 128) return launch_group<__half, 128>(p, group, stream);
  } else if (dtype == PA_BF16) {
    if (head_size == 64) return launch_group<__nv_bfloat16, 64>(p, group, stream);
    if (head_size == 128) return launch_group<__nv_bfloat16, 128>(p, group, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pkv
