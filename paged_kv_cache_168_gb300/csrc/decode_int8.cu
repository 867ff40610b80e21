// decode_int8.cu -- paged decode attention over an 8-bit cache, on CUDA cores.
//
// What is computed: the decode of the "vLLM" page, section "PageAttention"
// (softmax(scale * q . K_t) applied to V_t over the sequence's blocks, found
// through the block table), where the cache holds each K_t / V_t of a kv head
// as 8-bit codes c with one fp32 scale ("8bit KV Cache", the TurboMind section
// of the inference-framework notes): K_t = sk_t * c_K,t and V_t = sv_t * c_V,t.
// The scales are folded out of the inner loops:
//   z_t = sk_t * (scale * q . c_K,t),   o = sum_t (p_t * sv_t) c_V,t / sum_t p_t,
// so each code costs one byte permute, one subtraction (exact int8 -> fp32:
// the byte goes into the low mantissa bits of 2^23, then 2^23 + 128 is taken
// off) and one fma per query head.
//
// Structure (as the 16-bit CUDA-core kernel): CTA = (partition, kv head,
// sequence); warp 4 issues one bulk copy per (block, kv head) chunk -- codes and
// scales together, 2*bs*128 + 2*roundup16(4*bs) bytes -- into a 3-stage ring
// of 64-token stages; warps 0-3 consume with 8-lane groups, one token per group
// at a time, each lane owning one 16-byte piece (16 dims) of the 128-byte code
// rows.  Partitions produce (m, l, o~) merged by the shared log-sum-exp kernel.
// Every wait is bounded; a timeout sets PA_DEVERR_TIMEOUT.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pkv {

template <int G>
struct I8Cfg {
  static constexpr int D = 128;
  static constexpr int kConsumerWarps = 4;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int HPW = G == 1 ? 1 : 2;                    // query heads per warp
  static constexpr int NT = G / HPW;                            // head teams
  static constexpr int TW = kConsumerWarps / NT;                // token warps per team
  static constexpr int kStageTokens = 64;
  static constexpr int kStageBytes = kStageTokens * (2 * D + 32);   // the largest chunk per token (bs = 1)
  static constexpr int kStages = 3;
  static constexpr int kTokPerGroup = kStageTokens / (4 * TW);
  static constexpr int kRedFloats = TW * G * (D + 2);
  static_assert(NT * TW == kConsumerWarps, "head teams must tile the consumer warps");
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");
};

// 16 codes of one 16-byte piece -> exact fp32 values.
__device__ __forceinline__ void codes16(const uint4 u, float (&f)[16]) {
  const uint32_t w[4] = {u.x ^ 0x80808080u, u.y ^ 0x80808080u, u.z ^ 0x80808080u, u.w ^ 0x80808080u};
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int b = 0; b < 4; ++b)
      f[4 * k + b] = __uint_as_float(__byte_perm(w[k], 0x4B000000u, 0x7540 + b)) - 8388736.0f;
}

template <typename T>
__device__ __forceinline__ void load_q16(const T* p, float (&f)[16]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 v = Elem<T>::to_float2(u[k]);
    f[2 * k] = v.x;
    f[2 * k + 1] = v.y;
  }
}

template <typename T, int G>
__device__ void i8_zero_rows(const DecodeParams& p, int s, int kvh) {
  T* out = static_cast<T*>(p.out);
  for (int i = threadIdx.x; i < G * 128; i += blockDim.x)
    out[((int64_t)s * p.num_q_heads + kvh * G + i / 128) * 128 + i % 128] = Elem<T>::from_float(0.f);
}

template <typename T, int G>
__global__ void __launch_bounds__(I8Cfg<G>::kThreads, 3)
    decode_i8_kernel(const __grid_constant__ DecodeParams p) {
  using C = I8Cfg<G>;
  constexpr int D = C::D;
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
      i8_zero_rows<T, G>(p, s, kvh);
      if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_CONTEXT);
    }
    return;
  }
  if (ctx <= 0) {
    if (part == 0) i8_zero_rows<T, G>(p, s, kvh);
    return;
  }
  const int t_first = window_start(ctx, bs, p.window, p.ring_blocks);
  const int t_base = (t_first / bs) * bs;
  const int t0 = t_base + part * P;
  if (t0 >= ctx) return;
  const int t1 = min(ctx, t0 + P);
  const int n_parts = (ctx - t_base + P - 1) / P;
  const int j0 = t0 / bs;
  const int nblk = (t1 - t0 + bs - 1) / bs;
  const I8Layout L{bs, p.num_kv_heads};
  const int64_t chunk_bytes = L.chunk_bytes();
  const int64_t sbytes = L.scale_bytes();
  const int blocks_per_stage = C::kStageTokens / bs;
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

  const int64_t ws_row = ((int64_t)s * p.num_q_heads + kvh * G) * p.max_parts + part;
  if (flag_bad) {
    if (threadIdx.x == 0) report(p.dev_err, PA_DEVERR_BLOCK_ID);
    if (n_parts == 1) {
      i8_zero_rows<T, G>(p, s, kvh);
    } else if (threadIdx.x < G) {
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 0] = 0.f;
      p.ws_ml[(ws_row + (int64_t)threadIdx.x * p.max_parts) * 2 + 1] = -1.f;
    }
    return;
  }

  if (warp == C::kConsumerWarps) {
    // ---------------- producer
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
      for (int st = max(0, issued - C::kStages); st < issued; ++st)
        if (!mbar_wait(&full_bar[st % C::kStages], (st / C::kStages) & 1)) report(p.dev_err, PA_DEVERR_TIMEOUT);
    }
    return;
  }

  // ---------------- consumers
  const int team = warp / C::TW, tw = warp % C::TW;
  const int gi = lane >> 3, j = lane & 7;
  constexpr int HPW = C::HPW, TPG = C::kTokPerGroup;

  float q[HPW][16];
  {
    const T* qp = static_cast<const T*>(p.q) + (int64_t)s * p.q_seq_stride;
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      load_q16<T>(qp + (kvh * G + team * HPW + i) * D + j * 16, q[i]);
#pragma unroll
      for (int e = 0; e < 16; ++e) q[i][e] *= p.scale_log2;
    }
  }
  float m[HPW], l[HPW], acc[HPW][16];
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[i][e] = 0.f;
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
    const int lo = t_first - (t0 + st * C::kStageTokens);

    float sc[TPG][HPW];
#pragma unroll
    for (int k = 0; k < TPG; ++k) {
      const int pos = tw * 4 + gi + k * 4 * C::TW;
      const bool live = pos >= lo && pos < valid;
      float dot[HPW][4];
#pragma unroll
      for (int i = 0; i < HPW; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) dot[i][c] = 0.f;
      float sk = 0.f;
      if (live) {
        const int blk = pos / bs, tb = pos % bs;
        const uint8_t* cb = buf + blk * chunk_bytes;
        float f[16];
        codes16(*reinterpret_cast<const uint4*>(cb + tb * D + ((j ^ (tb & 7)) << 4)), f);
        sk = *reinterpret_cast<const float*>(cb + 2 * bs * D + 4 * tb);
#pragma unroll
        for (int i = 0; i < HPW; ++i)
#pragma unroll
          for (int e = 0; e < 16; ++e) dot[i][e & 3] = fmaf(q[i][e], f[e], dot[i][e & 3]);
      }
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        float v = (dot[i][0] + dot[i][1]) + (dot[i][2] + dot[i][3]);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        sc[k][i] = live ? v * sk : -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      float mt = sc[0][i];
#pragma unroll
      for (int k = 1; k < TPG; ++k) mt = fmaxf(mt, sc[k][i]);
      const float mn = fmaxf(m[i], mt);
      if (mn != -INFINITY) {
        const float alpha = exp2f(m[i] - mn);
        l[i] *= alpha;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[i][e] *= alpha;
        m[i] = mn;
      }
    }
#pragma unroll
    for (int k = 0; k < TPG; ++k) {
      const int pos = tw * 4 + gi + k * 4 * C::TW;
      if (pos >= lo && pos < valid) {
        const int blk = pos / bs, tb = pos % bs;
        const uint8_t* cb = buf + blk * chunk_bytes;
        float f[16];
        codes16(*reinterpret_cast<const uint4*>(cb + (bs + tb) * D + ((j ^ (tb & 7)) << 4)), f);
        const float sv = *reinterpret_cast<const float*>(cb + 2 * bs * D + sbytes + 4 * tb);
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
          const float w = exp2f(sc[k][i] - m[i]);
          l[i] += w;
          const float wv = w * sv;
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[i][e] = fmaf(wv, f[e], acc[i][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }

  // combine the four lane groups of the warp
#pragma unroll
  for (int i = 0; i < HPW; ++i) {
    float mw = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], 8));
    mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
    const float f = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - mw);
    l[i] *= f;
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 8);
    l[i] += __shfl_xor_sync(0xffffffffu, l[i], 16);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float v = acc[i][e] * f;
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      acc[i][e] = v;
    }
    m[i] = mw;
  }
  float* red_acc = red;
  float* red_m = red + C::TW * G * D;
  float* red_l = red_m + C::TW * G;
  if (gi == 0) {
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
      const int g = team * HPW + i;
#pragma unroll
      for (int e = 0; e < 16; ++e) red_acc[(tw * G + g) * D + j * 16 + e] = acc[i][e];
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
    float Lsum = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < C::TW; ++w) {
      const float mw = red_m[w * G + g];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      Lsum = fmaf(f, red_l[w * G + g], Lsum);
      O = fmaf(f, red_acc[(w * G + g) * D + d], O);
    }
    if (n_parts == 1) {
      out[((int64_t)s * p.num_q_heads + kvh * G + g) * D + d] = Elem<T>::from_float(O / Lsum);
    } else {
      const int64_t row = ws_row + (int64_t)g * p.max_parts;
      p.ws_o[row * D + d] = O;
      if (d == 0) {
        p.ws_ml[row * 2 + 0] = M;
        p.ws_ml[row * 2 + 1] = Lsum;
      }
    }
  }
}

template <typename T, int G>
static cudaError_t launch_i8_typed(const DecodeParams& p, int act_dtype, cudaStream_t stream) {
  using C = I8Cfg<G>;
  const int max_blk = (p.partition_size + p.block_size - 1) / p.block_size + 1;
  const size_t smem = (size_t)C::kStages * C::kStageBytes + (size_t)C::kRedFloats * 4 + (size_t)max_blk * 4;
  cudaError_t e = set_smem_attribute_once<decode_i8_kernel<T, G>>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.max_parts, (unsigned)p.num_kv_heads, (unsigned)p.num_seqs);
  decode_i8_kernel<T, G><<<grid, C::kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge(p, act_dtype, 128, stream);
}

template <typename T>
static cudaError_t launch_i8_group(const DecodeParams& p, int act_dtype, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_i8_typed<T, 1>(p, act_dtype, stream);
    case 2: return launch_i8_typed<T, 2>(p, act_dtype, stream);
    case 4: return launch_i8_typed<T, 4>(p, act_dtype, stream);
    case 8: return launch_i8_typed<T, 8>(p, act_dtype, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_i8(const DecodeParams& p, int act_dtype, int group, cudaStream_t stream) {
  if (act_dtype == PA_F16) return launch_i8_group<__half>(p, act_dtype, group, stream);
  if (act_dtype == PA_BF16) return launch_i8_group<__nv_bfloat16>(p, act_dtype, group, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
