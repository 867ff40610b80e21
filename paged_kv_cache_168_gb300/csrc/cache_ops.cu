// cache_ops.cu -- reshape_and_cache (slot scatter) and whole-block copies.
//
// reshape_and_cache restates store_kvcache (nano-vLLM article, section 5.2.3):
// token i's K and V vectors go to slot slot_mapping[i]; -1 skips the token.
// Here one thread moves one 16-byte piece (8 elements) of one head vector, so
// a token's 2 x Hkv x D elements are written by 2*Hkv*D/8 threads with 16-byte
// loads and stores; every piece lands in one 16-byte piece of the cache layout.
//
// The 8-bit cache has its own writer (quantisation per stored vector, below).
//
// Block copies serve both copy_blocks (copy-on-write inside the device pool)
// and swap_blocks (device pool <-> pinned host pool, addressed through its
// device mapping); "vLLM" page, section "CacheEngine".
#include "common.cuh"
#include "kernels.h"

namespace pkv {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    uint8_t* __restrict__ cache, Layout L, int64_t nslots, const uint8_t* __restrict__ key,
    int64_t key_stride_bytes, const uint8_t* __restrict__ value, int64_t value_stride_bytes,
    const int64_t* __restrict__ slot_mapping, int32_t n, uint32_t* dev_err) {
  const int pieces = L.D / 8;                       // 16-byte pieces per head vector
  const int64_t per_token = 2LL * L.Hkv * pieces;
  const int64_t total = per_token * n;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = idx / per_token;
    const int rem = (int)(idx - i * per_token);
    const int part = rem / (L.Hkv * pieces);
    const int h = (rem / pieces) % L.Hkv;
    const int c = rem % pieces;
    const int64_t slot = slot_mapping[i];
    if (slot == -1) continue;
    if (slot < 0 || slot >= nslots) {
      if (rem == 0) report(dev_err, PA_DEVERR_SLOT);
      continue;
    }
    const uint8_t* src = (part ? value + i * value_stride_bytes : key + i * key_stride_bytes) +
                         ((int64_t)h * L.D + c * 8) * 2;
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const int64_t block = slot / L.bs;
    const int t = (int)(slot - block * L.bs);
    *reinterpret_cast<uint4*>(cache + L.offset(block, h, part, t, c * 8) * 2) = v;
  }
}

cudaError_t launch_reshape_and_cache(uint8_t* layer_base, int32_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_size, const void* key,
                                     int64_t key_stride, const void* value, int64_t value_stride,
                                     const int64_t* slot_mapping, int32_t n, uint32_t* dev_err,
                                     cudaStream_t stream) {
  Layout L{block_size, head_size, num_kv_heads};
  const int64_t total = 2LL * num_kv_heads * (head_size / 8) * n;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  reshape_and_cache_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      layer_base, L, (int64_t)num_blocks * block_size, static_cast<const uint8_t*>(key),
      key_stride * 2, static_cast<const uint8_t*>(value), value_stride * 2, slot_mapping, n, dev_err);
  return cudaGetLastError();
}

// 8-bit cache writer: one warp per (token, part, kv head) vector of 128
// elements, 4 per lane.  amax by a warp max-reduction; scale = amax / 127 and
// code = round-half-even(x * (127 / amax)) clipped to +-127, with IEEE fp32
// division and multiplication (no contraction), so the codes are a pure
// function of the input bits.  A lane's 4 codes are one 4-byte store into the
// swizzled row (dims 4l..4l+3 lie in piece l / 4).
template <typename T>
__global__ void __launch_bounds__(256) reshape_and_cache_i8_kernel(
    uint8_t* __restrict__ cache, I8Layout L, int64_t nslots, const uint8_t* __restrict__ key,
    int64_t key_stride_bytes, const uint8_t* __restrict__ value, int64_t value_stride_bytes,
    const int64_t* __restrict__ slot_mapping, int32_t n, uint32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  const int64_t vectors = 2LL * L.Hkv * n;
  const int64_t warp_stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < vectors; w += warp_stride) {
    const int64_t i = w / (2 * L.Hkv);
    const int rem = (int)(w - i * 2 * L.Hkv);
    const int part = rem / L.Hkv, h = rem % L.Hkv;
    const int64_t slot = slot_mapping[i];
    if (slot == -1) continue;               // warp-uniform: the whole warp serves one vector
    if (slot < 0 || slot >= nslots) {
      if (rem == 0 && lane == 0) report(dev_err, PA_DEVERR_SLOT);
      continue;
    }
    const uint8_t* src = (part ? value + i * value_stride_bytes : key + i * key_stride_bytes) +
                         ((int64_t)h * I8Layout::D + lane * 4) * 2;
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const float2 a = Elem<T>::to_float2(u.x), b = Elem<T>::to_float2(u.y);
    const float x[4] = {a.x, a.y, b.x, b.y};
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    uint32_t packed = 0;
    float scale = 0.f;
    if (amax > 0.f) {
      const float inv = __fdiv_rn(127.f, amax);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = min(127, max(-127, __float2int_rn(__fmul_rn(x[e], inv))));
        packed |= (uint32_t)(c & 0xff) << (8 * e);
      }
      scale = __fdiv_rn(amax, 127.f);
    }
    const int64_t block = slot / L.bs;
    const int t = (int)(slot - block * L.bs);
    *reinterpret_cast<uint32_t*>(cache + L.code(block, h, part, t, lane * 4)) = packed;
    if (lane == 0) *reinterpret_cast<float*>(cache + L.scale(block, h, part, t)) = scale;
  }
}

cudaError_t launch_reshape_and_cache_i8(uint8_t* layer_base, int32_t num_blocks, int32_t block_size,
                                        int32_t num_kv_heads, int act_dtype, const void* key, int64_t key_stride,
                                        const void* value, int64_t value_stride, const int64_t* slot_mapping,
                                        int32_t n, uint32_t* dev_err, cudaStream_t stream) {
  I8Layout L{block_size, num_kv_heads};
  const int64_t warps = 2LL * num_kv_heads * n;
  const int threads = 256;
  int64_t blocks = (warps * 32 + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  const auto* k = static_cast<const uint8_t*>(key);
  const auto* v = static_cast<const uint8_t*>(value);
  const int64_t nslots = (int64_t)num_blocks * block_size;
  if (act_dtype == PA_F16)
    reshape_and_cache_i8_kernel<__half><<<(unsigned)blocks, threads, 0, stream>>>(
        layer_base, L, nslots, k, key_stride * 2, v, value_stride * 2, slot_mapping, n, dev_err);
  else if (act_dtype == PA_BF16)
    reshape_and_cache_i8_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, stream>>>(
        layer_base, L, nslots, k, key_stride * 2, v, value_stride * 2, slot_mapping, n, dev_err);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// grid = (pieces of a block, pairs, layers); each thread moves 4 x 16 bytes per
// round with all four loads issued before the stores.
__global__ void __launch_bounds__(256) block_copy_kernel(uint8_t* __restrict__ dst, int64_t dst_ls,
                                                         const uint8_t* __restrict__ src, int64_t src_ls,
                                                         int64_t block_bytes,
                                                         const __grid_constant__ PairList pairs) {
  const int pair = blockIdx.y;
  const int64_t layer = blockIdx.z;
  const uint4* s = reinterpret_cast<const uint4*>(src + layer * src_ls + pairs.src[pair] * block_bytes);
  uint4* d = reinterpret_cast<uint4*>(dst + layer * dst_ls + pairs.dst[pair] * block_bytes);
  const int64_t n16 = block_bytes / 16;
  const int64_t step = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x * 4 + threadIdx.x; i < n16; i += step) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * blockDim.x < n16) v[u] = s[i + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * blockDim.x < n16) d[i + u * blockDim.x] = v[u];
  }
}

cudaError_t launch_block_copy(uint8_t* dst, int64_t dst_layer_stride, const uint8_t* src,
                              int64_t src_layer_stride, int64_t block_bytes, int32_t layers,
                              const PairList& pairs, int32_t n, cudaStream_t stream) {
  const int threads = 256;
  const int64_t per_cta = threads * 4 * 16;
  const unsigned gx = (unsigned)((block_bytes + per_cta - 1) / per_cta);
  dim3 grid(gx, (unsigned)n, (unsigned)layers);
  block_copy_kernel<<<grid, threads, 0, stream>>>(dst, dst_layer_stride, src, src_layer_stride,
                                                  block_bytes, pairs);
  return cudaGetLastError();
}

}  // namespace pkv
