// common.cuh -- shared pieces of the sm_103a kernels: cache layout, element
// types, and inline-PTX wrappers for mbarriers and bulk (TMA) copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pagedkv.h"

namespace pkv {

// ------------------------------------------------------------------ layout
// One (block, kv head) chunk = 2 * bs * D elements.  Token slots are grouped by
// R = min(bs, 8); a group stores its K rows then its V rows, each as D/64 atoms
// of R rows x 64 dims; the 16-byte piece c of row r sits at piece (c ^ r).
struct Layout {
  int bs, D, Hkv;
  __host__ __device__ int rows() const { return bs < 8 ? bs : 8; }
  __host__ __device__ int64_t chunk_elems() const { return 2LL * bs * D; }
  // element offset inside a chunk
  __host__ __device__ int64_t in_chunk(int part, int t, int d) const {
    const int R = rows();
    const int g = t / R, r = t % R;
    const int atoms = D / 64;
    return (int64_t)(((g * 2 + part) * atoms + d / 64) * (R * 64)) + r * 64 +
           ((((d & 63) >> 3) ^ r) << 3) + (d & 7);
  }
  __host__ __device__ int64_t offset(int64_t block, int head, int part, int t, int d) const {
    return (block * Hkv + head) * chunk_elems() + in_chunk(part, t, d);
  }
};

// 8-bit cache (head_size 128): chunk = K codes [bs][128] | V codes [bs][128] |
// K scales fp32 [bs] | V scales fp32 [bs], each scale area padded to 16 bytes;
// the 16-byte piece c of the code row of slot t sits at piece (c ^ (t & 7)).
struct I8Layout {
  int bs, Hkv;
  static constexpr int D = 128;
  __host__ __device__ int64_t scale_bytes() const { return ((int64_t)bs * 4 + 15) / 16 * 16; }
  __host__ __device__ int64_t chunk_bytes() const { return 2LL * bs * D + 2 * scale_bytes(); }
  __host__ __device__ int64_t chunk(int64_t block, int head) const { return (block * Hkv + head) * chunk_bytes(); }
  __host__ __device__ int64_t code(int64_t block, int head, int part, int t, int d) const {
    return chunk(block, head) + (int64_t)(part * bs + t) * D + ((((d >> 4) ^ (t & 7)) << 4) | (d & 15));
  }
  __host__ __device__ int64_t scale(int64_t block, int head, int part, int t) const {
    return chunk(block, head) + 2LL * bs * D + part * scale_bytes() + 4LL * t;
  }
};

// ------------------------------------------------------------------ element types
template <typename T> struct Elem;
template <> struct Elem<__half> {
  static __device__ __forceinline__ float2 to_float2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
  static __device__ __forceinline__ __half from_float(float f) { return __float2half_rn(f); }
  static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float2 to_float2(uint32_t u) {
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_float(float f) { return __float2bfloat16_rn(f); }
  static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

// ------------------------------------------------------------------ launch set-up
// Raise kernel Kern's dynamic shared-memory limit once per device (the
// attribute is per function and device).  Doing it once keeps later launches
// free of non-stream runtime calls, so they can be captured into CUDA graphs.
// The size recorded is the largest requested so far.
template <auto Kern>
cudaError_t set_smem_attribute_once(size_t bytes) {
  static std::atomic<size_t> done[64];   // one set per kernel (Kern is a template argument)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (done[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) {
    size_t cur = done[dev].load();
    while (cur < bytes && !done[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

// ------------------------------------------------------------------ error word
__device__ __forceinline__ void report(uint32_t* dev_err, uint32_t bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// ------------------------------------------------------------------ PTX: mbarrier + bulk copy
// Bounded waits: a wait that does not complete within kSpinLimit polls gives up
// and returns false; callers then set PA_DEVERR_TIMEOUT and abandon the item.
constexpr uint32_t kSpinLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// A hint: bring the 128-byte line that holds *ptr into L2; nothing is returned.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Non-blocking test of phase `parity` (try_wait may suspend the thread for a
// while; a loop that polls several barriers in turn must not sleep on one).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// The same, polling with test_wait (never suspends): for a single-lane issuer
// that must react as soon as the phase completes.
__device__ __forceinline__ bool mbar_spin(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return false;
}

// An ordinary wait of a kernel whose launch carries a poll limit: polls == 0
// is mbar_wait (the default limit); otherwise at most `polls` non-suspending
// polls (try_wait may sleep until the phase completes, so only test_wait makes
// a small limit run out for certain).  Waits that drain a CTA's own copies or
// tensor-core operations before it exits never take a caller's limit: they
// always use mbar_wait, so a CTA never leaves work in flight.
__device__ __forceinline__ bool mbar_wait_polls(uint64_t* bar, uint32_t parity, uint32_t polls) {
  if (polls == 0) return mbar_wait(bar, parity);
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_test_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace pkv
