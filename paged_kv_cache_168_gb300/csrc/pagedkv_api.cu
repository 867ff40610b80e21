// pagedkv_api.cu -- the C ABI: argument validation on the host, then kernel
// dispatch on the caller's stream.  No memory is allocated and no state is kept
// between calls (the per-thread error message aside).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "pagedkv.h"

namespace {

thread_local char g_msg[512] = "";

pa_status fail(pa_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
pa_status fail(pa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Default partition sizes for the tensor-core kernels: the shortest, the longest
// for contexts up to kLongContext tokens, the longest beyond, and the work items
// (sequence, kv head, partition) wanted before a longer partition is taken --
// kItemsPerSm per SM of the current device (912 on a 152-SM GB300), below which
// the persistent kernels' last wave leaves SMs idle (a sweep of 512..8192 tokens
// on the 7B, 8B, 70B and beam decode shapes, 16- and 8-bit).  The CUDA-core
// kernel, one CTA per item, keeps 512 (1024 past kLongContext): longer
// partitions leave it too few CTAs.
constexpr int kMinPartition = 512;
constexpr int kMaxPartition = 4096;
constexpr int kMaxLongPartition = 8192;
constexpr int kLongContext = 32768;
constexpr int64_t kItemsPerSm = 6;
constexpr int kDefaultSms = 152;   // GB300; used where no device can be queried (host-only callers)

// SMs of the current device (looked up once per device), or kDefaultSms when no
// device is present.  The persistent decode kernels launch one CTA per SM, so
// their default partition size follows this count.
int device_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    (void)cudaGetLastError();
    return kDefaultSms;
  }
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    (void)cudaGetLastError();
    return kDefaultSms;
  }
  if (dev < 64) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Kernel choice: the tensor-core kernel serves head_size 128 (group sizes 1-16,
// up to pkv::kTcMaxSeqs sequences); the CUDA-core kernel serves the rest.  The
// environment variable PAGEDKV_DECODE_KERNEL=simt selects the CUDA-core kernel
// wherever it applies (used to test both kernels on the same inputs).
bool use_tensor_cores(int head_size, int block_size, int group, int num_seqs) {
  // the tensor-core operands need whole 8-token swizzle atoms: block_size >= 8
  if (head_size != 128 || block_size < 8 || num_seqs > pkv::kTcMaxSeqs) return false;
  if (group > 8) return true;
  const char* env = getenv("PAGEDKV_DECODE_KERNEL");
  return !(env && strcmp(env, "simt") == 0);
}

bool is_i8(const pa_cache_desc* d) { return d->dtype == PA_INT8_F16 || d->dtype == PA_INT8_BF16; }

// Default partition of the persistent tensor-core kernels for `units` long
// pieces of work per kv head (sequences, or shared prefixes) of up to
// max_context_len tokens: the longest of 4096..512 (8192 first past
// kLongContext) that still gives items_per_sm_x2 / 2 items per SM (six).
int32_t persistent_partition(const pa_cache_desc* desc, int64_t units, int32_t max_context_len,
                             int64_t items_per_sm_x2 = 2 * kItemsPerSm) {
  // Each partition writes (D + 2) floats per query head and the merge reads them
  // back, so longer partitions cost less -- until one item is so long that the
  // kernel's tail runs on a few SMs.  Long contexts have the per-SM work to
  // hide an 8192-token item; with contexts of at most 32768 tokens an item
  // stays at most 4096 tokens long.
  const int64_t pairs = (units > 0 ? units : 0) * (desc->num_kv_heads > 0 ? desc->num_kv_heads : 0);
  const int64_t ctx = max_context_len > 0 ? max_context_len : 0;
  for (int P = max_context_len > kLongContext ? kMaxLongPartition : kMaxPartition; P > kMinPartition; P /= 2)
    if (2 * pairs * ((ctx + P - 1) / P) >= items_per_sm_x2 * device_sm_count()) return P;
  return kMinPartition;
}

// Test hook for the timeout path: PAGEDKV_WAIT_POLLS=n (n >= 1) makes the
// ordinary waits of the CUDA-core decode kernels give up after n
// non-suspending polls instead of the default bound, so a test can make them
// run out and check PA_DEVERR_TIMEOUT and the abandoned items' zeroed rows.
// Unset (or invalid): 0, the default.
uint32_t test_wait_polls() {
  const char* env = getenv("PAGEDKV_WAIT_POLLS");
  if (!env || !*env) return 0;
  char* end = nullptr;
  const unsigned long v = strtoul(env, &end, 10);
  return (end && *end == 0 && v > 0 && v < (1ul << 24)) ? (uint32_t)v : 0;
}

// Whether these shapes get a tensor-core kernel by default (the environment
// switch aside): 16-bit caches as use_tensor_cores; 8-bit caches at head_size
// 128 up to pkv::kTcI8MaxSeqs sequences, any block size.
bool tc_by_default(const pa_cache_desc* d, int num_seqs) {
  if (d->head_size != 128) return false;
  return is_i8(d) ? num_seqs <= pkv::kTcI8MaxSeqs : d->block_size >= 8 && num_seqs <= pkv::kTcMaxSeqs;
}

// 16-bit type of q, key, value and out (and of a 16-bit cache).
int act_dtype(const pa_cache_desc* d) { return d->dtype == PA_INT8_BF16 || d->dtype == PA_BF16 ? PA_BF16 : PA_F16; }

int64_t block_bytes(const pa_cache_desc* d) {
  if (is_i8(d)) return (int64_t)d->num_kv_heads * pkv::I8Layout{d->block_size, d->num_kv_heads}.chunk_bytes();
  return (int64_t)d->num_kv_heads * 2 * d->block_size * d->head_size * 2;
}

pa_status check_desc(const pa_cache_desc* d) {
  if (!d) return fail(PA_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->num_layers <= 0)
    return fail(PA_ERR_INVALID_ARG, "num_blocks, num_kv_heads and num_layers must be > 0");
  if (d->dtype < PA_F16 || d->dtype > PA_INT8_BF16) return fail(PA_ERR_INVALID_ARG, "dtype %d", d->dtype);
  if (d->head_size != 64 && d->head_size != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_size %d (supported: 64, 128)", d->head_size);
  if (is_i8(d) && d->head_size != 128)
    return fail(PA_ERR_UNSUPPORTED, "8-bit cache with head_size %d (supported: 128)", d->head_size);
  if (d->block_size != 1 && d->block_size != 2 && d->block_size != 4 && d->block_size != 8 &&
      d->block_size != 16 && d->block_size != 32)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 1, 2, 4, 8, 16, 32)", d->block_size);
  const int64_t lb = block_bytes(d) * d->num_blocks;
  if (d->layer_stride_bytes != 0 && (d->layer_stride_bytes < lb || d->layer_stride_bytes % 16 != 0))
    return fail(PA_ERR_INVALID_ARG, "layer_stride_bytes %lld must be 0 or >= %lld and a multiple of 16",
                (long long)d->layer_stride_bytes, (long long)lb);
  return PA_OK;
}

int64_t layer_stride(const pa_cache_desc* d) {
  return d->layer_stride_bytes ? d->layer_stride_bytes : block_bytes(d) * d->num_blocks;
}

// Validate a host list of (src, dst) pairs.  Destinations must be distinct; when
// `same_pool`, no destination may also be a source (all pairs act at once).
pa_status check_pairs(const int64_t* pairs, int32_t n, int32_t src_blocks, int32_t dst_blocks,
                      bool same_pool) {
  if (n < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs %d < 0", n);
  if (n > 0 && !pairs) return fail(PA_ERR_INVALID_ARG, "pairs is NULL");
  std::vector<int64_t> dst(n), src(n);
  for (int32_t i = 0; i < n; ++i) {
    src[i] = pairs[2 * i];
    dst[i] = pairs[2 * i + 1];
    if (src[i] < 0 || src[i] >= src_blocks)
      return fail(PA_ERR_INVALID_ARG, "pair %d: src block %lld out of range [0, %d)", i, (long long)src[i],
                  src_blocks);
    if (dst[i] < 0 || dst[i] >= dst_blocks)
      return fail(PA_ERR_INVALID_ARG, "pair %d: dst block %lld out of range [0, %d)", i, (long long)dst[i],
                  dst_blocks);
  }
  std::sort(dst.begin(), dst.end());
  for (int32_t i = 1; i < n; ++i)
    if (dst[i] == dst[i - 1]) return fail(PA_ERR_INVALID_ARG, "dst block %lld repeated", (long long)dst[i]);
  if (same_pool) {
    for (int32_t i = 0; i < n; ++i)
      if (std::binary_search(dst.begin(), dst.end(), src[i]))
        return fail(PA_ERR_INVALID_ARG, "block %lld is both a src and a dst", (long long)src[i]);
  }
  return PA_OK;
}

pa_status run_pairs(uint8_t* dst, int64_t dst_ls, const uint8_t* src, int64_t src_ls, int64_t bb,
                    int32_t layers, const int64_t* pairs, int32_t n, cudaStream_t stream) {
  pkv::PairList list;
  for (int32_t i0 = 0; i0 < n; i0 += pkv::kMaxPairsPerLaunch) {
    const int32_t cnt = std::min<int32_t>(pkv::kMaxPairsPerLaunch, n - i0);
    for (int32_t i = 0; i < cnt; ++i) {
      list.src[i] = pairs[2 * (i0 + i)];
      list.dst[i] = pairs[2 * (i0 + i) + 1];
    }
    cudaError_t e = pkv::launch_block_copy(dst, dst_ls, src, src_ls, bb, layers, list, cnt, stream);
    if (e != cudaSuccess) return cuda_fail(e, "block copy launch");
  }
  return PA_OK;
}

}  // namespace

namespace pkv {
// Record a message for pa_last_error_message() (used by entry points defined in
// other translation units).
void set_last_error(const char* msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

// Every host-side check of pa_decode_window's arguments except the workspace
// (shared with pa_decode_static_workspace, whose workspace is the library's
// own): PA_OK with *need = the workspace bytes these shapes use, or the first
// failing check's status (message recorded).  num_seqs == 0 passes with
// *need = 0 (nothing to launch).
pa_status check_decode_args(const void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                            const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                            int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                            int32_t ring_blocks, int32_t partition_size, size_t* need) {
  *need = 0;
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (layer < 0 || layer >= desc->num_layers) return fail(PA_ERR_INVALID_ARG, "layer %d", layer);
  if (num_seqs < 0 || num_seqs > 65535) return fail(PA_ERR_INVALID_ARG, "num_seqs %d not in [0, 65535]", num_seqs);
  if (num_seqs == 0) return PA_OK;
  if (num_q_heads <= 0 || num_q_heads % desc->num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                num_q_heads, desc->num_kv_heads);
  const int group = num_q_heads / desc->num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8 &&
      !(group == 16 && desc->head_size == 128 && desc->block_size >= 8))
    return fail(PA_ERR_UNSUPPORTED,
                "query heads per kv head %d (supported: 1, 2, 4, 8; 16 at head_size 128 with block_size >= 8)", group);
  if (desc->num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads > 65535");
  if (is_i8(desc) && group > 8)
    return fail(PA_ERR_UNSUPPORTED, "8-bit cache with %d query heads per kv head (supported: 1, 2, 4, 8)", group);
  if (!out || !q || !kv_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "out, q, kv_cache, block_tables and context_lens must be non-NULL");
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q and kv_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3) || (reinterpret_cast<uintptr_t>(context_lens) & 3))
    return fail(PA_ERR_INVALID_ARG, "block_tables and context_lens must be 4-byte aligned");
  if (q_seq_stride < (int64_t)num_q_heads * desc->head_size || q_seq_stride % 8)
    return fail(PA_ERR_INVALID_ARG, "q_seq_stride must be >= num_q_heads*head_size and a multiple of 8");
  if (block_table_stride <= 0) return fail(PA_ERR_INVALID_ARG, "block_table_stride %d", block_table_stride);
  if (max_context_len <= 0) return fail(PA_ERR_INVALID_ARG, "max_context_len %d", max_context_len);
  if (window < 0) return fail(PA_ERR_INVALID_ARG, "window %d < 0", window);
  if (ring_blocks < 0 || ring_blocks > block_table_stride)
    return fail(PA_ERR_INVALID_ARG, "ring_blocks %d not in [0, block_table_stride %d]", ring_blocks,
                block_table_stride);
  const int32_t span = pa_decode_window_span(max_context_len, desc->block_size, window, ring_blocks);
  const int32_t P = pa_decode_partition_size(desc, num_seqs, span, partition_size);
  if (P % 128 || P < 128 || P > 8192)
    return fail(PA_ERR_INVALID_ARG, "partition_size %d must be a multiple of 128 in [128, 8192]", P);
  if (!(scale > 0.f) || scale != scale) return fail(PA_ERR_INVALID_ARG, "scale must be a positive number");
  *need = pa_decode_workspace_bytes(desc, num_seqs, num_q_heads, span, P);
  return PA_OK;
}
}  // namespace pkv

extern "C" {

size_t pa_cache_bytes(const pa_cache_desc* desc) {
  if (check_desc(desc) != PA_OK) return 0;
  return (size_t)(block_bytes(desc) * desc->num_blocks);
}

int64_t pa_cache_element_offset(const pa_cache_desc* desc, int64_t block, int32_t kv_head, int32_t part,
                                int32_t slot, int32_t dim) {
  if (check_desc(desc) != PA_OK) return -1;
  if (block < 0 || block >= desc->num_blocks || kv_head < 0 || kv_head >= desc->num_kv_heads || part < 0 ||
      part > 1 || slot < 0 || slot >= desc->block_size || dim < 0 || dim >= desc->head_size)
    return -1;
  if (is_i8(desc)) return pkv::I8Layout{desc->block_size, desc->num_kv_heads}.code(block, kv_head, part, slot, dim);
  pkv::Layout L{desc->block_size, desc->head_size, desc->num_kv_heads};
  return L.offset(block, kv_head, part, slot, dim);
}

int64_t pa_cache_scale_offset(const pa_cache_desc* desc, int64_t block, int32_t kv_head, int32_t part,
                              int32_t slot) {
  if (check_desc(desc) != PA_OK || !is_i8(desc)) return -1;
  if (block < 0 || block >= desc->num_blocks || kv_head < 0 || kv_head >= desc->num_kv_heads || part < 0 ||
      part > 1 || slot < 0 || slot >= desc->block_size)
    return -1;
  return pkv::I8Layout{desc->block_size, desc->num_kv_heads}.scale(block, kv_head, part, slot);
}

pa_status pa_reshape_and_cache(void* kv_cache, const pa_cache_desc* desc, int32_t layer, const void* key,
                               int64_t key_token_stride, const void* value, int64_t value_token_stride,
                               const int64_t* slot_mapping, int32_t num_tokens, uint32_t* dev_err,
                               void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (layer < 0 || layer >= desc->num_layers) return fail(PA_ERR_INVALID_ARG, "layer %d", layer);
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return PA_OK;
  if (!kv_cache || !key || !value || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "kv_cache, key, value and slot_mapping must be non-NULL");
  if (!aligned16(kv_cache) || !aligned16(key) || !aligned16(value))
    return fail(PA_ERR_INVALID_ARG, "kv_cache, key and value must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7) != 0)
    return fail(PA_ERR_INVALID_ARG, "slot_mapping must be 8-byte aligned");
  const int64_t row = (int64_t)desc->num_kv_heads * desc->head_size;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 || value_token_stride % 8)
    return fail(PA_ERR_INVALID_ARG, "token strides must be >= num_kv_heads*head_size and multiples of 8");
  uint8_t* base = static_cast<uint8_t*>(kv_cache) + layer * layer_stride(desc);
  if (is_i8(desc)) {
    cudaError_t e = pkv::launch_reshape_and_cache_i8(base, desc->num_blocks, desc->block_size, desc->num_kv_heads,
                                                     act_dtype(desc), key, key_token_stride, value,
                                                     value_token_stride, slot_mapping, num_tokens, dev_err,
                                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "reshape_and_cache launch");
  }
  cudaError_t e = pkv::launch_reshape_and_cache(base, desc->num_blocks, desc->block_size, desc->num_kv_heads,
                                                desc->head_size, key, key_token_stride, value,
                                                value_token_stride, slot_mapping, num_tokens, dev_err,
                                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e, "reshape_and_cache launch");
}

int32_t pa_decode_partition_size(const pa_cache_desc* desc, int32_t num_seqs, int32_t max_context_len,
                                 int32_t partition_size) {
  if (partition_size > 0) return partition_size;
  if (!desc || !tc_by_default(desc, num_seqs))
    return desc && max_context_len > kLongContext ? 2 * kMinPartition : kMinPartition;
  // Each partition writes (D + 2) floats per query head and the merge reads them
  // back, so longer partitions cost less -- until one item is so long that the
  // kernel's tail runs on a few SMs.  Long contexts have the per-SM work to
  // hide an 8192-token item; with contexts of at most 32768 tokens an item
  // stays at most 4096 tokens long.
  return persistent_partition(desc, num_seqs, max_context_len);
}

size_t pa_decode_workspace_bytes(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t max_context_len, int32_t partition_size) {
  if (!desc) return 0;
  const int64_t P = pa_decode_partition_size(desc, num_seqs, max_context_len, partition_size);
  const int64_t head_size = desc->head_size;
  if (num_seqs <= 0 || num_q_heads <= 0 || head_size <= 0 || max_context_len <= 0 || P <= 0) return 0;
  const int64_t parts = (max_context_len + P - 1) / P;
  if (parts <= 1) return 0;
  // saturate instead of wrapping: a wrapped (small) size would let a too-small
  // workspace pass pa_decode's check
  const unsigned __int128 need = (unsigned __int128)num_seqs * (unsigned __int128)num_q_heads *
                                 (unsigned __int128)parts * (unsigned __int128)((head_size + 2) * 4);
  return need > (unsigned __int128)(SIZE_MAX / 2) ? SIZE_MAX : (size_t)need;
}

int32_t pa_decode_window_span(int32_t max_context_len, int32_t block_size, int32_t window, int32_t ring_blocks) {
  int64_t span = max_context_len;
  if (window > 0 && (int64_t)window + block_size - 1 < span) span = (int64_t)window + block_size - 1;
  if (ring_blocks > 0 && (int64_t)ring_blocks * block_size < span) span = (int64_t)ring_blocks * block_size;
  return (int32_t)span;
}

pa_status pa_decode_window(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                           const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                           int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                           int32_t ring_blocks, int32_t partition_size, void* workspace, size_t workspace_bytes,
                           uint32_t* dev_err, void* stream) {
  size_t need = 0;
  pa_status st = pkv::check_decode_args(out, q, q_seq_stride, kv_cache, desc, layer, block_tables,
                                        block_table_stride, context_lens, num_seqs, num_q_heads, max_context_len,
                                        scale, window, ring_blocks, partition_size, &need);
  if (st != PA_OK || num_seqs == 0) return st;
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (need && (!workspace || !aligned16(workspace)))
    return fail(PA_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
  const int group = num_q_heads / desc->num_kv_heads;
  const int32_t span = pa_decode_window_span(max_context_len, desc->block_size, window, ring_blocks);
  const int32_t P = pa_decode_partition_size(desc, num_seqs, span, partition_size);

  pkv::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.q_seq_stride = q_seq_stride;
  p.cache = static_cast<const uint8_t*>(kv_cache) + layer * layer_stride(desc);
  p.num_blocks = desc->num_blocks;
  p.block_size = desc->block_size;
  p.num_kv_heads = desc->num_kv_heads;
  p.block_tables = block_tables;
  p.bt_stride = block_table_stride;
  p.context_lens = context_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.max_context_len = max_context_len;
  p.partition_size = P;
  p.max_parts = (span + P - 1) / P;
  p.window = window;
  p.ring_blocks = ring_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_polls = test_wait_polls();
  const int64_t parts = p.max_parts;
  p.ws_o = need ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = need ? static_cast<float*>(workspace) + (int64_t)num_seqs * num_q_heads * parts * desc->head_size
                 : nullptr;
  p.dev_err = dev_err;
  cudaError_t e;
  if (is_i8(desc)) {
    // tensor cores for every group (block sizes below 8 included: the converter
    // warps repack any block size into whole 8-token atoms); the CUDA-core
    // kernel serves more than kTcI8MaxSeqs sequences
    if (use_tensor_cores(desc->head_size, 8, group, num_seqs) && num_seqs <= pkv::kTcI8MaxSeqs) {
      int dev = 0, sms = 0;
      e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e == cudaSuccess)
        e = pkv::launch_decode_tc_i8(p, act_dtype(desc), group, sms, static_cast<cudaStream_t>(stream));
    } else {
      e = pkv::launch_decode_i8(p, act_dtype(desc), group, static_cast<cudaStream_t>(stream));
    }
  } else if (use_tensor_cores(desc->head_size, desc->block_size, group, num_seqs)) {
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = pkv::launch_decode_tc(p, desc->dtype, group, sms, static_cast<cudaStream_t>(stream));
  } else {
    e = pkv::launch_decode_simt(p, desc->dtype, desc->head_size, group, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? PA_OK : cuda_fail(e, "decode launch");
}


// Whether the shared-prefix tensor-core kernel serves these shapes (else
// pa_decode_shared_prefix runs pa_decode, which gives the same result).
static bool shared_prefix_kernel_serves(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads) {
  if (!desc || is_i8(desc) || desc->head_size != 128 || desc->block_size < 8 || desc->num_kv_heads <= 0) return false;
  if (num_seqs <= 0 || num_seqs > pkv::kTcSpMaxSeqs || num_q_heads <= 0 || num_q_heads % desc->num_kv_heads) return false;
  const int group = num_q_heads / desc->num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  return use_tensor_cores(desc->head_size, desc->block_size, group, num_seqs);
}

// Whether pa_decode_shared_prefix takes its dedicated kernel: served shapes,
// some groups, and partition counts that fit its 16-bit per-sequence tables.
static bool shared_prefix_path(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads, int32_t num_groups,
                               int32_t max_context_len, int64_t P) {
  return num_groups > 0 && P > 0 && shared_prefix_kernel_serves(desc, num_seqs, num_q_heads) &&
         ((int64_t)max_context_len + P - 1) / P + 1 <= 32767;
}

int32_t pa_decode_shared_prefix_partition_size(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_groups, int32_t max_context_len, int32_t partition_size) {
  if (partition_size > 0) return partition_size;
  if (!shared_prefix_kernel_serves(desc, num_seqs, num_q_heads) || num_groups <= 0)
    return pa_decode_partition_size(desc, num_seqs, max_context_len, 0);
  // the groups' prefixes are the long items; every sequence adds a (short)
  // tail item of its own, so 1.5 prefix items per SM keep the SMs busy to
  // the end while items stay long (fewer partial results to merge)
  return persistent_partition(desc, num_groups, max_context_len, 3);
}

size_t pa_decode_shared_prefix_workspace_bytes(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_groups, int32_t max_context_len, int32_t partition_size) {
  if (!desc) return 0;
  const int64_t P =
      pa_decode_shared_prefix_partition_size(desc, num_seqs, num_q_heads, num_groups, max_context_len, partition_size);
  if (!shared_prefix_path(desc, num_seqs, num_q_heads, num_groups, max_context_len, P))
    return pa_decode_workspace_bytes(desc, num_seqs, num_q_heads, max_context_len, (int32_t)P);
  if (max_context_len <= 0) return 0;
  // a sequence's prefix and its tail split into at most ceil(ctx / P) + 1
  // partitions; then three ints per sequence for the merge
  const int64_t parts = (max_context_len + P - 1) / P + 1;
  const int64_t floats = (int64_t)num_seqs * num_q_heads * parts * (desc->head_size + 2);
  return (size_t)((floats * 4 + 3 * (int64_t)num_seqs * 4 + 15) / 16 * 16);
}

pa_status pa_decode_shared_prefix(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                                  const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                                  int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                  const int32_t* group_start, const int32_t* prefix_lens, int32_t num_groups,
                                  int32_t partition_size, void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                  void* stream) {
  size_t need = 0;
  const int32_t P = desc ? pa_decode_shared_prefix_partition_size(desc, num_seqs, num_q_heads, num_groups,
                                                                   max_context_len, partition_size)
                         : partition_size;
  pa_status st = pkv::check_decode_args(out, q, q_seq_stride, kv_cache, desc, layer, block_tables,
                                        block_table_stride, context_lens, num_seqs, num_q_heads, max_context_len,
                                        scale, 0, 0, P, &need);
  if (st != PA_OK || num_seqs == 0) return st;
  if (num_groups < 0 || num_groups > num_seqs)
    return fail(PA_ERR_INVALID_ARG, "num_groups %d not in [0, num_seqs %d]", num_groups, num_seqs);
  if (num_groups > 0 && (!group_start || !prefix_lens))
    return fail(PA_ERR_INVALID_ARG, "group_start and prefix_lens must be non-NULL when num_groups > 0");
  if ((reinterpret_cast<uintptr_t>(group_start) & 3) || (reinterpret_cast<uintptr_t>(prefix_lens) & 3))
    return fail(PA_ERR_INVALID_ARG, "group_start and prefix_lens must be 4-byte aligned");
  if (!shared_prefix_path(desc, num_seqs, num_q_heads, num_groups, max_context_len, P))
    return pa_decode_window(out, q, q_seq_stride, kv_cache, desc, layer, block_tables, block_table_stride,
                            context_lens, num_seqs, num_q_heads, max_context_len, scale, 0, 0, P, workspace,
                            workspace_bytes, dev_err, stream);
  need = pa_decode_shared_prefix_workspace_bytes(desc, num_seqs, num_q_heads, num_groups, max_context_len, P);
  if (workspace_bytes < need)
    return fail(PA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (!workspace || !aligned16(workspace))
    return fail(PA_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");

  pkv::DecodeParams p{};
  p.out = out;
  p.q = q;
  p.q_seq_stride = q_seq_stride;
  p.cache = static_cast<const uint8_t*>(kv_cache) + layer * layer_stride(desc);
  p.num_blocks = desc->num_blocks;
  p.block_size = desc->block_size;
  p.num_kv_heads = desc->num_kv_heads;
  p.block_tables = block_tables;
  p.bt_stride = block_table_stride;
  p.context_lens = context_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.max_context_len = max_context_len;
  p.partition_size = P;
  p.max_parts = (max_context_len + P - 1) / P + 1;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_polls = test_wait_polls();
  const int64_t rows = (int64_t)num_seqs * num_q_heads * p.max_parts;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = p.ws_o + rows * desc->head_size;
  p.ws_seq = reinterpret_cast<int32_t*>(p.ws_ml + rows * 2);
  p.group_start = group_start;
  p.prefix_lens = prefix_lens;
  p.num_groups = num_groups;
  p.dev_err = dev_err;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = pkv::launch_decode_tc_sp(p, desc->dtype, num_q_heads / desc->num_kv_heads, sms,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e, "shared-prefix decode launch");
}

pa_status pa_decode(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                    const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                    int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                    int32_t num_q_heads, int32_t max_context_len, float scale, int32_t partition_size,
                    void* workspace, size_t workspace_bytes, uint32_t* dev_err, void* stream) {
  return pa_decode_window(out, q, q_seq_stride, kv_cache, desc, layer, block_tables, block_table_stride,
                          context_lens, num_seqs, num_q_heads, max_context_len, scale, 0, 0, partition_size,
                          workspace, workspace_bytes, dev_err, stream);
}

pa_status pa_prefill(void* out, const void* q, int64_t q_token_stride, const void* kv_cache,
                     const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                     int32_t block_table_stride, const int32_t* context_lens, const int32_t* query_start_loc,
                     int32_t num_seqs, int32_t num_q_heads, int32_t max_query_len, float scale, uint32_t* dev_err,
                     void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (is_i8(desc)) return fail(PA_ERR_UNSUPPORTED, "prefill over an 8-bit cache");
  if (desc->block_size < 8)
    return fail(PA_ERR_UNSUPPORTED, "prefill with block_size %d (supported: 8, 16, 32)", desc->block_size);
  if (layer < 0 || layer >= desc->num_layers) return fail(PA_ERR_INVALID_ARG, "layer %d", layer);
  if (num_seqs < 0 || num_seqs > 65535) return fail(PA_ERR_INVALID_ARG, "num_seqs %d not in [0, 65535]", num_seqs);
  if (num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (max_query_len < 0) return fail(PA_ERR_INVALID_ARG, "max_query_len %d < 0", max_query_len);
  if (num_q_heads <= 0 || num_q_heads % desc->num_kv_heads)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d",
                num_q_heads, desc->num_kv_heads);
  const int group = num_q_heads / desc->num_kv_heads;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
    return fail(PA_ERR_UNSUPPORTED, "query heads per kv head %d (supported: 1, 2, 4, 8, 16)", group);
  if (desc->num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "num_kv_heads > 65535");
  if (!out || !q || !kv_cache || !block_tables || !context_lens || !query_start_loc)
    return fail(PA_ERR_INVALID_ARG,
                "out, q, kv_cache, block_tables, context_lens and query_start_loc must be non-NULL");
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache))
    return fail(PA_ERR_INVALID_ARG, "out, q and kv_cache must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_tables) & 3) || (reinterpret_cast<uintptr_t>(context_lens) & 3) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3))
    return fail(PA_ERR_INVALID_ARG, "block_tables, context_lens and query_start_loc must be 4-byte aligned");
  if (q_token_stride < (int64_t)num_q_heads * desc->head_size || q_token_stride % 8)
    return fail(PA_ERR_INVALID_ARG, "q_token_stride must be >= num_q_heads*head_size and a multiple of 8");
  if (block_table_stride <= 0) return fail(PA_ERR_INVALID_ARG, "block_table_stride %d", block_table_stride);
  if (!(scale > 0.f) || scale != scale) return fail(PA_ERR_INVALID_ARG, "scale must be a positive number");
  const int rows_per_tile = 128 / group;
  if ((int64_t)(max_query_len + rows_per_tile - 1) / rows_per_tile > 0x7fffffff)
    return fail(PA_ERR_INVALID_ARG, "max_query_len too large");

  pkv::PrefillParams p{};
  p.out = out;
  p.q = q;
  p.q_token_stride = q_token_stride;
  p.cache = static_cast<const uint8_t*>(kv_cache) + layer * layer_stride(desc);
  p.num_blocks = desc->num_blocks;
  p.block_size = desc->block_size;
  p.num_kv_heads = desc->num_kv_heads;
  p.block_tables = block_tables;
  p.bt_stride = block_table_stride;
  p.context_lens = context_lens;
  p.query_start_loc = query_start_loc;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.max_query_len = max_query_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.dev_err = dev_err;
  cudaError_t e = pkv::launch_prefill_tc(p, desc->dtype, desc->head_size, group, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e, "prefill launch");
}

pa_status pa_copy_blocks(void* kv_cache, const pa_cache_desc* desc, const int64_t* pairs, int32_t num_pairs,
                         void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  st = check_pairs(pairs, num_pairs, desc->num_blocks, desc->num_blocks, true);
  if (st != PA_OK) return st;
  if (num_pairs == 0) return PA_OK;
  if (!kv_cache || !aligned16(kv_cache)) return fail(PA_ERR_INVALID_ARG, "kv_cache NULL or not 16-byte aligned");
  uint8_t* base = static_cast<uint8_t*>(kv_cache);
  return run_pairs(base, layer_stride(desc), base, layer_stride(desc), block_bytes(desc), desc->num_layers, pairs,
                   num_pairs, static_cast<cudaStream_t>(stream));
}

pa_status pa_swap_blocks(void* dst_pool, const pa_cache_desc* dst_desc, const void* src_pool,
                         const pa_cache_desc* src_desc, int32_t direction, const int64_t* pairs,
                         int32_t num_pairs, void* stream) {
  pa_status st = check_desc(dst_desc);
  if (st != PA_OK) return st;
  st = check_desc(src_desc);
  if (st != PA_OK) return st;
  if (dst_desc->block_size != src_desc->block_size || dst_desc->num_kv_heads != src_desc->num_kv_heads ||
      dst_desc->head_size != src_desc->head_size || dst_desc->dtype != src_desc->dtype ||
      dst_desc->num_layers != src_desc->num_layers)
    return fail(PA_ERR_INVALID_ARG, "src and dst pools differ in geometry");
  if (direction != 0 && direction != 1) return fail(PA_ERR_INVALID_ARG, "direction %d (0 = out, 1 = in)", direction);
  st = check_pairs(pairs, num_pairs, src_desc->num_blocks, dst_desc->num_blocks, false);
  if (st != PA_OK) return st;
  if (num_pairs == 0) return PA_OK;
  if (!dst_pool || !src_pool || !aligned16(dst_pool) || !aligned16(src_pool))
    return fail(PA_ERR_INVALID_ARG, "pools must be non-NULL and 16-byte aligned");
  const void* host = direction == 0 ? dst_pool : src_pool;
  const void* devp = direction == 0 ? src_pool : dst_pool;
  cudaPointerAttributes ah, ad;
  cudaError_t e = cudaPointerGetAttributes(&ah, host);
  if (e != cudaSuccess) return cuda_fail(e, "host pool attributes");
  if (ah.type != cudaMemoryTypeHost || ah.devicePointer == nullptr)
    return fail(PA_ERR_INVALID_ARG, "the host pool must be page-locked host memory mapped for the device");
  e = cudaPointerGetAttributes(&ad, devp);
  if (e != cudaSuccess) return cuda_fail(e, "device pool attributes");
  if (ad.type != cudaMemoryTypeDevice) return fail(PA_ERR_INVALID_ARG, "the device pool must be device memory");
  // the host pool is addressed through its device mapping
  const uint8_t* src = static_cast<const uint8_t*>(direction == 0 ? src_pool : ah.devicePointer);
  uint8_t* dst = static_cast<uint8_t*>(direction == 0 ? ah.devicePointer : dst_pool);
  return run_pairs(dst, layer_stride(dst_desc), src, layer_stride(src_desc), block_bytes(src_desc),
                   src_desc->num_layers, pairs, num_pairs, static_cast<cudaStream_t>(stream));
}

pa_status pa_read_device_errors(uint32_t* dev_err, uint32_t* host_bits, int32_t clear, void* stream) {
  if (!dev_err || !host_bits) return fail(PA_ERR_INVALID_ARG, "dev_err and host_bits must be non-NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_bits, dev_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(dev_err, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? PA_OK : cuda_fail(e, "read device errors");
}

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_OUT_OF_BLOCKS: return "out of blocks";
  }
  return "unknown status";
}

const char* pa_last_error_message(void) { return g_msg; }

}  // extern "C"
