// decode_static_workspace.cu -- pa_decode for callers that cannot allocate.
//
// pa_decode needs a caller-provided workspace whenever a context spans more
// than one partition.  Some callers have no way to provide one: a plugin
// running inside another framework whose allocator owns all device memory, a
// serving loop that forbids device allocation once it is running, or a foreign
// language binding that cannot keep a device buffer alive between calls.  For
// them this entry point uses a workspace that the library itself carries: a
// fixed-size array in the library's own device memory, created when the
// library's GPU code is loaded on a device and held until the process exits.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <mutex>

#include "pagedkv.h"

#include <cuda_runtime.h>

namespace pkv {
void set_last_error(const char* msg);
}

namespace {

static_assert(PA_STATIC_WORKSPACE_BYTES % 256 == 0, "static workspace size must keep 256-byte alignment");

// The shared workspace: one per device that loads this library.
__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (looked up once).
cudaError_t static_workspace_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(void* out, const void* q, int64_t q_seq_stride,
                                                const void* kv_cache, const pa_cache_desc* desc, int32_t layer,
                                                const int32_t* block_tables, int32_t block_table_stride,
                                                const int32_t* context_lens, int32_t num_seqs,
                                                int32_t num_q_heads, int32_t max_context_len, float scale,
                                                int32_t partition_size, uint32_t* dev_err, void* stream) {
  const size_t need = pa_decode_workspace_bytes(desc, num_seqs, num_q_heads, max_context_len, partition_size);
  if (need > (size_t)PA_STATIC_WORKSPACE_BYTES) {
    // Same status as pa_decode with a too-small workspace; nothing is launched.
    pkv::set_last_error(
        "pa_decode_static_workspace: these shapes need more workspace than the library's fixed "
        "PA_STATIC_WORKSPACE_BYTES; use a larger partition_size or pa_decode with your own workspace");
    return PA_ERR_WORKSPACE_TOO_SMALL;
  }
  void* ws = nullptr;
  if (need > 0) {
    const cudaError_t e = static_workspace_address(&ws);
    if (e != cudaSuccess) {
      pkv::set_last_error("pa_decode_static_workspace: cudaGetSymbolAddress of the static workspace failed");
      return PA_ERR_CUDA;
    }
  }
  return pa_decode(out, q, q_seq_stride, kv_cache, desc, layer, block_tables, block_table_stride, context_lens,
                   num_seqs, num_q_heads, max_context_len, scale, partition_size, ws,
                   need > 0 ? (size_t)PA_STATIC_WORKSPACE_BYTES : 0, dev_err, stream);
}
