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
// names a host-side stand-in), so the device address is looked up with
// cudaGetSymbolAddress, with the device current, and cached.  The cache is keyed
// by the CUDA context (its process-unique id), not only by the device: after
// cudaDeviceReset the device gets a new primary context, the library's module
// is loaded again and the array may sit at another address, so the first call
// in the new context looks it up afresh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pagedkv.h"

namespace pkv {
void set_last_error(const char* msg);
pa_status check_decode_args(const void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                            const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                            int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                            int32_t ring_blocks, int32_t partition_size, size_t* need);
}

namespace {

static_assert(PA_STATIC_WORKSPACE_BYTES % 256 == 0, "static workspace size must keep 256-byte alignment");

// The shared workspace: one per device that loads this library.
__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
struct Cached {
  unsigned long long ctx_id;   // context the address belongs to (0: none yet)
  void* addr;
};
Cached g_cache[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the current context, through the driver's entry points (the runtime is
// linked statically; the library does not link the driver library itself).
cudaError_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_current || !get_id) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult r0, r1;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &r0);
    if (e == cudaSuccess) e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &r1);
    if (e != cudaSuccess) return e;
    if (r0 != cudaDriverEntryPointSuccess || r1 != cudaDriverEntryPointSuccess || !f0 || !f1)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
    get_id = reinterpret_cast<CtxGetIdFn>(f1);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}

// Device address of g_static_workspace in the current context (looked up once
// per context).  With no context current yet, the lookup itself makes the
// device's primary context current, and the id is read after it.
cudaError_t static_workspace_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  unsigned long long id = 0;
  if (current_context_id(&id) == cudaSuccess && g_cache[dev].ctx_id == id && g_cache[dev].addr) {
    *out = g_cache[dev].addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e != cudaSuccess) return e;
  e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  g_cache[dev] = Cached{id, p};
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_static_workspace(void* out, const void* q, int64_t q_seq_stride,
                                                const void* kv_cache, const pa_cache_desc* desc, int32_t layer,
                                                const int32_t* block_tables, int32_t block_table_stride,
                                                const int32_t* context_lens, int32_t num_seqs,
                                                int32_t num_q_heads, int32_t max_context_len, float scale,
                                                int32_t partition_size, uint32_t* dev_err, void* stream) {
  // every argument check of pa_decode first, so a bad argument is reported as
  // such and not as a workspace that is too small
  size_t need = 0;
  const pa_status st = pkv::check_decode_args(out, q, q_seq_stride, kv_cache, desc, layer, block_tables,
                                              block_table_stride, context_lens, num_seqs, num_q_heads,
                                              max_context_len, scale, 0, 0, partition_size, &need);
  if (st != PA_OK) return st;
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
      pkv::set_last_error("pa_decode_static_workspace: looking up the static workspace's device address failed");
      return PA_ERR_CUDA;
    }
  }
  return pa_decode(out, q, q_seq_stride, kv_cache, desc, layer, block_tables, block_table_stride, context_lens,
                   num_seqs, num_q_heads, max_context_len, scale, partition_size, ws,
                   need > 0 ? (size_t)PA_STATIC_WORKSPACE_BYTES : 0, dev_err, stream);
}
