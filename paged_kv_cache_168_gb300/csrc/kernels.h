// kernels.h -- internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kMaxPairsPerLaunch = 1024;

// Block pairs passed by value in kernel parameter space (16 KiB).
struct PairList {
  int64_t src[kMaxPairsPerLaunch];
  int64_t dst[kMaxPairsPerLaunch];
};

struct DecodeParams {
  void* out;                  // [S, Hq, D] q dtype
  const void* q;              // [S, Hq, D] with sequence stride q_seq_stride
  int64_t q_seq_stride;       // elements
  const uint8_t* cache;       // this layer's pool
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  const int32_t* block_tables;
  int32_t bt_stride;
  const int32_t* context_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t max_context_len;
  int32_t partition_size;     // tokens per partition (multiple of 128)
  int32_t max_parts;          // ceil(max_context_len / partition_size)
  float scale_log2;           // scale * log2(e): scores are kept in base-2 units
  float* ws_o;                // [S, Hq, max_parts, D] unnormalised partition outputs
  float* ws_ml;               // [S, Hq, max_parts, 2] (running max in base-2 units, sum)
  uint32_t* dev_err;
  int32_t window;             // > 0: attend only positions >= ctx - window
  int32_t ring_blocks;        // > 0: table rows are rings; logical block j at entry j % ring_blocks
  uint32_t wait_polls;        // 0: default bounded waits; > 0: ordinary waits give up after this many
                              // polls (tests of the timeout path; CUDA-core kernels)
  // shared-prefix decode: group g = sequences group_start[g] .. group_start[g + 1] - 1,
  // whose first prefix_lens[g] tokens are the same physical blocks
  const int32_t* group_start; // [num_groups + 1]
  const int32_t* prefix_lens; // [num_groups]
  int32_t num_groups;
  int32_t* ws_seq;            // workspace [3][num_seqs]: partitions in all, effective prefix,
                              // first member of the sequence's prefix item (for the merge)
};

// First position a decode attends for context length ctx: inside the window
// (>= ctx - window when window > 0) and still held by a ring table (from the
// start of block (ctx-1)/bs - ring + 1 when ring > 0).
__host__ __device__ inline int window_start(int ctx, int bs, int window, int ring) {
  int t = 0;
  if (window > 0 && ctx - window > t) t = ctx - window;
  if (ring > 0) {
    const int held = ((ctx - 1) / bs - ring + 1) * bs;
    if (held > t) t = held;
  }
  return t;
}

// Table entry holding logical block j.
__host__ __device__ inline int table_index(int j, int ring) { return ring > 0 ? j % ring : j; }

// Whether a context length can be served: linear rows must hold it; every
// context must be within max_context_len.
__host__ __device__ inline bool context_ok(const DecodeParams& p, int ctx) {
  return (p.ring_blocks > 0 || (int64_t)ctx <= (int64_t)p.bt_stride * p.block_size) && ctx <= p.max_context_len;
}

// Partitions of a sequence: windows start at the block holding window_start.
__host__ __device__ inline int attended_from(const DecodeParams& p, int ctx) {
  return (window_start(ctx, p.block_size, p.window, p.ring_blocks) / p.block_size) * p.block_size;
}

cudaError_t launch_reshape_and_cache(uint8_t* layer_base, int32_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_size, const void* key,
                                     int64_t key_stride, const void* value, int64_t value_stride,
                                     const int64_t* slot_mapping, int32_t n, uint32_t* dev_err,
                                     cudaStream_t stream);

// 8-bit cache (head_size 128); key / value in act_dtype (PA_F16 or PA_BF16).
cudaError_t launch_reshape_and_cache_i8(uint8_t* layer_base, int32_t num_blocks, int32_t block_size,
                                        int32_t num_kv_heads, int act_dtype, const void* key, int64_t key_stride,
                                        const void* value, int64_t value_stride, const int64_t* slot_mapping,
                                        int32_t n, uint32_t* dev_err, cudaStream_t stream);

// Copies `pairs.n` whole blocks of `block_bytes` for each of `layers` layers.
cudaError_t launch_block_copy(uint8_t* dst, int64_t dst_layer_stride, const uint8_t* src,
                              int64_t src_layer_stride, int64_t block_bytes, int32_t layers,
                              const PairList& pairs, int32_t n, cudaStream_t stream);

// Paged decode on CUDA cores (all supported shapes).  Returns cudaErrorInvalidValue
// for an unsupported (dtype, head_size, group) combination.
cudaError_t launch_decode_simt(const DecodeParams& p, int dtype, int head_size, int group,
                               cudaStream_t stream);

// Log-sum-exp merge of partition results in the workspace (items whose context
// spans more than one partition); no-op launch when max_parts <= 1.
cudaError_t launch_merge(const DecodeParams& p, int dtype, int head_size, cudaStream_t stream);

// Paged decode on the tensor cores (tcgen05): head_size 128, group size 1-16,
// at most kTcMaxSeqs sequences.  Launches the decode kernel and the merge.
constexpr int kTcMaxSeqs = 8192;
cudaError_t launch_decode_tc(const DecodeParams& p, int dtype, int group, int num_sms, cudaStream_t stream);

// Causal prefill / extend over a 16-bit cache (tcgen05): head_size 64 or 128,
// block_size >= 8, group 1, 2, 4, 8 or 16.
struct PrefillParams {
  void* out;                      // [tokens, Hq, D] q dtype, contiguous
  const void* q;                  // [tokens, Hq, D], token stride q_token_stride elements
  int64_t q_token_stride;
  const uint8_t* cache;           // this layer's pool
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  const int32_t* block_tables;
  int32_t bt_stride;
  const int32_t* context_lens;    // [S], counts the new tokens
  const int32_t* query_start_loc; // [S + 1]
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t max_query_len;
  float scale_log2;
  uint32_t* dev_err;
};
cudaError_t launch_prefill_tc(const PrefillParams& p, int dtype, int head_size, int group, cudaStream_t stream);

// Paged decode over an 8-bit cache on the tensor cores: the same kernel with
// converter warps that turn each staged 8-bit tile into fp16 operands.
// group 1, 2, 4 or 8, at most kTcI8MaxSeqs sequences.  Launches decode and merge.
constexpr int kTcI8MaxSeqs = 1024;
cudaError_t launch_decode_tc_i8(const DecodeParams& p, int act_dtype, int group, int num_sms, cudaStream_t stream);

// Paged decode with shared prefixes on the tensor cores (16-bit cache, head_size
// 128, block_size >= 8, group 1, 2, 4 or 8, at most kTcSpMaxSeqs sequences): a
// group's prefix is streamed once for all its members.  Launches the decode
// kernel and the merge (which also checks the members' prefix block ids).
// (the item tables of 160 sequences keep static + dynamic shared memory within
// the 227 KiB a CTA may have)
constexpr int kTcSpMaxSeqs = 160;
cudaError_t launch_decode_tc_sp(const DecodeParams& p, int dtype, int group, int num_sms, cudaStream_t stream);
cudaError_t launch_merge_sp(const DecodeParams& p, int dtype, int head_size, cudaStream_t stream);

// Paged decode over an 8-bit cache on CUDA cores: head_size 128, group 1/2/4/8;
// q / out in act_dtype.  Launches the decode kernel and the merge.
cudaError_t launch_decode_i8(const DecodeParams& p, int act_dtype, int group, cudaStream_t stream);

}  // namespace pkv
