/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode library.
 *
 * The library implements the hot path of paged-attention decoding as the vLLM
 * and nano-vLLM write-ups describe it:
 *
 *   pa_reshape_and_cache  scatter each step's new K/V into cache slots
 *                         (nano-vLLM article, section 5.2.3 "KV Cache 写入":
 *                         store_kvcache writes token i to slot_mapping[i],
 *                         -1 means "skip").
 *   pa_decode             one query token per sequence attends over its
 *                         non-contiguous KV blocks found through a block table
 *                         ("vLLM" page, section "PageAttention": softmax(QK^T /
 *                         sqrt(d_k)) V; mlqm.cn article, section 二.2.2: block
 *                         table maps logical to physical blocks).  Long contexts
 *                         are split into partitions merged by log-sum-exp
 *                         ("vLLM" page, "Prefill vs decoding" item 5,
 *                         FlashDecoding).
 *   pa_copy_blocks        copy-on-write block copies ("vLLM" page, section
 *                         "CacheEngine": copy / copy_blocks; mlqm.cn article,
 *                         Copy-on-Write example).
 *   pa_prefill            several new query tokens per sequence (a prompt or
 *                         a chunk of one) attend causally over the paged cache
 *                         ("vLLM" page, prefill vs decoding; FAQ, chunked
 *                         prefill).
 *   pa_swap_blocks        whole-block moves between the GPU cache and a pinned
 *                         CPU cache ("vLLM" page, section "CacheEngine":
 *                         swap_in = CPU->GPU, swap_out = GPU->CPU; section
 *                         "Preemption").
 *
 * Conventions
 *   Ownership:  the caller allocates every buffer (cache pools, workspace,
 *               error word).  The library allocates no device memory and keeps
 *               no per-call state (pa_decode_static_workspace alone uses a
 *               fixed array the library carries; see its comment); the block
 *               manager keeps host memory for its own bookkeeping.
 *   Streams:    every call except pa_read_device_errors is asynchronous on the
 *               given CUDA stream (a cudaStream_t passed as void*; NULL = the
 *               legacy default stream) and performs no host synchronisation.
 *   Errors:     problems visible on the host (null or misaligned pointers,
 *               unsupported shapes, bad pair lists, small workspace) return a
 *               status synchronously and launch nothing; pa_last_error_message()
 *               then names the argument.  Problems only visible on the device
 *               (a block id or slot out of range, a context longer than the
 *               block table) set bits in the optional device error word
 *               `dev_err`; the affected item is skipped (its output zeroed).
 *               Kernels never trap.
 *   Types:      query, key, value and output elements are fp16 or bf16 (one
 *               dtype per call); the cache holds the same 16-bit type, or 8-bit
 *               codes with fp32 scales (PA_INT8_F16 / PA_INT8_BF16, below);
 *               arithmetic is fp32.
 *
 * Cache layout (one layer; a pool may hold several layers `layer_stride_bytes`
 * apart).  The pool is num_blocks blocks; block b holds, for each kv head h,
 * one contiguous chunk of 2 * block_size * head_size elements at element offset
 * (b * num_kv_heads + h) * 2 * block_size * head_size.  Inside a chunk the
 * block's token slots are grouped by R = min(block_size, 8); group g holds the K
 * rows of its R slots and then their V rows; each is head_size / 64 "atoms" of
 * R rows x 64 dims (128-byte rows); inside an atom the 16-byte piece c (dims
 * 8c..8c+7) of row r is stored at piece position c XOR r.  This is the
 * 128-byte-swizzled K-major operand layout of the sm_100-family tensor cores,
 * so one bulk copy per chunk stages a block ready for both CUDA-core and
 * tensor-core consumers.  pa_cache_element_offset() computes the position of
 * any element.
 *
 * 8-bit cache (dtype PA_INT8_F16 / PA_INT8_BF16; head_size 128).  The TurboMind
 * section of the inference-framework notes lists an "8bit KV Cache"; the scheme
 * here is per token and per kv head symmetric quantisation: each stored K or V
 * vector x gets scale = max|x| / 127 and codes round-half-even(x * (127 /
 * max|x|)) clipped to [-127, 127], both decided in IEEE fp32 (an all-zero
 * vector stores scale 0 and zero codes); the value a code stands for is
 * code * scale.  Chunk (block, kv head) holds, in bytes: K codes [block_size]
 * [128] row-major, V codes [block_size][128], K scales (fp32 [block_size]
 * padded to a multiple of 16 bytes), V scales (same).  Chunk bytes =
 * 2 * block_size * 128 + 2 * roundup16(4 * block_size); chunks are ordered by
 * (block, kv head) as above.  pa_cache_element_offset() gives code byte
 * offsets and pa_cache_scale_offset() scale byte offsets.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,        /* bad pointer, size, id or pair list */
    PA_ERR_UNSUPPORTED = 2,        /* valid but not implemented (head_size, block_size, group) */
    PA_ERR_CUDA = 3,               /* a CUDA runtime call failed (launch, copy, attribute query) */
    PA_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes < pa_decode_workspace_bytes(...) */
    PA_ERR_OUT_OF_BLOCKS = 5        /* block manager: not enough free blocks (nothing changed) */
} pa_status;

/* Element types.  PA_F16 / PA_BF16: cache, query, key, value and output all of
 * that type.  PA_INT8_F16 / PA_INT8_BF16: 8-bit cache (layout above) with
 * query, key, value and output in fp16 / bf16. */
typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1, PA_INT8_F16 = 2, PA_INT8_BF16 = 3 } pa_dtype;

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID 0x1u  /* a block-table entry that must be read is < 0 or >= num_blocks */
#define PA_DEVERR_SLOT 0x2u      /* a slot_mapping entry is not -1 and not in [0, num_blocks*block_size) */
#define PA_DEVERR_CONTEXT 0x4u   /* context_lens[s] > block_table_stride*block_size or > max_context_len */
#define PA_DEVERR_TIMEOUT 0x8u   /* a bounded wait inside a kernel ran out (the item was abandoned) */
#define PA_DEVERR_PREFIX 0x10u   /* pa_decode_shared_prefix: a member's block ids differ from its group's
                                    inside the shared prefix (its rows are zeroed), or the group
                                    starts are out of order (sharing is then ignored) */

/* Geometry of a cache pool.  head_size in {64, 128}; block_size in {1, 2, 4, 8, 16, 32}
 * (block_size 1 is token-granular paging);
 * dtype a pa_dtype.  layer_stride_bytes = distance between consecutive layers
 * (0 means layers are packed: pa_cache_bytes(desc)). */
typedef struct pa_cache_desc {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_size;
    int32_t dtype;
    int32_t num_layers;
    int64_t layer_stride_bytes;
} pa_cache_desc;

/* Bytes of one layer of the pool: num_blocks * num_kv_heads * 2 * block_size *
 * head_size * 2 (the KV-size formula of the mlqm.cn article, section 二.2.1,
 * rounded up to whole blocks); for an 8-bit cache num_blocks * num_kv_heads *
 * the chunk bytes given above.  Returns 0 for an invalid descriptor. */
size_t pa_cache_bytes(const pa_cache_desc* desc);

/* Element offset (from the start of a layer, in cache elements: 16-bit elements,
 * or bytes for an 8-bit cache) of dim `dim` of the K (part = 0) or V (part = 1)
 * vector stored in slot `slot` of block `block` for kv head `kv_head`.  Returns
 * -1 for out-of-range arguments.  Host only. */
int64_t pa_cache_element_offset(const pa_cache_desc* desc, int64_t block, int32_t kv_head,
                                int32_t part, int32_t slot, int32_t dim);

/* Byte offset (from the start of a layer) of the fp32 scale of the K (part = 0)
 * or V (part = 1) vector in slot `slot` of block `block`, kv head `kv_head`, of
 * an 8-bit cache.  Returns -1 for a 16-bit cache or out-of-range arguments.
 * Host only; this library's own addition (the notes name no layout). */
int64_t pa_cache_scale_offset(const pa_cache_desc* desc, int64_t block, int32_t kv_head,
                              int32_t part, int32_t slot);

/* Write each new token's K and V into the cache.
 * Follows store_kvcache (nano-vLLM article, section 5.2.3): for token i with
 * slot = slot_mapping[i] != -1, block = slot / block_size and offset =
 * slot % block_size, the num_kv_heads x head_size K and V elements are copied
 * bit for bit into that slot of layer `layer` (an 8-bit cache stores each head
 * vector's codes and scale instead, quantised as described above).
 *   kv_cache     device pool (see layout above), 16-byte aligned.
 *   key, value   device [num_tokens, num_kv_heads, head_size], heads and dims
 *                contiguous; token strides key_token_stride / value_token_stride
 *                in elements (multiples of 8); 16-byte aligned.
 *   slot_mapping device int64 [num_tokens].
 *   dev_err      optional device uint32; PA_DEVERR_SLOT is OR-ed in for a slot
 *                out of range (that token is skipped).
 * num_tokens == 0 launches nothing. */
pa_status pa_reshape_and_cache(void* kv_cache, const pa_cache_desc* desc, int32_t layer,
                               const void* key, int64_t key_token_stride, const void* value,
                               int64_t value_token_stride, const int64_t* slot_mapping,
                               int32_t num_tokens, uint32_t* dev_err, void* stream);

/* Workspace bytes pa_decode needs for these shapes (0 when no sequence can span
 * more than one partition, or desc is NULL; SIZE_MAX when the size does not fit
 * in half the address space).  partition_size 0 selects the default
 * (pa_decode_partition_size with the same desc, num_seqs and max_context_len). */
size_t pa_decode_workspace_bytes(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t max_context_len, int32_t partition_size);

/* The partition size pa_decode uses: `partition_size` itself when > 0, else a
 * default that depends on the kernel these shapes get.
 *   Tensor-core kernel (head_size 128 and either a 16-bit cache with
 *   block_size >= 8 and at most 8192 sequences, or an 8-bit cache with at most
 *   1024 sequences): it walks work items of one (sequence, kv head, partition),
 *   and the default is the longest of 4096, 2048, 1024 and 512 tokens (8192
 *   first when max_context_len > 32768) for which
 *     num_seqs * num_kv_heads * ceil(max_context_len / P) >= 6 * SMs
 *   (six items per SM of the current device: 912 on a 152-SM GB300; 152 is
 *   assumed when no device can be queried), else 512.  Longer partitions write and
 *   merge fewer partial results; shorter ones split the work finely enough to
 *   keep every SM busy to the end.
 *   CUDA-core kernel (the other shapes): 512, or 1024 when max_context_len >
 *   32768.
 * desc NULL gives 512. */
int32_t pa_decode_partition_size(const pa_cache_desc* desc, int32_t num_seqs, int32_t max_context_len,
                                 int32_t partition_size);

/* Paged decode attention: one query token per sequence.
 * For sequence s and query head h (kv head = h / (num_q_heads / num_kv_heads)):
 *   z_t = scale * q[s,h,:] . K_t   for t < ctx = context_lens[s], where token t
 *         lives in slot t % block_size of block block_tables[s*block_table_stride + t/block_size];
 *   out[s,h,:] = sum_t softmax(z)_t V_t     (fp32 accumulation, rounded to the
 *                                            dtype of q, round-to-nearest-even).
 * context_lens counts the new token, so pa_reshape_and_cache must run first.
 * ctx <= 0 gives a zero output row.  Contexts longer than partition_size are
 * split into partitions of partition_size tokens, each producing (max, sum,
 * unnormalised output) in the workspace, merged by log-sum-exp in a second
 * kernel on the same stream.
 *   out           device [num_seqs, num_q_heads, head_size], q's dtype, contiguous.
 *   q             device [num_seqs, num_q_heads, head_size]; sequence stride
 *                 q_seq_stride elements (multiple of 8); 16-byte aligned.
 *   block_tables  device int32 [num_seqs, block_table_stride]; entries past
 *                 ceil(ctx / block_size) are never read.
 *   context_lens  device int32 [num_seqs].
 *   max_context_len  an upper bound of context_lens (sizes the launch and the
 *                 workspace); a longer context sets PA_DEVERR_CONTEXT.
 *   partition_size   0 (default) or a multiple of 128 in [128, 8192].
 *   workspace     device, 16-byte aligned, >= pa_decode_workspace_bytes(...);
 *                 may be NULL when that is 0.  Contents need no initialisation.
 *   dev_err       optional device uint32 error word (PA_DEVERR_* bits).
 * Supported: head_size 64 or 128, block_size 1/2/4/8/16/32, num_q_heads a
 * multiple of num_kv_heads with group size 1, 2, 4 or 8, and 16 at head_size 128
 * with block_size >= 8 (PA_ERR_UNSUPPORTED otherwise).  An 8-bit cache
 * (PA_INT8_F16 / PA_INT8_BF16) attends over code * scale: head_size 128, group
 * size 1, 2, 4 or 8, any supported block_size (windows and ring tables
 * included); q and out are the dtype's 16-bit type. */
pa_status pa_decode(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                    const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                    int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                    int32_t num_q_heads, int32_t max_context_len, float scale,
                    int32_t partition_size, void* workspace, size_t workspace_bytes,
                    uint32_t* dev_err, void* stream);

/* Causal prefill / extend attention over the paged cache (several new tokens per
 * sequence: a whole prompt, or one chunk of it under chunked prefill -- the
 * "vLLM" page's prefill/decoding description and the FAQ's vLLM scheduler notes
 * on chunked prefill).  Sequence s owns the packed query tokens
 * query_start_loc[s] .. query_start_loc[s+1]-1 (q_len of them, possibly 0);
 * they are its newest q_len positions, already written into the cache by
 * pa_reshape_and_cache, so with ctx = context_lens[s] query j attends
 *   positions 0 .. ctx - q_len + j   (causal), found through the block table;
 *   out[token, h, :] = sum_t softmax(scale * q[token, h, :] . K_t) V_t
 * with fp32 accumulation, rounded to the dtype (round-to-nearest-even).
 *   out            device [total tokens, num_q_heads, head_size], contiguous.
 *   q              device [total tokens, num_q_heads, head_size]; token stride
 *                  q_token_stride elements (multiple of 8); 16-byte aligned.
 *   query_start_loc device int32 [num_seqs + 1], non-decreasing, starting at 0.
 *   context_lens   device int32 [num_seqs], counting the new tokens.
 *   max_query_len  an upper bound of every q_len (sizes the launch); a longer
 *                  sequence gets zero rows and PA_DEVERR_CONTEXT.
 *   dev_err        optional; PA_DEVERR_CONTEXT for q_len > ctx or ctx beyond the
 *                  table row, PA_DEVERR_BLOCK_ID for a bad block id (that query
 *                  tile's rows are zeroed).
 * Supported: a 16-bit cache, head_size 64 or 128, block_size 8, 16 or 32, group
 * size 1, 2, 4, 8 or 16 (PA_ERR_UNSUPPORTED otherwise).  No workspace. */
pa_status pa_prefill(void* out, const void* q, int64_t q_token_stride, const void* kv_cache,
                     const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                     int32_t block_table_stride, const int32_t* context_lens,
                     const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                     int32_t max_query_len, float scale, uint32_t* dev_err, void* stream);

/* Paged decode where groups of sequences share the first tokens of their
 * context physically: beams of one prompt, or parallel samples, whose prompt
 * blocks are the same physical blocks in every member's block table (the
 * mlqm.cn article's copy-on-write example, section 二.2.2: samples of one
 * request share the prompt's blocks until one writes; the "vLLM" page's
 * CacheEngine copies a block only when a beam writes into it).  The result is
 * pa_decode's; the shared blocks are read from memory once per group and kv
 * head instead of once per member.
 *   group_start  device int32 [num_groups + 1], non-decreasing in [0, num_seqs]:
 *                group g is sequences group_start[g] .. group_start[g+1] - 1
 *                (consecutive; sequences outside every group are decoded alone).
 *   prefix_lens  device int32 [num_groups]: tokens at the start of every member's
 *                context whose block-table entries are the same in all members.
 *                The kernel uses the largest whole number of blocks <= both
 *                prefix_lens[g] and the group's shortest context, so any value is
 *                safe; a group of one sequence shares nothing.
 *   num_groups   0 .. num_seqs (0: plain pa_decode).
 * The prefix is read through the table row of the first member of each chunk
 * of 16 / (num_q_heads / num_kv_heads) members (one tensor-core item serves a
 * chunk's query heads together).  A member whose table entries differ from
 * that row inside the prefix gets zero output rows and PA_DEVERR_PREFIX; group
 * starts out of order make the call ignore the groups (each sequence read
 * through its own row) and also set PA_DEVERR_PREFIX.
 * Other arguments as pa_decode; size the workspace with
 * pa_decode_shared_prefix_workspace_bytes and take the default partition size
 * from pa_decode_shared_prefix_partition_size (the same arguments).  Served by
 * a dedicated tensor-core kernel for a 16-bit cache, head_size 128,
 * block_size >= 8, 1, 2, 4 or 8 query heads per kv head and at most 160
 * sequences; other shapes run pa_decode (the same result, without the sharing).
 * No windows or ring tables. */
pa_status pa_decode_shared_prefix(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                                  const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                                  int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                  const int32_t* group_start, const int32_t* prefix_lens, int32_t num_groups,
                                  int32_t partition_size, void* workspace, size_t workspace_bytes,
                                  uint32_t* dev_err, void* stream);

/* The partition size pa_decode_shared_prefix uses: partition_size when > 0;
 * else, where its dedicated kernel serves the shapes and num_groups > 0, the
 * longest of 4096, 2048, 1024, 512 tokens (8192 first past 32768) for which
 * the groups' prefixes alone still give 1.5 items per SM
 * (num_groups * num_kv_heads * ceil(max_context_len / P) >= 1.5 * SMs; each
 * sequence adds its own tail item), else 512; otherwise
 * pa_decode_partition_size(desc, num_seqs, max_context_len, 0). */
int32_t pa_decode_shared_prefix_partition_size(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_groups, int32_t max_context_len, int32_t partition_size);

/* Workspace bytes pa_decode_shared_prefix needs (partition_size 0: the default
 * above).  Where the dedicated kernel serves the shapes: num_seqs *
 * num_q_heads * (ceil(max_context_len / P) + 1) * (head_size + 2) floats plus
 * 3 * num_seqs ints, rounded up to 16 bytes; otherwise pa_decode's. */
size_t pa_decode_shared_prefix_workspace_bytes(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_groups, int32_t max_context_len, int32_t partition_size);

/* Size of the workspace the library carries for pa_decode_static_workspace
 * (32 MiB on every device that loads the library, held until the process exits). */
#define PA_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)

/* Paged decode over a sliding window, with optional ring block tables.
 * The vLLM block manager ("推理框架知识点" page, vLLM BlockSpaceManagerV1) keeps a
 * sliding-window sequence in ceil(window / block_size) blocks and reuses
 * block_table[logical_block % that count]; such a table row is a ring.
 *   window       > 0: attend only positions >= ctx - window (0: no window).
 *   ring_blocks  > 0: logical block j of a sequence is at table entry
 *                j % ring_blocks (<= block_table_stride); the ring only still
 *                holds positions from the start of block (ctx-1)/bs - ring + 1,
 *                so the attended positions are [t, ctx) with
 *                t = max(0, ctx - window, ((ctx-1)/bs - ring_blocks + 1) * bs).
 *                The window is exact when ring_blocks >= ceil((window-1)/bs) + 1.
 *                0: linear rows (then ctx must fit the row, as in pa_decode).
 * Other arguments as pa_decode; size the workspace with
 * pa_decode_workspace_bytes(desc, num_seqs, num_q_heads,
 * pa_decode_window_span(max_context_len, block_size, window, ring_blocks),
 * partition_size).  pa_decode is this call with window = ring_blocks = 0. */
pa_status pa_decode_window(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                           const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                           int32_t block_table_stride, const int32_t* context_lens, int32_t num_seqs,
                           int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                           int32_t ring_blocks, int32_t partition_size, void* workspace, size_t workspace_bytes,
                           uint32_t* dev_err, void* stream);

/* Upper bound on the tokens one sequence's windowed decode spans (from the
 * block holding its first attended position): min(max_context_len,
 * window + block_size - 1 if window > 0, ring_blocks * block_size if
 * ring_blocks > 0).  Pass it as max_context_len to pa_decode_workspace_bytes. */
int32_t pa_decode_window_span(int32_t max_context_len, int32_t block_size, int32_t window, int32_t ring_blocks);

/* pa_decode for callers that cannot allocate device memory.  The pages describe
 * no such entry point; it exists for this library's users.  Some callers cannot
 * call cudaMalloc where they call decode: a plugin inside a framework whose
 * allocator owns all device memory, a serving loop that forbids allocation once
 * it runs, or a binding from another language that cannot keep a device buffer
 * between calls.  This call takes the same arguments as pa_decode minus the
 * workspace, and uses instead a fixed array of PA_STATIC_WORKSPACE_BYTES in the
 * library's own device memory.
 *   - Shapes whose pa_decode_workspace_bytes(...) exceeds
 *     PA_STATIC_WORKSPACE_BYTES are rejected with PA_ERR_WORKSPACE_TOO_SMALL
 *     (pa_last_error_message explains); nothing is launched.  A larger
 *     partition_size shrinks the need.
 *   - Every argument is checked as pa_decode checks it before the size test,
 *     so a bad argument returns its own status (PA_ERR_INVALID_ARG or
 *     PA_ERR_UNSUPPORTED), not PA_ERR_WORKSPACE_TOO_SMALL.
 *   - It allocates nothing.  The first call in a CUDA context that needs the
 *     array looks up its device address (cudaGetSymbolAddress) with the device
 *     current and caches it for that context; make that first call before any
 *     stream capture.  After cudaDeviceReset the device's new context gets a
 *     fresh lookup (the array may then sit at another address), so the first
 *     call after a reset must also come before any capture.
 *   - The array is shared by every call on a device and keeps the last call's
 *     contents (decode needs none of it zeroed).  Calls that may overlap on the
 *     GPU -- on different streams, or from different threads -- race on it:
 *     serialise them, or give each its own workspace through pa_decode. */
pa_status pa_decode_static_workspace(void* out, const void* q, int64_t q_seq_stride, const void* kv_cache,
                                     const pa_cache_desc* desc, int32_t layer, const int32_t* block_tables,
                                     int32_t block_table_stride, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                     float scale, int32_t partition_size, uint32_t* dev_err, void* stream);

/* Copy whole blocks inside one pool (every kv head, K and V, every layer):
 * for each pair i, block pairs[2i+1] receives block pairs[2i].  All pairs act
 * at once ("vLLM" page, CacheEngine copy; used for copy-on-write).
 *   pairs   HOST int64 [num_pairs][2] (src, dst), read before the call returns.
 * Rejected with PA_ERR_INVALID_ARG: an id out of range, a repeated dst, a dst
 * that is also a src.  num_pairs == 0 launches nothing. */
pa_status pa_copy_blocks(void* kv_cache, const pa_cache_desc* desc, const int64_t* pairs,
                         int32_t num_pairs, void* stream);

/* Move whole blocks (every layer) between the device pool and a pinned host
 * pool of the same geometry (num_blocks and layer stride may differ).
 *   direction 0 = swap_out (src device pool -> dst pinned host pool),
 *             1 = swap_in  (src pinned host pool -> dst device pool).
 *   pairs   HOST int64 [num_pairs][2] (src block, dst block); dst ids unique.
 * The host pool must be page-locked (cudaHostAlloc / pin_memory). */
pa_status pa_swap_blocks(void* dst_pool, const pa_cache_desc* dst_desc, const void* src_pool,
                         const pa_cache_desc* src_desc, int32_t direction, const int64_t* pairs,
                         int32_t num_pairs, void* stream);

/* ---------------------------------------------------------------- block manager
 * Host-side bookkeeping that turns sequences of token ids into the block
 * tables, slots, copy-on-write pairs and swap pairs the calls above consume --
 * the vLLM block manager of the "推理框架知识点" page (BlockSpaceManagerV1 with its
 * uncached and prefix-caching allocators and LRU evictor), with the mlqm.cn
 * article's copy-on-write example and nano-vLLM's chain-hashed prefix blocks
 * (section 5.2.1).  It holds only host memory (its own metadata); block ids are
 * indices into the device pool (and, for swapped sequences, the host pool).
 * Free blocks are handed out last-freed first, starting from the highest id.
 * Not thread-safe: one caller at a time per manager. */
typedef struct pa_block_manager pa_block_manager;

typedef enum pa_alloc_status { PA_ALLOC_OK = 0, PA_ALLOC_LATER = 1, PA_ALLOC_NEVER = 2 } pa_alloc_status;

/* num_cpu_blocks: host (swap) pool size.  watermark: fraction of device blocks
 * kept free by admission.  sliding_window > 0: logical block i of a sequence
 * reuses table entry i % ceil(sliding_window / block_size).  With
 * enable_prefix_caching, full blocks are shared between sequences whose token
 * ids agree up to and including that block (not combinable with a window). */
pa_status pa_bm_create(int32_t block_size, int32_t num_gpu_blocks, int32_t num_cpu_blocks, float watermark,
                       int32_t sliding_window, int32_t enable_prefix_caching, pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);

/* Admission of a prompt of num_tokens tokens: a pa_alloc_status. */
int32_t pa_bm_can_allocate(pa_block_manager* bm, int32_t num_tokens);

/* Blocks for a new sequence's prompt (token_ids[0..num_tokens-1]).  Returns
 * PA_ERR_OUT_OF_BLOCKS (and changes nothing) when the pool runs out. */
pa_status pa_bm_allocate(pa_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t num_tokens);

/* Room for one more token: *slot receives its cache slot (block * block_size +
 * offset, for pa_reshape_and_cache); when the last block was shared it is
 * copied first and (*cow_src, *cow_dst) name the pair for pa_copy_blocks, else
 * both are -1. */
pa_status pa_bm_append_slot(pa_block_manager* bm, int64_t seq_id, int32_t token_id, int64_t* slot,
                            int64_t* cow_src, int64_t* cow_dst);

/* The child shares every block of the parent (parallel sampling, beam search). */
pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Release a sequence's blocks. */
pa_status pa_bm_free(pa_block_manager* bm, int64_t seq_id);

/* A sequence's block table (capacity entries at `table`, may be NULL to query
 * sizes), its number of blocks and of tokens. */
pa_status pa_bm_block_table(pa_block_manager* bm, int64_t seq_id, int32_t* table, int32_t capacity,
                            int32_t* num_blocks, int32_t* num_tokens);

/* Move every block of the n sequences to the host pool (swap_out) or back
 * (swap_in); pairs receives [*num_pairs][2] (src, dst) ids for pa_swap_blocks
 * (may be NULL to count).  A block shared by several of them moves once. */
pa_status pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs, int32_t capacity,
                         int32_t* num_pairs);
pa_status pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs, int32_t capacity,
                        int32_t* num_pairs);

/* Whether num_running sequences can each take one more token now: 1 when
 * num_running <= the free device blocks (each may need a new block, or a copy
 * of a shared last block), else 0 -- the vLLM block manager's can_append_slots
 * ("推理框架知识点" page, running/swapped queues). */
int32_t pa_bm_can_append_slots(pa_block_manager* bm, int32_t num_running);

/* Admission of pa_bm_swap_in for the n (swapped-out) sequences: their distinct
 * blocks (a shared block counted once) against the free device blocks and the
 * watermark, as pa_bm_can_allocate: a pa_alloc_status, or -1 for an unknown or
 * not swapped-out sequence (pa_last_error_message says which). */
int32_t pa_bm_can_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n);

/* Whether the host pool has room for pa_bm_swap_out of the n (device-resident)
 * sequences: 1 or 0, or -1 for an unknown or swapped-out sequence. */
int32_t pa_bm_can_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n);

/* Free blocks (the evictor's cached blocks included) on the device (0) or host (1) side. */
int32_t pa_bm_num_free_blocks(pa_block_manager* bm, int32_t on_host);

/* Reference count of a block (-1 for an id out of range). */
int32_t pa_bm_ref_count(pa_block_manager* bm, int32_t on_host, int32_t block);

/* Synchronise `stream`, copy the device error word into *host_bits, and reset
 * it to 0 when `clear` is non-zero. */
pa_status pa_read_device_errors(uint32_t* dev_err, uint32_t* host_bits, int32_t clear, void* stream);

/* Static description of a status code. */
const char* pa_status_string(pa_status status);

/* Detail of the last failed call on this thread ("" if none). */
const char* pa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
