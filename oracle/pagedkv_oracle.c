/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA library; it restates from the pages
 * what the hot path computes, in the most direct way:
 *
 *   - "vLLM" (yang20150702.github.io agent-guide), section "PageAttention":
 *     attention Z = softmax(Q K^T / sqrt(d_k)) V.
 *   - "vLLM" page, section "CacheEngine": copy (copy_blocks) and
 *     swap_in / swap_out (swap_blocks) move whole cache blocks.
 *   - nano-vLLM article (cybasar.com), section 5.2.3 "KV Cache 写入":
 *     each new token i is written to cache slot slot_mapping[i]; -1 skips it.
 *   - mlqm.cn vLLM article, section 3 (Nano-vLLM): attention over a paged
 *     cache = gather the sequence's blocks by block table into a contiguous
 *     temporary, then run ordinary attention on it.
 *   - "vLLM" page, "Prefill vs decoding" item 5 (FlashDecoding): splitting the
 *     KV sequence into pieces; the pieces are merged with log-sum-exp algebra.
 *
 * Floating point: every 16-bit element is widened exactly to double; all
 * arithmetic is double.  Nothing here is blocked, fused or reordered beyond
 * what the definition states.
 *
 * Cache layout (the library's chosen layout, restated here independently):
 *   one layer = num_blocks chunks; chunk (block, kv_head) holds 2*bs*D elements.
 *   Inside a chunk, token slots are grouped by R = min(bs, 8) rows; each group
 *   holds the K part then the V part; each part is D/64 "atoms" of R rows x 64
 *   dims; inside an atom, the 8-element (16-byte) column piece c of row r is
 *   stored at piece position (c XOR r).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------- element decoding (IEEE 754 binary16, bfloat16) ---------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                  /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac | 0x400), expo - 25);  /* (1.frac) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem_to_double(uint16_t bits, int dtype) {
    return dtype == 0 ? half_bits_to_double(bits) : bf16_bits_to_double(bits);
}

double oracle_elem_to_double(uint16_t bits, int dtype) { return elem_to_double(bits, dtype); }

/* ---------------- cache geometry ---------------- */

typedef struct {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_size;
    int32_t dtype;          /* 0 = fp16, 1 = bf16 */
    int32_t num_layers;
    int64_t layer_stride;   /* elements between layers */
} oracle_geom;

static int64_t chunk_elems(const oracle_geom* g) {
    return 2 * (int64_t)g->block_size * g->head_size;
}

/* Offset, in elements from the start of a layer, of element (block, kv_head,
 * part (0 = K, 1 = V), slot t in the block, dim d). */
static int64_t cache_offset(const oracle_geom* g, int64_t block, int64_t head, int part,
                            int64_t t, int64_t d) {
    const int64_t R = g->block_size < 8 ? g->block_size : 8;
    const int64_t atoms = g->head_size / 64;
    const int64_t group = t / R, row = t % R;
    const int64_t atom = d / 64, piece = (d % 64) / 8, lane = d % 8;
    int64_t off = (block * g->num_kv_heads + head) * chunk_elems(g);
    off += ((group * 2 + part) * atoms + atom) * (R * 64);
    off += row * 64 + ((piece ^ row) * 8) + lane;
    return off;
}

int64_t oracle_cache_offset(const oracle_geom* g, int64_t block, int64_t head, int part,
                            int64_t t, int64_t d) {
    return cache_offset(g, block, head, part, t, d);
}

/* Error bits reported by the oracle (same meaning as the library's device error word). */
enum { ORC_ERR_BLOCK_ID = 1, ORC_ERR_SLOT = 2, ORC_ERR_CONTEXT = 4 };

/* ---------------- reshape_and_cache (store_kvcache) ---------------- */

/* For each new token i with slot_mapping[i] != -1, copy its K and V vectors
 * (num_kv_heads x head_size elements each, raw bits) into cache slot
 * slot = block * block_size + offset.  key/value rows are [num_kv_heads][head_size]
 * with the given token stride (elements). */
int oracle_reshape_and_cache(uint16_t* layer, const oracle_geom* g,
                             const uint16_t* key, int64_t key_stride,
                             const uint16_t* value, int64_t value_stride,
                             const int64_t* slot_mapping, int32_t n) {
    int err = 0;
    const int64_t nslots = (int64_t)g->num_blocks * g->block_size;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= nslots) { err |= ORC_ERR_SLOT; continue; }
        const int64_t block = slot / g->block_size, t = slot % g->block_size;
        for (int64_t h = 0; h < g->num_kv_heads; ++h)
            for (int64_t d = 0; d < g->head_size; ++d) {
                layer[cache_offset(g, block, h, 0, t, d)] = key[i * key_stride + h * g->head_size + d];
                layer[cache_offset(g, block, h, 1, t, d)] = value[i * value_stride + h * g->head_size + d];
            }
    }
    return err;
}

/* ---------------- gather by block table ---------------- */

/* Copy tokens t in [t0, t1) of one kv head into contiguous K[t1-t0][D],
 * V[t1-t0][D] (doubles), reading token t from slot t % bs of block
 * table_row[j] with j = t / bs, or j = (t / bs) % ring when the table row is a
 * ring of `ring` blocks (sliding window; the "vLLM" block manager of the FAQ
 * page reuses block_table[logical_idx % block_sliding_window]).
 * Returns ORC_ERR_BLOCK_ID if any needed table entry is out of range. */
int oracle_gather_range(const uint16_t* layer, const oracle_geom* g, const int32_t* table_row,
                        int32_t t0, int32_t t1, int32_t ring, int32_t kv_head, double* K, double* V) {
    for (int32_t t = t0; t < t1; ++t) {
        const int32_t j = ring > 0 ? (t / g->block_size) % ring : t / g->block_size;
        const int32_t block = table_row[j];
        if (block < 0 || block >= g->num_blocks) return ORC_ERR_BLOCK_ID;
        const int64_t slot = t % g->block_size;
        for (int32_t d = 0; d < g->head_size; ++d) {
            K[(int64_t)(t - t0) * g->head_size + d] =
                elem_to_double(layer[cache_offset(g, block, kv_head, 0, slot, d)], g->dtype);
            V[(int64_t)(t - t0) * g->head_size + d] =
                elem_to_double(layer[cache_offset(g, block, kv_head, 1, slot, d)], g->dtype);
        }
    }
    return 0;
}

/* All tokens 0..ctx-1 through a linear table row. */
int oracle_gather(const uint16_t* layer, const oracle_geom* g, const int32_t* table_row,
                  int32_t ctx, int32_t kv_head, double* K, double* V) {
    return oracle_gather_range(layer, g, table_row, 0, ctx, 0, kv_head, K, V);
}

/* First position attended for context length ctx: the window keeps positions
 * >= ctx - window (window > 0), and a ring of `ring` blocks only still holds
 * positions from the start of block (ctx-1)/bs - ring + 1 on. */
int32_t oracle_window_start(int32_t ctx, int32_t block_size, int32_t window, int32_t ring) {
    int32_t t = 0;
    if (window > 0 && ctx - window > t) t = ctx - window;
    if (ring > 0) {
        const int32_t held = ((ctx - 1) / block_size - ring + 1) * block_size;
        if (held > t) t = held;
    }
    return t;
}

/* ---------------- textbook attention on contiguous arrays ---------------- */

/* out[D] = softmax(scale * q . K[t]) over t < ctx, applied to V.  The maximum
 * score is subtracted before exponentiation (this changes nothing exactly and
 * keeps exp() finite).  ctx <= 0 gives zeros. */
void oracle_contiguous_attention(const double* q, const double* K, const double* V,
                                 int32_t ctx, int32_t D, double scale, double* out) {
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (ctx <= 0) return;
    double* z = (double*)malloc(sizeof(double) * (size_t)ctx);
    double m = -INFINITY;
    for (int32_t t = 0; t < ctx; ++t) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += q[d] * K[(int64_t)t * D + d];
        z[t] = scale * dot;
        if (z[t] > m) m = z[t];
    }
    double denom = 0.0;
    for (int32_t t = 0; t < ctx; ++t) {
        z[t] = exp(z[t] - m);
        denom += z[t];
    }
    for (int32_t t = 0; t < ctx; ++t)
        for (int32_t d = 0; d < D; ++d) out[d] += z[t] * V[(int64_t)t * D + d];
    for (int32_t d = 0; d < D; ++d) out[d] /= denom;
    free(z);
}

/* ---------------- paged decode attention ---------------- */

/* One new query per sequence.  For each (sequence s, query head h):
 * kv head = h / (Hq / Hkv); gather the sequence's ctx_s tokens of that kv head
 * through its block-table row, then contiguous attention.  Writes doubles to
 * out[s][h][D].  A sequence with ctx <= 0 gives zeros.  A (s, h) whose context
 * exceeds the table row (bt_stride * bs) or max_context_len, or whose table has
 * an out-of-range block id, gives zeros and sets an error bit.
 * If sel != NULL only the nsel (s, h) pairs listed in sel[2*i], sel[2*i+1] are
 * computed (out is then [nsel][D]).  Returns the OR of error bits. */
int oracle_decode_window(double* out, const uint16_t* q, int64_t q_seq_stride, const uint16_t* layer,
                         const oracle_geom* g, const int32_t* block_tables, int32_t bt_stride,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t max_context_len, double scale, int32_t window, int32_t ring,
                         const int32_t* sel, int32_t nsel, int32_t nthreads) {
    const int32_t D = g->head_size;
    const int32_t G = num_q_heads / g->num_kv_heads;
    const int64_t items = sel ? nsel : (int64_t)num_seqs * num_q_heads;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int64_t it = 0; it < items; ++it) {
        const int32_t s = sel ? sel[2 * it] : (int32_t)(it / num_q_heads);
        const int32_t h = sel ? sel[2 * it + 1] : (int32_t)(it % num_q_heads);
        double* o = out + it * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        const int32_t ctx = context_lens[s];
        if (ctx <= 0) continue;
        if ((ring <= 0 && (int64_t)ctx > (int64_t)bt_stride * g->block_size) || ctx > max_context_len) {
            err |= ORC_ERR_CONTEXT;
            continue;
        }
        const int32_t t0 = oracle_window_start(ctx, g->block_size, window, ring);
        const int32_t n = ctx - t0;
        double* K = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        const int e = oracle_gather_range(layer, g, block_tables + (int64_t)s * bt_stride, t0, ctx, ring, h / G,
                                          K, V);
        if (e) {
            err |= e;
        } else {
            for (int32_t d = 0; d < D; ++d)
                qd[d] = elem_to_double(q[(int64_t)s * q_seq_stride + (int64_t)h * D + d], g->dtype);
            oracle_contiguous_attention(qd, K, V, n, D, scale, o);
        }
        free(K);
        free(V);
        free(qd);
    }
    return err;
}

int oracle_decode(double* out, const uint16_t* q, int64_t q_seq_stride, const uint16_t* layer,
                  const oracle_geom* g, const int32_t* block_tables, int32_t bt_stride,
                  const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                  int32_t max_context_len, double scale, const int32_t* sel, int32_t nsel,
                  int32_t nthreads) {
    return oracle_decode_window(out, q, q_seq_stride, layer, g, block_tables, bt_stride, context_lens,
                                num_seqs, num_q_heads, max_context_len, scale, 0, 0, sel, nsel, nthreads);
}

/* ---------------- prefill / extend over the paged cache ---------------- */

/* Several new tokens per sequence (a whole prompt, or one chunk of it under
 * chunked prefill: the FAQ's vLLM scheduler notes and the "vLLM" page's
 * prefill/decoding description).  Sequence s owns query tokens
 * query_start_loc[s] .. query_start_loc[s+1]-1 (q_len of them); they are the
 * newest q_len positions of its context, already written to the cache, so
 * query j sits at position ctx - q_len + j and attends (causally) positions
 * 0 .. ctx - q_len + j through the block table.  For each (token, query head):
 * gather, then contiguous attention over those positions.  out is
 * [total tokens][num_q_heads][D] doubles.  q_len <= 0 writes nothing; a
 * sequence with q_len > ctx or ctx beyond its table row gives zeros and
 * ORC_ERR_CONTEXT; a bad block id gives zeros and ORC_ERR_BLOCK_ID. */
int oracle_prefill(double* out, const uint16_t* q, int64_t q_token_stride, const uint16_t* layer,
                   const oracle_geom* g, const int32_t* block_tables, int32_t bt_stride,
                   const int32_t* context_lens, const int32_t* query_start_loc, int32_t num_seqs,
                   int32_t num_q_heads, double scale, int32_t nthreads) {
    const int32_t D = g->head_size;
    const int32_t G = num_q_heads / g->num_kv_heads;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int64_t it = 0; it < (int64_t)num_seqs * num_q_heads; ++it) {
        const int32_t s = (int32_t)(it / num_q_heads), h = (int32_t)(it % num_q_heads);
        const int32_t first = query_start_loc[s], q_len = query_start_loc[s + 1] - first;
        const int32_t ctx = context_lens[s];
        if (q_len <= 0) continue;
        for (int32_t j = 0; j < q_len; ++j)
            for (int32_t d = 0; d < D; ++d) out[((int64_t)(first + j) * num_q_heads + h) * D + d] = 0.0;
        if (q_len > ctx || (int64_t)ctx > (int64_t)bt_stride * g->block_size) {
            err |= ORC_ERR_CONTEXT;
            continue;
        }
        double* K = (double*)malloc(sizeof(double) * (size_t)ctx * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)ctx * D);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        const int e = oracle_gather(layer, g, block_tables + (int64_t)s * bt_stride, ctx, h / G, K, V);
        if (e) {
            err |= e;
        } else {
            for (int32_t j = 0; j < q_len; ++j) {
                const int64_t tok = first + j;
                for (int32_t d = 0; d < D; ++d)
                    qd[d] = elem_to_double(q[tok * q_token_stride + (int64_t)h * D + d], g->dtype);
                oracle_contiguous_attention(qd, K, V, ctx - q_len + j + 1, D, scale,
                                            out + (tok * num_q_heads + h) * D);
            }
        }
        free(K);
        free(V);
        free(qd);
    }
    return err;
}

/* ---------------- 8-bit KV cache ---------------- */

/* An 8-bit cache ("8bit KV Cache" quantisation, the TurboMind section of the
 * inference-framework FAQ page) stores each token's K and V vector of one kv
 * head as signed 8-bit codes with one scale: scale = max|x| / 127 and
 * code = round-half-even(x * (127 / max|x|)) clipped to [-127, 127], the
 * decision taken in IEEE binary32 (as the writer on the device does); the
 * value a code stands for is code * scale.
 * Chunk (block, kv head) of head_size 128: K codes [bs][128], V codes
 * [bs][128], K scales [bs] (fp32, padded to 16 bytes), V scales [bs] (same).
 * Inside a 128-byte code row of slot t, the 16 codes of dims 16c..16c+15 sit at
 * piece position c XOR (t mod 8), like the rows of the 16-bit cache. */
static int64_t i8_scale_bytes(int64_t bs) { return ((bs * 4 + 15) / 16) * 16; }
static int64_t i8_chunk_bytes(const oracle_geom* g) {
    return 2 * (int64_t)g->block_size * g->head_size + 2 * i8_scale_bytes(g->block_size);
}
int64_t oracle_i8_chunk_bytes(const oracle_geom* g) { return i8_chunk_bytes(g); }

/* Byte position of dim d inside the code row of slot t. */
static int64_t i8_pos(int64_t t, int64_t d) { return ((((d >> 4) ^ (t & 7)) << 4) | (d & 15)); }

static double i8_value(const uint8_t* layer, const oracle_geom* g, int64_t block, int64_t head, int part,
                       int64_t t, int64_t d) {
    const uint8_t* chunk = layer + (block * g->num_kv_heads + head) * i8_chunk_bytes(g);
    const int8_t code = (int8_t)chunk[(part * g->block_size + t) * g->head_size + i8_pos(t, d)];
    float scale;
    memcpy(&scale, chunk + 2 * g->block_size * g->head_size + part * i8_scale_bytes(g->block_size) + t * 4, 4);
    return (double)code * (double)scale;
}

/* Quantise one vector of n 16-bit elements; codes to out[0..n-1], returns the scale. */
static float i8_quantise(const uint16_t* x, int dtype, int64_t n, int8_t* out) {
    float amax = 0.0f;
    for (int64_t d = 0; d < n; ++d) {
        const float v = (float)fabs(elem_to_double(x[d], dtype));
        if (v > amax) amax = v;
    }
    if (!(amax > 0.0f)) {
        for (int64_t d = 0; d < n; ++d) out[d] = 0;
        return 0.0f;
    }
    const float inv = 127.0f / amax;
    for (int64_t d = 0; d < n; ++d) {
        float y = (float)elem_to_double(x[d], dtype) * inv;
        long c = lrintf(y);
        if (c > 127) c = 127;
        if (c < -127) c = -127;
        out[d] = (int8_t)c;
    }
    return amax / 127.0f;
}

int oracle_reshape_and_cache_i8(uint8_t* layer, const oracle_geom* g, const uint16_t* key, int64_t key_stride,
                                const uint16_t* value, int64_t value_stride, const int64_t* slot_mapping,
                                int32_t n) {
    int err = 0;
    const int64_t nslots = (int64_t)g->num_blocks * g->block_size;
    const int64_t D = g->head_size;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot == -1) continue;
        if (slot < 0 || slot >= nslots) { err |= ORC_ERR_SLOT; continue; }
        const int64_t block = slot / g->block_size, t = slot % g->block_size;
        for (int64_t h = 0; h < g->num_kv_heads; ++h)
            for (int part = 0; part < 2; ++part) {
                const uint16_t* src = (part ? value + i * value_stride : key + i * key_stride) + h * D;
                uint8_t* chunk = layer + (block * g->num_kv_heads + h) * i8_chunk_bytes(g);
                int8_t codes[128];
                const float scale = i8_quantise(src, g->dtype, D, codes);
                for (int64_t d = 0; d < D; ++d) chunk[(part * g->block_size + t) * D + i8_pos(t, d)] = (uint8_t)codes[d];
                memcpy(chunk + 2 * g->block_size * D + part * i8_scale_bytes(g->block_size) + t * 4, &scale, 4);
            }
    }
    return err;
}

/* The 8-bit decode with the same attended set as oracle_decode_window:
 * positions oracle_window_start(ctx, bs, window, ring) .. ctx - 1, logical
 * block j found at table entry j % ring when ring > 0. */
int oracle_decode_i8_window(double* out, const uint16_t* q, int64_t q_seq_stride, const uint8_t* layer,
                            const oracle_geom* g, const int32_t* block_tables, int32_t bt_stride,
                            const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                            int32_t max_context_len, double scale, int32_t window, int32_t ring, int32_t nthreads) {
    const int32_t D = g->head_size;
    const int32_t G = num_q_heads / g->num_kv_heads;
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int64_t it = 0; it < (int64_t)num_seqs * num_q_heads; ++it) {
        const int32_t s = (int32_t)(it / num_q_heads), h = (int32_t)(it % num_q_heads);
        double* o = out + it * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        const int32_t ctx = context_lens[s];
        if (ctx <= 0) continue;
        if ((ring <= 0 && (int64_t)ctx > (int64_t)bt_stride * g->block_size) || ctx > max_context_len) {
            err |= ORC_ERR_CONTEXT;
            continue;
        }
        const int32_t t0 = oracle_window_start(ctx, g->block_size, window, ring);
        const int32_t n = ctx - t0;
        double* K = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)n * D);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        int bad = 0;
        for (int32_t t = t0; t < ctx && !bad; ++t) {
            const int32_t j = t / g->block_size;
            const int32_t block = block_tables[(int64_t)s * bt_stride + (ring > 0 ? j % ring : j)];
            if (block < 0 || block >= g->num_blocks) { bad = 1; break; }
            for (int32_t d = 0; d < D; ++d) {
                K[(int64_t)(t - t0) * D + d] = i8_value(layer, g, block, h / G, 0, t % g->block_size, d);
                V[(int64_t)(t - t0) * D + d] = i8_value(layer, g, block, h / G, 1, t % g->block_size, d);
            }
        }
        if (bad) {
            err |= ORC_ERR_BLOCK_ID;
        } else {
            for (int32_t d = 0; d < D; ++d)
                qd[d] = elem_to_double(q[(int64_t)s * q_seq_stride + (int64_t)h * D + d], g->dtype);
            oracle_contiguous_attention(qd, K, V, n, D, scale, o);
        }
        free(K);
        free(V);
        free(qd);
    }
    return err;
}

int oracle_decode_i8(double* out, const uint16_t* q, int64_t q_seq_stride, const uint8_t* layer,
                     const oracle_geom* g, const int32_t* block_tables, int32_t bt_stride,
                     const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                     double scale, int32_t nthreads) {
    return oracle_decode_i8_window(out, q, q_seq_stride, layer, g, block_tables, bt_stride, context_lens, num_seqs,
                                   num_q_heads, max_context_len, scale, 0, 0, nthreads);
}

int oracle_copy_blocks_bytes(uint8_t* pool, int64_t block_bytes, int32_t num_blocks, int32_t num_layers,
                             int64_t layer_stride, const int64_t* pairs, int32_t n) {
    for (int32_t i = 0; i < n; ++i)
        for (int k = 0; k < 2; ++k)
            if (pairs[2 * i + k] < 0 || pairs[2 * i + k] >= num_blocks) return ORC_ERR_BLOCK_ID;
    uint8_t* tmp = (uint8_t*)malloc((size_t)(block_bytes * (n > 0 ? n : 1)));
    for (int32_t l = 0; l < num_layers; ++l) {
        uint8_t* layer = pool + (int64_t)l * layer_stride;
        for (int32_t i = 0; i < n; ++i)
            memcpy(tmp + (int64_t)i * block_bytes, layer + pairs[2 * i] * block_bytes, (size_t)block_bytes);
        for (int32_t i = 0; i < n; ++i)
            memcpy(layer + pairs[2 * i + 1] * block_bytes, tmp + (int64_t)i * block_bytes, (size_t)block_bytes);
    }
    free(tmp);
    return 0;
}

/* ---------------- split-context partitions and log-sum-exp merge ---------------- */

/* For one (s, h): split tokens into consecutive partitions of P tokens.  For
 * partition p: m_p = max score, l_p = sum exp(z - m_p), o_p = sum exp(z - m_p) v
 * (unnormalised).  Writes n_part = ceil(ctx / P) entries of m[], l[], o[][D].
 * Returns n_part (0 when ctx <= 0), or -1 on a bad block id. */
int oracle_partition_stats(const uint16_t* q_row, const uint16_t* layer, const oracle_geom* g,
                           const int32_t* table_row, int32_t ctx, int32_t kv_head, double scale,
                           int32_t P, double* m, double* l, double* o) {
    const int32_t D = g->head_size;
    if (ctx <= 0) return 0;
    double* K = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)ctx * D);
    if (oracle_gather(layer, g, table_row, ctx, kv_head, K, V)) {
        free(K);
        free(V);
        return -1;
    }
    const int32_t n_part = (ctx + P - 1) / P;
    for (int32_t p = 0; p < n_part; ++p) {
        const int32_t t0 = p * P, t1 = (t0 + P < ctx) ? t0 + P : ctx;
        double mp = -INFINITY;
        for (int32_t t = t0; t < t1; ++t) {
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += elem_to_double(q_row[d], g->dtype) * K[(int64_t)t * D + d];
            if (scale * dot > mp) mp = scale * dot;
        }
        double lp = 0.0;
        for (int32_t d = 0; d < D; ++d) o[(int64_t)p * D + d] = 0.0;
        for (int32_t t = t0; t < t1; ++t) {
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += elem_to_double(q_row[d], g->dtype) * K[(int64_t)t * D + d];
            const double w = exp(scale * dot - mp);
            lp += w;
            for (int32_t d = 0; d < D; ++d) o[(int64_t)p * D + d] += w * V[(int64_t)t * D + d];
        }
        m[p] = mp;
        l[p] = lp;
    }
    free(K);
    free(V);
    return n_part;
}

/* Merge partition statistics: M = max m_p;
 * out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p. */
void oracle_merge_partitions(const double* m, const double* l, const double* o, int32_t n_part,
                             int32_t D, double* out) {
    for (int32_t d = 0; d < D; ++d) out[d] = 0.0;
    if (n_part <= 0) return;
    double M = -INFINITY;
    for (int32_t p = 0; p < n_part; ++p)
        if (m[p] > M) M = m[p];
    double denom = 0.0;
    for (int32_t p = 0; p < n_part; ++p) {
        const double w = exp(m[p] - M);
        denom += w * l[p];
        for (int32_t d = 0; d < D; ++d) out[d] += w * o[(int64_t)p * D + d];
    }
    for (int32_t d = 0; d < D; ++d) out[d] /= denom;
}

/* ---------------- copy_blocks and swap_blocks ---------------- */

/* Copy whole blocks (every kv head, K and V, every layer) for each (src, dst)
 * pair.  All pairs act at once: every source is read before any destination is
 * written.  pairs is [n][2] (src, dst).  Returns ORC_ERR_BLOCK_ID on an
 * out-of-range id (and copies nothing). */
int oracle_copy_blocks(uint16_t* pool, const oracle_geom* g, const int64_t* pairs, int32_t n) {
    const int64_t block_elems = (int64_t)g->num_kv_heads * chunk_elems(g);
    for (int32_t i = 0; i < n; ++i)
        for (int k = 0; k < 2; ++k)
            if (pairs[2 * i + k] < 0 || pairs[2 * i + k] >= g->num_blocks) return ORC_ERR_BLOCK_ID;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(block_elems * (n > 0 ? n : 1)));
    for (int32_t l = 0; l < g->num_layers; ++l) {
        uint16_t* layer = pool + (int64_t)l * g->layer_stride;
        for (int32_t i = 0; i < n; ++i)
            memcpy(tmp + (int64_t)i * block_elems, layer + pairs[2 * i] * block_elems,
                   sizeof(uint16_t) * (size_t)block_elems);
        for (int32_t i = 0; i < n; ++i)
            memcpy(layer + pairs[2 * i + 1] * block_elems, tmp + (int64_t)i * block_elems,
                   sizeof(uint16_t) * (size_t)block_elems);
    }
    free(tmp);
    return 0;
}

/* Move whole blocks from one pool to another (GPU cache <-> pinned CPU cache):
 * dst block pairs[i][1] of every layer receives src block pairs[i][0].  The two
 * pools share geometry except num_blocks and layer stride. */
int oracle_swap_blocks(uint16_t* dst, const oracle_geom* gd, const uint16_t* src,
                       const oracle_geom* gs, const int64_t* pairs, int32_t n) {
    const int64_t block_elems = (int64_t)gs->num_kv_heads * chunk_elems(gs);
    for (int32_t i = 0; i < n; ++i)
        if (pairs[2 * i] < 0 || pairs[2 * i] >= gs->num_blocks || pairs[2 * i + 1] < 0 ||
            pairs[2 * i + 1] >= gd->num_blocks)
            return ORC_ERR_BLOCK_ID;
    for (int32_t l = 0; l < gs->num_layers; ++l)
        for (int32_t i = 0; i < n; ++i)
            memcpy(dst + (int64_t)l * gd->layer_stride + pairs[2 * i + 1] * block_elems,
                   src + (int64_t)l * gs->layer_stride + pairs[2 * i] * block_elems,
                   sizeof(uint16_t) * (size_t)block_elems);
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
