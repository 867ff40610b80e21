// block_manager.cpp -- host-side block manager: the logical -> physical block
// bookkeeping that produces the block tables, slot numbers, copy-on-write pairs
// and swap pairs the device kernels consume.
//
// Restates the vLLM block manager as the pages describe it ("推理框架知识点",
// vLLM BlockSpaceManagerV1 / UncachedBlockAllocator / CachedBlockAllocator /
// LRUEvictor; mlqm.cn article, Copy-on-Write example; nano-vLLM article §5.2.1,
// chain-hashed prefix blocks):
//   * can_allocate: NEVER when even an empty pool could not hold the prompt
//     above the watermark, LATER when the free blocks cannot now, else OK;
//   * allocation: one block per logical block of the prompt; with a sliding
//     window of W tokens, logical block i >= ceil(W / bs) reuses table entry
//     i % ceil(W / bs); with prefix caching, a full block is identified by the
//     hash of (previous block's hash, its token ids) and shared when a cached
//     block with that hash and those token ids exists;
//   * append_slot: a new block when the table is one short (sliding: reuse),
//     then copy-on-write if the last block is shared (reference count > 1);
//   * fork: the child shares every block of the parent (reference counts + 1);
//   * free: reference counts - 1; unreferenced hashed blocks go to the evictor,
//     which gives back the least recently used one (ties: more hashed tokens);
//   * swap out / in: every block of the sequences moves to the other pool, a
//     block shared by several of them once.
// Free blocks are handed out last-freed first (a stack), starting from the
// highest id.  Not thread-safe: one caller at a time per manager.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace pkv {
void set_last_error(const char* msg);
}

namespace {

struct Block {
  int32_t ref = 0;
  bool hashed = false;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;      // token ids of a hashed block (guards against hash collisions)
  int64_t last_access = 0;
  int32_t num_hashed_tokens = 0;
  int64_t evict_order = 0;          // insertion order into the evictor (final tie-break)
  bool evictable = false;
};

struct Pool {
  std::vector<Block> blocks;
  std::vector<int32_t> free_stack;  // back() is handed out next
  std::unordered_multimap<uint64_t, int32_t> by_hash;
  int32_t n_evictable = 0;

  explicit Pool(int32_t n) : blocks(n) {
    free_stack.reserve(n);
    for (int32_t i = 0; i < n; ++i) free_stack.push_back(i);
  }
  int32_t total() const { return (int32_t)blocks.size(); }
  int32_t num_free() const { return (int32_t)free_stack.size() + n_evictable; }

  void unhash(int32_t id) {
    Block& b = blocks[id];
    if (!b.hashed) return;
    auto range = by_hash.equal_range(b.hash);
    for (auto it = range.first; it != range.second; ++it)
      if (it->second == id) {
        by_hash.erase(it);
        break;
      }
    b.hashed = false;
    b.tokens.clear();
    b.num_hashed_tokens = 0;
  }

  // A block with no content identity: the free stack first, else evict.
  int32_t take_fresh() {
    int32_t id = -1;
    if (!free_stack.empty()) {
      id = free_stack.back();
      free_stack.pop_back();
    } else if (n_evictable > 0) {
      for (int32_t i = 0; i < total(); ++i) {
        const Block& b = blocks[i];
        if (!b.evictable) continue;
        if (id < 0) {
          id = i;
          continue;
        }
        const Block& e = blocks[id];
        if (b.last_access < e.last_access ||
            (b.last_access == e.last_access &&
             (b.num_hashed_tokens > e.num_hashed_tokens ||
              (b.num_hashed_tokens == e.num_hashed_tokens && b.evict_order < e.evict_order))))
          id = i;
      }
      blocks[id].evictable = false;
      --n_evictable;
      unhash(id);
    }
    if (id >= 0) blocks[id].ref = 1;
    return id;
  }

  int32_t find_cached(uint64_t hash, const int32_t* tokens, int32_t n) const {
    auto range = by_hash.equal_range(hash);
    for (auto it = range.first; it != range.second; ++it) {
      const Block& b = blocks[it->second];
      if ((int32_t)b.tokens.size() == n && std::equal(b.tokens.begin(), b.tokens.end(), tokens)) return it->second;
    }
    return -1;
  }

  void release(int32_t id, int64_t now, int64_t* order) {
    Block& b = blocks[id];
    if (b.ref <= 0) return;   // already free
    if (--b.ref > 0) return;
    if (b.hashed) {
      b.evictable = true;
      b.last_access = now;
      b.evict_order = (*order)++;
      ++n_evictable;
    } else {
      free_stack.push_back(id);
    }
  }
};

// 64-bit FNV-1a over (previous hash, token ids).
uint64_t chain_hash(uint64_t prev, const int32_t* tokens, int32_t n) {
  uint64_t h = 1469598103934665603ull;
  auto mix = [&h](const void* p, size_t len) {
    const unsigned char* c = static_cast<const unsigned char*>(p);
    for (size_t i = 0; i < len; ++i) {
      h ^= c[i];
      h *= 1099511628211ull;
    }
  };
  mix(&prev, sizeof prev);
  mix(tokens, sizeof(int32_t) * (size_t)n);
  return h;
}

struct Seq {
  std::vector<int32_t> table;       // physical block per logical block
  std::vector<int32_t> tokens;      // every token id (prefix hashes)
  std::vector<uint64_t> hashes;     // chain hash of each full block
  bool swapped = false;             // table holds host-pool ids
};

std::vector<int32_t> unique_blocks(const std::vector<int32_t>& table) {
  std::vector<int32_t> u(table);
  std::sort(u.begin(), u.end());
  u.erase(std::unique(u.begin(), u.end()), u.end());
  return u;
}

pa_status bm_fail(pa_status st, const char* msg) {
  pkv::set_last_error(msg);
  return st;
}

}  // namespace

struct pa_block_manager {
  int32_t bs;
  int32_t window_blocks;            // ceil(window / bs), 0 without a sliding window
  bool caching;
  int32_t watermark_blocks;
  Pool gpu, cpu;
  std::map<int64_t, Seq> seqs;
  int64_t clock = 0;
  int64_t evict_order = 0;

  pa_block_manager(int32_t bs_, int32_t ngpu, int32_t ncpu, float watermark, int32_t window, bool caching_)
      : bs(bs_), window_blocks(window > 0 ? (window + bs_ - 1) / bs_ : 0), caching(caching_),
        watermark_blocks((int32_t)(watermark * ngpu)), gpu(ngpu), cpu(ncpu) {}

  Seq* find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }

  // Allocate the block for logical block i of s (whose tokens are already in s->tokens).
  int32_t alloc_logical(Seq* s, int32_t i) {
    if (window_blocks > 0 && i >= window_blocks) return s->table[i % window_blocks];
    const int32_t ntok = (int32_t)s->tokens.size();
    if (caching && (i + 1) * bs <= ntok) {
      const uint64_t prev = i > 0 ? s->hashes[i - 1] : 0;
      const uint64_t h = chain_hash(prev, s->tokens.data() + (int64_t)i * bs, bs);
      s->hashes.push_back(h);
      const int32_t hit = gpu.find_cached(h, s->tokens.data() + (int64_t)i * bs, bs);
      if (hit >= 0) {
        Block& b = gpu.blocks[hit];
        if (b.evictable) {
          b.evictable = false;
          --gpu.n_evictable;
        }
        ++b.ref;
        b.last_access = ++clock;
        return hit;
      }
      const int32_t id = gpu.take_fresh();
      if (id >= 0) register_hash(id, h, s->tokens.data() + (int64_t)i * bs, (i + 1) * bs);
      return id;
    }
    return gpu.take_fresh();
  }

  void register_hash(int32_t id, uint64_t h, const int32_t* tokens, int32_t num_hashed) {
    Block& b = gpu.blocks[id];
    b.hashed = true;
    b.hash = h;
    b.tokens.assign(tokens, tokens + bs);
    b.num_hashed_tokens = num_hashed;
    b.last_access = ++clock;
    gpu.by_hash.emplace(h, id);
  }

  void release_table(const std::vector<int32_t>& table, bool on_cpu) {
    for (int32_t b : unique_blocks(table)) (on_cpu ? cpu : gpu).release(b, ++clock, &evict_order);
  }
};

extern "C" {

pa_status pa_bm_create(int32_t block_size, int32_t num_gpu_blocks, int32_t num_cpu_blocks, float watermark,
                       int32_t sliding_window, int32_t enable_prefix_caching, pa_block_manager** out) {
  if (!out) return bm_fail(PA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (block_size <= 0 || num_gpu_blocks <= 0 || num_cpu_blocks < 0 || !(watermark >= 0.f) || sliding_window < 0)
    return bm_fail(PA_ERR_INVALID_ARG, "block_size and num_gpu_blocks must be > 0; watermark, window, cpu >= 0");
  if (enable_prefix_caching && sliding_window > 0)
    return bm_fail(PA_ERR_UNSUPPORTED, "prefix caching with a sliding window is not supported");
  pa_block_manager* bm =
      new (std::nothrow) pa_block_manager(block_size, num_gpu_blocks, num_cpu_blocks, watermark, sliding_window,
                                          enable_prefix_caching != 0);
  if (!bm) return bm_fail(PA_ERR_INVALID_ARG, "out of host memory");
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_can_allocate(pa_block_manager* bm, int32_t num_tokens) {
  int32_t need = (num_tokens + bm->bs - 1) / bm->bs;
  if (bm->window_blocks > 0) need = std::min(need, bm->window_blocks);
  if (bm->gpu.total() - need < bm->watermark_blocks) return PA_ALLOC_NEVER;
  if (bm->gpu.num_free() - need >= bm->watermark_blocks) return PA_ALLOC_OK;
  return PA_ALLOC_LATER;
}

pa_status pa_bm_allocate(pa_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t num_tokens) {
  if (num_tokens <= 0 || !token_ids) return bm_fail(PA_ERR_INVALID_ARG, "a prompt needs at least one token");
  if (bm->find(seq_id)) return bm_fail(PA_ERR_INVALID_ARG, "sequence id already allocated");
  Seq s;
  s.tokens.assign(token_ids, token_ids + num_tokens);
  const int32_t nblk = (num_tokens + bm->bs - 1) / bm->bs;
  for (int32_t i = 0; i < nblk; ++i) {
    const int32_t id = bm->alloc_logical(&s, i);
    if (id < 0) {
      bm->release_table(s.table, false);
      return bm_fail(PA_ERR_OUT_OF_BLOCKS, "no free device blocks for the prompt");
    }
    s.table.push_back(id);
  }
  bm->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

pa_status pa_bm_append_slot(pa_block_manager* bm, int64_t seq_id, int32_t token_id, int64_t* slot, int64_t* cow_src,
                            int64_t* cow_dst) {
  Seq* s = bm->find(seq_id);
  if (!s || s->swapped) return bm_fail(PA_ERR_INVALID_ARG, "unknown or swapped-out sequence");
  if (!slot || !cow_src || !cow_dst) return bm_fail(PA_ERR_INVALID_ARG, "output pointers must be non-NULL");
  *cow_src = *cow_dst = -1;
  const int32_t n = (int32_t)s->tokens.size() + 1;
  const int32_t need = (n + bm->bs - 1) / bm->bs;
  if ((int32_t)s->table.size() < need) {
    int32_t id;
    if (bm->window_blocks > 0 && (int32_t)s->table.size() >= bm->window_blocks) {
      id = s->table[s->table.size() % bm->window_blocks];
    } else {
      id = bm->gpu.take_fresh();
      if (id < 0) return bm_fail(PA_ERR_OUT_OF_BLOCKS, "no free device block to append");
    }
    s->table.push_back(id);
  } else {
    const int32_t last = s->table.back();
    if (bm->gpu.blocks[last].ref > 1) {   // shared: copy on write
      const int32_t id = bm->gpu.take_fresh();
      if (id < 0) return bm_fail(PA_ERR_OUT_OF_BLOCKS, "no free device block for copy-on-write");
      s->table.back() = id;
      bm->gpu.release(last, ++bm->clock, &bm->evict_order);
      *cow_src = last;
      *cow_dst = id;
    }
  }
  s->tokens.push_back(token_id);
  const int32_t last = s->table.back();
  *slot = (int64_t)last * bm->bs + (n - 1) % bm->bs;
  // a block that just became full gets its chain hash; a private one is
  // registered for prefix reuse
  if (bm->caching && n % bm->bs == 0) {
    const int32_t i = n / bm->bs - 1;
    const uint64_t prev = i > 0 ? s->hashes[i - 1] : 0;
    const uint64_t h = chain_hash(prev, s->tokens.data() + (int64_t)i * bm->bs, bm->bs);
    s->hashes.resize(i);
    s->hashes.push_back(h);
    const int32_t* blk_tokens = s->tokens.data() + (int64_t)i * bm->bs;
    if (!bm->gpu.blocks[last].hashed && bm->gpu.blocks[last].ref == 1 && bm->gpu.find_cached(h, blk_tokens, bm->bs) < 0)
      bm->register_hash(last, h, blk_tokens, n);
  }
  return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  Seq* parent = bm->find(parent_id);
  if (!parent || parent->swapped) return bm_fail(PA_ERR_INVALID_ARG, "unknown or swapped-out parent");
  if (bm->find(child_id)) return bm_fail(PA_ERR_INVALID_ARG, "child id already in use");
  Seq child = *parent;
  for (int32_t b : unique_blocks(child.table)) ++bm->gpu.blocks[b].ref;
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

pa_status pa_bm_free(pa_block_manager* bm, int64_t seq_id) {
  Seq* s = bm->find(seq_id);
  if (!s) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence");
  bm->release_table(s->table, s->swapped);
  bm->seqs.erase(seq_id);
  return PA_OK;
}

pa_status pa_bm_block_table(pa_block_manager* bm, int64_t seq_id, int32_t* table, int32_t capacity,
                            int32_t* num_blocks, int32_t* num_tokens) {
  Seq* s = bm->find(seq_id);
  if (!s) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence");
  if (num_blocks) *num_blocks = (int32_t)s->table.size();
  if (num_tokens) *num_tokens = (int32_t)s->tokens.size();
  if (table) {
    if (capacity < (int32_t)s->table.size()) return bm_fail(PA_ERR_INVALID_ARG, "table capacity too small");
    std::copy(s->table.begin(), s->table.end(), table);
  }
  return PA_OK;
}

static pa_status bm_swap(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs, int32_t capacity,
                         int32_t* num_pairs, bool out) {
  if (!num_pairs || (n > 0 && !seq_ids)) return bm_fail(PA_ERR_INVALID_ARG, "NULL argument");
  Pool& src = out ? bm->gpu : bm->cpu;
  Pool& dst = out ? bm->cpu : bm->gpu;
  std::set<int32_t> need;
  for (int32_t i = 0; i < n; ++i) {
    Seq* s = bm->find(seq_ids[i]);
    if (!s || s->swapped != !out) return bm_fail(PA_ERR_INVALID_ARG, "unknown sequence or wrong side");
    for (int32_t b : s->table) need.insert(b);
  }
  if (!pairs) {   // count only; nothing moves
    *num_pairs = (int32_t)need.size();
    return PA_OK;
  }
  if ((int32_t)dst.free_stack.size() + dst.n_evictable < (int32_t)need.size())
    return bm_fail(PA_ERR_OUT_OF_BLOCKS, "not enough free blocks on the destination side");
  if (capacity < (int32_t)need.size()) return bm_fail(PA_ERR_INVALID_ARG, "pair capacity too small");
  std::map<int32_t, int32_t> mapping;
  for (int32_t i = 0; i < n; ++i) {
    Seq* s = bm->find(seq_ids[i]);
    for (int32_t b : unique_blocks(s->table)) {
      auto it = mapping.find(b);
      if (it != mapping.end()) {
        ++dst.blocks[it->second].ref;
      } else {
        mapping[b] = dst.take_fresh();
      }
      src.release(b, ++bm->clock, &bm->evict_order);
    }
    for (int32_t& b : s->table) b = mapping[b];
    s->swapped = out;
  }
  int32_t k = 0;
  for (const auto& m : mapping) {
    pairs[2 * k] = m.first;
    pairs[2 * k + 1] = m.second;
    ++k;
  }
  *num_pairs = k;
  return PA_OK;
}

// Distinct blocks of the n sequences, all on the side given (-1: an unknown
// sequence, or one on the other side).
static int32_t bm_distinct_blocks(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, bool swapped) {
  if (n < 0 || (n > 0 && !seq_ids)) {
    bm_fail(PA_ERR_INVALID_ARG, "NULL argument");
    return -1;
  }
  std::set<int32_t> need;
  for (int32_t i = 0; i < n; ++i) {
    Seq* s = bm->find(seq_ids[i]);
    if (!s || s->swapped != swapped) {
      bm_fail(PA_ERR_INVALID_ARG, "unknown sequence or wrong side");
      return -1;
    }
    need.insert(s->table.begin(), s->table.end());
  }
  return (int32_t)need.size();
}

int32_t pa_bm_can_append_slots(pa_block_manager* bm, int32_t num_running) {
  // each running sequence may need one new block (or a copy of a shared last block)
  return num_running >= 0 && num_running <= bm->gpu.num_free() ? 1 : 0;
}

int32_t pa_bm_can_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n) {
  const int32_t need = bm_distinct_blocks(bm, seq_ids, n, true);
  if (need < 0) return -1;
  if (bm->gpu.total() - need < bm->watermark_blocks) return PA_ALLOC_NEVER;
  if (bm->gpu.num_free() - need >= bm->watermark_blocks) return PA_ALLOC_OK;
  return PA_ALLOC_LATER;
}

int32_t pa_bm_can_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n) {
  const int32_t need = bm_distinct_blocks(bm, seq_ids, n, false);
  if (need < 0) return -1;
  return need <= bm->cpu.num_free() ? 1 : 0;
}

pa_status pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs, int32_t capacity,
                         int32_t* num_pairs) {
  return bm_swap(bm, seq_ids, n, pairs, capacity, num_pairs, true);
}

pa_status pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs, int32_t capacity,
                        int32_t* num_pairs) {
  return bm_swap(bm, seq_ids, n, pairs, capacity, num_pairs, false);
}

int32_t pa_bm_num_free_blocks(pa_block_manager* bm, int32_t on_host) {
  return on_host ? bm->cpu.num_free() : bm->gpu.num_free();
}

int32_t pa_bm_ref_count(pa_block_manager* bm, int32_t on_host, int32_t block) {
  Pool& pool = on_host ? bm->cpu : bm->gpu;
  if (block < 0 || block >= pool.total()) return -1;
  return pool.blocks[block].ref;
}

}  // extern "C"
