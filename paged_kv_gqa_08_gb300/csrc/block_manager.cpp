// Host-side manager of the paged KV cache's blocks: which physical page each
// sequence's tokens live in, which pages are free, and which full pages hold
// a prefix that a new sequence can reuse.
//
// Semantics follow the nano-vLLM learning note (Block, BlockManager,
// compute_hash, can_allocate, allocate, deallocate, can_append, may_append
// and hash_blocks listings):
//   * a block has a reference count, and, once full and computed, a hash of
//     its tokens chained with the previous block's hash, plus the tokens;
//   * free blocks form a FIFO: allocation takes the oldest free block and a
//     released block goes to the back, so a released block keeps its hash
//     (and can be hit by a later prefix) for as long as possible;
//   * a new sequence walks its full blocks except the last one, hashing as it
//     goes, and stops at the first block whose hash is unknown or whose
//     stored tokens differ; the blocks before that are shared (reference
//     count + 1, or taken back from the free list when nobody holds them);
//   * a sequence that grows into a new block (length % block_size == 1) gets
//     a fresh block; releasing a sequence drops one reference per block, last
//     block first.
// What differs from the listings: the hash is a chained SplitMix64 mix of
// 32-bit token ids instead of xxHash64 (a hit is confirmed by comparing the
// stored tokens either way, so the hash only has to spread keys), a reused
// block's stale hash entry is erased when the block is handed out again, and
// the free list is an intrusive doubly-linked list so that taking a cached
// block back from the middle of it is O(1).
//
// Not thread-safe: one manager belongs to one scheduler thread.
#include <stdint.h>
#include <string.h>

#include <new>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

namespace {

// SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014).
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

constexpr uint64_t kHashSeed = 0x9e3779b97f4a7c15ull;

uint64_t chain_hash(bool has_prev, uint64_t prev, const int32_t* tokens, int32_t n) {
  uint64_t h = has_prev ? mix64(kHashSeed ^ prev) : kHashSeed;
  for (int32_t i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tokens[i]));
  return h;
}

struct Block {
  int32_t ref = 0;
  bool hashed = false;
  uint64_t hash = 0;
  std::vector<int32_t> tokens;  // the block's tokens once hashed
  int32_t prev = -1, next = -1; // free-list links
  bool is_free = true;
};

struct Seq {
  std::vector<int32_t> tokens;
  std::vector<int32_t> table;
  int64_t cached_tokens = 0;  // tokens whose KV came from shared blocks at allocation
  int64_t hashed_blocks = 0;  // leading blocks already registered in the hash table
};

}  // namespace

struct pa_block_manager {
  int32_t P = 0;
  std::vector<Block> blocks;
  int32_t head = -1, tail = -1;  // free list: head = oldest
  int64_t n_free = 0;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Seq> seqs;

  void push_free(int32_t id) {
    Block& b = blocks[id];
    b.is_free = true;
    b.prev = tail;
    b.next = -1;
    if (tail >= 0) blocks[tail].next = id;
    else head = id;
    tail = id;
    ++n_free;
  }

  void unlink_free(int32_t id) {
    Block& b = blocks[id];
    if (b.prev >= 0) blocks[b.prev].next = b.next;
    else head = b.next;
    if (b.next >= 0) blocks[b.next].prev = b.prev;
    else tail = b.prev;
    b.prev = b.next = -1;
    b.is_free = false;
    --n_free;
  }

  // The oldest free block, emptied: reference count 1, no hash.
  int32_t take_fresh() {
    const int32_t id = head;
    unlink_free(id);
    Block& b = blocks[id];
    if (b.hashed) {
      auto it = by_hash.find(b.hash);
      if (it != by_hash.end() && it->second == id) by_hash.erase(it);
    }
    b.hashed = false;
    b.tokens.clear();
    b.ref = 1;
    return id;
  }

  // The registered block holding exactly these tokens after this prefix, or -1.
  int32_t lookup(bool has_prev, uint64_t prev, const int32_t* tok, uint64_t* h_out) const {
    const uint64_t h = chain_hash(has_prev, prev, tok, P);
    *h_out = h;
    auto it = by_hash.find(h);
    if (it == by_hash.end()) return -1;
    const Block& b = blocks[it->second];
    if (!b.hashed || b.hash != h || static_cast<int32_t>(b.tokens.size()) != P ||
        memcmp(b.tokens.data(), tok, sizeof(int32_t) * P) != 0)
      return -1;
    return it->second;
  }

  // Leading full blocks (never the last block) reusable from the cache, and
  // how many fresh blocks the sequence needs on top of them.
  void plan(const int32_t* tok, int64_t n, int64_t* cached, int64_t* fresh, std::vector<int32_t>* ids) const {
    const int64_t nb = (n + P - 1) / P;
    int64_t hits = 0, need = nb;
    bool has_prev = false;
    uint64_t prev = 0;
    for (int64_t i = 0; i + 1 < nb; ++i) {
      uint64_t h;
      const int32_t id = lookup(has_prev, prev, tok + i * P, &h);
      if (id < 0) break;
      if (ids) ids->push_back(id);
      ++hits;
      if (!blocks[id].is_free) --need;  // held by another sequence: no new space
      has_prev = true;
      prev = h;
    }
    *cached = hits;
    *fresh = need;
  }
};

namespace {

pa_status guard(pa_block_manager* m) { return m ? PA_OK : PA_ERR_NULL; }

Seq* find_seq(pa_block_manager* m, int64_t id) {
  auto it = m->seqs.find(id);
  return it == m->seqs.end() ? nullptr : &it->second;
}

}  // namespace

extern "C" {

PA_API pa_status pa_bm_create(int64_t num_blocks, int32_t block_size, pa_block_manager** out) {
  if (!out) return PA_ERR_NULL;
  *out = nullptr;
  if (num_blocks < 1 || num_blocks > 0x7fffffff || block_size < 1) return PA_ERR_SHAPE;
  pa_block_manager* m = new (std::nothrow) pa_block_manager();
  if (!m) return PA_ERR_CAPACITY;
  try {
    m->P = block_size;
    m->blocks.resize(static_cast<size_t>(num_blocks));
    for (int32_t i = 0; i < static_cast<int32_t>(num_blocks); ++i) m->push_free(i);
  } catch (...) {
    delete m;
    return PA_ERR_CAPACITY;
  }
  *out = m;
  return PA_OK;
}

PA_API void pa_bm_destroy(pa_block_manager* m) { delete m; }

PA_API pa_status pa_bm_can_allocate(pa_block_manager* m, const int32_t* token_ids, int64_t num_tokens,
                                    int64_t* num_cached_blocks) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (!num_cached_blocks || (!token_ids && num_tokens > 0)) return PA_ERR_NULL;
  if (num_tokens < 1) return PA_ERR_SHAPE;
  int64_t cached, fresh;
  m->plan(token_ids, num_tokens, &cached, &fresh, nullptr);
  *num_cached_blocks = m->n_free < fresh ? -1 : cached;
  return PA_OK;
}

PA_API pa_status pa_bm_allocate(pa_block_manager* m, int64_t seq_id, const int32_t* token_ids, int64_t num_tokens,
                                int64_t* num_cached_tokens) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (!token_ids) return PA_ERR_NULL;
  if (num_tokens < 1) return PA_ERR_SHAPE;
  if (m->seqs.count(seq_id)) return PA_ERR_SHAPE;
  try {
    std::vector<int32_t> hit_ids;
    int64_t cached, fresh;
    m->plan(token_ids, num_tokens, &cached, &fresh, &hit_ids);
    if (m->n_free < fresh) return PA_ERR_CAPACITY;
    Seq s;
    s.tokens.assign(token_ids, token_ids + num_tokens);
    const int64_t nb = (num_tokens + m->P - 1) / m->P;
    s.table.reserve(static_cast<size_t>(nb));
    for (int32_t id : hit_ids) {
      Block& b = m->blocks[id];
      if (b.is_free) {
        m->unlink_free(id);
        b.ref = 1;
      } else {
        ++b.ref;
      }
      s.table.push_back(id);
    }
    for (int64_t i = cached; i < nb; ++i) s.table.push_back(m->take_fresh());
    s.cached_tokens = cached * m->P;
    s.hashed_blocks = cached;
    m->seqs.emplace(seq_id, std::move(s));
    if (num_cached_tokens) *num_cached_tokens = cached * m->P;
  } catch (...) {
    return PA_ERR_CAPACITY;
  }
  return PA_OK;
}

PA_API pa_status pa_bm_append_token(pa_block_manager* m, int64_t seq_id, int32_t token_id) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  Seq* s = find_seq(m, seq_id);
  if (!s) return PA_ERR_SHAPE;
  const bool new_block = s->tokens.size() % static_cast<size_t>(m->P) == 0;  // length % P == 1 after the push
  if (new_block && m->n_free < 1) return PA_ERR_CAPACITY;
  try {
    s->tokens.push_back(token_id);
    if (new_block) s->table.push_back(m->take_fresh());
  } catch (...) {
    return PA_ERR_CAPACITY;
  }
  return PA_OK;
}

PA_API pa_status pa_bm_hash_blocks(pa_block_manager* m, int64_t seq_id, int64_t num_computed_tokens) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  Seq* s = find_seq(m, seq_id);
  if (!s) return PA_ERR_SHAPE;
  if (num_computed_tokens < 0 || num_computed_tokens > static_cast<int64_t>(s->tokens.size())) return PA_ERR_SHAPE;
  const int64_t end = num_computed_tokens / m->P;
  try {
    for (int64_t i = s->hashed_blocks; i < end; ++i) {
      Block& b = m->blocks[s->table[i]];
      const bool has_prev = i > 0;
      const uint64_t prev = has_prev ? m->blocks[s->table[i - 1]].hash : 0;
      const int32_t* tok = s->tokens.data() + i * m->P;
      b.hash = chain_hash(has_prev, prev, tok, m->P);
      b.hashed = true;
      b.tokens.assign(tok, tok + m->P);
      m->by_hash[b.hash] = s->table[i];
    }
  } catch (...) {
    return PA_ERR_CAPACITY;
  }
  if (end > s->hashed_blocks) s->hashed_blocks = end;
  return PA_OK;
}

PA_API pa_status pa_bm_free(pa_block_manager* m, int64_t seq_id) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return PA_ERR_SHAPE;
  const std::vector<int32_t>& t = it->second.table;
  for (auto r = t.rbegin(); r != t.rend(); ++r) {
    Block& b = m->blocks[*r];
    if (--b.ref == 0) m->push_free(*r);
  }
  m->seqs.erase(it);
  return PA_OK;
}

PA_API pa_status pa_bm_block_tables(pa_block_manager* m, const int64_t* seq_ids, int32_t num_seqs,
                                    int32_t max_pages_per_seq, int32_t pad_page, int32_t* block_tables,
                                    int32_t* context_lens) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || max_pages_per_seq < 1) return PA_ERR_SHAPE;
  if (num_seqs > 0 && (!seq_ids || !block_tables)) return PA_ERR_NULL;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Seq* s = find_seq(m, seq_ids[i]);
    if (!s) return PA_ERR_SHAPE;
    if (static_cast<int64_t>(s->table.size()) > max_pages_per_seq) return PA_ERR_SHAPE;
  }
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Seq* s = find_seq(m, seq_ids[i]);
    int32_t* row = block_tables + static_cast<int64_t>(i) * max_pages_per_seq;
    const int32_t nt = static_cast<int32_t>(s->table.size());
    for (int32_t j = 0; j < max_pages_per_seq; ++j) row[j] = j < nt ? s->table[j] : pad_page;
    if (context_lens) context_lens[i] = static_cast<int32_t>(s->tokens.size());
  }
  return PA_OK;
}

PA_API pa_status pa_bm_slot_mapping(pa_block_manager* m, const int64_t* seq_ids, int32_t num_seqs,
                                    const int32_t* num_new_tokens, int64_t* slot_mapping) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (num_seqs < 0) return PA_ERR_SHAPE;
  if (num_seqs > 0 && (!seq_ids || !num_new_tokens || !slot_mapping)) return PA_ERR_NULL;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Seq* s = find_seq(m, seq_ids[i]);
    if (!s || num_new_tokens[i] < 0 || num_new_tokens[i] > static_cast<int64_t>(s->tokens.size()))
      return PA_ERR_SHAPE;
  }
  int64_t o = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const Seq* s = find_seq(m, seq_ids[i]);
    const int64_t len = static_cast<int64_t>(s->tokens.size());
    for (int64_t pos = len - num_new_tokens[i]; pos < len; ++pos)
      slot_mapping[o++] = static_cast<int64_t>(s->table[pos / m->P]) * m->P + pos % m->P;
  }
  return PA_OK;
}

PA_API pa_status pa_bm_query(pa_block_manager* m, int64_t* num_free_blocks, int64_t* num_seqs,
                             int64_t* num_hashed_blocks) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (num_free_blocks) *num_free_blocks = m->n_free;
  if (num_seqs) *num_seqs = static_cast<int64_t>(m->seqs.size());
  if (num_hashed_blocks) *num_hashed_blocks = static_cast<int64_t>(m->by_hash.size());
  return PA_OK;
}

PA_API pa_status pa_bm_block_ref_count(pa_block_manager* m, int32_t block_id, int32_t* ref_count) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  if (!ref_count) return PA_ERR_NULL;
  if (block_id < 0 || block_id >= static_cast<int32_t>(m->blocks.size())) return PA_ERR_SHAPE;
  *ref_count = m->blocks[block_id].ref;
  return PA_OK;
}

PA_API pa_status pa_bm_seq_info(pa_block_manager* m, int64_t seq_id, int64_t* num_tokens,
                                int64_t* num_cached_tokens, int32_t* num_blocks) {
  pa_status st = guard(m);
  if (st != PA_OK) return st;
  const Seq* s = find_seq(m, seq_id);
  if (!s) return PA_ERR_SHAPE;
  if (num_tokens) *num_tokens = static_cast<int64_t>(s->tokens.size());
  if (num_cached_tokens) *num_cached_tokens = s->cached_tokens;
  if (num_blocks) *num_blocks = static_cast<int32_t>(s->table.size());
  return PA_OK;
}

}  // extern "C"
