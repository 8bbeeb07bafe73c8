// Host block allocator: fixed-size blocks, free list, reference counts,
// fork and copy-on-write.
//
// "vLLM internals (2) - why PagedAttention splits the KV cache into pages",
// block-table section: blocks are handed out one at a time when needed, from
// anywhere in the pool.  "PagedAttention", section "Block Table 如何工作": a
// full block triggers a new allocation and the table is extended; blocks no
// longer referenced return to the free pool.  Same page, "支持块级共享", and
// "LLM KV cache 02 - serving engine KV" section 2: several sequences point at
// one physical block under a reference count, and a branch that has to write
// into a shared block first gets its own copy (copy-on-write).
//
// Policy where the pages leave it open: the free list starts in the caller's
// order; allocation pops the front; a block whose count reaches zero is
// pushed to the back; a sequence is released in table order (last block
// first when prefix caching is on).
#include <array>
#include <cstdint>
#include <cstring>
#include <list>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"
#include "sha256.h"

namespace pa {

// Automatic prefix caching ("llm-kv-cache-02-serving-engine-kv", section 4
// "프리픽스 캐시"), enabled per allocator:
//  * every full block of a tracked sequence gets a key, SHA-256 of the
//    previous block's key (32 zero bytes for the first block), the block's
//    token ids (little-endian int32) and the request's extra bytes (cache
//    salt, adapter, ... as the caller composes them); a key therefore stands
//    for the whole prefix up to and including its block;
//  * only full blocks are keyed; a key maps to the first block that held it;
//  * a new sequence reuses, block by block from the start, every block whose
//    key is cached, up to the first miss (those tokens need no prefill);
//  * a block whose count drops to zero keeps its key and content on the free
//    queue; allocation takes the queue's front and evicts that block's key,
//    so the least recently freed cached block goes first; a finished
//    sequence's blocks are queued last block first, so tails are evicted
//    before the prefixes they extend; a hit takes its block off the queue.
class BlockAllocator {
 public:
  using Key = std::array<uint8_t, 32>;
  struct KeyHash {
    size_t operator()(const Key& k) const {
      size_t h;
      std::memcpy(&h, k.data(), sizeof(h));
      return h;
    }
  };
  struct Seq {
    std::vector<int32_t> table;
    int32_t len = 0;
    // prefix caching: token ids and keys of the full blocks so far
    bool track = false;
    std::vector<int32_t> tokens;
    std::vector<uint8_t> extra;
    int32_t keyed = 0;  // leading full blocks whose key is known
    Key last_key{};
  };

  BlockAllocator(int32_t num_blocks, int32_t block_size)
      : num_blocks_(num_blocks),
        block_size_(block_size),
        ref_(num_blocks, 0),
        where_(num_blocks),
        in_free_(num_blocks, 0) {}

  bool init_free_list(const int32_t* order) {
    std::vector<char> seen(num_blocks_, 0);
    for (int32_t i = 0; i < num_blocks_; ++i) {
      int32_t b = order ? order[i] : i;
      if (b < 0 || b >= num_blocks_ || seen[b]) return false;
      seen[b] = 1;
      push_free(b);
    }
    return true;
  }

  int32_t num_blocks() const { return num_blocks_; }
  int32_t block_size() const { return block_size_; }
  int32_t num_free() const { return static_cast<int32_t>(free_.size()); }
  int32_t refcount(int32_t b) const { return valid_block(b) ? ref_[b] : -1; }
  bool valid_block(int32_t b) const { return b >= 0 && b < num_blocks_; }

  int32_t allocate() {
    if (free_.empty()) return -1;
    int32_t b = free_.front();
    free_.pop_front();
    in_free_[b] = 0;
    if (pc_ && keyed_[b]) {  // the least recently freed cached block gives up its key
      cached_.erase(key_[b]);
      keyed_[b] = 0;
    }
    ref_[b] = 1;
    return b;
  }

  pa_status incref(int32_t b) {
    if (!valid_block(b) || ref_[b] <= 0) return PA_ERR_INVALID_ARG;
    ++ref_[b];
    return PA_OK;
  }

  pa_status decref(int32_t b) {
    if (!valid_block(b) || ref_[b] <= 0) return PA_ERR_INVALID_ARG;
    if (--ref_[b] == 0) push_free(b);
    return PA_OK;
  }

  int32_t seq_create() {
    int32_t s = next_seq_++;
    seqs_[s] = Seq{};
    return s;
  }

  Seq* find(int32_t s) {
    auto it = seqs_.find(s);
    return it == seqs_.end() ? nullptr : &it->second;
  }
  const Seq* find(int32_t s) const {
    auto it = seqs_.find(s);
    return it == seqs_.end() ? nullptr : &it->second;
  }

  pa_status fork(int32_t parent, int32_t* child) {
    const Seq* p = find(parent);
    if (!p) return PA_ERR_INVALID_ARG;
    Seq copy = *p;  // copy before inserting: insertion may not move nodes, but be explicit
    for (int32_t b : copy.table) ++ref_[b];
    int32_t c = next_seq_++;
    seqs_[c] = std::move(copy);
    *child = c;
    return PA_OK;
  }

  // Reserve the next token's slot (see pa_alloc_append_slot).  A tracked
  // sequence appended to without its token id stops being keyed.
  pa_status append_slot(int32_t s, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    Seq* q = find(s);
    if (!q) return PA_ERR_INVALID_ARG;
    pa_status st = reserve(q, slot, cow_src, cow_dst);
    if (st == PA_OK && q->track) {
      q->track = false;
      q->tokens.clear();
    }
    return st;
  }

  pa_status append_tokens(int32_t s, int32_t n, int64_t* slots, const int32_t* ids = nullptr) {
    Seq* q = find(s);
    if (!q || n < 0) return PA_ERR_INVALID_ARG;
    // all-or-nothing: check the blocks needed and the sharing state first
    const int32_t pos = q->len;
    if (n == 0) return PA_OK;
    if (pos % block_size_ != 0 && ref_[q->table[pos / block_size_]] > 1) return PA_ERR_INVALID_ARG;
    const int64_t have = static_cast<int64_t>(q->table.size());
    const int64_t need = (static_cast<int64_t>(pos) + n + block_size_ - 1) / block_size_;
    if (need - have > static_cast<int64_t>(free_.size())) return PA_ERR_OOM;
    for (int32_t j = 0; j < n; ++j) {
      int32_t a, b;
      pa_status st = reserve(q, &slots[j], &a, &b);
      if (st != PA_OK) return st;  // unreachable after the checks above
    }
    if (q->track) {
      if (ids) {
        q->tokens.insert(q->tokens.end(), ids, ids + n);
        register_full_blocks(q);
      } else {
        q->track = false;
        q->tokens.clear();
      }
    }
    return PA_OK;
  }

  pa_status free_seq(int32_t s) {
    auto it = seqs_.find(s);
    if (it == seqs_.end()) return PA_ERR_INVALID_ARG;
    const std::vector<int32_t>& t = it->second.table;
    if (pc_) {
      for (auto b = t.rbegin(); b != t.rend(); ++b)  // tail first: evicted first
        if (--ref_[*b] == 0) push_free(*b);
    } else {
      for (int32_t b : t)
        if (--ref_[b] == 0) push_free(b);
    }
    seqs_.erase(it);
    return PA_OK;
  }

  // ---- prefix caching ----
  pa_status enable_prefix_cache() {
    if (pc_) return PA_OK;
    if (!seqs_.empty() || static_cast<int32_t>(free_.size()) != num_blocks_) return PA_ERR_INVALID_ARG;
    pc_ = true;
    key_.assign(num_blocks_, Key{});
    keyed_.assign(num_blocks_, 0);
    return PA_OK;
  }
  bool prefix_cache() const { return pc_; }
  int32_t num_cached() const { return static_cast<int32_t>(cached_.size()); }
  const Key* block_key(int32_t b) const { return valid_block(b) && pc_ && keyed_[b] ? &key_[b] : nullptr; }

  Key key_of(const Key* prev, const int32_t* ids, const std::vector<uint8_t>& extra) {
    // previous key || token ids (little-endian int32) || extra, hashed in one pass
    std::vector<uint8_t>& buf = key_buf_;
    buf.resize(32 + 4 * static_cast<size_t>(block_size_) + extra.size());
    if (prev) std::memcpy(buf.data(), prev->data(), 32);
    else std::memset(buf.data(), 0, 32);
    uint8_t* p = buf.data() + 32;
    for (int32_t j = 0; j < block_size_; ++j, p += 4) {
      const uint32_t v = static_cast<uint32_t>(ids[j]);
      p[0] = static_cast<uint8_t>(v);
      p[1] = static_cast<uint8_t>(v >> 8);
      p[2] = static_cast<uint8_t>(v >> 16);
      p[3] = static_cast<uint8_t>(v >> 24);
    }
    if (!extra.empty()) std::memcpy(p, extra.data(), extra.size());
    Sha256 h;
    h.update(buf.data(), buf.size());
    Key k;
    h.finish(k.data());
    return k;
  }

  pa_status seq_create_prefix(const int32_t* ids, int32_t n, const uint8_t* extra, int32_t extra_n,
                              int32_t* seq, int32_t* cached_tokens, int64_t* slots) {
    if (!pc_ || n < 0 || extra_n < 0 || (n > 0 && (!ids || !slots)) || (extra_n > 0 && !extra))
      return PA_ERR_INVALID_ARG;
    std::vector<uint8_t> ex(extra, extra + extra_n);
    // longest run of cached leading full blocks (lookups only)
    std::vector<int32_t> hits;
    std::vector<Key> keys;
    int32_t in_queue = 0;
    for (int32_t j = 0; (static_cast<int64_t>(j) + 1) * block_size_ <= n; ++j) {
      Key k = key_of(j ? &keys.back() : nullptr, ids + static_cast<int64_t>(j) * block_size_, ex);
      auto it = cached_.find(k);
      if (it == cached_.end()) break;
      hits.push_back(it->second);
      keys.push_back(k);
      if (ref_[it->second] == 0) ++in_queue;
    }
    const int64_t need = (static_cast<int64_t>(n) + block_size_ - 1) / block_size_ - hits.size();
    if (need > static_cast<int64_t>(free_.size()) - in_queue) return PA_ERR_OOM;
    const int32_t s = seq_create();
    Seq* q = find(s);
    q->track = true;
    q->extra = std::move(ex);
    for (int32_t b : hits) {
      if (ref_[b] == 0) take_free(b);
      ++ref_[b];
      q->table.push_back(b);
    }
    q->len = static_cast<int32_t>(hits.size()) * block_size_;
    q->keyed = static_cast<int32_t>(hits.size());
    if (!keys.empty()) q->last_key = keys.back();
    q->tokens.assign(ids, ids + n);
    for (int32_t t = q->len; t < n; ++t) {
      int32_t a, b;
      int64_t sl;
      reserve(q, &sl, &a, &b);  // fresh blocks only: cannot fail after the check above
    }
    for (int32_t t = 0; t < n; ++t)
      slots[t] = static_cast<int64_t>(q->table[t / block_size_]) * block_size_ + t % block_size_;
    register_full_blocks(q);
    *seq = s;
    if (cached_tokens) *cached_tokens = static_cast<int32_t>(hits.size()) * block_size_;
    return PA_OK;
  }

  const std::list<int32_t>& free_list() const { return free_; }
  const std::map<int32_t, Seq>& seqs() const { return seqs_; }

 private:
  void push_free(int32_t b) {
    free_.push_back(b);
    where_[b] = std::prev(free_.end());
    in_free_[b] = 1;
  }
  void take_free(int32_t b) {
    free_.erase(where_[b]);
    in_free_[b] = 0;
  }

  pa_status reserve(Seq* q, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    const int32_t pos = q->len;
    const int32_t li = pos / block_size_;
    int32_t src = -1, dst = -1;
    if (pos % block_size_ == 0) {
      int32_t nb = allocate();
      if (nb < 0) return PA_ERR_OOM;
      q->table.push_back(nb);
    } else {
      int32_t last = q->table[li];
      if (ref_[last] > 1) {
        int32_t nb = allocate();
        if (nb < 0) return PA_ERR_OOM;
        --ref_[last];  // still > 0: a shared block never reaches the free list here
        q->table[li] = nb;
        src = last;
        dst = nb;
      }
    }
    q->len = pos + 1;
    *slot = static_cast<int64_t>(q->table[li]) * block_size_ + pos % block_size_;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PA_OK;
  }

  // Key every newly full block of a tracked sequence; a key already cached
  // for another block leaves this block unkeyed (the first holder keeps it).
  void register_full_blocks(Seq* q) {
    if (!pc_ || !q->track) return;
    const int32_t full = q->len / block_size_;
    while (q->keyed < full) {
      const int32_t j = q->keyed;
      const Key k = key_of(j ? &q->last_key : nullptr,
                           q->tokens.data() + static_cast<int64_t>(j) * block_size_, q->extra);
      const int32_t b = q->table[j];
      if (!keyed_[b] && cached_.find(k) == cached_.end()) {
        key_[b] = k;
        keyed_[b] = 1;
        cached_.emplace(k, b);
      }
      q->last_key = k;
      ++q->keyed;
    }
  }

  int32_t num_blocks_;
  int32_t block_size_;
  std::vector<int32_t> ref_;
  std::list<int32_t> free_;
  std::vector<std::list<int32_t>::iterator> where_;
  std::vector<char> in_free_;
  std::map<int32_t, Seq> seqs_;
  int32_t next_seq_ = 0;
  // prefix cache
  bool pc_ = false;
  std::vector<Key> key_;
  std::vector<char> keyed_;
  std::unordered_map<Key, int32_t, KeyHash> cached_;
  std::vector<uint8_t> key_buf_;
};

}  // namespace pa

struct pa_allocator {
  pa::BlockAllocator impl;
  pa_allocator(int32_t nb, int32_t bs) : impl(nb, bs) {}
};

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                          pa_allocator** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_allocator* a = new (std::nothrow) pa_allocator(num_blocks, block_size);
  if (!a) return PA_ERR_OOM;
  if (!a->impl.init_free_list(free_order)) {
    delete a;
    return PA_ERR_INVALID_ARG;
  }
  *out = a;
  return PA_OK;
}

void pa_alloc_destroy(pa_allocator* a) { delete a; }

int32_t pa_alloc_num_blocks(const pa_allocator* a) { return a ? a->impl.num_blocks() : -1; }
int32_t pa_alloc_block_size(const pa_allocator* a) { return a ? a->impl.block_size() : -1; }
int32_t pa_alloc_num_free(const pa_allocator* a) { return a ? a->impl.num_free() : -1; }
int32_t pa_alloc_refcount(const pa_allocator* a, int32_t block) {
  return a ? a->impl.refcount(block) : -1;
}

pa_status pa_alloc_allocate(pa_allocator* a, int32_t* block) {
  if (!a || !block) return PA_ERR_INVALID_ARG;
  int32_t b = a->impl.allocate();
  if (b < 0) return PA_ERR_OOM;
  *block = b;
  return PA_OK;
}

pa_status pa_alloc_incref(pa_allocator* a, int32_t block) {
  return a ? a->impl.incref(block) : PA_ERR_INVALID_ARG;
}

pa_status pa_alloc_decref(pa_allocator* a, int32_t block) {
  return a ? a->impl.decref(block) : PA_ERR_INVALID_ARG;
}

pa_status pa_alloc_seq_create(pa_allocator* a, int32_t* seq) {
  if (!a || !seq) return PA_ERR_INVALID_ARG;
  *seq = a->impl.seq_create();
  return PA_OK;
}

pa_status pa_alloc_fork(pa_allocator* a, int32_t parent, int32_t* child) {
  if (!a || !child) return PA_ERR_INVALID_ARG;
  return a->impl.fork(parent, child);
}

pa_status pa_alloc_append_slot(pa_allocator* a, int32_t seq, int64_t* slot, int32_t* cow_src,
                               int32_t* cow_dst) {
  if (!a || !slot) return PA_ERR_INVALID_ARG;
  return a->impl.append_slot(seq, slot, cow_src, cow_dst);
}

pa_status pa_alloc_append_slots(pa_allocator* a, const int32_t* seqs, int32_t n, int64_t* slots,
                                int64_t* cow_pairs, int32_t* num_cow, int32_t* num_done) {
  if (num_done) *num_done = 0;
  if (num_cow) *num_cow = 0;
  if (!a || n < 0 || (n > 0 && (!seqs || !slots || !cow_pairs))) return PA_ERR_INVALID_ARG;
  int32_t ncow = 0;
  for (int32_t j = 0; j < n; ++j) {
    int32_t src = -1, dst = -1;
    pa_status st = a->impl.append_slot(seqs[j], &slots[j], &src, &dst);
    if (st != PA_OK) {
      if (num_cow) *num_cow = ncow;
      return st;
    }
    if (src >= 0) {
      cow_pairs[2 * ncow] = src;
      cow_pairs[2 * ncow + 1] = dst;
      ++ncow;
    }
    if (num_done) *num_done = j + 1;
  }
  if (num_cow) *num_cow = ncow;
  return PA_OK;
}

pa_status pa_alloc_append_tokens(pa_allocator* a, int32_t seq, int32_t n, int64_t* slots) {
  if (!a || n < 0 || (n > 0 && !slots)) return PA_ERR_INVALID_ARG;
  return a->impl.append_tokens(seq, n, slots);
}

pa_status pa_alloc_free_seq(pa_allocator* a, int32_t seq) {
  return a ? a->impl.free_seq(seq) : PA_ERR_INVALID_ARG;
}

int32_t pa_alloc_seq_len(const pa_allocator* a, int32_t seq) {
  if (!a) return -1;
  const pa::BlockAllocator::Seq* q = a->impl.find(seq);
  return q ? q->len : -1;
}

int32_t pa_alloc_num_seqs(const pa_allocator* a) {
  return a ? static_cast<int32_t>(a->impl.seqs().size()) : -1;
}

pa_status pa_alloc_block_table(const pa_allocator* a, int32_t seq, int32_t* out, int32_t cap,
                               int32_t* n) {
  if (!a || !n || cap < 0) return PA_ERR_INVALID_ARG;
  const pa::BlockAllocator::Seq* q = a->impl.find(seq);
  if (!q) return PA_ERR_INVALID_ARG;
  const int32_t len = static_cast<int32_t>(q->table.size());
  *n = len;
  if (len > cap || (len > 0 && !out)) return PA_ERR_INVALID_ARG;
  for (int32_t k = 0; k < len; ++k) out[k] = q->table[k];
  return PA_OK;
}

pa_status pa_alloc_export_tables(const pa_allocator* a, const int32_t* seqs, int32_t n,
                                 int32_t* tables, int32_t max_blocks, int32_t* lens,
                                 int32_t pad_value) {
  if (!a || n < 0 || max_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (n > 0 && (!seqs || !tables || !lens)) return PA_ERR_INVALID_ARG;
  for (int32_t j = 0; j < n; ++j) {
    const pa::BlockAllocator::Seq* q = a->impl.find(seqs[j]);
    if (!q) return PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(q->table.size()) > max_blocks) return PA_ERR_INVALID_ARG;
  }
  for (int32_t j = 0; j < n; ++j) {
    const pa::BlockAllocator::Seq* q = a->impl.find(seqs[j]);
    int32_t* row = tables + static_cast<int64_t>(j) * max_blocks;
    const int32_t len = static_cast<int32_t>(q->table.size());
    for (int32_t k = 0; k < len; ++k) row[k] = q->table[k];
    for (int32_t k = len; k < max_blocks; ++k) row[k] = pad_value;
    lens[j] = q->len;
  }
  return PA_OK;
}

pa_status pa_alloc_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n) {
  if (!a || !n || cap < 0) return PA_ERR_INVALID_ARG;
  const auto& fl = a->impl.free_list();
  *n = static_cast<int32_t>(fl.size());
  if (*n > cap || (*n > 0 && !out)) return PA_ERR_INVALID_ARG;
  int32_t k = 0;
  for (int32_t b : fl) out[k++] = b;
  return PA_OK;
}

pa_status pa_alloc_enable_prefix_cache(pa_allocator* a) {
  return a ? a->impl.enable_prefix_cache() : PA_ERR_INVALID_ARG;
}

pa_status pa_alloc_seq_create_prefix(pa_allocator* a, const int32_t* token_ids, int32_t num_tokens,
                                     const void* extra, int32_t extra_bytes, int32_t* seq,
                                     int32_t* cached_tokens, int64_t* slots) {
  if (!a || !seq) return PA_ERR_INVALID_ARG;
  return a->impl.seq_create_prefix(token_ids, num_tokens, static_cast<const uint8_t*>(extra),
                                   extra_bytes, seq, cached_tokens, slots);
}

pa_status pa_alloc_append_token_ids(pa_allocator* a, int32_t seq, const int32_t* token_ids,
                                    int32_t n, int64_t* slots) {
  if (!a || n < 0 || (n > 0 && (!slots || !token_ids))) return PA_ERR_INVALID_ARG;
  return a->impl.append_tokens(seq, n, slots, token_ids);
}

int32_t pa_alloc_num_cached(const pa_allocator* a) { return a ? a->impl.num_cached() : -1; }

pa_status pa_alloc_block_key(const pa_allocator* a, int32_t block, uint8_t key[32]) {
  if (!a || !key) return PA_ERR_INVALID_ARG;
  const pa::BlockAllocator::Key* k = a->impl.block_key(block);
  if (!k) return PA_ERR_INVALID_ARG;
  std::memcpy(key, k->data(), 32);
  return PA_OK;
}

pa_status pa_alloc_live_seqs(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n) {
  if (!a || !n || cap < 0) return PA_ERR_INVALID_ARG;
  const auto& m = a->impl.seqs();
  *n = static_cast<int32_t>(m.size());
  if (*n > cap || (*n > 0 && !out)) return PA_ERR_INVALID_ARG;
  int32_t k = 0;
  for (const auto& kv : m) out[k++] = kv.first;
  return PA_OK;
}

}  // extern "C"
