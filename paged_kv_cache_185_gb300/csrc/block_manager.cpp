// block_manager.cpp -- prefix-caching manager of the physical KV blocks (host).
//
// The allocation side of the paged cache: which physical block holds which
// tokens of which sequence.  Sequences that share a prompt prefix share the
// physical blocks of that prefix ("wLLM" project page, "Features / Core
// engine": prefix sharing is a block-table operation; "mini-vLLM" README,
// "What changed": a block keeps a reference count for it).
//
//   * A full block is identified by the chain hash of every token up to and
//     including its last one, and keeps its tokens, so a hit is checked token
//     for token (no false sharing on a hash collision).  New sequences reuse
//     cached full blocks of their prompt; only the rest needs K/V written.
//   * Every block has a reference count (sequences whose table names it).  A
//     sequence about to write into a block that others also name gets its own
//     copy first (copy-on-write): the call reports the (source, destination)
//     pair and the caller copies the first `len % block_size` slots.
//   * Freed full blocks stay cached (evictable, least recently freed first)
//     until their block is needed again; other freed blocks are reused first.
//
// Single-threaded per manager; calls that fail leave the manager unchanged.
#include <cstdint>
#include <list>
#include <unordered_map>
#include <vector>

#include "wllm.h"

namespace {

uint64_t mix64(uint64_t x) {  // a splitmix64-style finaliser
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ULL;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebULL;
  x ^= x >> 31;
  return x;
}

uint64_t chain_hash(uint64_t prev, const int32_t* tok, int n) {
  uint64_t h = mix64(prev ^ 0x9e3779b97f4a7c15ULL);
  for (int i = 0; i < n; ++i) h = mix64(h ^ static_cast<uint32_t>(tok[i]));
  return h | 1;  // 0 means "not cached"
}

struct Seq {
  std::vector<int32_t> blocks;
  std::vector<int32_t> tail;  // tokens of the last, partly filled block
  int64_t len = 0;
  uint64_t last_full_hash = 0;  // chain hash of the last full block (0: none)
};

}  // namespace

struct wllm_block_manager {
  int num_blocks = 0, block_size = 0;
  std::vector<int32_t> ref;                     // sequences naming each block
  std::vector<uint64_t> hash;                   // chain hash of a cached full block, else 0
  std::vector<std::vector<int32_t>> tokens;     // tokens of a cached full block
  std::unordered_map<uint64_t, int32_t> cache;  // chain hash -> cached block
  std::vector<int32_t> free_plain;              // unreferenced, not cached
  std::list<int32_t> free_cached;               // unreferenced, cached: oldest first
  std::vector<std::list<int32_t>::iterator> lru_pos;
  std::vector<char> in_lru;
  std::unordered_map<int64_t, Seq> seqs;

  int64_t available() const { return static_cast<int64_t>(free_plain.size() + free_cached.size()); }

  void uncache(int32_t b) {
    if (hash[b] != 0) {
      auto it = cache.find(hash[b]);
      if (it != cache.end() && it->second == b) cache.erase(it);
      hash[b] = 0;
      tokens[b].clear();
    }
  }
  // take an unreferenced block: a plain one first, else the oldest cached one
  int32_t take() {
    int32_t b;
    if (!free_plain.empty()) {
      b = free_plain.back();
      free_plain.pop_back();
    } else {
      b = free_cached.front();
      free_cached.pop_front();
      in_lru[b] = 0;
      uncache(b);
    }
    ref[b] = 1;
    return b;
  }
  // one more reference to b (which may be an unreferenced cached block)
  void acquire(int32_t b) {
    if (ref[b] == 0 && in_lru[b]) {
      free_cached.erase(lru_pos[b]);
      in_lru[b] = 0;
    }
    ++ref[b];
  }
  void release(int32_t b) {
    if (--ref[b] > 0) return;
    if (hash[b] != 0) {
      free_cached.push_back(b);
      lru_pos[b] = std::prev(free_cached.end());
      in_lru[b] = 1;
    } else {
      free_plain.push_back(b);
    }
  }
  // register a block that just became full with these tokens under hash h
  void publish(int32_t b, uint64_t h, const int32_t* tok) {
    if (cache.count(h) != 0) return;  // an equal block is already cached
    hash[b] = h;
    tokens[b].assign(tok, tok + block_size);
    cache.emplace(h, b);
  }
  // a cached block holding exactly these tokens under hash h, or -1
  int32_t lookup(uint64_t h, const int32_t* tok) const {
    auto it = cache.find(h);
    if (it == cache.end()) return -1;
    const std::vector<int32_t>& t = tokens[it->second];
    for (int i = 0; i < block_size; ++i)
      if (t[i] != tok[i]) return -1;
    return it->second;
  }
};

extern "C" {

int wllm_bm_create(int num_blocks, int block_size, wllm_block_manager** out) {
  if (out == nullptr || num_blocks < 1 || block_size < 1) return WLLM_ERR_INVALID_ARG;
  auto* m = new wllm_block_manager();
  m->num_blocks = num_blocks;
  m->block_size = block_size;
  m->ref.assign(num_blocks, 0);
  m->hash.assign(num_blocks, 0);
  m->tokens.resize(num_blocks);
  m->lru_pos.resize(num_blocks);
  m->in_lru.assign(num_blocks, 0);
  m->free_plain.reserve(num_blocks);
  for (int b = num_blocks - 1; b >= 0; --b) m->free_plain.push_back(b);  // block 0 is taken first
  *out = m;
  return WLLM_OK;
}

void wllm_bm_destroy(wllm_block_manager* m) { delete m; }

int wllm_bm_add_sequence(wllm_block_manager* m, int64_t seq_id, const int32_t* tokens, int64_t n, int64_t* slots,
                         int64_t* cached_tokens) {
  if (m == nullptr || n < 0 || (n > 0 && tokens == nullptr) || m->seqs.count(seq_id) != 0)
    return WLLM_ERR_INVALID_ARG;
  const int bs = m->block_size;
  const int64_t full = n / bs, nblk = (n + bs - 1) / bs;
  // cached prefix: leading full blocks found in the cache, in order
  std::vector<int32_t> hit;
  std::vector<uint64_t> hashes(full);
  uint64_t h = 0;
  bool hitting = true;
  for (int64_t i = 0; i < full; ++i) {
    h = chain_hash(h, tokens + i * bs, bs);
    hashes[i] = h;
    if (hitting) {
      const int32_t b = m->lookup(h, tokens + i * bs);
      if (b >= 0) hit.push_back(b);
      else hitting = false;
    }
  }
  // blocks to take: the rest; unreferenced cached hits also leave the free pool
  int64_t hit_free = 0;
  for (int32_t b : hit) hit_free += m->ref[b] == 0 ? 1 : 0;
  if (nblk - static_cast<int64_t>(hit.size()) > m->available() - hit_free) return WLLM_ERR_OUT_OF_RANGE;
  Seq s;
  for (int32_t b : hit) {
    m->acquire(b);
    s.blocks.push_back(b);
  }
  for (int64_t i = static_cast<int64_t>(hit.size()); i < nblk; ++i) {
    const int32_t b = m->take();
    s.blocks.push_back(b);
    if (i < full) m->publish(b, hashes[i], tokens + i * bs);
  }
  s.len = n;
  s.last_full_hash = full > 0 ? hashes[full - 1] : 0;
  s.tail.assign(tokens + full * bs, tokens + n);
  if (slots != nullptr)
    for (int64_t t = 0; t < n; ++t) slots[t] = static_cast<int64_t>(s.blocks[t / bs]) * bs + t % bs;
  if (cached_tokens != nullptr) *cached_tokens = static_cast<int64_t>(hit.size()) * bs;
  m->seqs.emplace(seq_id, std::move(s));
  return WLLM_OK;
}

int wllm_bm_append_token(wllm_block_manager* m, int64_t seq_id, int32_t token, int64_t* slot, int32_t* copy_src,
                         int32_t* copy_dst) {
  if (m == nullptr) return WLLM_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return WLLM_ERR_INVALID_ARG;
  Seq& s = it->second;
  const int bs = m->block_size;
  const int off = static_cast<int>(s.len % bs);
  int32_t src = -1, dst = -1;
  if (off == 0) {  // the last block is full (or there is none): a fresh block
    if (m->available() < 1) return WLLM_ERR_OUT_OF_RANGE;
    s.blocks.push_back(m->take());
  } else if (m->ref[s.blocks.back()] > 1) {  // shared partial block: copy on write
    if (m->available() < 1) return WLLM_ERR_OUT_OF_RANGE;
    src = s.blocks.back();
    dst = m->take();
    m->release(src);
    s.blocks.back() = dst;
  }
  const int32_t b = s.blocks.back();
  if (slot != nullptr) *slot = static_cast<int64_t>(b) * bs + off;
  if (copy_src != nullptr) *copy_src = src;
  if (copy_dst != nullptr) *copy_dst = dst;
  s.tail.push_back(token);
  ++s.len;
  if (off + 1 == bs) {  // the block just filled: cache it for later prompts
    s.last_full_hash = chain_hash(s.last_full_hash, s.tail.data(), bs);
    m->publish(b, s.last_full_hash, s.tail.data());
    s.tail.clear();
  }
  return WLLM_OK;
}

int wllm_bm_fork(wllm_block_manager* m, int64_t parent, int64_t child) {
  if (m == nullptr || m->seqs.count(child) != 0) return WLLM_ERR_INVALID_ARG;
  auto it = m->seqs.find(parent);
  if (it == m->seqs.end()) return WLLM_ERR_INVALID_ARG;
  Seq s = it->second;
  for (int32_t b : s.blocks) m->acquire(b);
  m->seqs.emplace(child, std::move(s));
  return WLLM_OK;
}

int wllm_bm_free_sequence(wllm_block_manager* m, int64_t seq_id) {
  if (m == nullptr) return WLLM_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return WLLM_ERR_INVALID_ARG;
  // release the last block first, so the older (prefix) blocks stay cached longest
  for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) m->release(*b);
  m->seqs.erase(it);
  return WLLM_OK;
}

int wllm_bm_block_table(const wllm_block_manager* m, int64_t seq_id, int32_t* row, int max_blocks,
                        int64_t* context_len) {
  if (m == nullptr || max_blocks < 0 || (max_blocks > 0 && row == nullptr)) return WLLM_ERR_INVALID_ARG;
  auto it = m->seqs.find(seq_id);
  if (it == m->seqs.end()) return WLLM_ERR_INVALID_ARG;
  const Seq& s = it->second;
  if (static_cast<int64_t>(s.blocks.size()) > max_blocks) return WLLM_ERR_OUT_OF_RANGE;
  for (int j = 0; j < max_blocks; ++j) row[j] = j < static_cast<int>(s.blocks.size()) ? s.blocks[j] : -1;
  if (context_len != nullptr) *context_len = s.len;
  return WLLM_OK;
}

int64_t wllm_bm_num_free_blocks(const wllm_block_manager* m) { return m == nullptr ? -1 : m->available(); }

int64_t wllm_bm_num_cached_blocks(const wllm_block_manager* m) {
  return m == nullptr ? -1 : static_cast<int64_t>(m->cache.size());
}

int wllm_bm_block_ref(const wllm_block_manager* m, int32_t block) {
  if (m == nullptr || block < 0 || block >= m->num_blocks) return -1;
  return m->ref[block];
}

}  // extern "C"
