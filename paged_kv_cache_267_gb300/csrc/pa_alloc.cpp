// Host block allocator of libpa: a fixed pool of physical KV blocks with a
// seeded shuffled free list, reference-counted sharing (fork), copy-on-write
// of a shared partial last block on append, deferred reclamation, a hard
// capacity ("vLLM 0.5 深度解析" §2.1; "vLLM 0.7.2深度解析" §2.1 and §5.3), and
// release of blocks that a sliding window has left behind ("vLLM 0.7.2深度解析"
// §2.3). A released table entry is -1.
#include <algorithm>
#include <cstdint>
#include <memory>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pa.h"

struct pa_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_list;  // allocation pops from the back
  std::vector<int32_t> pending;    // ref count reached zero, not yet reclaimed
  std::vector<int32_t> ref;
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
  };
  std::unordered_map<int32_t, Seq> seqs;
  int32_t next_id = 0;
  // prefix cache: key -> block, and block -> (key, token ids of the block)
  std::unordered_map<uint64_t, int32_t> cache;
  std::unordered_map<int32_t, std::pair<uint64_t, std::vector<int32_t>>> cached;
};

namespace {

// SplitMix64 (Steele, Lea and Flood; public-domain reference by Vigna).
struct SplitMix64 {
  uint64_t s;
  uint64_t next() {
    s += 0x9E3779B97F4A7C15ull;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
};

int64_t blocks_for(int64_t n, int32_t bs) { return n / bs + (n % bs != 0); }  // no overflow

// FNV-1a, 64-bit (Fowler, Noll, Vo): per byte, xor then multiply.
uint64_t fnv1a64_bytes(const unsigned char* p, size_t n, uint64_t h) {
  for (size_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001B3ull;
  }
  return h;
}

// Key of a full block: FNV-1a-64 over the previous key (8 bytes, little
// endian) followed by the block's token ids (4 bytes each, little endian).
uint64_t block_key(uint64_t prev, const int32_t* tok, int32_t bs) {
  unsigned char buf[8];
  for (int i = 0; i < 8; ++i) buf[i] = static_cast<unsigned char>(prev >> (8 * i));
  uint64_t h = fnv1a64_bytes(buf, 8, 0xCBF29CE484222325ull);
  for (int32_t j = 0; j < bs; ++j) {
    const uint32_t t = static_cast<uint32_t>(tok[j]);
    unsigned char b4[4] = {static_cast<unsigned char>(t), static_cast<unsigned char>(t >> 8),
                           static_cast<unsigned char>(t >> 16),
                           static_cast<unsigned char>(t >> 24)};
    h = fnv1a64_bytes(b4, 4, h);
  }
  return h;
}

int32_t pop_block(pa_alloc* a) {
  int32_t b = a->free_list.back();
  a->free_list.pop_back();
  a->ref[b] = 1;
  return b;
}

}  // namespace

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, uint64_t seed,
                          pa_alloc** out) try {
  if (!out || num_blocks < 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  std::unique_ptr<pa_alloc> a(new pa_alloc());
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->ref.assign(num_blocks, 0);
  a->free_list.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) a->free_list[i] = i;
  // Fisher-Yates, Durstenfeld's form: i from n-1 down to 1, j uniform-ish in [0, i]
  SplitMix64 rng{seed};
  for (int64_t i = static_cast<int64_t>(num_blocks) - 1; i > 0; --i) {
    const uint64_t j = rng.next() % static_cast<uint64_t>(i + 1);
    std::swap(a->free_list[i], a->free_list[j]);
  }
  *out = a.release();
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

pa_status pa_alloc_add(pa_alloc* a, int64_t n_tokens, int32_t* seq_out) try {
  if (!a || !seq_out || n_tokens < 0) return PA_ERR_INVALID_ARG;
  const int64_t need = blocks_for(n_tokens, a->block_size);
  if (need > static_cast<int64_t>(a->free_list.size())) return PA_ERR_OUT_OF_BLOCKS;
  pa_alloc::Seq s;
  s.len = n_tokens;
  s.blocks.reserve(need);
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(pop_block(a));
  const int32_t id = a->next_id++;
  a->seqs.emplace(id, std::move(s));
  *seq_out = id;
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

pa_status pa_alloc_fork(pa_alloc* a, int32_t src, int32_t* seq_out) try {
  if (!a || !seq_out) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(src);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  pa_alloc::Seq s = it->second;
  for (int32_t b : s.blocks)
    if (b >= 0) a->ref[b] += 1;
  const int32_t id = a->next_id++;
  a->seqs.emplace(id, std::move(s));
  *seq_out = id;
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

pa_status pa_alloc_append(pa_alloc* a, int32_t seq, int64_t n_tokens, int32_t* cow_src,
                          int32_t* cow_dst) try {
  if (!a || n_tokens < 0) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  pa_alloc::Seq& s = it->second;
  if (n_tokens > INT64_MAX - s.len) return PA_ERR_INVALID_ARG;
  int32_t src = -1, dst = -1;
  if (n_tokens > 0) {
    const bool partial = s.len % a->block_size != 0;
    const bool cow = partial && a->ref[s.blocks.back()] > 1;
    const int64_t extra =
        blocks_for(s.len + n_tokens, a->block_size) - static_cast<int64_t>(s.blocks.size());
    if (extra + (cow ? 1 : 0) > static_cast<int64_t>(a->free_list.size()))
      return PA_ERR_OUT_OF_BLOCKS;
    if (cow) {
      src = s.blocks.back();
      dst = pop_block(a);
      a->ref[src] -= 1;
      s.blocks.back() = dst;
    }
    for (int64_t i = 0; i < extra; ++i) s.blocks.push_back(pop_block(a));
    s.len += n_tokens;
  }
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

pa_status pa_alloc_free(pa_alloc* a, int32_t seq) try {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  for (int32_t b : it->second.blocks) {
    if (b >= 0 && --a->ref[b] == 0) a->pending.push_back(b);
  }
  a->seqs.erase(it);
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

pa_status pa_alloc_trim_window(pa_alloc* a, int32_t seq, int32_t window,
                               int32_t* n_released) try {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  int32_t n = 0;
  if (window > 0) {
    pa_alloc::Seq& s = it->second;
    const int64_t start = s.len > window ? s.len - window : 0;
    const int64_t first_live = start / a->block_size;
    for (int64_t i = 0; i < first_live && i < static_cast<int64_t>(s.blocks.size()); ++i) {
      const int32_t b = s.blocks[i];
      if (b < 0) continue;
      s.blocks[i] = -1;
      if (--a->ref[b] == 0) a->pending.push_back(b);
      ++n;
    }
  }
  if (n_released) *n_released = n;
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

pa_status pa_alloc_add_cached(pa_alloc* a, const int32_t* tokens, int64_t n_tokens,
                              int32_t* seq_out, int64_t* n_cached) try {
  if (!a || !seq_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
  const int32_t bs = a->block_size;
  const int64_t nblk = blocks_for(n_tokens, bs), nfull = n_tokens / bs;
  std::vector<uint64_t> keys(static_cast<size_t>(nfull));
  std::vector<int32_t> reuse;
  uint64_t prev = 0;
  bool matching = true;
  for (int64_t i = 0; i < nfull; ++i) {
    const int32_t* tok = tokens + i * bs;
    keys[i] = block_key(prev, tok, bs);
    prev = keys[i];
    if (!matching) continue;
    auto it = a->cache.find(keys[i]);
    if (it != a->cache.end()) {
      const auto& stored = a->cached[it->second].second;
      if (std::equal(stored.begin(), stored.end(), tok)) {
        reuse.push_back(it->second);
        continue;
      }
    }
    matching = false;
  }
  if (nblk - static_cast<int64_t>(reuse.size()) > static_cast<int64_t>(a->free_list.size()))
    return PA_ERR_OUT_OF_BLOCKS;
  pa_alloc::Seq s;
  s.len = n_tokens;
  s.blocks.reserve(static_cast<size_t>(nblk));
  for (int32_t b : reuse) {
    if (a->ref[b] == 0) a->pending.erase(std::find(a->pending.begin(), a->pending.end(), b));
    a->ref[b] += 1;
    s.blocks.push_back(b);
  }
  for (int64_t i = static_cast<int64_t>(reuse.size()); i < nblk; ++i) {
    const int32_t b = pop_block(a);
    s.blocks.push_back(b);
    if (i < nfull && a->cache.find(keys[i]) == a->cache.end()) {
      a->cache.emplace(keys[i], b);
      a->cached[b] = {keys[i], std::vector<int32_t>(tokens + i * bs, tokens + (i + 1) * bs)};
    }
  }
  const int32_t id = a->next_id++;
  a->seqs.emplace(id, std::move(s));
  *seq_out = id;
  if (n_cached) *n_cached = static_cast<int64_t>(reuse.size()) * bs;
  return PA_OK;
} catch (const std::bad_alloc&) {
  return PA_ERR_HOST_MEMORY;
}

int32_t pa_alloc_reclaim(pa_alloc* a) {
  if (!a) return 0;
  for (int32_t b : a->pending) {
    auto it = a->cached.find(b);
    if (it != a->cached.end()) {
      a->cache.erase(it->second.first);
      a->cached.erase(it);
    }
  }
  const int32_t n = static_cast<int32_t>(a->pending.size());
  a->free_list.insert(a->free_list.end(), a->pending.begin(), a->pending.end());
  a->pending.clear();
  return n;
}

pa_status pa_alloc_block_table(const pa_alloc* a, int32_t seq, int32_t* out, int32_t capacity,
                               int32_t* n_out) {
  if (!a || !n_out) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  const auto& bl = it->second.blocks;
  *n_out = static_cast<int32_t>(bl.size());
  if (static_cast<int64_t>(bl.size()) > capacity || (!out && !bl.empty())) return PA_ERR_INVALID_ARG;
  for (size_t i = 0; i < bl.size(); ++i) out[i] = bl[i];
  return PA_OK;
}

pa_status pa_alloc_seq_len(const pa_alloc* a, int32_t seq, int64_t* len_out) {
  if (!a || !len_out) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
  *len_out = it->second.len;
  return PA_OK;
}

pa_status pa_alloc_fill_tables(const pa_alloc* a, const int32_t* seqs, int32_t n,
                               int32_t* tables, int32_t max_blocks, int32_t* lens_out) {
  if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seqs || !tables || !lens_out)))
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seqs[i]);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    if (static_cast<int64_t>(it->second.blocks.size()) > max_blocks ||
        it->second.len > INT32_MAX)
      return PA_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const auto& s = a->seqs.find(seqs[i])->second;
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    for (int32_t j = 0; j < max_blocks; ++j)
      row[j] = j < static_cast<int32_t>(s.blocks.size()) ? s.blocks[j] : -1;
    lens_out[i] = static_cast<int32_t>(s.len);
  }
  return PA_OK;
}

int32_t pa_alloc_refcount(const pa_alloc* a, int32_t block) {
  if (!a || block < 0 || block >= a->num_blocks) return -1;
  return a->ref[block];
}

int32_t pa_alloc_num_free(const pa_alloc* a) {
  return a ? static_cast<int32_t>(a->free_list.size()) : 0;
}

int32_t pa_alloc_num_pending(const pa_alloc* a) {
  return a ? static_cast<int32_t>(a->pending.size()) : 0;
}

}  // extern "C"
