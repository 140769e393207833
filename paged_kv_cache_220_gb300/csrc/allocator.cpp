// Host block allocator for the paged KV cache.
//
// Sources: "How vLLM gets real throughput on H100s ...", sections
// "PagedAttention borrows from operating systems" (fixed-size blocks, a block
// table per sequence, blocks taken only as tokens are produced, copy-on-write
// sharing of a prompt's blocks among rollouts) and "Continuous batching
// removes straggler bubbles" (a finished sequence's blocks return to the pool
// at once); "vLLM architecture, memory and benchmarks deep dive", section
// "PagedAttention: a 1960s idea for modern GPUs" (only the last block of a
// running sequence has free slots; memory is cloned only where rollouts
// diverge); "Dissecting vLLM ...", section "PagedAttention: Virtual Memory
// for KV Cache" (freed blocks go to the next request; shared prefixes point
// at the same physical blocks); "High-Throughput LLM Inference & Training: A
// Deep Dive into vLLM", Figures 1 and 2 (the slot accounting).
//
// Every call is transactional: it checks everything it needs (free blocks,
// output room) before it changes any state.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <random>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_allocator {
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // stack: back() is popped next
  std::vector<int32_t> refcount;   // 0 = free
  std::vector<int32_t> fill;       // slots written in the block
  std::unordered_map<int, Seq> seqs;
  int next_id = 0;

  int32_t pop() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    refcount[b] = 1;
    fill[b] = 0;
    return b;
  }
  void release(int32_t b) {
    if (--refcount[b] == 0) {
      fill[b] = 0;
      free_list.push_back(b);
    }
  }
};

extern "C" int pkv_alloc_create(int num_blocks, int block_size, uint64_t seed,
                                pkv_allocator** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_allocator* a = new (std::nothrow) pkv_allocator();
  if (!a) return PKV_ERR_OUT_OF_BLOCKS;
  try {
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->free_list.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) a->free_list[i] = i;
    // Seeded Fisher-Yates; the bounded draw is a plain modulo so the order is
    // the same with every standard library.
    std::mt19937_64 rng(seed);
    for (int i = num_blocks - 1; i > 0; --i) {
      const int j = static_cast<int>(rng() % static_cast<uint64_t>(i + 1));
      std::swap(a->free_list[i], a->free_list[j]);
    }
    a->refcount.assign(num_blocks, 0);
    a->fill.assign(num_blocks, 0);
  } catch (...) {
    delete a;
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  *out = a;
  return PKV_OK;
}

extern "C" void pkv_alloc_destroy(pkv_allocator* a) { delete a; }

extern "C" int pkv_seq_new(pkv_allocator* a, int* seq_id) {
  if (!a || !seq_id) return PKV_ERR_INVALID_ARG;
  try {
    const int id = a->next_id;
    a->seqs.emplace(id, pkv_allocator::Seq{});
    a->next_id = id + 1;
    *seq_id = id;
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

extern "C" int pkv_seq_fork(pkv_allocator* a, int parent, int* child) {
  if (!a || !child) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
  try {
    pkv_allocator::Seq c = it->second;  // copy of the parent's table
    const int id = a->next_id;
    a->seqs.emplace(id, std::move(c));
    a->next_id = id + 1;
    for (int32_t b : a->seqs[id].table) ++a->refcount[b];
    *child = id;
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

extern "C" int pkv_seq_append(pkv_allocator* a, int seq, int n_tokens, int64_t* slots_out,
                              int32_t* cow_pairs_out, int* n_cow) {
  if (!a || n_tokens < 0 || (n_tokens > 0 && !slots_out)) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
  if (n_cow) *n_cow = 0;
  if (n_tokens == 0) return PKV_OK;
  pkv_allocator::Seq& s = it->second;
  const int B = a->block_size;
  const int64_t len = s.len;
  const int64_t have = static_cast<int64_t>(s.table.size());
  const int64_t need_total = (len + n_tokens + B - 1) / B;
  // The last block is written into only if it is partially filled; if it is
  // shared, this holder first takes a private copy.
  const bool cow = (len % B != 0) && a->refcount[s.table.back()] > 1;
  const int64_t new_blocks = (need_total - have) + (cow ? 1 : 0);
  if (new_blocks > static_cast<int64_t>(a->free_list.size())) return PKV_ERR_OUT_OF_BLOCKS;
  if (cow && !cow_pairs_out) return PKV_ERR_INVALID_ARG;
  try {
    s.table.reserve(need_total);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  if (cow) {
    const int32_t old = s.table.back();
    const int32_t fresh = a->pop();
    a->fill[fresh] = a->fill[old];
    --a->refcount[old];  // still > 0: another holder keeps it
    s.table.back() = fresh;
    cow_pairs_out[0] = old;
    cow_pairs_out[1] = fresh;
    if (n_cow) *n_cow = 1;
  }
  for (int i = 0; i < n_tokens; ++i) {
    const int64_t pos = len + i;
    const int64_t bi = pos / B;
    if (bi == static_cast<int64_t>(s.table.size())) s.table.push_back(a->pop());
    const int32_t b = s.table[bi];
    slots_out[i] = static_cast<int64_t>(b) * B + pos % B;
    ++a->fill[b];
  }
  s.len = len + n_tokens;
  return PKV_OK;
}

extern "C" int pkv_seq_free(pkv_allocator* a, int seq) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
  // Release in reverse so the sequence's first block is reused first.
  const std::vector<int32_t>& t = it->second.table;
  for (auto b = t.rbegin(); b != t.rend(); ++b) a->release(*b);
  a->seqs.erase(it);
  return PKV_OK;
}

extern "C" int pkv_seq_block_table(const pkv_allocator* a, int seq, int32_t* out, int cap,
                                   int* n_blocks) {
  if (!a || !n_blocks || cap < 0) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
  const std::vector<int32_t>& t = it->second.table;
  *n_blocks = static_cast<int>(t.size());
  if (static_cast<int64_t>(t.size()) > cap) return PKV_ERR_INVALID_ARG;
  if (!t.empty() && !out) return PKV_ERR_INVALID_ARG;
  for (size_t i = 0; i < t.size(); ++i) out[i] = t[i];
  return PKV_OK;
}

extern "C" int pkv_seq_len(const pkv_allocator* a, int seq, int* len) {
  if (!a || !len) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PKV_ERR_NOT_FOUND;
  *len = static_cast<int>(it->second.len);
  return PKV_OK;
}

extern "C" int pkv_block_refcount(const pkv_allocator* a, int block, int* refcount) {
  if (!a || !refcount || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID_ARG;
  *refcount = a->refcount[block];
  return PKV_OK;
}

extern "C" int pkv_alloc_stats(const pkv_allocator* a, int* free_blocks, int* used_blocks,
                               long long* used_slots) {
  if (!a) return PKV_ERR_INVALID_ARG;
  const int nfree = static_cast<int>(a->free_list.size());
  if (free_blocks) *free_blocks = nfree;
  if (used_blocks) *used_blocks = a->num_blocks - nfree;
  if (used_slots) {
    long long u = 0;
    for (int b = 0; b < a->num_blocks; ++b)
      if (a->refcount[b] > 0) u += a->fill[b];
    *used_slots = u;
  }
  return PKV_OK;
}

// ---------------------------------------------------------------- checkpoint
//
// The whole allocator state as a flat little-endian int64 record:
//   magic, version, num_blocks, block_size, next_id,
//   free list size, free list (bottom to top),
//   refcount[num_blocks], fill[num_blocks],
//   number of sequences, then per sequence (ascending id):
//   id, length, table size, table.
// Loading checks the record against itself (sizes, ranges, every block either
// free with refcount 0 or held by exactly refcount tables, fill within the
// block) and returns PKV_ERR_INVALID_ARG otherwise, building nothing.

namespace {

constexpr int64_t kMagic = 0x31414b5650LL;  // "PVKA1"

void put(std::vector<int64_t>& v, int64_t x) { v.push_back(x); }

}  // namespace

extern "C" int pkv_alloc_save(const pkv_allocator* a, void* buf, size_t cap, size_t* n) {
  if (!a || !n) return PKV_ERR_INVALID_ARG;
  std::vector<int64_t> r;
  try {
    put(r, kMagic);
    put(r, 1);
    put(r, a->num_blocks);
    put(r, a->block_size);
    put(r, a->next_id);
    put(r, static_cast<int64_t>(a->free_list.size()));
    for (int32_t b : a->free_list) put(r, b);
    for (int32_t c : a->refcount) put(r, c);
    for (int32_t f : a->fill) put(r, f);
    std::vector<int> ids;
    ids.reserve(a->seqs.size());
    for (const auto& kv : a->seqs) ids.push_back(kv.first);
    std::sort(ids.begin(), ids.end());
    put(r, static_cast<int64_t>(ids.size()));
    for (int id : ids) {
      const pkv_allocator::Seq& q = a->seqs.at(id);
      put(r, id);
      put(r, q.len);
      put(r, static_cast<int64_t>(q.table.size()));
      for (int32_t b : q.table) put(r, b);
    }
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  *n = r.size() * sizeof(int64_t);
  if (!buf) return PKV_OK;  // size query
  if (cap < *n) return PKV_ERR_INVALID_ARG;
  std::memcpy(buf, r.data(), *n);
  return PKV_OK;
}

extern "C" int pkv_alloc_load(const void* buf, size_t n, pkv_allocator** out) {
  if (!buf || !out || n % sizeof(int64_t) != 0) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  const size_t words = n / sizeof(int64_t);
  std::vector<int64_t> r(words);
  std::memcpy(r.data(), buf, n);
  size_t i = 0;
  auto get = [&](int64_t* x) -> bool {
    if (i >= words) return false;
    *x = r[i++];
    return true;
  };
  int64_t magic, version, nb, bs, next_id, nfree;
  if (!get(&magic) || !get(&version) || !get(&nb) || !get(&bs) || !get(&next_id) ||
      !get(&nfree))
    return PKV_ERR_INVALID_ARG;
  if (magic != kMagic || version != 1 || nb <= 0 || nb > INT32_MAX || bs <= 0 || bs > INT32_MAX ||
      next_id < 0 || next_id > INT32_MAX || nfree < 0 || nfree > nb)
    return PKV_ERR_INVALID_ARG;
  pkv_allocator* a = new (std::nothrow) pkv_allocator();
  if (!a) return PKV_ERR_OUT_OF_BLOCKS;
  auto fail = [&](int rc) {
    delete a;
    return rc;
  };
  try {
    a->num_blocks = static_cast<int>(nb);
    a->block_size = static_cast<int>(bs);
    a->next_id = static_cast<int>(next_id);
    a->free_list.resize(nfree);
    a->refcount.resize(nb);
    a->fill.resize(nb);
    for (int64_t k = 0; k < nfree; ++k) {
      int64_t b;
      if (!get(&b) || b < 0 || b >= nb) return fail(PKV_ERR_INVALID_ARG);
      a->free_list[k] = static_cast<int32_t>(b);
    }
    for (int64_t k = 0; k < nb; ++k) {
      int64_t c;
      if (!get(&c) || c < 0 || c > INT32_MAX) return fail(PKV_ERR_INVALID_ARG);
      a->refcount[k] = static_cast<int32_t>(c);
    }
    for (int64_t k = 0; k < nb; ++k) {
      int64_t f;
      if (!get(&f) || f < 0 || f > bs) return fail(PKV_ERR_INVALID_ARG);
      a->fill[k] = static_cast<int32_t>(f);
    }
    int64_t nseq;
    if (!get(&nseq) || nseq < 0) return fail(PKV_ERR_INVALID_ARG);
    std::vector<int64_t> held(nb, 0);
    for (int64_t k = 0; k < nseq; ++k) {
      int64_t id, len, nt;
      if (!get(&id) || !get(&len) || !get(&nt)) return fail(PKV_ERR_INVALID_ARG);
      if (id < 0 || id >= next_id || a->seqs.count(static_cast<int>(id)) || len < 0 || nt < 0 ||
          nt > nb || nt != (len + bs - 1) / bs)
        return fail(PKV_ERR_INVALID_ARG);
      pkv_allocator::Seq q;
      q.len = len;
      q.table.resize(nt);
      for (int64_t t = 0; t < nt; ++t) {
        int64_t b;
        if (!get(&b) || b < 0 || b >= nb) return fail(PKV_ERR_INVALID_ARG);
        q.table[t] = static_cast<int32_t>(b);
        ++held[b];
      }
      a->seqs.emplace(static_cast<int>(id), std::move(q));
    }
    if (i != words) return fail(PKV_ERR_INVALID_ARG);
    // every block: free (refcount 0, on the free list once) or held by
    // exactly refcount tables
    std::vector<char> on_free(nb, 0);
    for (int32_t b : a->free_list) {
      if (on_free[b] || a->refcount[b] != 0) return fail(PKV_ERR_INVALID_ARG);
      on_free[b] = 1;
    }
    for (int64_t b = 0; b < nb; ++b) {
      if (!on_free[b] && (a->refcount[b] == 0 || held[b] != a->refcount[b]))
        return fail(PKV_ERR_INVALID_ARG);
      if (on_free[b] && held[b] != 0) return fail(PKV_ERR_INVALID_ARG);
    }
  } catch (...) {
    return fail(PKV_ERR_OUT_OF_BLOCKS);
  }
  *out = a;
  return PKV_OK;
}
