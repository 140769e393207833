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
#include <cstdint>
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
