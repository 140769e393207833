// Iteration-level (continuous) batching over the block allocator.
//
// Sources: "How vLLM gets real throughput on H100s ...", section "Continuous
// batching removes straggler bubbles" (scheduling at every forward pass; a
// sequence that ends returns its blocks at once and a queued request takes
// its place on the next iteration); "Dissecting vLLM ...", section
// "Continuous Batching: Breaking the Sequence Barrier" (after each iteration:
// eject finished sequences, admit waiting requests into the freed room,
// preempt under memory pressure); "vLLM architecture, memory and benchmarks
// deep dive", section "Continuous batching and the straggler problem".
//
// One call of pkv_sched_step is one iteration:
//   1. eject: running requests that produced their last token in the previous
//      iteration are finished and their sequences freed (blocks back to the
//      free list);
//   2. admit: waiting requests, first come first served, while the batch has
//      room (max_num_seqs) and the free blocks cover the prompt plus its first
//      new token on top of the blocks the running sequences need this
//      iteration; an admitted request's prompt slots are reported so the
//      caller can store its K/V (the prefill, outside this library);
//   3. grow: every running request takes one slot for this iteration's token.
//      If the pool cannot supply a block, the most recently admitted running
//      request is preempted: its sequence is freed and it goes back to the
//      front of the queue to be recomputed from its prompt later, or, in swap
//      mode, its block list is reported so the caller can copy the blocks to
//      host memory before they are reused ("Dissecting vLLM ...", sections
//      "Continuous Batching: Breaking the Sequence Barrier" and "FAQ": the
//      preempted sequence's blocks go to CPU RAM and come back later).
// Swapped requests are resumed before new ones are admitted: a resumed
// request gets fresh blocks for its whole length (reported, for the copy
// back) and continues where it stopped; nothing is recomputed.
// EOS is a request's own token budget (max_new_tokens), known up front.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

struct Req {
  int64_t id;
  int prompt_len;
  int max_new;
  int generated;  // tokens produced so far (the one of this iteration included)
  int seq;        // allocator sequence id while running
  std::vector<int64_t> prompt_slots;  // reported in the admitting iteration
  std::vector<int32_t> swap_blocks;   // swap mode: blocks to copy out / back in
  int samples;    // waiting: sequences to fork from the prompt at admission
  bool shared_tail = false;  // a sample whose last block is still the shared prompt's
};

}  // namespace

struct pkv_scheduler {
  pkv_allocator* alloc = nullptr;
  int block_size = 0;
  int max_num_seqs = 0;
  std::deque<Req> waiting;
  std::vector<Req> running;                 // admission order
  std::vector<int64_t> finished;            // ejected in the last step
  std::vector<int64_t> preempted;           // preempted in the last step
  std::vector<int64_t> admitted;            // ids admitted in the last step
  std::vector<int64_t> new_slots;           // per running request, last step
  int64_t steps = 0;
  int preempt_mode = PKV_PREEMPT_RECOMPUTE;
  std::deque<Req> swapped;                  // swapped-out requests, resume order
  std::vector<Req> swapped_out;             // swapped out in the last step (for their blocks)
  std::vector<int64_t> swapped_in;          // ids resumed in the last step
  int batch_order = PKV_BATCH_ADMISSION;    // row order of the exported batch
  std::vector<int32_t> cow_pairs;           // (src, dst) of the last step's growth
};

namespace {

// Rows of the exported batch: indices into running, in admission order or
// by decreasing context length (ties in admission order).
std::vector<int> export_order(const pkv_scheduler* s) {
  std::vector<int> idx(s->running.size());
  for (size_t i = 0; i < idx.size(); ++i) idx[i] = static_cast<int>(i);
  if (s->batch_order == PKV_BATCH_LONGEST_FIRST) {
    std::stable_sort(idx.begin(), idx.end(), [s](int a, int b) {
      const Req& x = s->running[a];
      const Req& y = s->running[b];
      return x.prompt_len + x.generated > y.prompt_len + y.generated;
    });
  }
  return idx;
}

}  // namespace

extern "C" int pkv_sched_create(pkv_allocator* alloc, int block_size, int max_num_seqs,
                                pkv_scheduler** out) {
  if (!alloc || !out || block_size <= 0 || max_num_seqs <= 0) return PKV_ERR_INVALID_ARG;
  pkv_scheduler* s = new (std::nothrow) pkv_scheduler();
  if (!s) return PKV_ERR_OUT_OF_BLOCKS;
  s->alloc = alloc;
  s->block_size = block_size;
  s->max_num_seqs = max_num_seqs;
  *out = s;
  return PKV_OK;
}

extern "C" void pkv_sched_destroy(pkv_scheduler* s) { delete s; }

namespace {

// Whether an id in [lo, hi) belongs to a request that is waiting (with its
// samples' ids), running or swapped out. Finished ids may be reused.
bool ids_in_use(const pkv_scheduler* s, int64_t lo, int64_t hi) {
  auto hit = [lo, hi](int64_t a, int64_t b) { return a < hi && lo < b; };
  for (const Req& r : s->waiting)
    if (hit(r.id, r.id + std::max(1, r.samples))) return true;
  for (const Req& r : s->running)
    if (hit(r.id, r.id + 1)) return true;
  for (const Req& r : s->swapped)
    if (hit(r.id, r.id + 1)) return true;
  return false;
}

}  // namespace

extern "C" int pkv_sched_add_request_n(pkv_scheduler* s, int64_t request_id, int prompt_len,
                                       int max_new_tokens, int n) {
  if (!s || prompt_len < 0 || max_new_tokens <= 0 || n < 1 || n > s->max_num_seqs)
    return PKV_ERR_INVALID_ARG;
  // the samples take ids request_id .. request_id + n - 1: none may be taken
  // by a live request (the lookups by id would then find the wrong one)
  if (request_id < 0 || request_id > INT64_MAX - n ||
      ids_in_use(s, request_id, request_id + n))
    return PKV_ERR_INVALID_ARG;
  try {
    s->waiting.push_back(Req{request_id, prompt_len, max_new_tokens, 0, -1, {}, {}, n});
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

extern "C" int pkv_sched_add_request(pkv_scheduler* s, int64_t request_id, int prompt_len,
                                     int max_new_tokens) {
  return pkv_sched_add_request_n(s, request_id, prompt_len, max_new_tokens, 1);
}

namespace {

int blocks_for(int64_t tokens, int B) { return static_cast<int>((tokens + B - 1) / B); }

int free_blocks(const pkv_scheduler* s) {
  int f = 0;
  pkv_alloc_stats(s->alloc, &f, nullptr, nullptr);
  return f;
}

// Blocks the running requests need to grow by one token each.
int growth_blocks(const pkv_scheduler* s) {
  int n = 0;
  for (const Req& r : s->running) {
    const int64_t len = static_cast<int64_t>(r.prompt_len) + r.generated;
    if (len % s->block_size == 0 || r.shared_tail) ++n;  // a new block or a copy
  }
  return n;
}

int preempt_last(pkv_scheduler* s) {
  Req r = std::move(s->running.back());
  s->running.pop_back();
  s->preempted.push_back(r.id);
  r.prompt_slots.clear();
  r.shared_tail = false;
  // admitted in this very step: its prompt K/V is not stored yet, so there is
  // nothing to copy out; it waits to be admitted (and prefilled) again
  if (std::find(s->admitted.begin(), s->admitted.end(), r.id) != s->admitted.end()) {
    pkv_seq_free(s->alloc, r.seq);
    r.seq = -1;
    r.generated = 0;
    s->waiting.push_front(std::move(r));
    return PKV_OK;
  }
  if (s->preempt_mode == PKV_PREEMPT_SWAP) {
    // resumed in this very step: its blocks were never filled and the host
    // copy is still the valid one, so it goes back without a copy-out
    auto it = std::find(s->swapped_in.begin(), s->swapped_in.end(), r.id);
    if (it != s->swapped_in.end()) {
      s->swapped_in.erase(it);
      pkv_seq_free(s->alloc, r.seq);
      r.seq = -1;
      r.swap_blocks.clear();
      s->swapped.push_front(std::move(r));
      return PKV_OK;
    }
    // the block list in logical order: the caller copies these blocks out
    // before anything is written this iteration
    const int64_t len = static_cast<int64_t>(r.prompt_len) + r.generated;
    const int nb = blocks_for(len, s->block_size);
    r.swap_blocks.assign(nb > 0 ? nb : 1, -1);
    int n = 0;
    const int rc = pkv_seq_block_table(s->alloc, r.seq, r.swap_blocks.data(), nb > 0 ? nb : 1, &n);
    if (rc != PKV_OK) return rc;
    r.swap_blocks.resize(n);
    pkv_seq_free(s->alloc, r.seq);
    r.seq = -1;
    s->swapped_out.push_back(r);  // keeps the block list for pkv_sched_swap_blocks
    r.swap_blocks.clear();
    s->swapped.push_front(std::move(r));
    return PKV_OK;
  }
  pkv_seq_free(s->alloc, r.seq);
  r.seq = -1;
  r.generated = 0;  // recomputed from the prompt when it is admitted again
  s->waiting.push_front(std::move(r));
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_sched_step(pkv_scheduler* s, int* num_running, int* num_admitted,
                              int* num_finished) {
  if (!s) return PKV_ERR_INVALID_ARG;
  try {
    s->finished.clear();
    s->preempted.clear();
    s->admitted.clear();
    s->swapped_out.clear();
    s->swapped_in.clear();
    s->cow_pairs.clear();
    // 1. eject
    std::vector<Req> keep;
    keep.reserve(s->running.size());
    for (Req& r : s->running) {
      if (r.generated >= r.max_new) {
        pkv_seq_free(s->alloc, r.seq);
        s->finished.push_back(r.id);
      } else {
        r.prompt_slots.clear();
        keep.push_back(std::move(r));
      }
    }
    s->running.swap(keep);
    // 2a. resume swapped requests first: fresh blocks for their whole length
    while (!s->swapped.empty() && static_cast<int>(s->running.size()) < s->max_num_seqs) {
      Req& w = s->swapped.front();
      const int64_t len = static_cast<int64_t>(w.prompt_len) + w.generated;
      const int need = blocks_for(len + 1, s->block_size);
      if (need + growth_blocks(s) > free_blocks(s)) break;
      Req r = std::move(w);
      s->swapped.pop_front();
      int sid = -1;
      int rc = pkv_seq_new(s->alloc, &sid);
      if (rc != PKV_OK) return rc;
      r.seq = sid;
      if (len > 0) {
        std::vector<int64_t> slots(static_cast<size_t>(len));
        rc = pkv_seq_append(s->alloc, sid, static_cast<int>(len), slots.data(), nullptr, nullptr);
        if (rc != PKV_OK) {
          pkv_seq_free(s->alloc, sid);
          return rc;
        }
      }
      const int nb = blocks_for(len, s->block_size);
      r.swap_blocks.assign(nb > 0 ? nb : 1, -1);
      int n = 0;
      rc = pkv_seq_block_table(s->alloc, sid, r.swap_blocks.data(), nb > 0 ? nb : 1, &n);
      if (rc != PKV_OK) return rc;
      r.swap_blocks.resize(n);
      s->swapped_in.push_back(r.id);
      s->running.push_back(std::move(r));
    }
    // 2b. admit (a request of n samples: the prompt once, then n - 1 forks
    // sharing its blocks; each sample's first token may need a block of its
    // own, a copy of the shared last prompt block or a fresh one)
    while (s->swapped.empty() && !s->waiting.empty()) {
      Req& w = s->waiting.front();
      const int n = w.samples;
      if (static_cast<int>(s->running.size()) + n > s->max_num_seqs) break;
      const int need = n == 1 ? blocks_for(static_cast<int64_t>(w.prompt_len) + 1, s->block_size)
                              : blocks_for(w.prompt_len, s->block_size) + n;
      if (need + growth_blocks(s) > free_blocks(s)) break;
      Req r = std::move(w);
      s->waiting.pop_front();
      int sid = -1;
      int rc = pkv_seq_new(s->alloc, &sid);
      if (rc != PKV_OK) return rc;
      r.seq = sid;
      r.generated = 0;
      r.samples = 1;
      r.prompt_slots.assign(r.prompt_len, -1);
      if (r.prompt_len > 0) {
        rc = pkv_seq_append(s->alloc, sid, r.prompt_len, r.prompt_slots.data(), nullptr, nullptr);
        if (rc != PKV_OK) {
          pkv_seq_free(s->alloc, sid);
          return rc;
        }
      }
      std::vector<Req> forks;
      for (int k = 1; k < n; ++k) {
        int child = -1;
        rc = pkv_seq_fork(s->alloc, sid, &child);
        if (rc != PKV_OK) {
          for (Req& f : forks) pkv_seq_free(s->alloc, f.seq);
          pkv_seq_free(s->alloc, sid);
          return rc;
        }
        forks.push_back(Req{r.id + k, r.prompt_len, r.max_new, 0, child, {}, {}, 1});
        forks.back().shared_tail = true;
      }
      r.shared_tail = n > 1;
      s->admitted.push_back(r.id);
      s->running.push_back(std::move(r));
      for (Req& f : forks) {
        s->admitted.push_back(f.id);
        s->running.push_back(std::move(f));
      }
    }
    // 3. grow by one token each; preempt the newest on exhaustion
    s->new_slots.clear();
    for (size_t i = 0; i < s->running.size();) {
      Req& r = s->running[i];
      int64_t slot = -1;
      int32_t pair[2] = {-1, -1};
      int ncow = 0;
      const int rc = pkv_seq_append(s->alloc, r.seq, 1, &slot, pair, &ncow);
      if (rc == PKV_OK) {
        ++r.generated;
        r.shared_tail = false;
        s->new_slots.push_back(slot);
        if (ncow > 0) {
          s->cow_pairs.push_back(pair[0]);
          s->cow_pairs.push_back(pair[1]);
        }
        ++i;
        continue;
      }
      if (rc != PKV_ERR_OUT_OF_BLOCKS) return rc;
      // the request being grown may itself be the newest one
      const bool self = (i + 1 == s->running.size());
      const int prc = preempt_last(s);
      if (prc != PKV_OK) return prc;
      if (self) break;
    }
    // a preempted request may have been admitted or resumed in this very step
    auto still_running = [&](std::vector<int64_t>& ids) {
      std::vector<int64_t> keep_ids;
      for (int64_t id : ids)
        for (const Req& r : s->running)
          if (r.id == id) keep_ids.push_back(id);
      ids.swap(keep_ids);
    };
    still_running(s->admitted);
    still_running(s->swapped_in);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  ++s->steps;
  if (num_running) *num_running = static_cast<int>(s->running.size());
  if (num_admitted) *num_admitted = static_cast<int>(s->admitted.size());
  if (num_finished) *num_finished = static_cast<int>(s->finished.size());
  return PKV_OK;
}

extern "C" int pkv_sched_running(const pkv_scheduler* s, int64_t* request_ids,
                                 int32_t* context_lens, int64_t* new_slots, int cap) {
  if (!s) return PKV_ERR_INVALID_ARG;
  const int n = static_cast<int>(s->running.size());
  if (cap < n) return PKV_ERR_INVALID_ARG;
  try {
    const std::vector<int> order = export_order(s);
    for (int i = 0; i < n; ++i) {
      const Req& r = s->running[order[i]];
      if (request_ids) request_ids[i] = r.id;
      if (context_lens) context_lens[i] = r.prompt_len + r.generated;
      if (new_slots) new_slots[i] = s->new_slots[order[i]];
    }
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  return PKV_OK;
}

extern "C" int pkv_sched_block_tables(const pkv_scheduler* s, int32_t* tables, int max_blocks,
                                      int rows) {
  if (!s || !tables || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
  const int n = static_cast<int>(s->running.size());
  if (rows < n) return PKV_ERR_INVALID_ARG;
  std::vector<int> order;
  try {
    order = export_order(s);
  } catch (...) {
    return PKV_ERR_OUT_OF_BLOCKS;
  }
  for (int i = 0; i < n; ++i) {
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    int nb = 0;
    const int rc = pkv_seq_block_table(s->alloc, s->running[order[i]].seq, row, max_blocks, &nb);
    if (rc != PKV_OK) return rc;
    std::fill(row + nb, row + max_blocks, -1);
  }
  return PKV_OK;
}

extern "C" int pkv_sched_prompt_slots(const pkv_scheduler* s, int64_t request_id,
                                      int64_t* slots, int cap, int* n) {
  if (!s || !n) return PKV_ERR_INVALID_ARG;
  for (const Req& r : s->running) {
    if (r.id != request_id) continue;
    *n = static_cast<int>(r.prompt_slots.size());
    if (cap < *n || (*n > 0 && !slots)) return PKV_ERR_INVALID_ARG;
    std::copy(r.prompt_slots.begin(), r.prompt_slots.end(), slots);
    return PKV_OK;
  }
  return PKV_ERR_NOT_FOUND;
}

extern "C" int pkv_sched_events(const pkv_scheduler* s, int kind, int64_t* ids, int cap,
                                int* n) {
  if (!s || !n) return PKV_ERR_INVALID_ARG;
  std::vector<int64_t> out_ids;
  const std::vector<int64_t>* v = kind == 0 ? &s->admitted
                                  : kind == 1 ? &s->finished
                                  : kind == 2 ? &s->preempted
                                  : kind == 4 ? &s->swapped_in : nullptr;
  if (kind == 3) {
    for (const Req& r : s->swapped_out) out_ids.push_back(r.id);
    v = &out_ids;
  }
  if (!v) return PKV_ERR_INVALID_ARG;
  *n = static_cast<int>(v->size());
  if (cap < *n || (*n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
  std::copy(v->begin(), v->end(), ids);
  return PKV_OK;
}

extern "C" int pkv_sched_set_preemption(pkv_scheduler* s, int mode) {
  if (!s || (mode != PKV_PREEMPT_RECOMPUTE && mode != PKV_PREEMPT_SWAP)) return PKV_ERR_INVALID_ARG;
  s->preempt_mode = mode;
  return PKV_OK;
}

extern "C" int pkv_sched_cow_pairs(const pkv_scheduler* s, int32_t* pairs, int cap, int* n) {
  if (!s || !n) return PKV_ERR_INVALID_ARG;
  *n = static_cast<int>(s->cow_pairs.size() / 2);
  if (cap < *n || (*n > 0 && !pairs)) return PKV_ERR_INVALID_ARG;
  std::copy(s->cow_pairs.begin(), s->cow_pairs.end(), pairs);
  return PKV_OK;
}

extern "C" int pkv_sched_set_batch_order(pkv_scheduler* s, int order) {
  if (!s || (order != PKV_BATCH_ADMISSION && order != PKV_BATCH_LONGEST_FIRST))
    return PKV_ERR_INVALID_ARG;
  s->batch_order = order;
  return PKV_OK;
}

extern "C" int pkv_sched_swap_blocks(const pkv_scheduler* s, int64_t request_id,
                                     int32_t* blocks, int cap, int* n) {
  if (!s || !n) return PKV_ERR_INVALID_ARG;
  const std::vector<int32_t>* v = nullptr;
  for (const Req& r : s->swapped_out)
    if (r.id == request_id) v = &r.swap_blocks;
  if (!v)
    for (int64_t id : s->swapped_in)
      if (id == request_id)
        for (const Req& r : s->running)
          if (r.id == request_id) v = &r.swap_blocks;
  if (!v) return PKV_ERR_NOT_FOUND;
  *n = static_cast<int>(v->size());
  if (cap < *n || (*n > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
  std::copy(v->begin(), v->end(), blocks);
  return PKV_OK;
}

extern "C" int pkv_sched_counts(const pkv_scheduler* s, int* waiting, int* running,
                                long long* steps) {
  if (!s) return PKV_ERR_INVALID_ARG;
  if (waiting) *waiting = static_cast<int>(s->waiting.size() + s->swapped.size());
  if (running) *running = static_cast<int>(s->running.size());
  if (steps) *steps = s->steps;
  return PKV_OK;
}
