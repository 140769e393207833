"""Build the device state of a decode workload through the library itself.

The allocator hands out slots (seeded random placement), the cache is filled
with the history rows [0, ctx - 1) through ``kv_cache_write``, and the state
for one decode step is kept ready: the new token's K/V rows and slots, the
query, the block tables and context lengths. Layers share one block table
(every layer's pool uses the same block ids) and have their own pools.

Shared prefixes (``Workload.prefix_len > 0``): the first rollout of each prompt
is created and filled with the prompt rows, the others are forks of it; then
every rollout appends its first completion token in one step, which is where
copy-on-write pairs appear (a prompt whose last block is partly filled); those
pairs are executed with ``copy_blocks`` before the completion rows are
written.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, NamedTuple, Optional

import numpy as np
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import synth


@dataclass
class LayerState:
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor                 # [S, Hq, D] bf16
    k_new: torch.Tensor             # [S, Hk, D] bf16, row ctx-1 of each sequence
    v_new: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None


@dataclass
class PagedWorkload:
    w: synth.Workload
    alloc: pkv.BlockAllocator
    seqs: List[int]
    block_tables: torch.Tensor      # [S, MB] int32 (device)
    context_lens: torch.Tensor      # [S] int32 (device)
    slot_mapping: torch.Tensor      # [S] int64 (device): slot of row ctx-1
    max_context: int
    layers: List[LayerState] = field(default_factory=list)
    cow_pairs: Optional[torch.Tensor] = None   # [n, 2] int32 from the divergence step
    cow_pairs_host: Optional[np.ndarray] = None
    tables_host: Optional[np.ndarray] = None
    history_slots: Optional[List[np.ndarray]] = None
    # [S] int32 (device): the order in which step() has the decode take the
    # sequences, longest context first; None: batch order (all contexts equal,
    # or set by the caller)
    visit_order: Optional[torch.Tensor] = None

    @property
    def num_seqs(self):
        return self.w.num_seqs


def _write_rows(w, layer, st, seq, slots, t0, t1, device, k_scale, v_scale):
    """Generate logical rows [t0, t1) of `seq` and store them at `slots`."""
    if t1 <= t0:
        return
    k = w.rows(synth.KIND_K, layer, seq, t0, t1, device)
    v = w.rows(synth.KIND_V, layer, seq, t0, t1, device)
    sm = torch.as_tensor(np.ascontiguousarray(slots[: t1 - t0]), device=device)
    pkv.kv_cache_write(k, v, sm, st.k_cache, st.v_cache, k_scale, v_scale)


def fp8_scales(w: synth.Workload, layer: int, device) -> tuple:
    """Per-KV-head scales amax_h / 448 (fp32) over every logical row of every
    sequence (history and the new token) of the layer."""
    Hk = w.num_kv_heads
    amax = []
    for kind in (synth.KIND_K, synth.KIND_V):
        m = torch.zeros(Hk, dtype=torch.float32, device=device)
        for s in range(w.num_seqs):
            r = w.rows(kind, layer, s, 0, w.ctx[s], device).float().abs()
            m = torch.maximum(m, r.amax(dim=(0, 2)))
        amax.append(m)
    # an IEEE fp32 quotient (a tensor divisor: torch turns division by a
    # Python scalar into a product with its rounded reciprocal)
    d = torch.full_like(amax[0], 448.0)
    return torch.div(amax[0], d), torch.div(amax[1], d)


def build(w: synth.Workload, device="cuda", layers: Optional[int] = None,
          alloc_seed: Optional[int] = None, share_prefix: bool = True) -> PagedWorkload:
    """share_prefix=False gives every rollout a private copy of its prompt
    (same logical rows, no shared blocks), for aliasing comparisons."""
    device = torch.device(device)
    L = w.layers if layers is None else layers
    B = w.block_size
    nb = w.pool_blocks()
    if w.prefix_len > 0 and not share_prefix:
        nb = sum(-(-c // B) for c in w.ctx) + w.slack_blocks
    alloc = pkv.BlockAllocator(nb, B, seed=w.seed if alloc_seed is None else alloc_seed)
    S = w.num_seqs
    Hk, D = w.num_kv_heads, w.head_dim
    cache_dtype = torch.uint8 if w.fp8 else torch.bfloat16
    states = []
    for layer in range(L):
        kc = torch.zeros(alloc.num_blocks, Hk, B, D, dtype=cache_dtype, device=device)
        vc = torch.zeros_like(kc)
        ks = vs = None
        if w.fp8:
            ks, vs = fp8_scales(w, layer, device)
        states.append(LayerState(kc, vc, w.q(layer, device), None, None, ks, vs))

    seqs: List[int] = []
    hist_slots: List[Optional[np.ndarray]] = [None] * S
    cow_pairs = np.zeros((0, 2), dtype=np.int32)
    if w.prefix_len > 0 and not share_prefix:
        for s in range(S):
            sid = alloc.new_seq()
            seqs.append(sid)
            slots, _ = alloc.append(sid, w.ctx[s])
            for layer in range(L):
                _write_rows(w, layer, states[layer], s, slots, 0, w.ctx[s] - 1, device,
                            states[layer].k_scale, states[layer].v_scale)
    elif w.prefix_len > 0:
        G, P = w.group, w.prefix_len
        n_prompt = S // G
        seqs = [0] * S
        slot_parts = [[] for _ in range(S)]
        for p in range(n_prompt):
            s0 = alloc.new_seq()
            slots, _ = alloc.append(s0, P)
            for layer in range(L):
                _write_rows(w, layer, states[layer], p * G, slots, 0, P, device,
                            states[layer].k_scale, states[layer].v_scale)
            ids = [s0] + [alloc.fork(s0) for _ in range(G - 1)]
            for r in range(G):
                seqs[p * G + r] = ids[r]
                slot_parts[p * G + r].append(slots)
        # divergence: every rollout appends its first completion token; the
        # first G-1 rollouts of a prompt clone a partly filled last block
        pairs = []
        first = [None] * S
        order = []
        for p in range(n_prompt):
            order += [p * G + r for r in range(1, G)] + [p * G]
        for s in order:
            sl, pr = alloc.append(seqs[s], 1)
            first[s] = sl
            pairs += [tuple(x) for x in pr.tolist()]
        cow_pairs = np.array(pairs, dtype=np.int32).reshape(-1, 2)
        if len(pairs):
            cp = torch.as_tensor(cow_pairs, device=device)
            for st in states:
                pkv.copy_blocks(st.k_cache, st.v_cache, cp)
        for s in range(S):
            rest = w.ctx[s] - P - 1                      # further tokens after the first
            more, pr = alloc.append(seqs[s], rest) if rest > 0 else (np.zeros(0, np.int64), [])
            assert len(pr) == 0
            full = np.concatenate(slot_parts[s] + [first[s], more])
            hist_slots[s] = full
            for layer in range(L):
                _write_rows(w, layer, states[layer], s, full[P:], P, w.ctx[s] - 1, device,
                            states[layer].k_scale, states[layer].v_scale)
    else:
        for s in range(S):
            sid = alloc.new_seq()
            seqs.append(sid)
            slots, _ = alloc.append(sid, w.ctx[s])
            hist_slots[s] = slots
            for layer in range(L):
                _write_rows(w, layer, states[layer], s, slots, 0, w.ctx[s] - 1, device,
                            states[layer].k_scale, states[layer].v_scale)

    MB = max(1, max(-(-c // B) for c in w.ctx))
    tables = alloc.block_tables(seqs, MB)
    # final slot of every logical position, read off the final block tables
    # (a cloned block moves the positions it holds)
    for s in range(S):
        pos = np.arange(w.ctx[s], dtype=np.int64)
        hist_slots[s] = tables[s][pos // B].astype(np.int64) * B + pos % B
    slot_new = np.array([hist_slots[s][w.ctx[s] - 1] for s in range(S)], dtype=np.int64)
    for layer, st in enumerate(states):
        st.k_new = torch.stack([w.rows(synth.KIND_K, layer, s, w.ctx[s] - 1, w.ctx[s], device)[0]
                                for s in range(S)])
        st.v_new = torch.stack([w.rows(synth.KIND_V, layer, s, w.ctx[s] - 1, w.ctx[s], device)[0]
                                for s in range(S)])
    pw = PagedWorkload(
        w=w, alloc=alloc, seqs=seqs,
        block_tables=torch.as_tensor(tables, device=device),
        context_lens=torch.as_tensor(np.array(w.ctx, dtype=np.int32), device=device),
        slot_mapping=torch.as_tensor(slot_new, device=device),
        max_context=w.max_context, layers=states,
        cow_pairs=torch.as_tensor(cow_pairs, device=device) if len(cow_pairs) else None,
        cow_pairs_host=cow_pairs, tables_host=tables, history_slots=hist_slots,
        visit_order=visit_order(w.ctx, device))
    return pw


def visit_order(lengths, device="cuda") -> Optional[torch.Tensor]:
    """Longest first (pkv.longest_first_order) as a device tensor, or None
    when all lengths are equal (the identity order needs no table)."""
    a = np.asarray(lengths, dtype=np.int64)
    if a.size == 0 or np.all(a == a[0]):
        return None
    return torch.as_tensor(pkv.longest_first_order(a), device=device)


def step(pw: PagedWorkload, out: List[torch.Tensor], workspace: Optional[torch.Tensor],
         partition_size: Optional[int] = None, stream=None) -> None:
    """One decode step over every layer: write the new token, attend, merge."""
    P = pw.w.partition_size if partition_size is None else partition_size
    for layer, st in enumerate(pw.layers):
        pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                           st.k_scale, st.v_scale, stream)
        pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens,
                            pw.w.scale, pw.max_context, P, st.k_scale, st.v_scale,
                            out=out[layer], workspace=workspace, stream=stream,
                            seq_order=pw.visit_order)


def capture_step(pw: PagedWorkload, out: List[torch.Tensor], workspace: Optional[torch.Tensor],
                 partition_size: Optional[int] = None, copy_pairs: bool = False, groups=None):
    """Record one decode step (every layer's cache write, decode and merge;
    with copy_pairs also the copy-on-write block copies) as a CUDA graph, so a
    step is replayed with one launch from the host instead of 3-4 per layer
    ("vLLM architecture, memory and benchmarks deep dive", section
    "Hardware-level optimizations": per-kernel dispatch cost on the CPU
    exceeds small kernels' run time; a recorded graph replays the whole
    sequence in one dispatch).

    The graph reads the tensors it was recorded with: update q, the new K/V,
    slots, block tables and context lengths in place, then replay().
    copy_pairs records the copy-on-write copies too; that is only right for
    the divergence iteration itself, since a clone later also holds tokens
    written after the copy. With groups (from prefix_groups) the step uses the
    shared-prefix decode.
    Every kernel is run once eagerly first (on the capture stream), so the
    library's one-time per-device set-up happens outside the capture."""

    def one():
        if copy_pairs and pw.cow_pairs is not None:
            for st in pw.layers:
                pkv.copy_blocks(st.k_cache, st.v_cache, pw.cow_pairs)
        if groups is not None:
            step_shared_prefix(pw, out, groups, workspace, partition_size)
        else:
            step(pw, out, workspace, partition_size)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        one()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        one()
    return g


class ContinuousBatch:
    """Decode iterations driven by the continuous-batching scheduler.

    Every iteration: the scheduler ejects finished requests (their blocks go
    back to the pool), admits waiting ones (their prompt K/V rows are written
    to the prompt slots, standing in for the prefill) and gives each running
    request the slot of this iteration's token; then the new K/V rows are
    written and the split decode + merge runs over the running batch. K/V rows
    and queries come from per-request streams (synth.request_rows /
    request_query), so any iteration can be checked on the host.

    preemption="swap": a request preempted under memory pressure keeps its
    progress: its blocks are copied to pinned host memory (swap_out) before
    anything is written in that iteration, and copied back into fresh blocks
    (swap_in) when it is resumed; without it, preempted requests are
    recomputed from their prompts.

    batch_order="longest_first": the scheduler reports the batch by
    decreasing context length (the decode's longest rows launch first).

    A request (id, prompt, budget, n) asks for n samples of one prompt: they
    run as ids id .. id + n - 1, share the prompt's blocks (and rows), and
    the scheduler's copy-on-write pairs are applied with copy_blocks after
    the prompts are stored and before the iteration's tokens."""

    def __init__(self, seed, requests, num_blocks, block_size=32, num_heads=24,
                 num_kv_heads=4, head_dim=256, max_num_seqs=64, partition_size=512,
                 device="cuda", alloc_seed=None, preemption="recompute",
                 batch_order="admission"):
        self.seed = seed
        self.B = block_size
        self.Hq, self.Hk, self.D = num_heads, num_kv_heads, head_dim
        self.P = partition_size
        self.device = torch.device(device)
        self.alloc = pkv.BlockAllocator(num_blocks, block_size,
                                        seed=seed if alloc_seed is None else alloc_seed)
        self.sched = pkv.Scheduler(self.alloc, max_num_seqs)
        if preemption not in ("recompute", "swap"):
            raise ValueError("preemption: 'recompute' or 'swap'")
        if preemption == "swap":
            self.sched.set_preemption(pkv.PKV_PREEMPT_SWAP)
        if batch_order not in ("admission", "longest_first"):
            raise ValueError("batch_order: 'admission' or 'longest_first'")
        if batch_order == "longest_first":
            self.sched.set_batch_order(pkv.PKV_BATCH_LONGEST_FIRST)
        self.saved = {}       # request id -> pinned host (K, V) blocks
        self.retired = []     # host buffers whose swap_in may still be in flight
        self.swaps = 0
        self.max_num_seqs = max_num_seqs
        # (id, prompt, budget) or (id, prompt, budget, samples): n samples run
        # as ids id .. id + n - 1 and share the prompt's rows
        reqs = [tuple(r) + (1,) * (4 - len(r)) for r in requests]
        self.max_context = max(p + g for _, p, g, _ in reqs)
        self.max_blocks = -(-self.max_context // block_size)
        self.base_of, self.prompt_of = {}, {}
        for rid, p, g, n in reqs:
            self.sched.add_request(rid, p, g, n=n)
            for k in range(n):
                self.base_of[rid + k], self.prompt_of[rid + k] = rid, p
        self.cow_copies = 0
        self.k_cache = torch.zeros(num_blocks, num_kv_heads, block_size, head_dim,
                                   dtype=torch.bfloat16, device=self.device)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.out = torch.empty(max_num_seqs, num_heads, head_dim, dtype=torch.bfloat16,
                               device=self.device)
        self.ws = pkv.alloc_workspace(max_num_seqs, num_heads, head_dim, self.max_context,
                                      partition_size, device=self.device) \
            if partition_size else None
        self.scale = float(torch.tensor(1.0 / (head_dim ** 0.5), dtype=torch.float32))
        self.tokens = 0

    def rows(self, kind, rid, t0, t1, device=None):
        """K or V rows [t0, t1) of request rid: the prompt's rows (shared by
        the samples of one prompt) below its prompt length, its own after."""
        p, base = self.prompt_of[rid], self.base_of[rid]
        dev = device if device is not None else self.device
        parts = []
        if t0 < min(t1, p):
            parts.append(synth.request_rows(self.seed, kind, 0, base, t0, min(t1, p), self.Hk,
                                            self.D, dev))
        if t1 > max(t0, p):
            parts.append(synth.request_rows(self.seed, kind, 0, rid, max(t0, p), t1, self.Hk,
                                            self.D, dev))
        return torch.cat(parts) if len(parts) > 1 else parts[0]

    def done(self) -> bool:
        c = self.sched.counts()
        return c["running"] == 0 and c["waiting"] == 0

    def step(self):
        """One iteration; returns (request_ids, context_lens, out[:n]) or None
        when nothing is running."""
        n, na, _ = self.sched.step()
        dev = self.device
        if self.retired:
            torch.cuda.current_stream(dev).synchronize()
            self.retired.clear()
        # swapped-out blocks are already free: save them before any write
        for rid in self.sched.events(3):
            blocks = torch.as_tensor(self.sched.swap_blocks(int(rid)), device=dev)
            shape = (blocks.numel(),) + tuple(self.k_cache.shape[1:])
            kb = torch.empty(shape, dtype=self.k_cache.dtype, pin_memory=True)
            vb = torch.empty(shape, dtype=self.v_cache.dtype, pin_memory=True)
            pkv.swap_out(self.k_cache, self.v_cache, blocks, kb, vb)
            self.saved[int(rid)] = (kb, vb)
            self.swaps += 1
        for rid in self.sched.events(4):
            blocks = torch.as_tensor(self.sched.swap_blocks(int(rid)), device=dev)
            kb, vb = self.saved.pop(int(rid))
            pkv.swap_in(self.k_cache, self.v_cache, blocks, kb, vb)
            self.retired.append((kb, vb))
        if n == 0:
            return None
        for rid in self.sched.events(0):
            slots = self.sched.prompt_slots(int(rid))
            if len(slots) == 0:
                continue
            k = self.rows(synth.KIND_K, int(rid), 0, len(slots))
            v = self.rows(synth.KIND_V, int(rid), 0, len(slots))
            pkv.kv_cache_write(k, v, torch.as_tensor(slots, device=dev), self.k_cache,
                               self.v_cache)
        # samples writing into a block still shared take a copy of it first
        pairs = self.sched.cow_pairs()
        if len(pairs):
            pkv.copy_blocks(self.k_cache, self.v_cache, torch.as_tensor(pairs, device=dev))
            self.cow_copies += len(pairs)
        ids, ctx, slots = self.sched.running()
        k_new = torch.stack([self.rows(synth.KIND_K, int(r), int(c) - 1, int(c))[0]
                             for r, c in zip(ids, ctx)])
        v_new = torch.stack([self.rows(synth.KIND_V, int(r), int(c) - 1, int(c))[0]
                             for r, c in zip(ids, ctx)])
        q = torch.stack([synth.request_query(self.seed, 0, int(r), int(c) - 1, self.Hq, self.D,
                                             dev) for r, c in zip(ids, ctx)])
        pkv.kv_cache_write(k_new, v_new, torch.as_tensor(slots, device=dev), self.k_cache,
                           self.v_cache)
        bt = torch.as_tensor(self.sched.block_tables(self.max_blocks), device=dev)
        cl = torch.as_tensor(ctx, device=dev)
        out = self.out[:n]
        mc = int(ctx.max())
        pkv.paged_attention(q, self.k_cache, self.v_cache, bt, cl, self.scale, mc, self.P,
                            out=out, workspace=self.ws, seq_order=visit_order(ctx, dev))
        self.tokens += n
        return ids, ctx, out


class PrefixGroups(NamedTuple):
    group_start: torch.Tensor       # int32 [G + 1] (device)
    prefix_blocks: torch.Tensor     # int32 [S] (device)
    max_prefix_blocks: int
    max_own_context: int
    max_group_members: int
    # the members' own-block decode order: longest own part first (None:
    # all own parts equal)
    visit_order: Optional[torch.Tensor] = None


def prefix_groups(pw: PagedWorkload, device="cuda") -> PrefixGroups:
    """Group metadata of a shared-prefix workload. The shared prefix of a
    group is the run of leading full blocks whose physical ids every member's
    table has in common (a partly filled prompt block is cloned on divergence
    and so is private); max_own_context is the longest context past its
    sequence's shared prefix; max_group_members the largest group;
    visit_order the members' own-block decode order, longest own part
    first."""
    w = pw.w
    S = w.num_seqs
    ctx = np.asarray(w.ctx, dtype=np.int64)
    if w.prefix_len <= 0:
        return PrefixGroups(torch.zeros(1, dtype=torch.int32, device=device),
                            torch.zeros(S, dtype=torch.int32, device=device), 0,
                            int(ctx.max()) if S else 0, 1, visit_order(ctx, device))
    G = w.group
    n_prompt = S // G
    tables = pw.tables_host
    pre = np.zeros(S, dtype=np.int32)
    for p in range(n_prompt):
        rows = tables[p * G:(p + 1) * G]
        full = w.prefix_len // w.block_size
        k = 0
        while k < full and np.all(rows[:, k] == rows[0, k]):
            k += 1
        pre[p * G:(p + 1) * G] = k
    starts = np.arange(0, n_prompt * G + 1, G, dtype=np.int32)
    own = ctx - pre.astype(np.int64) * w.block_size
    return PrefixGroups(torch.as_tensor(starts, device=device), torch.as_tensor(pre, device=device),
                        int(pre.max()) if S else 0, int(own.max()) if S else 0, G,
                        visit_order(own, device))


def step_shared_prefix(pw: PagedWorkload, out: List[torch.Tensor], groups, workspace,
                       partition_size: Optional[int] = None, stream=None) -> None:
    """One decode step over every layer with the shared-prefix decode."""
    P = pw.w.partition_size if partition_size is None else partition_size
    for layer, st in enumerate(pw.layers):
        pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                           st.k_scale, st.v_scale, stream)
        pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                          pw.context_lens, pw.w.scale, groups.max_own_context,
                                          groups.group_start, groups.prefix_blocks,
                                          groups.max_prefix_blocks, P,
                                          groups.max_group_members, out=out[layer],
                                          workspace=workspace, k_scale=st.k_scale,
                                          v_scale=st.v_scale, stream=stream,
                                          seq_order=groups.visit_order)


# ---- several GPUs: sequences are independent, so every rank runs its own
# batch (weak scaling, no collective on the data path); only the timing is
# combined across ranks.
def rank_workload(w: synth.Workload, rank: int, world: int) -> synth.Workload:
    """The batch of one rank: the same shapes with the rank's own seed."""
    import dataclasses
    if world <= 1:
        return w
    return dataclasses.replace(w, seed=w.seed + 100 * rank)


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of the ranks' values (e.g. elapsed milliseconds)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's step time."""
    return bytes_per_rank_step * world / (ms_per_step / 1e3) / 1e9
