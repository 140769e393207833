"""Host block allocator: the worked example of Figures 1-2, the invariants the
pages state, copy-on-write, exhaustion and determinism."""
import json
import os

import numpy as np
import pytest

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build, synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _check_invariants(a, seqs):
    """blocks(seq) = ceil(len/B); sum of refcounts = sum of table lengths;
    free + used = NB; a block is held by as many tables as its refcount."""
    B = a.block_size
    held = {}
    for s in seqs:
        t = a.block_table(s)
        assert len(t) == -(-a.seq_len(s) // B)
        for b in t:
            held[int(b)] = held.get(int(b), 0) + 1
    for b in range(a.num_blocks):
        assert a.refcount(b) == held.get(b, 0)
    st = a.stats()
    assert st["free_blocks"] + st["used_blocks"] == a.num_blocks
    assert st["used_blocks"] == len(held)


def test_figures_1_2_worked_example():
    g = json.load(open(os.path.join(GOLD, "figure_1_2_allocation.json")))
    B = g["block_size"]
    a = pkv.BlockAllocator(g["contiguous_reserved"] // B, B, seed=7)
    seqs = []
    for n in g["lengths"]:
        s = a.new_seq()
        a.append(s, n)
        seqs.append(s)
    st = a.stats()
    assert [len(a.block_table(s)) for s in seqs] == g["paged_blocks_per_request"]
    assert st["used_blocks"] * B == g["paged_reserved"]
    assert st["used_slots"] == g["used"]
    assert st["used_blocks"] * B - st["used_slots"] == g["paged_unused"]
    assert g["contiguous_reserved"] - st["used_blocks"] * B == g["freed_vs_contiguous"]
    ref = oracle.contiguous_vs_paged(g["lengths"], g["max_len"], B)
    assert ref["paged_reserved"] == st["used_blocks"] * B
    _check_invariants(a, seqs)


def test_only_last_block_has_free_slots_under_random_appends():
    rng = np.random.default_rng(0)
    a = pkv.BlockAllocator(4096, 16, seed=1)
    seqs = [a.new_seq() for _ in range(20)]
    for _ in range(200):
        s = seqs[rng.integers(len(seqs))]
        a.append(s, int(rng.integers(1, 40)))
    _check_invariants(a, seqs)
    # slots are distinct and land in the sequence's own table
    seen = set()
    for s in seqs:
        t = a.block_table(s)
        for pos in range(a.seq_len(s)):
            slot = int(t[pos // 16]) * 16 + pos % 16
            assert slot not in seen
            seen.add(slot)


def test_slots_follow_block_table():
    a = pkv.BlockAllocator(64, 16, seed=3)
    s = a.new_seq()
    slots, pairs = a.append(s, 40)
    t = a.block_table(s)
    assert len(pairs) == 0
    assert slots.tolist() == [int(t[p // 16]) * 16 + p % 16 for p in range(40)]
    more, _ = a.append(s, 1)
    assert int(more[0]) == int(t[2]) * 16 + 8


def test_fork_and_copy_on_write():
    B = 16
    a = pkv.BlockAllocator(64, B, seed=5)
    p = a.new_seq()
    a.append(p, 40)                       # 2 full blocks + 8 tokens
    kids = [a.fork(p) for _ in range(3)]
    last = a.block_table(p)[-1]
    assert a.refcount(int(last)) == 4
    _check_invariants(a, [p] + kids)
    # every sibling but the last to write clones the shared partial block
    emitted = []
    for s in kids + [p]:
        slots, pairs = a.append(s, 1)
        emitted.append([tuple(x) for x in pairs.tolist()])
        t = a.block_table(s)
        assert int(slots[0]) == int(t[2]) * B + 8
    assert [len(e) for e in emitted] == [1, 1, 1, 0]
    assert all(e[0][0] == int(last) for e in emitted[:3])
    assert a.refcount(int(last)) == 1 and int(a.block_table(p)[-1]) == int(last)
    # the full prefix blocks stay shared
    assert a.refcount(int(a.block_table(p)[0])) == 4
    _check_invariants(a, [p] + kids)
    # full shared last block: no copy, a new block
    q = a.new_seq()
    a.append(q, 32)
    r = a.fork(q)
    _, pairs = a.append(r, 1)
    assert len(pairs) == 0


def test_free_returns_blocks_lifo():
    a = pkv.BlockAllocator(32, 16, seed=9)
    s = a.new_seq()
    a.append(s, 48)
    t = a.block_table(s).tolist()
    a.free(s)
    assert a.stats()["free_blocks"] == 32
    s2 = a.new_seq()
    a.append(s2, 48)
    assert a.block_table(s2).tolist() == t       # last freed, first reused
    with pytest.raises(pkv.PagedKVError):
        a.free(s)                                 # already gone


def test_shared_blocks_survive_until_last_holder_frees():
    a = pkv.BlockAllocator(16, 16, seed=2)
    p = a.new_seq()
    a.append(p, 20)
    c = a.fork(p)
    a.free(p)
    assert a.stats()["used_blocks"] == 2
    assert all(a.refcount(int(b)) == 1 for b in a.block_table(c))
    a.free(c)
    assert a.stats()["used_blocks"] == 0


def test_out_of_blocks_leaves_state_unchanged():
    a = pkv.BlockAllocator(4, 16, seed=4)
    s = a.new_seq()
    a.append(s, 50)                               # 4 blocks
    before = (a.block_table(s).tolist(), a.seq_len(s), a.stats())
    with pytest.raises(pkv.PagedKVError) as e:
        a.append(s, 20)
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert (a.block_table(s).tolist(), a.seq_len(s), a.stats()) == before
    a.append(s, 14)                               # fills the last block exactly
    # copy-on-write needs a free block too
    b = pkv.BlockAllocator(3, 16, seed=4)
    p = b.new_seq()
    b.append(p, 40)
    c = b.fork(p)
    with pytest.raises(pkv.PagedKVError):
        b.append(c, 1)
    assert b.seq_len(c) == 40 and b.refcount(int(b.block_table(p)[-1])) == 2


def test_seeded_placement_is_deterministic():
    def tables(seed):
        a = pkv.BlockAllocator(256, 16, seed=seed)
        out = []
        for n in (50, 120, 240, 1024):
            s = a.new_seq()
            a.append(s, n)
            out.append(a.block_table(s).tolist())
        return out
    assert tables(11) == tables(11)
    assert tables(11) != tables(12)
    # the placement is a permutation, not the identity
    flat = sum(tables(11), [])
    assert flat != sorted(flat)


def test_unknown_sequence_and_bad_args():
    a = pkv.BlockAllocator(8, 16)
    with pytest.raises(pkv.PagedKVError) as e:
        a.append(99, 1)
    assert e.value.status == pkv.PKV_ERR_NOT_FOUND
    with pytest.raises(pkv.PagedKVError):
        pkv.BlockAllocator(0, 16)


def test_footprint_of_one_sequence_matches_closed_form():
    """One 8,192-token sequence of the 16-layer, 4-KV-head, d=256 BF16 layout
    occupies exactly the bytes of the footprint equation."""
    w = synth.qwen_like(num_seqs=1)
    a = pkv.BlockAllocator(w.pool_blocks(), w.block_size, seed=1)
    s = a.new_seq()
    a.append(s, 8192)
    page = w.block_size * w.num_kv_heads * w.head_dim * 2           # one block, all heads
    total = a.stats()["used_blocks"] * page * 2 * w.layers            # K and V, 16 layers
    assert total == oracle.kv_bytes(16, 4, 256, 8192, 2) == 2 ** 29


def test_mixed_lengths_internal_fragmentation():
    """Blocks allocated on demand leave only the last block part-empty: for
    the mixed-length workload (B = 32) the waste is far under 4 %."""
    w = synth.mixed()
    a = pkv.BlockAllocator(w.pool_blocks(), w.block_size, seed=w.seed)
    for c in w.ctx:
        s = a.new_seq()
        a.append(s, c)
    st = a.stats()
    frag = 1 - st["used_slots"] / (st["used_blocks"] * w.block_size)
    assert st["used_slots"] == sum(w.ctx)
    assert frag < 0.04


def _churn(a, rng, seqs, steps):
    """Random appends, forks and frees; returns the live sequences."""
    for _ in range(steps):
        op = rng.integers(0, 10)
        try:
            if op < 5 and seqs:
                a.append(seqs[int(rng.integers(0, len(seqs)))], int(rng.integers(1, 40)))
            elif op < 7 and seqs:
                seqs.append(a.fork(seqs[int(rng.integers(0, len(seqs)))]))
            elif op < 8 and seqs:
                a.free(seqs.pop(int(rng.integers(0, len(seqs)))))
            else:
                seqs.append(a.new_seq())
        except pkv.PagedKVError:
            pass                                 # pool exhausted: state unchanged
    return seqs


def test_checkpoint_round_trip_continues_identically():
    """A restored allocator holds the same tables, lengths, refcounts and
    free-list order: the same operations afterwards give the same slots and
    copy-on-write pairs on both."""
    rng = np.random.default_rng(21)
    a = pkv.BlockAllocator(96, 16, seed=9)
    seqs = _churn(a, rng, [], 300)
    rec = a.save()
    b = pkv.BlockAllocator.load(rec)
    assert b.save() == rec
    assert b.stats() == a.stats()
    for s in seqs:
        assert np.array_equal(a.block_table(s), b.block_table(s))
        assert a.seq_len(s) == b.seq_len(s)
    for blk in range(a.num_blocks):
        assert a.refcount(blk) == b.refcount(blk)
    _check_invariants(b, seqs)
    # identical futures
    def try_append(x, s, n):
        try:
            slots, pairs = x.append(s, n)
            return slots.tolist(), pairs.tolist()
        except pkv.PagedKVError as e:
            return str(e)

    for step in range(200):
        if not seqs:
            break
        s = seqs[step % len(seqs)]
        assert try_append(a, s, 1 + step % 7) == try_append(b, s, 1 + step % 7)
        if step % 50 == 49:
            a.free(seqs[0])
            b.free(seqs[0])
            seqs.pop(0)
    assert a.save() == b.save()


def test_checkpoint_rejects_inconsistent_records():
    a = pkv.BlockAllocator(32, 16, seed=2)
    s = a.new_seq()
    a.append(s, 40)
    a.fork(s)
    rec = np.frombuffer(a.save(), dtype="<i8").copy()

    def load(words):
        return pkv.BlockAllocator.load(words.astype("<i8").tobytes())

    load(rec)                                    # the record itself is fine
    bad = []
    r = rec.copy(); r[0] ^= 1; bad.append(r)                      # magic
    r = rec.copy(); r[2] = 0; bad.append(r)                       # num_blocks
    nfree = int(rec[5])
    r = rec.copy(); r[6] = rec[7]; bad.append(r)                  # a block free twice
    r = rec.copy(); r[6 + nfree + int(rec[6 + nfree - 1] if nfree else 0)] += 1; bad.append(r)
    r = rec.copy(); r[6 + nfree] += 1; bad.append(r)              # refcount of a block
    bad.append(rec[:-1])                                          # truncated
    bad.append(np.concatenate([rec, [0]]))                        # trailing data
    for r in bad:
        with pytest.raises(pkv.PagedKVError):
            load(r)


def test_random_operations_keep_every_sequence_readable():
    """A random mix of new / fork / append / free on a small pool, checked
    against a model of the pool's contents: every slot holds the label of
    the token last written there, copy-on-write pairs copy whole blocks (as
    copy_blocks does) before the new token is written, and after every
    operation each live sequence reads its own tokens through its block
    table (a fork's shared prefix reads the parent's tokens). A call that
    fails for lack of blocks leaves the whole state unchanged (compared
    through the checkpoint record); the invariants hold throughout."""
    B, NB = 4, 48
    a = pkv.BlockAllocator(NB, B, seed=13)
    rng = np.random.default_rng(2024)
    content = {}          # slot -> token label
    toks = {}             # live sequence -> its token labels, logical order
    next_label = [0]

    def label():
        next_label[0] += 1
        return next_label[0]

    def check():
        for s, tl in toks.items():
            t = a.block_table(s)
            assert a.seq_len(s) == len(tl)
            for i, lab in enumerate(tl):
                assert content.get(int(t[i // B]) * B + i % B) == lab, (s, i)
        _check_invariants(a, list(toks))

    failed = 0
    for _ in range(3000):
        op = rng.integers(0, 10)
        live = list(toks)
        if op == 0 or not live:
            toks[a.new_seq()] = []
        elif op == 1 and len(live) < 16:
            p = live[rng.integers(len(live))]
            toks[a.fork(p)] = list(toks[p])
        elif op == 2:
            s = live[rng.integers(len(live))]
            a.free(s)
            del toks[s]
        else:
            s = live[rng.integers(len(live))]
            n = int(rng.integers(1, 3 * B))
            before = a.save()
            try:
                slots, pairs = a.append(s, n)
            except pkv.PagedKVError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
                assert a.save() == before
                failed += 1
                continue
            for src, dst in pairs.tolist():
                for r in range(B):
                    if src * B + r in content:
                        content[dst * B + r] = content[src * B + r]
            for sl in slots.tolist():
                lab = label()
                content[int(sl)] = lab
                toks[s].append(lab)
        check()
    assert failed > 0 and next_label[0] > 1000
    for s in list(toks):
        a.free(s)
    assert a.stats()["free_blocks"] == NB
