"""Continuous-batching scheduler on the host: iteration-level admission and
ejection, blocks returned at EOS, invariants, preemption under pressure."""
import numpy as np
import pytest

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build, synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _check(alloc, sched, B):
    ids, ctx, slots = sched.running()
    tables = sched.block_tables(4096)
    assert len(set(slots.tolist())) == len(slots)
    for i in range(len(ids)):
        nb = int((tables[i] >= 0).sum())
        assert nb == -(-int(ctx[i]) // B)
        pos = int(ctx[i]) - 1
        assert int(slots[i]) == int(tables[i][pos // B]) * B + pos % B
    st = alloc.stats()
    assert st["free_blocks"] + st["used_blocks"] == alloc.num_blocks
    assert st["used_slots"] == int(ctx.sum())


def test_iteration_level_eject_and_admit():
    """The pages' straggler example: budgets 50, 120, 240 and 1024 tokens with
    room for two at a time. A finished request's slot is taken by the next
    waiting request in the very next iteration."""
    B = 16
    alloc = pkv.BlockAllocator(1024, B, seed=1)
    sched = pkv.Scheduler(alloc, max_num_seqs=2)
    budgets = [50, 120, 240, 1024]
    for i, g in enumerate(budgets):
        sched.add_request(i, 10, g)
    admitted_at, finished_at = {}, {}
    step = 0
    while True:
        n, na, nf = sched.step()
        step += 1
        for r in sched.events(0):
            admitted_at[int(r)] = step
        for r in sched.events(1):
            finished_at[int(r)] = step
        if n == 0 and sched.counts()["waiting"] == 0:
            break
        _check(alloc, sched, B)
        assert n <= 2
    assert admitted_at == {0: 1, 1: 1, 2: 51, 3: 121}
    assert finished_at == {0: 51, 1: 121, 2: 291, 3: 1145}
    assert alloc.stats()["used_blocks"] == 0 and alloc.stats()["free_blocks"] == 1024


def test_context_grows_one_token_per_iteration():
    alloc = pkv.BlockAllocator(64, 4, seed=2)
    sched = pkv.Scheduler(alloc, max_num_seqs=8)
    for i, (p, g) in enumerate([(3, 2), (5, 1), (2, 3)]):
        sched.add_request(i, p, g)
    sched.step()
    ids, ctx, _ = sched.running()
    assert ids.tolist() == [0, 1, 2] and ctx.tolist() == [4, 6, 3]
    for i in ids:
        assert len(sched.prompt_slots(int(i))) == [3, 5, 2][int(i)]
    sched.step()
    ids, ctx, _ = sched.running()
    assert ids.tolist() == [0, 2] and ctx.tolist() == [5, 4]
    assert sched.events(1).tolist() == [1]
    sched.step()
    ids, ctx, _ = sched.running()
    assert ids.tolist() == [2] and ctx.tolist() == [5]
    n, _, nf = sched.step()
    assert n == 0 and nf == 1
    assert alloc.stats()["used_blocks"] == 0


def test_admission_waits_for_free_blocks():
    B = 16
    alloc = pkv.BlockAllocator(10, B, seed=3)
    sched = pkv.Scheduler(alloc, max_num_seqs=16)
    sched.add_request(0, 100, 5)     # 7 blocks with its first token
    sched.add_request(1, 60, 5)      # needs 4 more: waits
    n, na, _ = sched.step()
    assert (n, na) == (1, 1)
    for _ in range(5):
        sched.step()
    assert 1 in sched.events(0).tolist()


def test_preemption_requeues_and_everything_finishes():
    B = 16
    alloc = pkv.BlockAllocator(40, B, seed=4)
    sched = pkv.Scheduler(alloc, max_num_seqs=8)
    reqs = synth.request_mix(7, 24, prompt_lo=16, prompt_hi=200, gen_lo=16, gen_hi=300)
    for rid, p, g in reqs:
        sched.add_request(rid, p, g)
    done, preempted = set(), 0
    for _ in range(20000):
        n, _, _ = sched.step()
        done |= set(sched.events(1).tolist())
        preempted += len(sched.events(2))
        if n:
            _check(alloc, sched, B)
        if n == 0 and sched.counts()["waiting"] == 0:
            break
    assert done == set(range(24))
    assert preempted > 0
    assert alloc.stats()["free_blocks"] == 40


def test_bad_arguments():
    alloc = pkv.BlockAllocator(8, 16)
    sched = pkv.Scheduler(alloc, 4)
    with pytest.raises(pkv.PagedKVError):
        sched.add_request(0, 10, 0)
    with pytest.raises(pkv.PagedKVError):
        sched.prompt_slots(5)


def test_swap_preemption_keeps_progress_and_cache_contents():
    """Swap mode on a host model of the pool: every slot holds the identity
    of the token written there. Swapped-out blocks are saved before this
    iteration's writes, restored into the fresh blocks on resume, and every
    running request's table always reads back its own tokens 0..ctx-1; no
    request is admitted (prefilled) twice."""
    B = 16
    NB = 40
    alloc = pkv.BlockAllocator(NB, B, seed=5)
    sched = pkv.Scheduler(alloc, max_num_seqs=8)
    sched.set_preemption(pkv.PKV_PREEMPT_SWAP)
    reqs = synth.request_mix(11, 24, prompt_lo=16, prompt_hi=200, gen_lo=16, gen_hi=300)
    for rid, p, g in reqs:
        sched.add_request(rid, p, g)
    pool = np.full((NB, B), -1, dtype=np.int64)
    saved = {}

    def tok(rid, pos):
        return int(rid) * 1_000_000 + int(pos)

    admitted, done = [], set()
    swaps_out = swaps_in = 0
    for _ in range(20000):
        n, _, _ = sched.step()
        for rid in sched.events(3):
            blocks = sched.swap_blocks(int(rid))
            saved[int(rid)] = pool[blocks].copy()
            swaps_out += 1
        for rid in sched.events(4):
            blocks = sched.swap_blocks(int(rid))
            rows = saved.pop(int(rid))
            assert rows.shape[0] == len(blocks)
            pool[blocks] = rows
            swaps_in += 1
        for rid in sched.events(0):
            admitted.append(int(rid))
            for pos, slot in enumerate(sched.prompt_slots(int(rid))):
                pool[slot // B, slot % B] = tok(rid, pos)
        done |= set(sched.events(1).tolist())
        if n:
            ids, ctx, slots = sched.running()
            for rid, c, slot in zip(ids, ctx, slots):
                pool[slot // B, slot % B] = tok(rid, c - 1)
            tables = sched.block_tables(4096)
            for i, (rid, c) in enumerate(zip(ids, ctx)):
                got = [pool[tables[i][pos // B], pos % B] for pos in range(int(c))]
                assert got == [tok(rid, pos) for pos in range(int(c))]
            _check(alloc, sched, B)
        if n == 0 and sched.counts()["waiting"] == 0:
            break
    assert done == set(range(24))
    assert swaps_out > 0 and swaps_in == swaps_out and not saved
    assert sorted(admitted) == list(range(24))       # nothing prefilled twice
    assert alloc.stats()["free_blocks"] == NB


def test_swap_mode_arguments():
    alloc = pkv.BlockAllocator(8, 16)
    sched = pkv.Scheduler(alloc, 4)
    with pytest.raises(pkv.PagedKVError):
        sched.set_preemption(7)
    with pytest.raises(pkv.PagedKVError):
        sched.swap_blocks(3)


def test_longest_first_batch_order():
    """Two schedulers on the same requests and the same seeded pool, one
    reporting in admission order and one longest first: every iteration gives
    the same rows (request, context, slot, block-table row), the second
    sorted by decreasing context with ties in admission order; preemption
    and completion are unchanged."""
    B = 16
    reqs = synth.request_mix(11, 30, prompt_lo=16, prompt_hi=400, gen_lo=8, gen_hi=200)
    runs = []
    for order in (pkv.PKV_BATCH_ADMISSION, pkv.PKV_BATCH_LONGEST_FIRST):
        alloc = pkv.BlockAllocator(120, B, seed=5)
        sched = pkv.Scheduler(alloc, max_num_seqs=12)
        sched.set_batch_order(order)
        for rid, p, g in reqs:
            sched.add_request(rid, p, g)
        runs.append((alloc, sched))
    steps = 0
    while True:
        rows = []
        for alloc, sched in runs:
            n, _, _ = sched.step()
            ids, ctx, slots = sched.running()
            tables = sched.block_tables(64)
            rows.append((n, ids, ctx, slots, tables, sched.events(2).tolist()))
            if n:
                _check(alloc, sched, B)
        (n0, i0, c0, s0, t0, p0), (n1, i1, c1, s1, t1, p1) = rows
        assert n0 == n1 and p0 == p1
        if n0 == 0 and runs[0][1].counts()["waiting"] == 0:
            break
        key = sorted(range(n0), key=lambda k: -int(c0[k]))  # stable: ties keep admission order
        assert i1.tolist() == [int(i0[k]) for k in key]
        assert c1.tolist() == [int(c0[k]) for k in key]
        assert s1.tolist() == [int(s0[k]) for k in key]
        assert np.array_equal(t1, t0[key])
        assert all(c1[k] >= c1[k + 1] for k in range(n1 - 1))
        steps += 1
    assert steps > 50
    with pytest.raises(pkv.PagedKVError):
        runs[0][1].set_batch_order(7)


@pytest.mark.parametrize("mode", [pkv.PKV_PREEMPT_RECOMPUTE, pkv.PKV_PREEMPT_SWAP])
def test_sampled_requests_share_the_prompt_with_copy_on_write(mode):
    """Requests of n samples on a host model of the pool (every slot holds
    the identity of the token written there), under preemption: the prompt
    is stored once and shared by the samples' tables; the copy-on-write
    pairs, applied as whole-block copies after the prompts and before this
    iteration's tokens, keep every sample reading the prompt's tokens
    followed by its own through its table, swapped samples included."""
    B, NB = 8, 48
    alloc = pkv.BlockAllocator(NB, B, seed=21)
    sched = pkv.Scheduler(alloc, max_num_seqs=12)
    sched.set_preemption(mode)
    rng = np.random.default_rng(5)
    base_of, plen_of, total = {}, {}, 0
    for g in range(14):
        base, p, n = 16 * g, int(rng.integers(3, 40)), int(rng.integers(1, 5))
        gen = int(rng.integers(4, 120))
        sched.add_request(base, p, gen, n=n)
        for k in range(n):
            base_of[base + k], plen_of[base + k] = base, p
        total += n
    pool = np.full((NB, B), -1, dtype=np.int64)
    saved = {}

    def want(rid, pos):
        if pos < plen_of[rid]:
            return -(base_of[rid] * 1_000_000 + pos) - 1   # the shared prompt
        return rid * 1_000_000 + pos

    done, pairs_seen, shared_seen, prefills, preempted = set(), 0, 0, 0, 0
    for _ in range(20000):
        n, _, _ = sched.step()
        preempted += len(sched.events(2))
        for rid in sched.events(3):
            saved[int(rid)] = pool[sched.swap_blocks(int(rid))].copy()
        for rid in sched.events(4):
            pool[sched.swap_blocks(int(rid))] = saved.pop(int(rid))
        for rid in sched.events(0):
            slots = sched.prompt_slots(int(rid))
            prefills += len(slots) > 0
            for pos, slot in enumerate(slots):
                pool[slot // B, slot % B] = want(int(rid), pos)
        pairs = sched.cow_pairs()
        pairs_seen += len(pairs)
        for src, dst in pairs.tolist():
            pool[dst] = pool[src]
        done |= set(sched.events(1).tolist())
        if n:
            ids, ctx, slots = sched.running()
            assert len(set(slots.tolist())) == len(slots)
            for rid, c, slot in zip(ids, ctx, slots):
                pool[slot // B, slot % B] = want(int(rid), int(c) - 1)
            tables = sched.block_tables(256)
            for i, (rid, c) in enumerate(zip(ids, ctx)):
                assert len([b for b in tables[i] if b >= 0]) == -(-int(c) // B)
                got = [int(pool[tables[i][pos // B], pos % B]) for pos in range(int(c))]
                assert got == [want(int(rid), pos) for pos in range(int(c))], int(rid)
            st = alloc.stats()
            assert st["free_blocks"] + st["used_blocks"] == NB
            shared_seen += st["used_slots"] < int(ctx.sum())
        if n == 0 and sched.counts()["waiting"] == 0:
            break
    assert done == set(base_of)
    assert pairs_seen > 0 and shared_seen > 0 and not saved
    assert prefills >= 14
    assert sched.counts()["running"] == 0 and alloc.stats()["free_blocks"] == NB
    assert preempted > 0


def test_sampled_request_arguments():
    alloc = pkv.BlockAllocator(8, 16)
    sched = pkv.Scheduler(alloc, 4)
    with pytest.raises(pkv.PagedKVError):
        sched.add_request(0, 10, 5, n=0)
    with pytest.raises(pkv.PagedKVError):
        sched.add_request(0, 10, 5, n=5)        # more samples than batch rows
    assert sched.cow_pairs().shape == (0, 2)


def test_request_ids_must_not_collide_with_live_requests():
    """Samples take ids id .. id + n - 1; an id still waiting, running or
    swapped out is rejected (the id lookups would find the wrong request),
    a finished one may be reused."""
    a = pkv.BlockAllocator(64, 4, seed=3)
    s = pkv.Scheduler(a, 8)
    s.add_request(10, 6, 2, n=3)                        # ids 10, 11, 12
    for rid, n in ((12, 1), (8, 3), (11, 2), (-1, 1)):
        with pytest.raises(pkv.PagedKVError) as e:
            s.add_request(rid, 4, 2, n=n)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    s.add_request(13, 4, 1)                             # adjacent ids are fine
    s.step()                                            # all admitted: running now
    with pytest.raises(pkv.PagedKVError):
        s.add_request(11, 4, 2)
    while not (s.counts()["running"] == 0 and s.counts()["waiting"] == 0):
        s.step()
    s.add_request(11, 4, 2)                             # finished ids are free again
    s.close()
    a.close()
