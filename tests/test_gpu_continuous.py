"""Decode iterations driven by the continuous-batching scheduler: requests
arrive, run, finish and free their blocks while others are admitted; the
outputs of every running request match the oracle at sampled iterations and
the pool is whole again at the end."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, bits16

pytestmark = pytest.mark.gpu


def _oracle(cb, ids, ctx):
    q = np.stack([bits16(synth.request_query(cb.seed, 0, int(r), int(c) - 1, cb.Hq, cb.D))
                  for r, c in zip(ids, ctx)])
    ks = [bits16(synth.request_rows(cb.seed, synth.KIND_K, 0, int(r), 0, int(c), cb.Hk, cb.D))
          for r, c in zip(ids, ctx)]
    vs = [bits16(synth.request_rows(cb.seed, synth.KIND_V, 0, int(r), 0, int(c), cb.Hk, cb.D))
          for r, c in zip(ids, ctx)]
    return oracle.decode(q, ks, vs, cb.scale)


@pytest.mark.parametrize("P,pool,order", [(512, 400, "admission"), (0, 160, "admission"),
                                          (512, 400, "longest_first")])
def test_continuous_batching_iterations_match_oracle(P, pool, order):
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    reqs = synth.request_mix(11, 40, prompt_lo=16, prompt_hi=1500, gen_lo=4, gen_hi=200)
    cb = workload.ContinuousBatch(31, reqs, num_blocks=pool, block_size=32, max_num_seqs=12,
                                  partition_size=P, batch_order=order)
    it, checked, preempted = 0, 0, 0
    while not cb.done() and it < 5000:
        r = cb.step()
        it += 1
        preempted += len(cb.sched.events(2))
        if r is None:
            continue
        ids, ctx, out = r
        if order == "longest_first":
            assert all(int(ctx[k]) >= int(ctx[k + 1]) for k in range(len(ctx) - 1))
        if it % 37 == 1:
            torch.cuda.synchronize()
            assert_close(out.cpu(), _oracle(cb, ids, ctx), "iteration %d" % it)
            checked += 1
    assert cb.done() and checked >= 3
    assert cb.alloc.stats()["free_blocks"] == pool
    assert cb.tokens == sum(g for _, _, g in reqs) + 0 or preempted > 0
    assert int(flag.item()) == 0
    pkv.set_device_check(None)


def test_continuous_batching_with_swap_preemption():
    """Swap-mode preemption: preempted requests' blocks go to pinned host
    memory and come back into fresh blocks; decode outputs of every checked
    iteration match the oracle and no request is prefilled twice."""
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    # long generations on a small pool: running requests outgrow what their
    # admission reserved, so the pool runs dry and requests are swapped
    reqs = synth.request_mix(13, 40, prompt_lo=16, prompt_hi=600, gen_lo=100, gen_hi=600)
    cb = workload.ContinuousBatch(37, reqs, num_blocks=100, block_size=32, max_num_seqs=12,
                                  partition_size=512, preemption="swap")
    it, checked, admitted = 0, 0, []
    while not cb.done() and it < 5000:
        r = cb.step()
        it += 1
        admitted += cb.sched.events(0).tolist()
        if r is None:
            continue
        ids, ctx, out = r
        if it % 23 == 1 or len(cb.sched.events(4)):
            torch.cuda.synchronize()
            assert_close(out.cpu(), _oracle(cb, ids, ctx), "iteration %d" % it)
            checked += 1
    torch.cuda.synchronize()
    assert cb.done() and checked >= 3
    assert cb.swaps > 0 and not cb.saved
    assert sorted(admitted) == sorted(r for r, _, _ in reqs)     # nothing recomputed
    assert cb.tokens == sum(g for _, _, g in reqs)
    assert cb.alloc.stats()["free_blocks"] == 100
    assert int(flag.item()) == 0
    pkv.set_device_check(None)


@pytest.mark.parametrize("preemption", ["recompute", "swap"])
def test_sampled_requests_share_prompt_blocks(preemption):
    """Requests of 1-4 samples of one prompt: the samples share the prompt's
    blocks, copy-on-write clones are made with copy_blocks, and the decode
    of every checked iteration matches the oracle on each sample's logical
    rows (the prompt's, then its own), under preemption."""
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    rng = np.random.default_rng(17)
    reqs = [(8 * i, int(rng.integers(20, 300)), int(rng.integers(4, 120)),
             int(rng.integers(1, 5))) for i in range(16)]
    cb = workload.ContinuousBatch(43, reqs, num_blocks=90, block_size=16, max_num_seqs=12,
                                  partition_size=64, preemption=preemption)
    it, checked, preempted = 0, 0, 0
    while not cb.done() and it < 5000:
        r = cb.step()
        it += 1
        preempted += len(cb.sched.events(2))
        if r is None:
            continue
        ids, ctx, out = r
        if it % 23 == 1:
            torch.cuda.synchronize()
            q = np.stack([bits16(synth.request_query(cb.seed, 0, int(i), int(c) - 1, cb.Hq,
                                                     cb.D)) for i, c in zip(ids, ctx)])
            ks = [bits16(cb.rows(synth.KIND_K, int(i), 0, int(c), "cpu"))
                  for i, c in zip(ids, ctx)]
            vs = [bits16(cb.rows(synth.KIND_V, int(i), 0, int(c), "cpu"))
                  for i, c in zip(ids, ctx)]
            assert_close(out.cpu(), oracle.decode(q, ks, vs, cb.scale), "iteration %d" % it)
            checked += 1
    assert cb.done() and checked >= 3
    assert cb.cow_copies > 0 and preempted > 0
    assert cb.alloc.stats()["free_blocks"] == 90
    assert int(flag.item()) == 0
    pkv.set_device_check(None)
