"""The decode's visit order (seq_order): the CTAs take the sequences in the
given order, and nothing else changes.

Each sequence's arithmetic is the same whatever the order, so every ordered
result must equal the batch-order result bit for bit: the split decode + merge,
the one-pass decode, and the shared-prefix decode, on bf16 and E4M3 pools,
for the longest-first order, its reverse and a random permutation. The
longest-first result is also compared with the oracle. An entry outside the
batch is reported in the error word and its CTAs write nothing."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, expected, host_fp8_scales

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _orders(lengths, seed):
    S = len(lengths)
    lf = pkv.longest_first_order(lengths)
    rnd = np.random.default_rng(seed).permutation(S).astype(np.int32)
    return {"longest first": lf, "shortest first": lf[::-1].copy(), "random": rnd}


@pytest.mark.parametrize("fp8,B,P", [(False, 16, 64), (False, 32, 512), (True, 32, 64),
                                     (True, 16, 48), (False, 16, 0), (True, 32, 0), (True, 16, 0)])
def test_order_gives_the_same_bits(fp8, B, P, _lib):
    ctx = [1, 700, 31, 2000, B, 5, 1500, 64, 333, 1200, 17, 900]
    w = synth.Workload("order", 1500 + B + P + (3 if fp8 else 0), 24, 4, 256, B, ctx, fp8=fp8,
                       partition_size=P, slack_blocks=8)
    pw = workload.build(w)
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                       st.k_scale, st.v_scale)

    def run(order):
        return pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                   pw.context_lens, w.scale, pw.max_context, P, st.k_scale,
                                   st.v_scale, seq_order=order)

    base = run(None)
    torch.cuda.synchronize()
    for name, order in _orders(ctx, B + P).items():
        got = run(torch.as_tensor(order, device="cuda"))
        torch.cuda.synchronize()
        assert _same_bits(got, base), name
    assert int(_lib.item()) == 0
    ks = vs = None
    if fp8:
        ks, vs = host_fp8_scales(w, 0)
    assert_close(got.cpu(), expected(w, 0, range(w.num_seqs), ks, vs), "ordered vs oracle")


@pytest.mark.parametrize("fp8", [False, True])
def test_shared_prefix_order_gives_the_same_bits(fp8, _lib):
    w = synth.cow(prompt_len=300, prompts=3, rollouts=8)
    comp = w.extra["completion"]
    w = dataclasses.replace(w, ctx=[300 + (c % 500) + 1 for c in comp], fp8=fp8)
    pw = workload.build(w)
    groups = workload.prefix_groups(pw)
    assert groups.visit_order is not None
    own = np.asarray(w.ctx) - groups.prefix_blocks.cpu().numpy() * w.block_size
    assert groups.visit_order.cpu().numpy().tolist() == pkv.longest_first_order(own).tolist()
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                       st.k_scale, st.v_scale)
    P = 64

    def run(order):
        return pkv.paged_attention_shared_prefix(
            st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens, w.scale,
            groups.max_own_context, groups.group_start, groups.prefix_blocks,
            groups.max_prefix_blocks, P, groups.max_group_members, k_scale=st.k_scale,
            v_scale=st.v_scale, seq_order=order)

    base = run(None)
    torch.cuda.synchronize()
    for name, order in _orders(own, 7).items():
        got = run(torch.as_tensor(order, device="cuda"))
        torch.cuda.synchronize()
        assert _same_bits(got, base), name
    assert int(_lib.item()) == 0
    ks = vs = None
    if fp8:
        ks, vs = host_fp8_scales(w, 0)
    assert_close(base.cpu(), expected(w, 0, range(w.num_seqs), ks, vs), "shared prefix")


def test_order_entry_outside_the_batch_is_reported(_lib):
    """One entry names a sequence past the batch: the error word says so, the
    CTAs of that entry write nothing, every other sequence is unchanged."""
    pw = workload.build(synth.tiny())
    w = pw.w
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache)
    base = pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens,
                               w.scale, pw.max_context, 0)
    torch.cuda.synchronize()
    S = w.num_seqs
    order = np.arange(S, dtype=np.int32)[::-1].copy()
    skipped = int(order[1])
    order[1] = S                                   # outside [0, S)
    out = torch.full_like(st.q, float("nan"))
    pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens,
                        w.scale, pw.max_context, 0, out=out,
                        seq_order=torch.as_tensor(order, device="cuda"))
    torch.cuda.synchronize()
    assert int(_lib.item()) == pkv.DEVERR_ORDER
    _lib.zero_()
    keep = [s for s in range(S) if s != skipped]
    assert _same_bits(out[keep], base[keep])
    assert torch.isnan(out[skipped].float()).all()
