"""Shared-prefix decode: rollouts of one prompt read the prompt's pages once
per group; the output matches the oracle and the plain split decode."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import (MAX_ABS, REL_L2, assert_close, bits16, errors, expected,
                          host_fp8_scales, host_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


@pytest.mark.parametrize("prompt,B,P,rollouts,d", [(40, 16, 32, 4, 256), (48, 16, 16, 16, 256),
                                                    (2040, 16, 512, 16, 256), (200, 32, 64, 3, 256),
                                                    (100, 16, 512, 21, 256), (300, 16, 64, 16, 128),
                                                    (330, 32, 128, 5, 128),
                                                    (300, 16, 64, 32, 256),
                                                    (130, 32, 64, 64, 128)])
def test_shared_prefix_matches_oracle(prompt, B, P, rollouts, d, _lib):
    w = synth.cow(prompt_len=prompt, prompts=2, rollouts=rollouts)
    comp = w.extra["completion"][:2 * rollouts]
    w = dataclasses.replace(w, block_size=B, head_dim=d, ctx=[prompt + (c % 300) + 1 for c in comp],
                            slack_blocks=64)
    pw = workload.build(w)
    groups = workload.prefix_groups(pw)
    assert groups.max_prefix_blocks == prompt // B
    assert groups.max_group_members == rollouts     # > 128 query rows: several row tiles
    out = [torch.empty_like(pw.layers[0].q)]
    workload.step_shared_prefix(pw, out, groups, None, P)
    torch.cuda.synchronize()
    ref = expected(w, 0, range(w.num_seqs))
    assert_close(out[0].cpu(), ref, "shared prefix %d" % prompt)
    # the plain split decode over the same state agrees within tolerance
    ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, P)
    plain = torch.empty_like(out[0])
    st = pw.layers[0]
    pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens, w.scale,
                        pw.max_context, P, out=plain, workspace=ws)
    torch.cuda.synchronize()
    ma, rl = errors(out[0].cpu(), plain.cpu().double().numpy())
    assert ma <= MAX_ABS and rl <= REL_L2
    assert int(_lib.item()) == 0


def test_shared_prefix_mixed_with_ungrouped_and_exact_prefix(_lib):
    """Groups of one, a member whose context ends right at the prefix."""
    w = synth.cow(prompt_len=64, prompts=2, rollouts=4)
    w = dataclasses.replace(w, ctx=[65, 66, 90, 65, 70, 71, 72, 200])
    pw = workload.build(w)
    gs, pre, mp, _, _, _ = workload.prefix_groups(pw)
    # split the second prompt's group into singletons without a shared prefix
    gs2 = torch.tensor([0, 4], dtype=torch.int32, device="cuda")
    pre2 = pre.clone()
    pre2[4:] = 0
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache)
    out = pkv.paged_attention_shared_prefix(pw.layers[0].q, pw.layers[0].k_cache,
                                            pw.layers[0].v_cache, pw.block_tables,
                                            pw.context_lens, w.scale, pw.max_context, gs2, pre2,
                                            mp, 32, 4)
    torch.cuda.synchronize()
    assert_close(out.cpu(), expected(w, 0, range(w.num_seqs)), "mixed groups")


def test_shared_prefix_graph_replay_matches_eager(_lib):
    """The prefix kernel and the members' own-block decode may run at the same
    time (the decode is a programmatic dependent launch); recorded in a CUDA
    graph, the step replays bit-identical to eager launches, twice in a row,
    and agrees with the oracle."""
    w = synth.cow(prompt_len=2040, prompts=4, rollouts=16)
    pw = workload.build(w)
    groups = workload.prefix_groups(pw)
    P = w.partition_size
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, groups.max_own_context,
                                     groups.max_prefix_blocks * w.block_size, P)
    eager = [torch.empty_like(pw.layers[0].q)]
    workload.step_shared_prefix(pw, eager, groups, ws, P)
    torch.cuda.synchronize()
    ref = eager[0].clone()
    out = [torch.empty_like(ref)]
    g = workload.capture_step(pw, out, ws, P, groups=groups)
    for _ in range(2):
        out[0].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out[0].view(torch.int16), ref.view(torch.int16))
    assert_close(out[0].cpu(), expected(w, 0, range(w.num_seqs)), "shared prefix graph")
    assert int(_lib.item()) == 0


def test_shared_prefix_own_part_bound(_lib):
    """max_own_context sizes the own-part grid: the longest own part gives
    the bits of the loose bound (the longest context); a bound below an own
    part is reported (PKV_DEVERR_CONTEXT), and nothing past the launched
    partitions is read."""
    w = synth.cow(prompt_len=2040, prompts=2, rollouts=16)
    pw = workload.build(w)
    gs, pre, mp, own, mm, _ = workload.prefix_groups(pw)
    assert own < pw.max_context - 2000
    P = 512                               # own parts in two partitions
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache)
    outs = [pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                              pw.context_lens, w.scale, bound, gs, pre, mp, P, mm)
            for bound in (own, pw.max_context)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert int(_lib.item()) == 0
    assert_close(outs[0].cpu(), expected(w, 0, range(w.num_seqs)), "own-part bound")
    short = pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                              pw.context_lens, w.scale, own - P, gs, pre, mp, P,
                                              mm)
    torch.cuda.synchronize()
    assert int(_lib.item()) == pkv.DEVERR_CONTEXT
    assert torch.isfinite(short.float()).all()
    _lib.zero_()


def test_shared_prefix_group_above_declared_bound(_lib):
    """A group with more members than max_group_members: the error word says
    so, the members a row tile covers are exact, and the uncovered members'
    result is the attention over their own rows only (their shared partials
    are written empty), never stale workspace."""
    w = synth.cow(prompt_len=256, prompts=2, rollouts=32)
    comp = w.extra["completion"]
    w = dataclasses.replace(w, ctx=[256 + (c % 200) + 1 for c in comp])
    pw = workload.build(w)
    gs, pre, mp, own, mm, _ = workload.prefix_groups(pw)
    assert mm == 32
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache)
    per_tile = 128 // (w.num_heads // w.num_kv_heads)            # 21 members at g = 6
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, own,
                                     mp * w.block_size, 64)
    ws.view(torch.float32).fill_(float("nan"))
    out = pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                            pw.context_lens, w.scale, own, gs, pre, mp, 64,
                                            per_tile, workspace=ws)
    torch.cuda.synchronize()
    assert int(_lib.item()) == pkv.DEVERR_CONTEXT
    _lib.zero_()
    got = out.cpu()
    covered = [p * 32 + r for p in range(2) for r in range(per_tile)]
    assert_close(got[covered], expected(w, 0, covered), "covered members")
    uncovered = [p * 32 + r for p in range(2) for r in range(per_tile, 32)]
    B = w.block_size
    q = bits16(w.q(0, "cpu"))[uncovered]
    ks, vs = [], []
    for s in uncovered:
        K, V = host_rows(w, 0, s)
        t0 = int(pre[s]) * B
        ks.append(bits16(K)[t0:])
        vs.append(bits16(V)[t0:])
    own_only = oracle.decode(q, ks, vs, w.scale)
    assert_close(got[uncovered], own_only, "uncovered members: own rows only")


@pytest.mark.parametrize("prompt,B,P,rollouts,d", [(40, 16, 32, 4, 256), (2040, 16, 512, 16, 256),
                                                    (200, 32, 64, 3, 256), (300, 16, 64, 32, 256),
                                                    (330, 32, 128, 5, 128), (100, 32, 64, 8, 128)])
def test_shared_prefix_fp8_matches_oracle(prompt, B, P, rollouts, d, _lib):
    """E4M3 pools: the shared pages' codes become f16 operands of the
    group product; the result matches the oracle on the same codes (scales
    recomputed on the host) and the plain split decode over the same pool."""
    w = synth.cow(prompt_len=prompt, prompts=2, rollouts=rollouts)
    comp = w.extra["completion"][:2 * rollouts]
    w = dataclasses.replace(w, block_size=B, head_dim=d, fp8=True,
                            ctx=[prompt + (c % 300) + 1 for c in comp], slack_blocks=64)
    pw = workload.build(w)
    st = pw.layers[0]
    ks, vs = host_fp8_scales(w, 0)
    assert np.array_equal(ks.view(np.uint32), st.k_scale.cpu().numpy().view(np.uint32))
    groups = workload.prefix_groups(pw)
    assert groups.max_prefix_blocks == prompt // B
    out = [torch.empty_like(st.q)]
    workload.step_shared_prefix(pw, out, groups, None, P)
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    ref = expected(w, 0, range(w.num_seqs), ks, vs)
    assert_close(out[0].cpu(), ref, "fp8 shared prefix %d" % prompt)
    plain = pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens,
                                w.scale, pw.max_context, P, st.k_scale, st.v_scale)
    torch.cuda.synchronize()
    ma, rl = errors(out[0].cpu(), plain.cpu().double().numpy())
    assert ma <= MAX_ABS and rl <= REL_L2
