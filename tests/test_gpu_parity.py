"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Cache writes, block copies and gathers are compared bit for bit; attention
outputs within MAX_ABS / REL_L2 (see _oracle_side). Small cases cover several
blocks, partitions and ragged tails; the edge sweep covers the degenerate
lengths.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import (assert_close, bits16, expected, expected_pool, errors, MAX_ABS,
                          REL_L2)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    pkv.lib()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


def _run_step(pw, P=None):
    out = [torch.empty_like(st.q) for st in pw.layers]
    P = pw.w.partition_size if P is None else P
    ws = None
    if P > 0:
        w = pw.w
        ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, P)
    workload.step(pw, out, ws, P)
    torch.cuda.synchronize()
    return out


def _scales(pw, layer):
    st = pw.layers[layer]
    if st.k_scale is None:
        return None, None
    return st.k_scale.cpu().numpy(), st.v_scale.cpu().numpy()


def _raw(t):
    return bits16(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _small(name, **kw):
    base = {"tiny": synth.tiny()}.get(name)
    return dataclasses.replace(base, **kw)


def test_generator_bit_identical_on_gpu_and_host():
    w = synth.mixed(num_seqs=4)
    for s in range(4):
        a = w.rows(synth.KIND_V, 0, s, 0, w.ctx[s], "cuda").cpu()
        b = w.rows(synth.KIND_V, 0, s, 0, w.ctx[s], "cpu")
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(w.q(0, "cuda").cpu().view(torch.int16), w.q(0, "cpu").view(torch.int16))


@pytest.mark.parametrize("fp8", [False, True])
def test_cache_write_bit_exact(fp8, _lib):
    w = dataclasses.replace(synth.tiny(), fp8=fp8)
    pw = workload.build(w)
    _run_step(pw, 0)                      # also writes row ctx-1 of every sequence
    for layer in range(w.layers):
        ks, vs = _scales(pw, layer)
        pk, pv = expected_pool(w, layer, pw.alloc.num_blocks, pw.history_slots, ks, vs)
        st = pw.layers[layer]
        got_k = _raw(st.k_cache)
        got_v = _raw(st.v_cache)
        assert np.array_equal(got_k, pk)
        assert np.array_equal(got_v, pv)
    assert int(_lib.item()) == 0


def test_cache_write_fp8_distinct_head_scales():
    """Hand-set per-head scales: head h must be divided by its own scale."""
    Hk, D, B, NB = 4, 256, 32, 8
    g = torch.Generator().manual_seed(3)
    k = (torch.randn(40, Hk, D, generator=g) * 50).to(torch.bfloat16)
    v = (torch.randn(40, Hk, D, generator=g) * 0.01).to(torch.bfloat16)
    slots = torch.randperm(NB * B, generator=g)[:40].to(torch.int64)
    slots[3] = -1
    ks = torch.tensor([0.01, 0.1, 1.0, 0.37], dtype=torch.float32)
    vs = torch.tensor([1e-4, 3e-5, 2e-3, 0.5], dtype=torch.float32)
    kc = torch.zeros(NB, Hk, B, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    pkv.kv_cache_write(k.cuda(), v.cuda(), slots.cuda(), kc, vc, ks.cuda(), vs.cuda())
    ek = np.zeros((NB, Hk, B, D), dtype=np.uint8)
    ev = np.zeros_like(ek)
    from _oracle_side import quantize
    oracle.scatter_rows(ek, quantize(k, ks.numpy()), slots.tolist())
    oracle.scatter_rows(ev, quantize(v, vs.numpy()), slots.tolist())
    assert np.array_equal(kc.cpu().numpy(), ek)
    assert np.array_equal(vc.cpu().numpy(), ev)


def test_fp8_encoder_matches_cuda_conversion_exhaustively():
    """All 65,536 bf16 inputs through the cache write (scale 1 and 0.37):
    the device codes equal the oracle's E4M3 encoder."""
    D = 128
    x = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = x[torch.isfinite(x.float())]
    n = (x.numel() // (2 * D)) * 2 * D
    x = x[:n].reshape(-1, 2, D)            # [T, Hk=2, D]
    T = x.shape[0]
    B = 16
    NB = -(-T // B)
    for sc in (1.0, 0.37):
        s = torch.full((2,), sc, dtype=torch.float32)
        kc = torch.zeros(NB, 2, B, D, dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        slots = torch.arange(T, dtype=torch.int64)
        pkv.kv_cache_write(x.cuda(), x.cuda(), slots.cuda(), kc, vc, s.cuda(), s.cuda())
        ek = np.zeros((NB, 2, B, D), dtype=np.uint8)
        from _oracle_side import quantize
        oracle.scatter_rows_fast(ek, quantize(x, s.numpy()), slots.numpy())
        assert np.array_equal(kc.cpu().numpy(), ek)


def test_copy_blocks_bit_exact(_lib):
    NB, Hk, B, D = 64, 4, 16, 256
    g = torch.Generator().manual_seed(5)
    kc = torch.randint(0, 65536, (NB, Hk, B, D), generator=g, dtype=torch.int32).to(torch.int16)
    vc = torch.randint(0, 65536, (NB, Hk, B, D), generator=g, dtype=torch.int32).to(torch.int16)
    perm = torch.randperm(NB, generator=g).tolist()
    pairs = np.array([[perm[i], perm[i + 20]] for i in range(20)], dtype=np.int32)
    ek, ev = bits16(kc.view(torch.bfloat16)).copy(), bits16(vc.view(torch.bfloat16)).copy()
    oracle.copy_blocks(ek, pairs.tolist())
    oracle.copy_blocks(ev, pairs.tolist())
    dk, dv = kc.view(torch.bfloat16).cuda(), vc.view(torch.bfloat16).cuda()
    pkv.copy_blocks(dk, dv, torch.as_tensor(pairs).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits16(dk), ek) and np.array_equal(bits16(dv), ev)
    # fp8 pools copy the same way
    k8, v8 = kc.view(torch.uint8).reshape(NB, Hk, B, 2 * D), vc.view(torch.uint8).reshape(NB, Hk, B, 2 * D)
    e8 = k8.numpy().copy()
    oracle.copy_blocks(e8, pairs.tolist())
    d8 = k8[:, :, :, :256].contiguous().cuda()
    e8 = e8[:, :, :, :256]
    pkv.copy_blocks(d8, v8[:, :, :, :256].contiguous().cuda(), torch.as_tensor(pairs).cuda())
    assert np.array_equal(d8.cpu().numpy(), e8)
    assert int(_lib.item()) == 0


@pytest.mark.parametrize("prompt_len", [40, 48])
def test_shared_prefix_pool_image_bit_exact(prompt_len, _lib):
    """Forked rollouts, copy-on-write of a partly filled last prompt block
    (prompt 40 with B=16), completion writes: the pool equals the oracle's
    image of every logical row at its final slot."""
    w = synth.cow(prompt_len=prompt_len, prompts=3, rollouts=4)
    w = dataclasses.replace(w, ctx=[prompt_len + (c % 37) + 1 for c in w.extra["completion"][:12]])
    pw = workload.build(w)
    n_pairs = 0 if pw.cow_pairs_host is None else len(pw.cow_pairs_host)
    assert n_pairs == (9 if prompt_len % 16 else 0)      # 3 prompts x (4 - 1) clones
    _run_step(pw, 0)
    pk, pv = expected_pool(w, 0, pw.alloc.num_blocks, pw.history_slots)
    # the shared prompt blocks are written once; clones hold copies
    st = pw.layers[0]
    assert np.array_equal(bits16(st.k_cache), pk)
    assert np.array_equal(bits16(st.v_cache), pv)
    assert int(_lib.item()) == 0


def test_gather_one_hot_positions_bit_exact():
    """A dominant logit on one logical position makes the output equal that
    position's V row exactly, so each chosen position checks the gather."""
    w = dataclasses.replace(synth.tiny(), ctx=[1000, 333, 17, 1024], num_blocks=None,
                            slack_blocks=8)
    pw = workload.build(w)
    st = pw.layers[0]
    S, Hq, D = st.q.shape
    Hk = w.num_kv_heads
    q = torch.zeros(S, Hq, D, dtype=torch.bfloat16)
    q[:, :, 0] = 1.0
    st.q.copy_(q)
    picks = [[0, 15, 16, 999], [332, 100, 31, 32], [16, 0, 5, 8], [1023, 512, 511, 1]]
    B = w.block_size
    for s, ps in enumerate(picks):
        for h, t in enumerate(ps[:Hk]):
            slot = int(pw.history_slots[s][t])
            krow = torch.zeros(D, dtype=torch.bfloat16, device="cuda")
            krow[0] = 16384.0
            st.k_cache[slot // B, h, slot % B] = krow
    # the new token must not overwrite a pick: write the same rows it has
    out = torch.empty_like(st.q)
    pkv.paged_attention_decode(out, st.q, st.k_cache, st.v_cache, pw.block_tables,
                               pw.context_lens, w.scale, pw.max_context, 0)
    torch.cuda.synchronize()
    g = Hq // Hk
    for s, ps in enumerate(picks):
        for h, t in enumerate(ps[:Hk]):
            slot = int(pw.history_slots[s][t])
            want = bits16(st.v_cache[slot // B, h, slot % B])
            for j in range(g):
                assert np.array_equal(bits16(out[s, h * g + j]), want), (s, h, t)


@pytest.mark.parametrize("P", [0, 64, 512])
def test_decode_tiny(P):
    w = synth.tiny()
    pw = workload.build(w)
    out = _run_step(pw, P)
    assert_close(out[0].cpu(), expected(w, 0, range(w.num_seqs)), "tiny P=%d" % P)


def _edge_cases():
    cases = []
    for d in (128, 256):
        for B in (16, 32):
            P = 4 * B
            for g in (1, 4, 6, 8):
                lens = [1, B - 1, B, B + 1, P - 1, P, P + 1, 3 * P + 5]
                cases.append((d, B, g, tuple(lens), P))
    return cases


@pytest.mark.parametrize("d,B,g,lens,P", _edge_cases())
def test_decode_edge_sweep(d, B, g, lens, P):
    Hk = 2
    w = synth.Workload("edge", 77 + d + B + g, g * Hk, Hk, d, B, list(lens), slack_blocks=3)
    pw = workload.build(w)
    ref = expected(w, 0, range(w.num_seqs))
    for part in (0, P):
        out = _run_step(pw, part)
        assert_close(out[0].cpu(), ref, "edge d=%d B=%d g=%d P=%d" % (d, B, g, part))


def test_decode_large_logits():
    """q x 30 pushes the logits far past exp's range without max subtraction."""
    w = dataclasses.replace(synth.tiny(), ctx=[300, 64, 1024, 7])
    pw = workload.build(w)
    st = pw.layers[0]
    st.q.mul_(30.0)
    q_host = w.q(0, "cpu").float().mul(30.0).to(torch.bfloat16)
    assert torch.equal(st.q.cpu().view(torch.int16), q_host.view(torch.int16))
    out = _run_step(pw, 0)[0].cpu()
    from _oracle_side import host_rows
    ks = [bits16(host_rows(w, 0, s)[0]) for s in range(4)]
    vs = [bits16(host_rows(w, 0, s)[1]) for s in range(4)]
    ref = oracle.decode(bits16(q_host), ks, vs, w.scale)
    assert_close(out, ref, "large logits")
    out2 = _run_step(pw, 128)[0].cpu()
    assert_close(out2, ref, "large logits split")


def test_split_matches_unsplit_and_single_partition_is_bit_identical():
    """One partition per sequence reproduces the one-pass output bit for bit
    when the one-pass launch uses a single CTA per sequence (contexts of at
    most four blocks); longer one-pass launches merge a cluster of CTAs and
    agree with the split form within the tolerance."""
    short = dataclasses.replace(synth.tiny(), ctx=[1, 17, 40, 64])
    pw = workload.build(short)
    a = _run_step(pw, 0)[0]
    b = _run_step(pw, 64)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    w = synth.tiny()
    pw = workload.build(w)
    ref = expected(w, 0, range(w.num_seqs))
    one = _run_step(pw, 0)[0]
    for P in (1024, 32):
        c = _run_step(pw, P)[0]
        ma, rl = errors(c.cpu(), one.cpu().double().numpy())
        assert ma <= MAX_ABS and rl <= REL_L2
        assert_close(c.cpu(), ref, "split P=%d" % P)


def test_one_pass_cluster_ranks_without_pages():
    """A batch whose longest context spreads one pass over 16 CTAs while the
    other sequences give most ranks no page at all."""
    w = dataclasses.replace(synth.tiny(), ctx=[1, 3, 1024, 70], num_blocks=None, slack_blocks=4)
    pw = workload.build(w)
    out = _run_step(pw, 0)[0]
    assert_close(out.cpu(), expected(w, 0, range(w.num_seqs)), "cluster ranks")


def test_physical_permutation_invariance_bit_identical():
    w = synth.tiny()
    outs = []
    for seed in (1, 2, 3):
        pw = workload.build(w, alloc_seed=seed)
        outs.append([o.cpu() for o in (_run_step(pw, 0)[0], _run_step(pw, 64)[0])])
    tabs = [workload.build(w, alloc_seed=s).tables_host for s in (1, 2)]
    assert not np.array_equal(tabs[0], tabs[1])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_aliasing_bit_identical_to_private_copies():
    w = synth.cow(prompt_len=104, prompts=2, rollouts=4)
    w = dataclasses.replace(w, ctx=[104 + (c % 70) + 1 for c in w.extra["completion"][:8]])
    shared = workload.build(w)
    private = workload.build(w, share_prefix=False)
    assert shared.alloc.stats()["used_blocks"] < private.alloc.stats()["used_blocks"]
    for P in (0, 64):
        a = _run_step(shared, P)[0]
        b = _run_step(private, P)[0]
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_close(a.cpu(), expected(w, 0, range(w.num_seqs)), "shared prefix")


def test_decode_fp8_small():
    w = synth.long_fp8(num_seqs=3, ctx=2500)
    w = dataclasses.replace(w, ctx=[2500, 700, 33])
    pw = workload.build(w)
    ks, vs = _scales(pw, 0)
    ref = expected(w, 0, range(3), ks, vs)
    for P in (0, 512):
        out = _run_step(pw, P)[0]
        assert_close(out.cpu(), ref, "fp8 P=%d" % P)


def test_decode_mixed_small():
    w = synth.mixed(num_seqs=24)
    pw = workload.build(w)
    ref = expected(w, 0, range(w.num_seqs))
    for P in (0, 512):
        assert_close(_run_step(pw, P)[0].cpu(), ref, "mixed P=%d" % P)


def test_context_zero_and_device_check(_lib):
    w = synth.tiny()
    pw = workload.build(w)
    st = pw.layers[0]
    ctx = pw.context_lens.clone()
    ctx[1] = 0
    for P in (0, 64):
        out = torch.full_like(st.q, 7.0)
        ws = pkv.alloc_workspace(4, 8, 128, pw.max_context, 64) if P else None
        pkv.paged_attention_decode(out, st.q, st.k_cache, st.v_cache, pw.block_tables, ctx,
                                   w.scale, pw.max_context, P, ws)
        if P:
            pkv.paged_attention_reduce(out, ws, ctx, pw.max_context, P)
        torch.cuda.synchronize()
        assert torch.all(out[1] == 0)
    assert int(_lib.item()) == 0
    # an out-of-range block id is skipped and reported, not dereferenced
    bt = pw.block_tables.clone()
    bt[2, 3] = pw.alloc.num_blocks + 5
    out = torch.empty_like(st.q)
    pkv.paged_attention_decode(out, st.q, st.k_cache, st.v_cache, bt, pw.context_lens,
                               w.scale, pw.max_context, 0)
    torch.cuda.synchronize()
    assert int(_lib.item()) == pkv.DEVERR_BLOCK_ID
    _lib.zero_()
    bad = torch.tensor([10 ** 9], dtype=torch.int64, device="cuda")
    pkv.kv_cache_write(st.k_new[:1], st.v_new[:1], bad, st.k_cache, st.v_cache)
    torch.cuda.synchronize()
    assert int(_lib.item()) == pkv.DEVERR_SLOT
    _lib.zero_()


@pytest.mark.parametrize("P", [0, 64, 32, 16])
def test_one_call_entry_equals_decode_then_reduce(P, _lib):
    """pkv_paged_attention (decode, then the merge for the split form) gives
    the bits of the two calls made one after the other, rows with an empty
    context included (zeros); a failed decode launches no merge."""
    w = dataclasses.replace(synth.tiny(), ctx=[50, 120, 240, 1024])
    pw = workload.build(w)
    st = pw.layers[0]
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache)
    ctx = pw.context_lens.clone()
    ctx[2] = 0
    outs = []
    for one_call in (True, False):
        ws = pkv.alloc_workspace(4, 8, 128, pw.max_context, P) if P else None
        if ws is not None:
            ws.fill_(0xFF)
        out = torch.full_like(st.q, 3.0)
        if one_call:
            pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, ctx, w.scale,
                                pw.max_context, P, out=out, workspace=ws)
        else:
            pkv.paged_attention_decode(out, st.q, st.k_cache, st.v_cache, pw.block_tables, ctx,
                                       w.scale, pw.max_context, P, ws)
            if P:
                pkv.paged_attention_reduce(out, ws, ctx, pw.max_context, P)
        torch.cuda.synchronize()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.all(outs[0][2] == 0)
    assert_close(outs[0][[0, 1, 3]].cpu(), expected(w, 0, [0, 1, 3]), "one call P=%d" % P)
    if P:
        out = torch.full_like(st.q, 3.0)
        with pytest.raises(pkv.PagedKVError):
            pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, ctx, w.scale,
                                pw.max_context, P + 1, out=out, workspace=ws)
        torch.cuda.synchronize()
        assert torch.all(out == 3.0)
    assert int(_lib.item()) == 0
