"""Parity at the full workload sizes, in the launch configuration the
benchmark times (split decode + reduce, every layer; the shared-prefix decode
replayed from a CUDA graph for the copy-on-write rollouts).

Every output of a whole layer is compared with the oracle: all 64 sequences
of layer 0 of the Qwen-like batch (plus 4 sampled sequences of each other
layer), all 256 mixed-length sequences, all 512 rollouts of both
copy-on-write variants (through the plain split decode and through the
shared-prefix decode), the 512 rollouts over an E4M3 cache (shared-prefix
decode), the 128 rollouts of 8184-token prompts (shared-prefix decode), and
all 8 long FP8 sequences. The cache writes of
layer 0 of the Qwen-like batch and of the FP8 batch are checked bit for bit
over the whole pool, and the FP8 scales are recomputed on the host from the
host rows. Host rows come from the seeded generator; nothing but the outputs
under test is read back from the device."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import (RowCache, assert_close, bits16, expected, host_fp8_scales, host_rows,
                          quantize)

pytestmark = pytest.mark.gpu

CHUNK = 16      # sequences per oracle call (bounds host memory)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


def _step(pw):
    w = pw.w
    out = [torch.empty_like(st.q) for st in pw.layers]
    ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context,
                             w.partition_size) if w.partition_size else None
    workload.step(pw, out, ws)
    torch.cuda.synchronize()
    return [o.cpu() for o in out]


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return sorted(set(rng.choice(n, size=k, replace=False).tolist()))


def _check_all(got, w, layer, rows, what, k_scale=None, v_scale=None, seqs=None):
    """Compare every sequence (or `seqs`) of got [S, Hq, D] with the oracle,
    CHUNK sequences per oracle call."""
    seqs = list(range(w.num_seqs)) if seqs is None else list(seqs)
    for i in range(0, len(seqs), CHUNK):
        part = seqs[i:i + CHUNK]
        ref = expected(w, layer, part, k_scale, v_scale, rows=rows)
        assert_close(got[part], ref, "%s seqs %d..%d" % (what, part[0], part[-1]))


def _pool_image(w, layer, pw, rows, num_blocks, k_scale=None, v_scale=None):
    """Expected (K, V) pool images of a layer: every logical row of every
    sequence at its slot (the oracle's scatter)."""
    dt = np.uint8 if w.fp8 else np.uint16
    shape = (num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    pk, pv = np.zeros(shape, dtype=dt), np.zeros(shape, dtype=dt)
    for s in range(w.num_seqs):
        K, V = rows(s)
        if w.fp8:
            k, v = quantize(K, k_scale), quantize(V, v_scale)
        else:
            k, v = bits16(K), bits16(V)
        oracle.scatter_rows_fast(pk, k, pw.history_slots[s])
        oracle.scatter_rows_fast(pv, v, pw.history_slots[s])
    return pk, pv


def _memo(fn):
    """Rows of a sequence generated once (the whole-layer checks read each
    sequence's rows twice: the oracle, then the pool image)."""
    cache = {}

    def get(s):
        if s not in cache:
            cache[s] = fn(s)
        return cache[s]
    return get


def _pool_bits(t):
    return t.cpu().numpy() if t.dtype == torch.uint8 else bits16(t)


def test_qwen_like_16_layers(_lib):
    w = synth.qwen_like()
    pw = workload.build(w)
    assert pw.alloc.stats()["free_blocks"] == 0          # the pool fits exactly
    out = _step(pw)
    assert int(_lib.item()) == 0
    # layer 0: every sequence, and the whole pool after the step's write
    rows = _memo(RowCache(w, 0).rows)
    _check_all(out[0], w, 0, rows, "layer 0")
    st = pw.layers[0]
    pk, pv = _pool_image(w, 0, pw, rows, st.k_cache.shape[0])
    assert np.array_equal(_pool_bits(st.k_cache), pk), "layer 0 K pool"
    del pk
    assert np.array_equal(_pool_bits(st.v_cache), pv), "layer 0 V pool"
    del pv
    for layer in range(1, w.layers):
        seqs = _sample(w.num_seqs, 4, layer)
        _check_all(out[layer], w, layer, None, "layer %d" % layer, seqs=seqs)
    del pw
    torch.cuda.empty_cache()


def test_mixed_lengths(_lib):
    w = synth.mixed()
    pw = workload.build(w)
    out = _step(pw)[0]
    assert int(_lib.item()) == 0
    _check_all(out, w, 0, None, "mixed")


@pytest.mark.parametrize("prompt_len", [2048, 2040])
def test_cow_rollouts(prompt_len, _lib):
    w = synth.cow(prompt_len=prompt_len)
    pw = workload.build(w)
    pairs = pw.cow_pairs_host
    rows = RowCache(w, 0).rows
    if prompt_len % w.block_size == 0:
        assert pairs is None or len(pairs) == 0
    else:
        assert len(pairs) == 32 * 15
        # every clone of every prompt holds the prompt's tail rows bit for bit
        B, tail = w.block_size, prompt_len % w.block_size
        kc = bits16(pw.layers[0].k_cache)
        for p in range(32):
            K, _ = rows(p * w.group)
            want = bits16(K)[prompt_len - tail:prompt_len]          # [tail, Hk, D]
            for r in range(w.group):
                s = p * w.group + r
                blk = int(pw.tables_host[s][prompt_len // B])
                got = kc[blk][:, :tail, :].transpose(1, 0, 2)
                assert np.array_equal(got, want)
        del kc
    out = _step(pw)[0]
    # the shared-prefix decode as the benchmark runs it (a replayed CUDA graph,
    # own parts split by split_partition_size)
    groups = workload.prefix_groups(pw)
    P = pkv.split_partition_size(groups.max_own_context, w.block_size, w.partition_size)
    assert P == 1040                      # each own part in one partition
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, groups.max_own_context,
                                     groups.max_prefix_blocks * w.block_size, P)
    sp = [torch.empty_like(pw.layers[0].q)]
    g = workload.capture_step(pw, sp, ws, P, groups=groups)
    g.replay()
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    sp = sp[0].cpu()
    for i in range(0, w.num_seqs, CHUNK):
        part = list(range(i, i + CHUNK))
        ref = expected(w, 0, part, rows=rows)
        assert_close(out[part], ref, "cow %d split, seqs %d.." % (prompt_len, i))
        assert_close(sp[part], ref, "cow %d shared prefix, seqs %d.." % (prompt_len, i))


def test_long_context_fp8(_lib):
    w = synth.long_fp8()
    pw = workload.build(w)
    st = pw.layers[0]
    # the scales, recomputed on the host from every row of the layer
    rows = _memo(lambda s: host_rows(w, 0, s))
    ks, vs = host_fp8_scales(w, 0, rows)
    assert np.array_equal(ks.view(np.uint32), st.k_scale.cpu().numpy().view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), st.v_scale.cpu().numpy().view(np.uint32))
    out = _step(pw)[0]
    assert int(_lib.item()) == 0
    # every sequence, on the oracle's own E4M3 codes of the host rows
    _check_all(out, w, 0, rows, "long fp8", ks, vs)
    # the whole pool after the step's write: the oracle's encoding at every slot
    pk, pv = _pool_image(w, 0, pw, rows, st.k_cache.shape[0], ks, vs)
    assert np.array_equal(_pool_bits(st.k_cache), pk), "fp8 K pool"
    del pk
    assert np.array_equal(_pool_bits(st.v_cache), pv), "fp8 V pool"


def test_cow_rollouts_over_fp8_cache(_lib):
    """All 512 rollouts of the 2040-token prompts over an E4M3 cache, through
    the shared-prefix decode as the benchmark runs it (a replayed CUDA graph,
    own parts longest first, split by split_partition_size; 16-token E4M3
    blocks two to a decode page), against the oracle on its own E4M3 codes of
    the host rows; the per-head scales recomputed on the host."""
    import dataclasses
    w = dataclasses.replace(synth.cow(prompt_len=2040), fp8=True)
    pw = workload.build(w)
    st = pw.layers[0]
    rows = _memo(RowCache(w, 0).rows)
    ks, vs = host_fp8_scales(w, 0, rows)
    assert np.array_equal(ks.view(np.uint32), st.k_scale.cpu().numpy().view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), st.v_scale.cpu().numpy().view(np.uint32))
    groups = workload.prefix_groups(pw)
    assert groups.visit_order is not None
    P = pkv.split_partition_size(groups.max_own_context, w.block_size, w.partition_size)
    assert P == 1040
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, groups.max_own_context,
                                     groups.max_prefix_blocks * w.block_size, P)
    sp = [torch.empty_like(st.q)]
    g = workload.capture_step(pw, sp, ws, P, groups=groups)
    g.replay()
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    _check_all(sp[0].cpu(), w, 0, rows, "cow fp8 shared prefix", ks, vs)


def test_long_prompt_rollouts(_lib):
    """128 rollouts of 8 prompts of 8184 tokens (own parts of at most 129
    tokens): the shared prefix spans several prefix partitions, read by the
    full prefix CTA; every output against the oracle, through the replayed
    shared-prefix step as the benchmark runs it."""
    import bench
    w = bench.workload_for("cow_long_prompts")
    pw = workload.build(w)
    groups = workload.prefix_groups(pw)
    P = pkv.split_partition_size(groups.max_own_context, w.block_size, w.partition_size)
    Pp = pkv.shared_prefix_partition_size(int(groups.group_start.shape[0]) - 1,
                                          groups.max_group_members, w.num_kv_heads, w.num_heads,
                                          w.block_size, groups.max_prefix_blocks, P)
    assert -(-groups.max_prefix_blocks * w.block_size // Pp) > 1     # several prefix partitions
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, groups.max_own_context,
                                     groups.max_prefix_blocks * w.block_size, P)
    sp = [torch.empty_like(pw.layers[0].q)]
    g = workload.capture_step(pw, sp, ws, P, groups=groups)
    g.replay()
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    _check_all(sp[0].cpu(), w, 0, RowCache(w, 0).rows, "long-prompt rollouts")
