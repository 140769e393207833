"""Parity at the full workload sizes, in the launch configuration the
benchmark times (split decode + reduce, every layer; the shared-prefix decode
replayed from a CUDA graph for the copy-on-write rollouts). The oracle checks a
seeded sample of sequences one by one; copy-on-write clones are checked bit
for bit."""
import numpy as np
import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, bits16, expected, host_rows, quantize

pytestmark = pytest.mark.gpu


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
    return sorted(set([0, n - 1] + rng.choice(n, size=k, replace=False).tolist()))


def test_qwen_like_16_layers(_lib):
    w = synth.qwen_like()
    pw = workload.build(w)
    assert pw.alloc.stats()["free_blocks"] == 0          # the pool fits exactly
    out = _step(pw)
    for layer in range(w.layers):
        seqs = _sample(w.num_seqs, 4, layer) if layer == 0 else [(5 * layer) % w.num_seqs]
        ref = expected(w, layer, seqs)
        assert_close(out[layer][seqs], ref, "layer %d" % layer)
    assert int(_lib.item()) == 0
    del pw
    torch.cuda.empty_cache()


def test_mixed_lengths(_lib):
    w = synth.mixed()
    pw = workload.build(w)
    out = _step(pw)[0]
    order = np.argsort(w.ctx)
    seqs = sorted(set(order[:4].tolist() + order[-4:].tolist() + _sample(w.num_seqs, 24, 3)))
    assert_close(out[seqs], expected(w, 0, seqs), "mixed")
    assert int(_lib.item()) == 0


@pytest.mark.parametrize("prompt_len", [2048, 2040])
def test_cow_rollouts(prompt_len, _lib):
    w = synth.cow(prompt_len=prompt_len)
    pw = workload.build(w)
    pairs = pw.cow_pairs_host
    if prompt_len % w.block_size == 0:
        assert pairs is None or len(pairs) == 0
    else:
        assert len(pairs) == 32 * 15
        # every clone holds the prompt's tail rows bit for bit
        B, tail = w.block_size, prompt_len % w.block_size
        st = pw.layers[0]
        kc = bits16(st.k_cache)
        for p in range(0, 32, 7):
            K, _ = host_rows(w, 0, p * w.group, prompt_len)
            want = bits16(K)[prompt_len - tail:prompt_len]          # [tail, Hk, D]
            for r in range(w.group):
                s = p * w.group + r
                blk = int(pw.tables_host[s][prompt_len // B])
                got = kc[blk][:, :tail, :].transpose(1, 0, 2)
                assert np.array_equal(got, want)
    out = _step(pw)[0]
    seqs = _sample(w.num_seqs, 30, 4)
    ref = expected(w, 0, seqs)
    assert_close(out[seqs], ref, "cow %d" % prompt_len)
    # the shared-prefix decode as the benchmark runs it (a replayed CUDA graph)
    groups = workload.prefix_groups(pw)
    P = w.partition_size
    ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim, groups[3],
                                     groups[2] * w.block_size, P)
    sp = [torch.empty_like(pw.layers[0].q)]
    g = workload.capture_step(pw, sp, ws, P, groups=groups)
    g.replay()
    torch.cuda.synchronize()
    assert_close(sp[0].cpu()[seqs], ref, "cow %d shared prefix" % prompt_len)
    assert int(_lib.item()) == 0


def test_long_context_fp8(_lib):
    w = synth.long_fp8()
    pw = workload.build(w)
    st = pw.layers[0]
    ks, vs = st.k_scale.cpu().numpy(), st.v_scale.cpu().numpy()
    # the stored codes of a sampled block equal the oracle's encoding
    s, t0 = 5, 77 * w.block_size
    K, V = host_rows(w, 0, s, t0 + w.block_size)
    blk = int(pw.tables_host[s][t0 // w.block_size])
    got = st.k_cache[blk].cpu().numpy().transpose(1, 0, 2)
    assert np.array_equal(got, quantize(K[t0:], ks))
    out = _step(pw)[0]
    seqs = [0, 7]
    assert_close(out[seqs], expected(w, 0, seqs, ks, vs), "long fp8")
    assert int(_lib.item()) == 0
