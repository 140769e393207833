"""CUDA Graph replay of a whole decode step (cache write, decode, merge, and
copy-on-write copies) gives bit-identical outputs to the same launches made
eagerly, also after the inputs were updated in place between replays."""
import dataclasses

import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, expected

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


def _eager(pw, P):
    out = [torch.empty_like(st.q) for st in pw.layers]
    ws = pkv.alloc_workspace(pw.w.num_seqs, pw.w.num_heads, pw.w.head_dim, pw.max_context, P) \
        if P else None
    workload.step(pw, out, ws, P)
    torch.cuda.synchronize()
    return [o.clone() for o in out]


@pytest.mark.parametrize("name,P", [("tiny", 0), ("mixed", 512), ("fp8", 256), ("qwen2", 1024)])
def test_graph_replay_matches_eager(name, P, _lib):
    if name == "tiny":
        w = synth.tiny()
    elif name == "mixed":
        w = synth.mixed(num_seqs=20)
    elif name == "fp8":
        w = dataclasses.replace(synth.long_fp8(num_seqs=2, ctx=3000), ctx=[3000, 999])
    else:
        w = synth.qwen_like(layers=2, num_seqs=4, ctx=2048)
    pw = workload.build(w)
    out = [torch.empty_like(st.q) for st in pw.layers]
    ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, P) if P else None
    g = workload.capture_step(pw, out, ws, P)
    g.replay()
    torch.cuda.synchronize()
    ref = _eager(pw, P)
    for a, b in zip(out, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for layer in range(len(pw.layers)):
        assert_close(out[layer].cpu(), expected(w, layer, range(w.num_seqs),
                                                *([pw.layers[layer].k_scale.cpu().numpy(),
                                                   pw.layers[layer].v_scale.cpu().numpy()]
                                                  if w.fp8 else [])), name)
    # new queries written in place are picked up by the next replay
    for st in pw.layers:
        st.q.mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    ref2 = _eager(pw, P)
    for a, b, c in zip(out, ref2, ref):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    assert int(_lib.item()) == 0


def test_graph_with_copy_on_write_pairs(_lib):
    """The divergence iteration itself (every rollout writes its first token
    right after the prompt): copy, write and decode can be replayed exactly.
    (Later iterations must not replay the copies: a clone also holds the
    tokens written after the divergence.)"""
    w = synth.cow(prompt_len=40, prompts=2, rollouts=4)
    w = dataclasses.replace(w, ctx=[41] * 8)
    pw = workload.build(w)
    assert pw.cow_pairs is not None and len(pw.cow_pairs_host) == 6
    out = [torch.empty_like(pw.layers[0].q)]
    g = workload.capture_step(pw, out, None, 0, copy_pairs=True)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_close(out[0].cpu(), expected(w, 0, range(w.num_seqs)), "cow graph")
