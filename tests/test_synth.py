"""The shared input generator: host and tensor forms agree bit for bit, and
its output looks like N(0, 1)."""
import numpy as np
import torch

from paged_kv_cache_220_gb300 import synth


def test_mix64_tensor_matches_python_ints():
    xs = [0, 1, 2, 12345, (1 << 62) - 1, (1 << 40) + 77]
    t = synth.mix64_tensor(torch.tensor(xs, dtype=torch.int64))
    for x, z in zip(xs, t.tolist()):
        assert z & ((1 << 64) - 1) == synth.mix64_int(x)


def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF
    assert synth.mix64_int(0) == 0xE220A8397B1DCDAF


def test_normal_table_moments():
    tab = synth.normal_table().to(torch.float64)
    assert abs(float(tab.mean())) < 1e-3
    assert abs(float(tab.std()) - 1.0) < 5e-3
    assert torch.all(tab[1:] >= tab[:-1])


def test_stream_values_deterministic_and_offsettable():
    w = synth.tiny()
    a = w.rows(synth.KIND_K, 0, 2, 0, 100)
    b = w.rows(synth.KIND_K, 0, 2, 40, 100)
    assert torch.equal(a[40:].view(torch.int16), b.view(torch.int16))
    x = a.to(torch.float64)
    assert abs(float(x.mean())) < 0.05 and abs(float(x.std()) - 1) < 0.05


def test_shared_prefix_rows():
    w = synth.cow(prompt_len=40, prompts=2, rollouts=3)
    r0 = w.rows(synth.KIND_V, 0, 0, 0, 45)
    r1 = w.rows(synth.KIND_V, 0, 1, 0, 45)
    r3 = w.rows(synth.KIND_V, 0, 3, 0, 45)
    assert torch.equal(r0[:40].view(torch.int16), r1[:40].view(torch.int16))
    assert not torch.equal(r0[40:].view(torch.int16), r1[40:].view(torch.int16))
    assert not torch.equal(r0[:40].view(torch.int16), r3[:40].view(torch.int16))


def test_workload_shapes():
    assert synth.tiny().ctx == [50, 120, 240, 1024]
    q = synth.qwen_like()
    assert q.num_seqs == 64 and q.layers == 16 and q.pool_blocks() == 64 * 512
    m = synth.mixed()
    assert len(m.ctx) == 256 and min(m.ctx) >= 16 and max(m.ctx) <= 16384
    c = synth.cow()
    assert c.num_seqs == 512 and all(2049 <= x <= 2048 + 1025 for x in c.ctx)
    f = synth.long_fp8()
    assert f.fp8 and f.ctx == [131072] * 8
    assert abs(q.scale - 0.0625) == 0.0


def test_normal_bf16_equals_elementwise_definition():
    # the vectorised stream against SplitMix64 on Python ints, element by
    # element, with counters near the top of the key range
    key = (1 << 62) - 5000
    vals = synth.normal_bf16(key, 64, 4000)
    tab = synth.normal_table()
    for i in range(64):
        z = synth.mix64_int(key + 4000 + i)
        assert vals[i].view(torch.int16).item() == tab[z >> 48].view(torch.int16).item()
