"""bench.py pieces that run without a GPU: the reference arm's JSON line,
the byte accounting of the metric, the code hash that keeps a stored ncu
traffic figure tied to the decode sources, and the host iteration timing."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_220_gb300 import build, synth  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    d = json.loads(lines[-1])
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == synth.tiny().name
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_metric_bytes_follow_the_definition():
    """Per layer: the K and V rows of every cached token, Q and out, and the
    block tables (S x max blocks, int32); the Qwen-like layer is
    2,149,187,584 B; the shared-prefix figure counts each group's prefix
    rows once."""
    w = synth.tiny()
    B, Hk, d, Hq = w.block_size, w.num_kv_heads, w.head_dim, w.num_heads
    S = len(w.ctx)
    mb = max(-(-c // B) for c in w.ctx)
    want = sum(w.ctx) * Hk * d * 2 * 2 + 2 * S * Hq * d * 2 + S * mb * 4
    assert bench.decode_bytes(w) == want
    assert bench.decode_bytes(synth.qwen_like()) == 2149187584
    f8 = synth.long_fp8()
    assert bench.decode_bytes(f8) == (sum(f8.ctx) * 4 * 256 * 1 * 2 + 2 * 8 * 24 * 256 * 2
                                      + 8 * (131072 // 32) * 4)
    cow = synth.cow(prompt_len=2048, prompts=2, rollouts=4)
    per_tok = cow.num_kv_heads * cow.head_dim * 2 * 2
    assert bench.unique_decode_bytes(cow) == bench.decode_bytes(cow) - 2 * 3 * 2048 * per_tok
    assert bench.unique_decode_bytes(w) == bench.decode_bytes(w)


def test_code_hash_ignores_comments_and_spacing(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cu"
    c = tmp_path / "c.cu"
    a.write_text('int f(int x) {  // one\n  return x + 1; /* two */\n}\nconst char* s = "//k";\n')
    b.write_text('/* header */\nint f(int x) {\n\n  return x + 1;\n}\nconst char* s = "//k";\n')
    c.write_text('int f(int x) {\n  return x + 2;\n}\nconst char* s = "//k";\n')
    assert bench.strip_comments(a.read_text()) == bench.strip_comments(b.read_text())
    assert '"//k"' in bench.strip_comments(a.read_text())
    old = bench.ROOT
    try:
        bench.ROOT = str(tmp_path)
        assert bench.source_hash(["a.cu"]) == bench.source_hash(["b.cu"])
        assert bench.source_hash(["a.cu"]) != bench.source_hash(["c.cu"])
    finally:
        bench.ROOT = old


def test_host_iteration_timing_runs_the_whole_batch():
    build.build()
    w = synth.mixed(num_seqs=40)
    h = bench.host_iteration_timing(w, iters=20)
    assert h["running"] == 40 and h["iterations"] == 20
    assert h["sched_step_us"] > 0 and h["block_tables_us"] > 0


def test_visit_order_is_longest_first_or_none():
    """The workload helpers' visit order: longest first (ties in batch order)
    as a permutation of the batch, none when every length is equal."""
    import numpy as np
    from paged_kv_cache_220_gb300 import workload
    assert workload.visit_order([8192] * 64, device="cpu") is None
    lens = [5, 900, 17, 900, 3000, 1]
    order = workload.visit_order(lens, device="cpu").numpy().tolist()
    assert sorted(order) == list(range(len(lens)))
    assert order == [4, 1, 3, 2, 0, 5]
    ctx = np.asarray(synth.mixed().ctx)
    order = workload.visit_order(ctx, device="cpu").numpy()
    assert np.all(np.diff(ctx[order]) <= 0)


@pytest.mark.parametrize("name", ["tiny", "qwen_like", "mixed", "cow", "cow2040", "cow2040_fp8",
                                  "cow_long_prompts", "long_fp8", "long_fp8_b16"])
def test_every_bench_configuration_is_a_valid_workload(name):
    """The named workloads bench.py runs: shapes the kernels take, a split
    size that is a multiple of the block size, contexts within the pool, and
    shared prompts of whole groups."""
    w = bench.workload_for(name)
    assert w.num_seqs >= 1 and all(c >= 1 for c in w.ctx)
    assert w.head_dim in (128, 256) and w.block_size in (16, 32)
    assert w.num_heads % w.num_kv_heads == 0 and w.num_heads // w.num_kv_heads <= 8
    assert w.partition_size % w.block_size == 0
    if w.prefix_len > 0:
        assert w.num_seqs % w.group == 0
        assert all(c > w.prefix_len for c in w.ctx)
    assert bench.decode_bytes(w) > 0
