"""Benchmark of the paged decode step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

NAME: qwen_like (default), tiny, mixed, cow, cow2040, cow2040_fp8 (the 2040-token rollouts
over an E4M3 cache), long_fp8.

A step is one pass of the whole hot path over the workload's batch: for every
layer the new token's K/V are written into their slots (kv_cache_write), the
split decode attends over the paged cache (paged_attention_decode) and the
partitions are merged (paged_attention_reduce); shared-prefix workloads use
the shared-prefix decode, and their copy-on-write block copies (copy_blocks,
the divergence iteration's) are timed on their own. Inputs
are resident in HBM; the default workload (64 sequences x 8192 tokens x 16
layers, 34 GB of K/V per step) is far larger than L2, smaller workloads flush
L2 before every step.

Prints one JSON line (rank 0). value = algorithmic bytes of the step (K/V
pages touched + Q + out + block tables, per layer) / step time, in GB/s.
`--impl reference` times the CPU oracle instead, on a bounded sample of the
same workload, and prints the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode-attention HBM GB/s (% of GB300 peak) and decode tokens/s per layer"
L2_BYTES = 129 * 1024 * 1024
DECODE_SOURCES = ["paged_kv_cache_220_gb300/csrc/decode.cu",
                  "paged_kv_cache_220_gb300/csrc/decode_tc.cu",
                  "paged_kv_cache_220_gb300/csrc/decode_params.h",
                  "paged_kv_cache_220_gb300/csrc/common.cuh",
                  "paged_kv_cache_220_gb300/csrc/tc_common.cuh"]


def _long_prompt_rollouts():
    """8 prompts of 8184 tokens x 16 rollouts, completion lengths (the copy-on-
    write workload's draws) mod 129."""
    import dataclasses
    from paged_kv_cache_220_gb300 import synth
    w = synth.cow(prompt_len=8184, prompts=8, rollouts=16)
    comp = [c % 129 for c in w.extra["completion"]]
    return dataclasses.replace(w, ctx=[8184 + c + 1 for c in comp], extra={"completion": comp},
                               name="cow_long_prompts_8184")


def workload_for(name: str):
    from paged_kv_cache_220_gb300 import synth
    table = {
        "qwen_like": lambda: synth.qwen_like(),
        "tiny": lambda: synth.tiny(),
        "mixed": lambda: synth.mixed(),
        "cow": lambda: synth.cow(prompt_len=2048),
        "cow2040": lambda: synth.cow(prompt_len=2040),
        "cow2040_fp8": lambda: __import__("dataclasses").replace(
            synth.cow(prompt_len=2040), fp8=True, name="cow_shared_prefix_2040_fp8"),
        "long_fp8": lambda: synth.long_fp8(),
        # the same shapes and bytes in 16-token blocks
        "long_fp8_b16": lambda: __import__("dataclasses").replace(
            synth.long_fp8(), block_size=16, name="long_context_fp8_splitk_b16"),
        # rollouts of long prompts with short completions: the shared prefix
        # is most of the bytes
        "cow_long_prompts": lambda: _long_prompt_rollouts(),
    }
    w = table[name]()
    if name == "tiny":
        import dataclasses
        w = dataclasses.replace(w, partition_size=0)
    return w


def decode_bytes(w) -> int:
    """Algorithmic bytes of one decode launch (one layer): K/V pages touched,
    Q, out and the block tables."""
    esz = 1 if w.fp8 else 2
    B = w.block_size
    kv = sum(w.ctx) * w.num_kv_heads * w.head_dim * esz * 2
    qo = 2 * w.num_seqs * w.num_heads * w.head_dim * 2
    mb = max(-(-c // B) for c in w.ctx)
    bt = w.num_seqs * mb * 4
    return kv + qo + bt


def unique_decode_bytes(w) -> int:
    """Shared prefixes counted once (the bytes a reader of unique pages moves)."""
    if w.prefix_len <= 0:
        return decode_bytes(w)
    esz = 1 if w.fp8 else 2
    per_tok = w.num_kv_heads * w.head_dim * esz * 2
    n_prompt = w.num_seqs // w.group
    tokens = n_prompt * w.prefix_len + sum(c - w.prefix_len for c in w.ctx)
    return decode_bytes(w) - sum(w.ctx) * per_tok + tokens * per_tok


NOMINAL_HBM_GBS = 8000.0    # GB300 HBM3e, nominal (~8 TB/s)


def peaks():
    """The roofline's HBM peak: the measured copy bandwidth of this machine's
    GB300s (MEASURED_PEAKS.json), else the profiling fallback of 6.8 TB/s."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer and part numbers, with the part's name where known)."""
    arm_parts = {"0xd4f": "Neoverse-V2", "0xd40": "Neoverse-V1", "0xd0c": "Neoverse-N1",
                 "0xd49": "Neoverse-N2", "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    imp, part = fields.get("CPU implementer"), fields.get("CPU part")
    if imp or part:
        name = arm_parts.get(part, "")
        return ("Arm implementer %s part %s %s" % (imp, part, name)).strip()
    return "unknown"


def strip_comments(src: str) -> str:
    """C/C++ source without comments and blank space, so that comment-only
    edits leave the hash of the code alone (string and character literals
    are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(paths) -> str:
    """Hash of the code (comments and spacing ignored) of the given sources."""
    h = hashlib.sha256()
    for rel in paths:
        h.update(strip_comments(open(os.path.join(ROOT, rel), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """dram bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode source."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None, None
    d = json.load(open(p))
    ent = d.get(config)
    if not ent or ent.get("source_hash") != source_hash(DECODE_SOURCES):
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("note")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms during the
    timed region (the `with` block). The sampler is started, and its first
    sample awaited, before the region begins; the summary keeps the samples
    written while the region ran (the nearest one on each side if it was
    shorter than a sampling period)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "pkv_clocks_%d_%d.csv" % (os.getpid(), gpu_index))
        self.n0 = self.n1 = 0

    def _rows(self):
        try:
            return [l for l in open(self.path).read().splitlines() if l.count(",") >= 8]
        except OSError:
            return []

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        t0 = time.time()
        while not self._rows() and time.time() - t0 < 3.0 and self.proc.poll() is None:
            time.sleep(0.01)
        self.n0 = len(self._rows())
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.n1 = len(self._rows())
            time.sleep(0.05)               # one more sample after the region
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        allrows = self._rows()
        inside = allrows[self.n0:self.n1]
        note = "samples taken during the timed region"
        if not inside:
            inside = allrows[max(0, self.n0 - 1):self.n1 + 1]
            note = "region shorter than the 20 ms sampling period: nearest samples"
        rows = [[x.strip() for x in r.split(",")] for r in inside]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "note": note}


def fp8_scales_host(w, layer=0):
    """Per-KV-head E4M3 scales from every row of every sequence of the layer:
    fp32 max |x| / 448 (an IEEE fp32 quotient), as the GPU arm's cache uses."""
    import numpy as np
    from paged_kv_cache_220_gb300 import synth
    amax = [np.zeros(w.num_kv_heads, dtype=np.float32) for _ in range(2)]
    for s in range(w.num_seqs):
        for i, kind in enumerate((synth.KIND_K, synth.KIND_V)):
            r = w.rows(kind, layer, s, 0, w.ctx[s], "cpu").float().abs().amax(dim=(0, 2))
            amax[i] = np.maximum(amax[i], r.numpy())
    return amax[0] / np.float32(448.0), amax[1] / np.float32(448.0)


def run_reference(args, w, rank, single_thread=False):
    """The CPU oracle on a bounded sample of the workload (same metric)."""
    import numpy as np
    import oracle
    from paged_kv_cache_220_gb300 import synth

    def bits(t):
        return t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)

    # sample: the first n sequences of layer 0, n sized for ~10-20 s of work
    budget_tokens = int(os.environ.get("PKV_ORACLE_TOKENS", "131072"))
    seqs, tok = [], 0
    for s in range(w.num_seqs):
        if tok >= budget_tokens and seqs:
            break
        seqs.append(s)
        tok += w.ctx[s]
    q = bits(w.q(0, "cpu"))[seqs]
    ks, vs = [], []
    ksc = vsc = None
    if w.fp8:
        ksc, vsc = fp8_scales_host(w, 0)
    for s in seqs:
        K = w.rows(synth.KIND_K, 0, s, 0, w.ctx[s], "cpu")
        V = w.rows(synth.KIND_V, 0, s, 0, w.ctx[s], "cpu")
        if w.fp8:
            ks.append(oracle.e4m3_encode_bf16(bits(K), ksc))
            vs.append(oracle.e4m3_encode_bf16(bits(V), vsc))
        else:
            ks.append(bits(K))
            vs.append(bits(V))
    import dataclasses
    sub = dataclasses.replace(w, ctx=[w.ctx[s] for s in seqs])
    sample_bytes = decode_bytes(sub)

    def one():
        if w.fp8:
            oracle.decode(q, ks, vs, w.scale, ksc.astype(np.float64), vsc.astype(np.float64))
        else:
            oracle.decode(q, ks, vs, w.scale)

    def timed(target_s, max_reps, min_reps):
        times = []
        while True:
            t0 = time.perf_counter()
            one()
            times.append(time.perf_counter() - t0)
            if len(times) >= min_reps and (sum(times) >= target_s or len(times) >= max_reps):
                return times

    # the reference arm times K steps; the baseline inside our own line
    # repeats the sample until about 10 s of CPU work have been timed
    cores = oracle.num_threads()
    if args.impl == "reference":
        times = timed(0.0, args.steps, args.steps)
    else:
        times = timed(10.0, 200, 1)
    t = sum(times) / len(times)
    out = {
        "value": round(sample_bytes / t / 1e9, 4), "unit": "GB/s", "cores": cores,
        "kind": "oracle",
        "sample": "layer 0, sequences %d..%d (%d tokens) of the workload, fp64 C oracle, "
                  "%d repetition(s), %.3f s each" % (seqs[0], seqs[-1], tok, len(times), t),
        "seconds": round(t, 4), "nproc": os.cpu_count(), "cpu_model": cpu_model(),
    }
    if single_thread:
        # the same sample on one thread (at most ~10 s)
        oracle.set_num_threads(1)
        try:
            t1 = timed(5.0, 3, 1)
        finally:
            oracle.set_num_threads(cores)
        t1 = sum(t1) / len(t1)
        out["single_thread"] = {"value": round(sample_bytes / t1 / 1e9, 4), "unit": "GB/s",
                                "cores": 1, "seconds": round(t1, 4)}
    return out


def make_step(pw, out, ws, cascade, stream):
    """One step of the hot path over every layer: the cache write of the new
    token, then the decode (shared-prefix decode with `cascade`) and, for the
    split decode, the merge. With ev, events are recorded on `stream` around
    each layer's decode launch (the roofline's kernel)."""
    import paged_kv_cache_220_gb300 as pkv
    w = pw.w
    P = w.partition_size

    def one_step(ev=None):
        for layer, st in enumerate(pw.layers):
            pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                               st.k_scale, st.v_scale)
            if ev is not None:
                ev[layer][0].record(stream)
            if cascade is not None:
                pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                                  pw.context_lens, w.scale,
                                                  cascade.max_own_context, cascade.group_start,
                                                  cascade.prefix_blocks,
                                                  cascade.max_prefix_blocks, P,
                                                  cascade.max_group_members,
                                                  out=out[layer], workspace=ws,
                                                  k_scale=st.k_scale, v_scale=st.v_scale,
                                                  seq_order=cascade.visit_order)
                if ev is not None:
                    ev[layer][1].record(stream)
                continue
            # the decode kernel alone (the roofline's kernel), then the merge
            pkv.paged_attention_decode(out[layer], st.q, st.k_cache, st.v_cache, pw.block_tables,
                                       pw.context_lens, w.scale, pw.max_context, P, ws,
                                       st.k_scale, st.v_scale, seq_order=pw.visit_order)
            if ev is not None:
                ev[layer][1].record(stream)
            if P:
                pkv.paged_attention_reduce(out[layer], ws, pw.context_lens, pw.max_context, P)
    return one_step


def step_launches(pw, cascade):
    """Kernels of one step: per layer the cache write and the decode, plus the
    merge of a split decode; the shared-prefix decode is three kernels."""
    L = len(pw.layers)
    P = pw.w.partition_size
    return L * ((4 if cascade is not None else 2) + (1 if P and cascade is None else 0))


def measure_other(name, steps=10, warmup=3):
    """A short run of another workload, for the same JSON line: device-timed
    step (graph replay) after `warmup` steps, the decode kernel's launch time
    from an eager pass, clocks sampled during the timed steps."""
    import dataclasses
    import torch
    import paged_kv_cache_220_gb300 as pkv
    from paged_kv_cache_220_gb300 import workload
    w = workload_for(name)
    pw = workload.build(w)
    L = len(pw.layers)
    P = w.partition_size
    out = [torch.empty_like(st.q) for st in pw.layers]
    ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, P) if P else None
    cascade = None
    if w.prefix_len > 0 and P:
        cascade = workload.prefix_groups(pw)
        # own parts: the split size without a nearly empty last partition
        P = pkv.split_partition_size(cascade.max_own_context, w.block_size, P)
        w = dataclasses.replace(w, partition_size=P)
        pw.w = w
        ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim,
                                         cascade.max_own_context,
                                         cascade.max_prefix_blocks * w.block_size, P)
    stream = torch.cuda.current_stream()
    one_step = make_step(pw, out, ws, cascade, stream)
    step_bytes = decode_bytes(w) * L
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") \
        if step_bytes < 4 * L2_BYTES else None
    for _ in range(warmup):
        one_step()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        one_step(evs[i])
    torch.cuda.synchronize()
    dec_ms = sum(evs[i][l][0].elapsed_time(evs[i][l][1]) for i in range(steps)
                 for l in range(L)) / (steps * L)
    graph = workload.capture_step(pw, out, ws, P, groups=cascade)
    for _ in range(warmup):
        graph.replay()
    # enough steps for ~0.3 s of timed work (the clock sampler's period is 20 ms)
    eager_ms = sum(evs[i][0][0].elapsed_time(evs[i][L - 1][1]) for i in range(steps)) / steps
    steps = max(steps, int(0.3 / max(eager_ms / 1e3, 1e-6)))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = sum(per) / steps
    peak, peak_kind = peaks()
    dec_bytes = decode_bytes(w) if cascade is None else unique_decode_bytes(w)
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    r = {"workload": w.name, "steps": steps, "warmup": warmup, "ms_per_step": round(ms, 4),
         "ms_per_step_median": round(statistics.median(per), 4),
         "value": round(step_bytes / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
         "roofline": {"kernel": "paged_attention_decode" if cascade is None else
                      "paged_attention_decode_shared_prefix (3 kernels, unique bytes)",
                      "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                      "frac": round(achieved / peak, 4), "bytes_per_launch": dec_bytes,
                      "launch_ms": round(dec_ms, 5)},
         "gpu_launches": step_launches(pw, cascade) * steps,
         "l2": "flushed before every step" if flush is not None else "inputs larger than L2",
         "clocks": clk.summary()}
    if w.prefix_len > 0:
        r["unique_bytes_gbs"] = round(unique_decode_bytes(w) * L / (ms / 1e3) / 1e9, 2)
        r["unique_frac_of_peak"] = round(unique_decode_bytes(w) * L / (ms / 1e3) / 1e9 / peak, 4)
    del graph, pw, out, ws
    torch.cuda.empty_cache()
    return r


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="qwen_like")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--other-configs", default="tiny,mixed,cow,cow2040,cow2040_fp8,long_fp8",
                    help="comma list of workloads timed briefly (10 steps) after the main one "
                         "and reported under other_configs ('' for none; 1 GPU only)")
    ap.add_argument("--shared-prefix", type=int, default=1,
                    help="1: workloads with shared prompts use the shared-prefix decode")
    ap.add_argument("--graph", type=int, default=1,
                    help="1: the timed steps replay a CUDA graph of the step (default)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (profiling of a smaller case)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="override the number of sequences (profiling of a smaller case)")
    ap.add_argument("--partition", type=int, default=-1,
                    help="override the partition size (0 = one pass)")
    ap.add_argument("--visit-order", default="longest", choices=["longest", "batch"],
                    help="order in which the decode takes the sequences: longest context "
                         "(own part, with the shared-prefix decode) first, or batch order "
                         "(workloads whose contexts are all equal always run in batch order)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = workload_for(args.config)
    import dataclasses
    if args.layers > 0:
        w = dataclasses.replace(w, layers=args.layers)
    if args.seqs > 0:
        w = dataclasses.replace(w, ctx=w.ctx[:args.seqs])
    if args.partition >= 0:
        w = dataclasses.replace(w, partition_size=args.partition)

    if args.impl == "reference":
        if rank != 0:
            return 0
        cb = run_reference(args, w, rank)
        line = {"metric": METRIC, "value": cb["value"], "unit": "GB/s", "impl": "reference",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(cb["seconds"] * 1000, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "sample": cb["sample"]},
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                    "nproc", "cpu_model")},
                "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    import paged_kv_cache_220_gb300 as pkv
    from paged_kv_cache_220_gb300 import build as pkv_build
    from paged_kv_cache_220_gb300 import workload

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    if rank == 0:
        pkv_build.build()
    if dist is not None:
        dist.barrier()
    pkv.lib()

    # weak scaling: every rank runs its own batch of the workload
    w = workload.rank_workload(w, rank, world)
    pw = workload.build(w)
    L = len(pw.layers)
    P = w.partition_size
    out = [torch.empty_like(st.q) for st in pw.layers]
    ws = pkv.alloc_workspace(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, P) if P else None
    flush = None
    per_step_bytes = decode_bytes(w) * L
    if per_step_bytes < 4 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    cow = pw.cow_pairs

    cascade = None
    if w.prefix_len > 0 and args.shared_prefix and P:
        cascade = workload.prefix_groups(pw)
        # own parts: the split size without a nearly empty last partition
        # (1033-token own parts at 512: 528, two partitions instead of three)
        P = pkv.split_partition_size(cascade.max_own_context, w.block_size, P)
        w = dataclasses.replace(w, partition_size=P)
        pw.w = w
        ws = pkv.shared_prefix_workspace(w.num_seqs, w.num_heads, w.head_dim,
                                         cascade.max_own_context,
                                         cascade.max_prefix_blocks * w.block_size, P)
    if args.visit_order == "batch":
        pw.visit_order = None
        if cascade is not None:
            cascade = cascade._replace(visit_order=None)
    order = pw.visit_order if cascade is None else cascade.visit_order

    one_step = make_step(pw, out, ws, cascade, stream)

    launches_per_step = step_launches(pw, cascade)
    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
           for _ in range(K)]
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    # (1) eager steps with events around every decode launch: the roofline of
    # the decode kernel, measured live on the launching stream
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        step_ev[i][0].record(stream)
        one_step(evs[i])
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    dec_ms = [evs[i][l][0].elapsed_time(evs[i][l][1]) for i in range(K) for l in range(L)]
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    # (2) the timed steps: replays of a CUDA graph of the whole step (one host
    # dispatch per step), or eager launches with --graph 0
    graph = None
    if args.graph:
        graph = workload.capture_step(pw, out, ws, P, groups=cascade)
        for _ in range(args.warmup):
            graph.replay()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        for i in range(K):
            if flush is not None:
                flush.fill_(i & 0xFF)
            step_ev[i][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                one_step()
            step_ev[i][1].record(stream)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    total_ms = sum(step_ms)
    total_ms = workload.max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / K
    value = workload.job_throughput(per_step_bytes, world, ms_per_step)

    # copy-on-write copies of the divergence iteration, timed on a scratch
    # pool with the same block geometry (replaying them on the live pool would
    # overwrite the tokens the clones received after the divergence)
    cow_copy = None
    if cow is not None and len(pw.cow_pairs_host):
        cow_copy = time_copy_blocks(pw, args)
    host = host_iteration_timing(w) if rank == 0 else None

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, pw, w, out, ws, P, per_step_bytes, world, dist, cascade)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    other = None
    if args.other_configs and world == 1:
        other = {}
        for name in args.other_configs.split(","):
            if name and name != args.config:
                other[name] = measure_other(name)
    peak, peak_kind = peaks()
    dec_bytes = decode_bytes(w) if cascade is None else unique_decode_bytes(w)
    achieved = dec_bytes / (dec_avg_ms / 1e3) / 1e9
    traffic, traffic_note = ncu_traffic(args.config)
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cb = run_reference(args, w, rank, single_thread=True)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "nproc",
                                  "cpu_model", "single_thread")}
    tok_per_s_layer = w.num_seqs * world / (ms_per_step / 1e3 / L)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "ms_per_step_median": round(statistics.median(step_ms), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3" if w.fp8 else "bf16", "data": "synthetic",
        "config": {
            "workload": w.name, "layers": L, "num_seqs": w.num_seqs,
            "context": w.ctx[0] if len(set(w.ctx)) == 1 else "mixed (sum %d)" % sum(w.ctx),
            "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "partition_size": P,
            "kv_dtype": "fp8_e4m3" if w.fp8 else "bf16",
            "l2": "flushed before every step" if flush is not None else
                  "inputs larger than L2 (%.1f GB of K/V per step)" % (per_step_bytes / 1e9),
            "parallelism": "replicas/weak: each GPU its own batch" if world > 1 else "1 GPU",
            "cuda_graph": bool(graph is not None),
            "visit_order": "batch order" if order is None else
                           "longest %s first" % ("context" if cascade is None else "own part"),
        },
        "eager_ms_per_step": round(eager_ms / K, 4),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "pct_of_peak_basis": "%s HBM copy bandwidth %.1f GB/s" % (peak_kind, peak),
        "pct_of_nominal": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_nominal_basis": "GB300 nominal HBM3e %.0f GB/s" % NOMINAL_HBM_GBS,
        "tokens_per_s_per_layer": round(tok_per_s_layer, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": peak_kind,
                     "kernel": "paged_attention_decode" if cascade is None else
                               "paged_attention_decode_shared_prefix (3 kernels, unique bytes)",
                     "bytes_per_launch": dec_bytes, "launch_ms": round(dec_avg_ms, 5),
                     "traffic": traffic},
        "cpu_baseline": cpu, "e2e": e2e, "copy_blocks": cow_copy, "host": host,
        "other_configs": other,
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
    }
    if w.prefix_len > 0:
        line["unique_bytes_gbs"] = round(unique_decode_bytes(w) * L * world / (ms_per_step / 1e3) / 1e9, 2)
    if traffic:
        line["roofline"]["traffic_over_bytes"] = round(traffic / dec_bytes, 4)
    # the pages' memory claims, on this workload's allocation: slots held in
    # partly filled blocks, and the slots a contiguous max-length reservation
    # per sequence would take
    st = pw.alloc.stats()
    held = st["used_blocks"] * w.block_size
    line["memory"] = {
        "internal_fragmentation": round(1 - st["used_slots"] / held, 4) if held else 0.0,
        "contiguous_over_paged_slots": round(w.num_seqs * pw.max_context / held, 3) if held else None,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def host_iteration_timing(w, iters: int = 100):
    """Host side of a decode iteration on this workload's batch, off the GPU
    clock: the scheduler step (one new slot per running sequence, a block
    taken from the free list when one fills) and the export of the batch's
    block tables, on a scheduler of its own holding the workload's lengths."""
    import paged_kv_cache_220_gb300 as pkv
    B = w.block_size
    S = w.num_seqs
    mb = max(-(-(c + iters + 1) // B) for c in w.ctx)
    blocks = sum(-(-(c + iters + 1) // B) for c in w.ctx) + S
    alloc = pkv.BlockAllocator(blocks, B, seed=7)
    sched = pkv.Scheduler(alloc, S)
    for i, c in enumerate(w.ctx):
        sched.add_request(i, max(c - 1, 1), iters + 10)
    sched.step()  # admits every prompt
    t_step, t_tab = [], []
    for _ in range(iters):
        t0 = time.perf_counter()
        sched.step()
        t1 = time.perf_counter()
        sched.block_tables(mb)
        t_tab.append(time.perf_counter() - t1)
        t_step.append(t1 - t0)
    running = sched.counts()["running"]
    sched.close()
    alloc.close()
    return {"sched_step_us": round(statistics.median(t_step) * 1e6, 2),
            "block_tables_us": round(statistics.median(t_tab) * 1e6, 2),
            "running": running, "iterations": iters,
            "note": "median host time per iteration (Python call included)"}


def time_copy_blocks(pw, args):
    """copy_blocks over the workload's divergence pairs (e.g. 480 for the
    2040-token prompts), remapped into a scratch pool of 2 x pairs blocks."""
    import torch
    import paged_kv_cache_220_gb300 as pkv
    n = len(pw.cow_pairs_host)
    st = pw.layers[0]
    shape = (2 * n,) + tuple(st.k_cache.shape[1:])
    kc = torch.empty(shape, dtype=st.k_cache.dtype, device="cuda")
    vc = torch.empty_like(kc)
    kc.view(torch.uint8).random_(0, 255)
    vc.view(torch.uint8).random_(0, 255)
    perm = torch.randperm(2 * n, generator=torch.Generator().manual_seed(5))
    pairs = torch.stack([perm[:n], perm[n:]], dim=1).to(torch.int32).cuda()
    for _ in range(3):
        pkv.copy_blocks(kc, vc, pairs)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    K = max(10, args.steps)
    torch.cuda.synchronize()
    a.record()
    for _ in range(K):
        pkv.copy_blocks(kc, vc, pairs)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    block_bytes = kc[0].numel() * kc.element_size()
    moved = n * block_bytes * 2 * 2          # K and V, read + write
    return {"pairs": n, "ms": round(ms, 5), "bytes": moved,
            "gbs": round(moved / (ms / 1e3) / 1e9, 1), "layers": 1}


def run_e2e(args, pw, w, out, ws, P, per_step_bytes, world, dist, cascade=None):
    """Same step through the public API, inputs copied from pinned host
    memory every step (q, new K/V, slots, block tables, context lengths, the
    visit order where the lengths differ) and
    the outputs copied back. The copies run on two streams of their own (in,
    out), layer by layer, overlapped with the compute of other layers; device
    buffers are double buffered across steps. The timed region ends after the
    last copy back of the last step. Shared-prefix workloads go through the
    shared-prefix call, their group metadata copied in with the rest."""
    import torch
    import paged_kv_cache_220_gb300 as pkv
    L = len(pw.layers)
    keys = ("q", "k_new", "v_new")
    host = [{k: getattr(st, k).cpu().pin_memory() for k in keys} for st in pw.layers]
    meta = [pw.slot_mapping, pw.block_tables, pw.context_lens]
    if cascade is not None:
        meta += [cascade.group_start, cascade.prefix_blocks]
    # the visit order (host-computed from the lengths, like the tables) last
    order = pw.visit_order if cascade is None else cascade.visit_order
    if order is not None:
        meta.append(order)
    h_meta = [t.cpu().pin_memory() for t in meta]
    h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in out]
    # two sets of device buffers: step i uses set i % 2
    dev = [[{k: torch.empty_like(getattr(st, k)) for k in keys} for st in pw.layers]
           for _ in range(2)]
    d_meta = [[torch.empty_like(t) for t in meta] for _ in range(2)]
    d_out = [[torch.empty_like(o) for o in out] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for hl in host for t in hl.values()) + \
        sum(t.numel() * t.element_size() for t in h_meta)
    d2h = sum(o.numel() * o.element_size() for o in out)
    main = torch.cuda.current_stream()
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(L)]
    ev_meta = torch.cuda.Event()
    ev_out = [torch.cuda.Event() for _ in range(L)]
    # set b is free again once its step's compute and copies back are done
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]
    ev_free[0].record(main)
    ev_free[1].record(main)
    it = [0]

    def step():
        b = it[0] & 1
        it[0] += 1
        dv, dm, do = dev[b], d_meta[b], d_out[b]
        # set b was last used two steps ago: its compute and copies back are done
        copy_in.wait_event(ev_free[b])
        with torch.cuda.stream(copy_in):
            for d, h in zip(dm, h_meta):
                d.copy_(h, non_blocking=True)
            ev_meta.record(copy_in)
            for layer in range(L):
                for k in keys:
                    dv[layer][k].copy_(host[layer][k], non_blocking=True)
                ev_in[layer].record(copy_in)
        main.wait_event(ev_meta)
        d_sm, d_bt, d_cl = dm[:3]
        for layer, st in enumerate(pw.layers):
            main.wait_event(ev_in[layer])
            pkv.kv_cache_write(dv[layer]["k_new"], dv[layer]["v_new"], d_sm, st.k_cache,
                               st.v_cache, st.k_scale, st.v_scale)
            if cascade is not None:
                pkv.paged_attention_shared_prefix(dv[layer]["q"], st.k_cache, st.v_cache, d_bt,
                                                  d_cl, w.scale, cascade.max_own_context, dm[3],
                                                  dm[4], cascade.max_prefix_blocks, P,
                                                  cascade.max_group_members, out=do[layer],
                                                  workspace=ws, k_scale=st.k_scale,
                                                  v_scale=st.v_scale,
                                                  seq_order=dm[-1] if order is not None else None)
            else:
                pkv.paged_attention(dv[layer]["q"], st.k_cache, st.v_cache, d_bt, d_cl, w.scale,
                                    pw.max_context, P, st.k_scale, st.v_scale, out=do[layer],
                                    workspace=ws,
                                    seq_order=dm[-1] if order is not None else None)
            ev_out[layer].record(main)
            copy_out.wait_event(ev_out[layer])
            with torch.cuda.stream(copy_out):
                h_out[layer].copy_(do[layer], non_blocking=True)
        ev_free[b].record(copy_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    K = args.steps
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    a.record(main)
    for _ in range(K):
        step()
    main.wait_stream(copy_out)
    e.record(main)
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t0) * 1e3
    ms = max(a.elapsed_time(e), wall_ms) / K
    if dist is not None:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": round(per_step_bytes * world / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 4), "copies": "own streams, overlapped with compute"}


if __name__ == "__main__":
    sys.exit(main())
