"""Oracle-side inputs and comparisons for the GPU parity tests.

Everything here is computed on the host from the seeded generator (the same
element streams the device side generates) and the oracle; nothing is read
back from the CUDA library except the outputs under test.
"""
import numpy as np
import torch

import oracle
from paged_kv_cache_220_gb300 import synth

# Tolerances for bf16 attention outputs (and FP8-KV outputs against the
# oracle on the same FP8 codes): maximum absolute error and relative L2 error.
MAX_ABS = 1e-2
REL_L2 = 5e-3


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def host_rows(w: synth.Workload, layer: int, s: int, t1: int = None):
    t1 = w.ctx[s] if t1 is None else t1
    return (w.rows(synth.KIND_K, layer, s, 0, t1, "cpu"),
            w.rows(synth.KIND_V, layer, s, 0, t1, "cpu"))


class RowCache:
    """Host rows of one layer, the shared prompt rows of a shared-prefix
    workload generated once per prompt instead of once per member."""

    def __init__(self, w: synth.Workload, layer: int):
        self.w, self.layer = w, layer
        self.prompts = {}

    def rows(self, s: int):
        """(K, V) bf16 [ctx_s, Hk, d] of sequence s."""
        w = self.w
        if w.prefix_len <= 0:
            return host_rows(w, self.layer, s)
        p = s // w.group
        if p not in self.prompts:
            self.prompts = {p: host_rows(w, self.layer, p * w.group, w.prefix_len)}
        pk, pv = self.prompts[p]
        t1 = w.ctx[s]
        if t1 <= w.prefix_len:
            return pk[:t1], pv[:t1]
        k = w.rows(synth.KIND_K, self.layer, s, w.prefix_len, t1, "cpu")
        v = w.rows(synth.KIND_V, self.layer, s, w.prefix_len, t1, "cpu")
        return torch.cat([pk, k]), torch.cat([pv, v])


def host_fp8_scales(w: synth.Workload, layer: int, rows=None):
    """Per-KV-head E4M3 scales computed on the host: the fp32 maximum of |x|
    over every logical row of every sequence of the layer (history and the
    new token), divided by 448 in fp32. `rows(s)` may supply the rows."""
    amax_k = np.zeros(w.num_kv_heads, dtype=np.float32)
    amax_v = np.zeros(w.num_kv_heads, dtype=np.float32)
    for s in range(w.num_seqs):
        K, V = rows(s) if rows is not None else host_rows(w, layer, s)
        amax_k = np.maximum(amax_k, K.float().abs().amax(dim=(0, 2)).numpy())
        amax_v = np.maximum(amax_v, V.float().abs().amax(dim=(0, 2)).numpy())
    return amax_k / np.float32(448.0), amax_v / np.float32(448.0)


def quantize(rows_bf16: torch.Tensor, scale: np.ndarray) -> np.ndarray:
    """E4M3 codes of x / scale[h] (fp32 quotient) with the oracle's encoder."""
    return oracle.e4m3_encode_bf16(bits16(rows_bf16), scale)


def expected(w: synth.Workload, layer: int, seqs, k_scale=None, v_scale=None,
             rows=None) -> np.ndarray:
    """fp64 oracle output [len(seqs), Hq, D] for the given sequences.
    `rows(s)` may supply the host rows (e.g. RowCache(w, layer).rows)."""
    q = bits16(w.q(layer, "cpu"))[list(seqs)]
    ks, vs = [], []
    for s in seqs:
        K, V = rows(s) if rows is not None else host_rows(w, layer, s)
        if w.fp8:
            ks.append(quantize(K, k_scale))
            vs.append(quantize(V, v_scale))
        else:
            ks.append(bits16(K))
            vs.append(bits16(V))
    if w.fp8:
        return oracle.decode(q, ks, vs, w.scale, k_scale.astype(np.float64),
                             v_scale.astype(np.float64))
    return oracle.decode(q, ks, vs, w.scale)


def expected_pool(w: synth.Workload, layer: int, num_blocks: int, slots_per_seq,
                  k_scale=None, v_scale=None):
    """Pool images (K, V) after every logical row of every sequence has been
    written to its slot: the block-table definition applied by the oracle."""
    dt = np.uint8 if w.fp8 else np.uint16
    shape = (num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    pk, pv = np.zeros(shape, dtype=dt), np.zeros(shape, dtype=dt)
    for s in range(w.num_seqs):
        K, V = host_rows(w, layer, s)
        if w.fp8:
            k, v = quantize(K, k_scale), quantize(V, v_scale)
        else:
            k, v = bits16(K), bits16(V)
        oracle.scatter_rows_fast(pk, k, slots_per_seq[s])
        oracle.scatter_rows_fast(pv, v, slots_per_seq[s])
    return pk, pv


def errors(got_bf16: torch.Tensor, ref: np.ndarray):
    g = bf16_to_f64(bits16(got_bf16))
    diff = g - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / den if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got_bf16, ref, what=""):
    ma, rl = errors(got_bf16, ref)
    assert ma <= MAX_ABS and rl <= REL_L2, "%s: max_abs=%.3e rel_l2=%.3e" % (what, ma, rl)
    return ma, rl
