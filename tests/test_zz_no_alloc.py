"""The allocation-free decode entry point.

Some callers cannot allocate device memory (a framework that owns the whole
device budget, C callers without a device allocator, latency-critical paths
where an allocation may synchronise the device). For them the library offers
pkv_paged_attention_decode_noalloc, which keeps the split-decode partials in
a fixed array of its own. This test calls it through the C ABI twice in a row,
on two different workloads, and compares each result with the workspace
entry points (decode + reduce) within the parity tolerance.

The file name makes pytest collect it last.
"""
import ctypes
import dataclasses

import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import MAX_ABS, REL_L2, errors

pytestmark = pytest.mark.gpu


def _noalloc_call(pw, out, P):
    """Raw C-ABI call (pointers, sizes and the current stream)."""
    st = pw.layers[0]
    w = pw.w
    L = pkv.lib()
    P_ = ctypes.c_void_p
    rc = L.pkv_paged_attention_decode_noalloc(
        P_(out.data_ptr()), P_(st.q.data_ptr()), P_(st.k_cache.data_ptr()),
        P_(st.v_cache.data_ptr()), pkv.cache_desc(st.k_cache),
        P_(st.k_scale.data_ptr()) if st.k_scale is not None else None,
        P_(st.v_scale.data_ptr()) if st.v_scale is not None else None,
        P_(pw.block_tables.data_ptr()), int(pw.block_tables.shape[1]),
        P_(pw.context_lens.data_ptr()), w.num_seqs, w.num_heads, pw.max_context,
        ctypes.c_float(w.scale), P, P_(torch.cuda.current_stream().cuda_stream))
    return rc


def _workspace_result(pw, P):
    st = pw.layers[0]
    w = pw.w
    return pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, pw.context_lens,
                               w.scale, pw.max_context, P, st.k_scale, st.v_scale)


def test_noalloc_matches_workspace_entry_points_two_calls():
    pkv_build.build()
    a = workload.build(synth.mixed(num_seqs=40))
    b = workload.build(dataclasses.replace(synth.long_fp8(num_seqs=2, ctx=3000), ctx=[3000, 1111]))
    for pw, P in ((a, 512), (b, 256)):
        out = torch.full_like(pw.layers[0].q, float("nan"))
        assert _noalloc_call(pw, out, P) == pkv.PKV_OK
        ref = _workspace_result(pw, P)
        torch.cuda.synchronize()
        ma, rl = errors(out.cpu(), ref.cpu().double().numpy())
        assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)


def test_noalloc_rejects_partials_larger_than_its_scratch():
    pkv_build.build()
    pw = workload.build(synth.tiny())
    out = torch.empty_like(pw.layers[0].q)
    w = pw.w
    need = pkv.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, pw.max_context, 16)
    assert need <= pkv.NOALLOC_SCRATCH_BYTES          # tiny fits
    # a context bound that would need more partials than the scratch holds
    S, Hq, D = 4, 8, 128
    too_long = (pkv.NOALLOC_SCRATCH_BYTES // (S * Hq * (D + 2) * 4) + 1) * 16
    L = pkv.lib()
    P_ = ctypes.c_void_p
    st = pw.layers[0]
    rc = L.pkv_paged_attention_decode_noalloc(
        P_(out.data_ptr()), P_(st.q.data_ptr()), P_(st.k_cache.data_ptr()),
        P_(st.v_cache.data_ptr()), pkv.cache_desc(st.k_cache), None, None,
        P_(pw.block_tables.data_ptr()), too_long // 16 + 1, P_(pw.context_lens.data_ptr()),
        S, Hq, too_long, ctypes.c_float(w.scale), 16, None)
    assert rc == pkv.PKV_ERR_UNSUPPORTED
    assert L.pkv_paged_attention_decode_noalloc(
        P_(out.data_ptr()), P_(st.q.data_ptr()), P_(st.k_cache.data_ptr()),
        P_(st.v_cache.data_ptr()), pkv.cache_desc(st.k_cache), None, None,
        P_(pw.block_tables.data_ptr()), 64, P_(pw.context_lens.data_ptr()),
        S, Hq, pw.max_context, ctypes.c_float(w.scale), 0, None) == pkv.PKV_ERR_INVALID_ARG
