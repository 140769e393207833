"""The allocation-free decode entry point.

Some callers cannot allocate device memory: code running inside a framework
that owns the whole device-memory budget, C callers without a device
allocator, and latency-critical paths where an allocation may synchronise the
device. For them the library offers pkv_paged_attention_decode_noalloc, which
keeps the split-decode partials in a fixed array of its own.

The calls here go through the C ABI. The entry point runs the same kernels on
the same partitions as the workspace entry points, so its output must equal
theirs bit for bit; it is also compared with the oracle. The calls come in a
row on different workloads, the later one with shorter contexts and fewer
partitions than the one before, so a partial left in the shared array by an
earlier call would show. All contexts empty give zeros; partials larger than
the array are rejected.

The file name makes pytest collect it last.
"""
import ctypes
import dataclasses

import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, expected, host_fp8_scales

pytestmark = pytest.mark.gpu


def _noalloc_call(pw, out, P, context_lens=None, max_context=None):
    """Raw C-ABI call (pointers, sizes and the current stream)."""
    st = pw.layers[0]
    w = pw.w
    cl = pw.context_lens if context_lens is None else context_lens
    mc = pw.max_context if max_context is None else max_context
    L = pkv.lib()
    P_ = ctypes.c_void_p
    return L.pkv_paged_attention_decode_noalloc(
        P_(out.data_ptr()), P_(st.q.data_ptr()), P_(st.k_cache.data_ptr()),
        P_(st.v_cache.data_ptr()), pkv.cache_desc(st.k_cache),
        P_(st.k_scale.data_ptr()) if st.k_scale is not None else None,
        P_(st.v_scale.data_ptr()) if st.v_scale is not None else None,
        P_(pw.block_tables.data_ptr()), int(pw.block_tables.shape[1]),
        P_(cl.data_ptr()), w.num_seqs, w.num_heads, mc,
        ctypes.c_float(w.scale), P, P_(torch.cuda.current_stream().cuda_stream))


def _workspace_result(pw, P, context_lens=None, max_context=None):
    st = pw.layers[0]
    w = pw.w
    cl = pw.context_lens if context_lens is None else context_lens
    mc = pw.max_context if max_context is None else max_context
    return pkv.paged_attention(st.q, st.k_cache, st.v_cache, pw.block_tables, cl, w.scale, mc, P,
                               st.k_scale, st.v_scale)


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_noalloc_matches_workspace_entry_points_calls_in_a_row():
    pkv_build.build()
    a = workload.build(synth.mixed(num_seqs=40))
    b = workload.build(dataclasses.replace(synth.long_fp8(num_seqs=2, ctx=3000), ctx=[3000, 1111]))
    for pw in (a, b):
        st = pw.layers[0]
        pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                           st.k_scale, st.v_scale)
    torch.cuda.synchronize()
    # the second mixed call attends over a third of each context: fewer
    # partitions than the call before it left in the shared array
    short_ctx = [max(1, c // 3) for c in a.w.ctx]
    short = torch.tensor(short_ctx, dtype=torch.int32, device="cuda")
    runs = [(a, 512, None, None), (b, 256, None, None), (a, 512, short, max(short_ctx))]
    for pw, P, cl, mc in runs:
        out = torch.full_like(pw.layers[0].q, float("nan"))
        assert _noalloc_call(pw, out, P, cl, mc) == pkv.PKV_OK
        ref = _workspace_result(pw, P, cl, mc)
        torch.cuda.synchronize()
        assert _same_bits(out, ref), "noalloc differs from the workspace entry points"
        w = pw.w if cl is None else dataclasses.replace(pw.w, ctx=short_ctx)
        ks = vs = None
        if w.fp8:
            ks, vs = host_fp8_scales(w, 0)
        assert_close(out.cpu(), expected(w, 0, range(w.num_seqs), ks, vs), "noalloc vs oracle")


def test_noalloc_empty_contexts_give_zeros():
    pkv_build.build()
    pw = workload.build(synth.tiny())
    zero = torch.zeros_like(pw.context_lens)
    out = torch.full_like(pw.layers[0].q, float("nan"))
    assert _noalloc_call(pw, out, 16, zero, 0) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert torch.equal(out.float(), torch.zeros_like(out.float()))


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
