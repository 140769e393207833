"""Swapping a sequence's blocks to pinned host memory and back: the blocks
come back byte for byte into fresh blocks, and decode over the restored
sequence gives the same output bit for bit as before the swap."""
import numpy as np
import pytest
import torch

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import assert_close, bits16, expected

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp8", [False, True])
def test_swap_out_free_reuse_swap_in(fp8):
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    import dataclasses
    w = dataclasses.replace(synth.tiny(), fp8=fp8, num_blocks=None, slack_blocks=80)
    pw = workload.build(w)
    st = pw.layers[0]
    out0 = workload_step(pw)
    a = pw.alloc
    victim = 3                                   # the 1024-token sequence
    seq = pw.seqs[victim]
    table = a.block_table(seq)
    n, ctx = len(table), a.seq_len(seq)
    blocks = torch.as_tensor(table).pin_memory()
    kb = torch.empty((n,) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype).pin_memory()
    vb = torch.empty_like(kb).pin_memory()
    pkv.swap_out(st.k_cache, st.v_cache, blocks, kb, vb)
    torch.cuda.synchronize()
    assert torch.equal(kb.view(torch.uint8), st.k_cache[table.tolist()].cpu().view(torch.uint8))
    a.free(seq)
    # other requests take the freed blocks and overwrite them
    other = a.new_seq()
    slots, _ = a.append(other, len(table) * w.block_size)
    junk = torch.full((len(slots), w.num_kv_heads, w.head_dim), -7.0, dtype=torch.bfloat16,
                      device="cuda")
    pkv.kv_cache_write(junk, junk, torch.as_tensor(slots, device="cuda"), st.k_cache,
                       st.v_cache, st.k_scale, st.v_scale)
    # bring the sequence back into fresh blocks
    back = a.new_seq()
    a.append(back, ctx)
    new_table = a.block_table(back)
    assert len(set(new_table.tolist()) & set(table.tolist())) < len(table)
    pkv.swap_in(st.k_cache, st.v_cache, torch.as_tensor(new_table).pin_memory(), kb, vb)
    bt = pw.block_tables.clone()
    bt[victim, :n] = torch.as_tensor(new_table, device="cuda")
    out1 = torch.empty_like(st.q)
    pkv.paged_attention_decode(out1, st.q, st.k_cache, st.v_cache, bt, pw.context_lens,
                               w.scale, pw.max_context, 0, None, st.k_scale, st.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(out1[victim].view(torch.int16), out0[victim].view(torch.int16))
    assert int(flag.item()) == 0
    pkv.set_device_check(None)


def workload_step(pw):
    out = [torch.empty_like(st.q) for st in pw.layers]
    workload.step(pw, out, None, 0)
    torch.cuda.synchronize()
    return out[0].clone()


def test_whole_cache_checkpoint_and_resume():
    """Checkpoint of a whole cache state: the allocator record plus every used
    block (shared blocks once) swapped to pinned host memory; the pools are
    wiped and the allocator dropped; a loaded allocator and a swap-in into the
    same block ids give the same decode output bit for bit."""
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    w = synth.cow(prompt_len=40, prompts=2, rollouts=4)
    pw = workload.build(w)
    st = pw.layers[0]
    out0 = workload_step(pw)
    record = pw.alloc.save()
    used = sorted({int(b) for s in pw.seqs for b in pw.alloc.block_table(s)})
    blocks = torch.as_tensor(used, dtype=torch.int32).pin_memory()
    kb = torch.empty((len(used),) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype).pin_memory()
    vb = torch.empty_like(kb).pin_memory()
    pkv.swap_out(st.k_cache, st.v_cache, blocks, kb, vb)
    torch.cuda.synchronize()
    st.k_cache.zero_()
    st.v_cache.zero_()
    pw.alloc.close()
    alloc = pkv.BlockAllocator.load(record)
    tables = alloc.block_tables(pw.seqs, pw.block_tables.shape[1])
    assert np.array_equal(tables, pw.block_tables.cpu().numpy())
    pkv.swap_in(st.k_cache, st.v_cache, blocks, kb, vb)
    out1 = torch.empty_like(st.q)
    pkv.paged_attention_decode(out1, st.q, st.k_cache, st.v_cache,
                               torch.as_tensor(tables, device="cuda"), pw.context_lens, w.scale,
                               pw.max_context, 0, None, st.k_scale, st.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out0.view(torch.int16))
    assert int(flag.item()) == 0
    pkv.set_device_check(None)
