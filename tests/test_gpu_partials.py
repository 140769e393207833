"""The split decode's per-partition partials, read back from the workspace and
compared with the oracle's per-partition statistics one by one.

The decode's partial p of a (sequence, query head) row covers logical tokens
[p*P, min((p+1)*P, ctx)) and holds the partition's largest logit m (natural
log units), its exponential sum l = sum exp(z - m) and the normalised output
sum exp(z - m) V / l. End-to-end tests see these only through the merge, where
a compensating pair of mistakes (a unit of m, a slot offset) could hide; here
each one is checked against the oracle directly, and every slot the decode
must not write is checked to be untouched.

The shared-prefix decode stores, per row, the shared partitions (size Pp, from
token 0) in slots [0, NPP) and the member's own partitions (size P, from token
prefix_blocks * B) in slots [NPP, NPP + NPS); both ranges are checked the same
way."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build as pkv_build
from paged_kv_cache_220_gb300 import synth, workload
from _oracle_side import bits16, host_fp8_scales, host_rows, quantize

pytestmark = pytest.mark.gpu

M_ABS = 1e-3        # largest logit, natural-log units
L_REL = 5e-3        # exponential sum
O_MAX_ABS = 1e-2    # normalised partial output, per (row, partition)
O_REL_L2 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.set_device_check(flag)
    yield flag
    pkv.set_device_check(None)


def _views(ws, S, Hq, NP, D):
    """(tmp_out [S,Hq,NP,D], max_logits [S,Hq,NP], exp_sums [S,Hq,NP]) on the host."""
    f = ws.view(torch.float32).cpu().numpy().astype(np.float64)
    R = S * Hq * NP
    return (f[:R * D].reshape(S, Hq, NP, D), f[R * D:R * D + R].reshape(S, Hq, NP),
            f[R * D + R:R * D + 2 * R].reshape(S, Hq, NP))


def _oracle_rows(w, rows, t0, t1, ks=None, vs=None):
    K, V = rows
    K, V = K[t0:t1], V[t0:t1]
    if ks is not None:
        return quantize(K, ks), quantize(V, vs)
    return bits16(K), bits16(V)


def _check_slots(got, ref, slots, what, exact_max=True):
    """got/ref: (tmp, ml, es) of one sequence [Hq, NP(, D)]; slots: pairs
    (slot in got, partition in ref). exact_max: m is the partition's largest
    logit; otherwise m may be any reference value at most 8 log2-units below
    it (the shared-prefix kernel rescales only when the maximum grows by more
    than 2^8), so the log-sum-exp m + ln l is what must agree."""
    gt, gm, ge = got
    rt, rm, re_ = ref
    for gs, rs in slots:
        lse_g = gm[:, gs] + np.log(ge[:, gs])
        lse_r = rm[:, rs] + np.log(re_[:, rs])
        dz = np.abs(lse_g - lse_r)
        assert np.all(dz <= L_REL), "%s slot %d: log-sum-exp off by %.3e" % (what, gs, dz.max())
        if exact_max:
            dm = np.abs(gm[:, gs] - rm[:, rs])
            assert np.all(dm <= M_ABS), "%s slot %d: max logit off by %.3e" % (what, gs, dm.max())
            dl = np.abs(ge[:, gs] - re_[:, rs]) / re_[:, rs]
            assert np.all(dl <= L_REL), "%s slot %d: exp sum rel %.3e" % (what, gs, dl.max())
        else:
            assert np.all(gm[:, gs] <= rm[:, rs] + M_ABS), "%s slot %d: m above max" % (what, gs)
            assert np.all(gm[:, gs] >= rm[:, rs] - 8 * np.log(2) - M_ABS), "%s slot %d" % (what, gs)
        d = gt[:, gs, :] - rt[:, rs, :]
        ma = float(np.abs(d).max())
        rl = float(np.linalg.norm(d) / np.linalg.norm(rt[:, rs, :]))
        assert ma <= O_MAX_ABS and rl <= O_REL_L2, "%s slot %d: o max_abs %.3e rel %.3e" % (
            what, gs, ma, rl)


CASES = [(False, 16, 16), (False, 16, 32), (False, 16, 64), (False, 16, 512), (False, 32, 32),
         (False, 32, 512), (True, 32, 32), (True, 32, 64), (True, 32, 512), (True, 16, 64),
         (True, 16, 48), (True, 16, 528)]


@pytest.mark.parametrize("fp8,B,P", CASES)
def test_split_partials_match_oracle(fp8, B, P, _lib):
    ctx = sorted({1, B - 1, B + 1, P - 1 if P > 1 else 1, P, P + 1, 3 * P + 5, 2000})
    ctx = [c for c in ctx if c >= 1]
    w = synth.Workload("partials", 1100 + B + P + (7 if fp8 else 0), 24, 4, 256, B, ctx,
                       fp8=fp8, partition_size=P, slack_blocks=8)
    pw = workload.build(w)
    st = pw.layers[0]
    S, Hq, D = w.num_seqs, w.num_heads, w.head_dim
    ks = vs = None
    if fp8:
        ks, vs = host_fp8_scales(w, 0)
        assert np.array_equal(ks.view(np.uint32), st.k_scale.cpu().numpy().view(np.uint32))
        assert np.array_equal(vs.view(np.uint32), st.v_scale.cpu().numpy().view(np.uint32))
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                       st.k_scale, st.v_scale)
    NP = -(-pw.max_context // P)
    ws = pkv.alloc_workspace(S, Hq, D, pw.max_context, P)
    ws.view(torch.float32).fill_(float("nan"))
    pkv.paged_attention_decode(None, st.q, st.k_cache, st.v_cache, pw.block_tables,
                               pw.context_lens, w.scale, pw.max_context, P, ws,
                               st.k_scale, st.v_scale)
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    tmp, ml, es = _views(ws, S, Hq, NP, D)
    q = bits16(w.q(0, "cpu"))
    for s in range(S):
        kk, vv = _oracle_rows(w, host_rows(w, 0, s), 0, w.ctx[s], ks, vs)
        args = (q[s:s + 1], [kk], [vv], w.scale, P, NP)
        if fp8:
            args += (ks.astype(np.float64), vs.astype(np.float64))
        rm, rl, ro = oracle.decode_partials(*args)
        n = -(-w.ctx[s] // P)
        _check_slots((tmp[s], ml[s], es[s]), (ro[0], rm[0], rl[0]),
                     [(p, p) for p in range(n)], "ctx %d" % w.ctx[s])
        # partitions past the context are never written
        assert np.all(np.isnan(ml[s, :, n:])) and np.all(np.isnan(tmp[s, :, n:]))


@pytest.mark.parametrize("prompt,prompts,rollouts,P,fp8", [(2040, 2, 16, 512, False),
                                                          (1024, 8, 4, 64, False),
                                                          (300, 2, 32, 64, False),
                                                          (1024, 8, 4, 64, True),
                                                          (300, 2, 32, 64, True)])
def test_shared_prefix_slots_match_oracle(prompt, prompts, rollouts, P, fp8, _lib):
    w = synth.cow(prompt_len=prompt, prompts=prompts, rollouts=rollouts)
    comp = w.extra["completion"]
    w = dataclasses.replace(w, ctx=[prompt + (c % 700) + 1 for c in comp], fp8=fp8)
    pw = workload.build(w)
    ks = vs = None
    if fp8:
        ks, vs = host_fp8_scales(w, 0)
    gr = workload.prefix_groups(pw)
    st = pw.layers[0]
    B = w.block_size
    S, Hq, Hk, D = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim
    G = int(gr.group_start.shape[0]) - 1
    Pp = pkv.shared_prefix_partition_size(G, gr.max_group_members, Hk, Hq, B,
                                          gr.max_prefix_blocks, P)
    assert Pp >= P and Pp % P == 0
    NPP = -(-(gr.max_prefix_blocks * B) // Pp)
    NPS = -(-gr.max_own_context // P)
    NPT = NPP + NPS
    ws = pkv.shared_prefix_workspace(S, Hq, D, gr.max_own_context, gr.max_prefix_blocks * B, P)
    ws.view(torch.float32).fill_(float("nan"))
    pkv.kv_cache_write(st.k_new, st.v_new, pw.slot_mapping, st.k_cache, st.v_cache,
                       st.k_scale, st.v_scale)
    pkv.paged_attention_shared_prefix(st.q, st.k_cache, st.v_cache, pw.block_tables,
                                      pw.context_lens, w.scale, gr.max_own_context,
                                      gr.group_start, gr.prefix_blocks, gr.max_prefix_blocks, P,
                                      gr.max_group_members, workspace=ws, k_scale=st.k_scale,
                                      v_scale=st.v_scale)
    torch.cuda.synchronize()
    assert int(_lib.item()) == 0
    tmp, ml, es = _views(ws, S, Hq, NPT, D)
    pre = gr.prefix_blocks.cpu().numpy()
    q = bits16(w.q(0, "cpu"))
    for s in range(S):
        rows = host_rows(w, 0, s)
        t_pre = int(pre[s]) * B
        npre = -(-t_pre // Pp)
        nown = -(-(w.ctx[s] - t_pre) // P)
        sc = (ks.astype(np.float64), vs.astype(np.float64)) if fp8 else ()
        kk, vv = _oracle_rows(w, rows, 0, t_pre, ks, vs)
        rm, rl, ro = oracle.decode_partials(q[s:s + 1], [kk], [vv], w.scale, Pp, NPP, *sc)
        _check_slots((tmp[s], ml[s], es[s]), (ro[0], rm[0], rl[0]),
                     [(p, p) for p in range(npre)], "seq %d shared" % s, exact_max=False)
        kk, vv = _oracle_rows(w, rows, t_pre, w.ctx[s], ks, vs)
        rm, rl, ro = oracle.decode_partials(q[s:s + 1], [kk], [vv], w.scale, P, NPS, *sc)
        _check_slots((tmp[s], ml[s], es[s]), (ro[0], rm[0], rl[0]),
                     [(NPP + p, p) for p in range(nown)], "seq %d own" % s)
        assert np.all(np.isnan(ml[s, :, npre:NPP])) and np.all(np.isnan(ml[s, :, NPP + nown:]))
