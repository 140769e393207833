"""Pins of the CPU oracle against things other than itself.

Each check below ties one oracle function to a fixed point that does not come
from the oracle: a library routine that computes the same quantity
(torch scaled-dot-product attention in float64, torch's float8 conversion), a
closed form (one row, zero query, equal keys, a dominant logit), a
mathematical identity (log-sum-exp merging of partitions), values the pages
print (the allocation example of Figures 1 and 2, the KV footprint), or the
OCP E4M3 definition. The last test plants each of the oracle's known
mistakes in turn and checks that some pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _random_case(seed, S=3, Hq=8, Hk=2, d=32, lens=(1, 7, 40), qmul=1.0):
    g = torch.Generator().manual_seed(seed)
    q = _bf16_bits(torch.randn(S, Hq, d, generator=g) * qmul)
    ks = [_bf16_bits(torch.randn(T, Hk, d, generator=g)) for T in lens[:S]]
    vs = [_bf16_bits(torch.randn(T, Hk, d, generator=g)) for T in lens[:S]]
    return q, ks, vs


def _sdpa_reference(q_bits, k_rows, v_rows, scale):
    """torch.nn.functional.scaled_dot_product_attention in float64 per sequence."""
    q = torch.from_numpy(_bf16_values(q_bits))
    S, Hq, d = q.shape
    out = torch.zeros(S, Hq, d, dtype=torch.float64)
    for s in range(S):
        K = torch.from_numpy(_bf16_values(k_rows[s]))  # [T, Hk, d]
        V = torch.from_numpy(_bf16_values(v_rows[s]))
        T, Hk, _ = K.shape
        if T == 0:
            continue
        g = Hq // Hk
        Kq = K.permute(1, 0, 2).repeat_interleave(g, dim=0)  # [Hq, T, d]
        Vq = V.permute(1, 0, 2).repeat_interleave(g, dim=0)
        qs = q[s].unsqueeze(1)  # [Hq, 1, d]
        o = torch.nn.functional.scaled_dot_product_attention(qs, Kq, Vq, scale=scale)
        out[s] = o[:, 0, :]
    return out.numpy()


# ---------------------------------------------------------------- pins as functions
def pin_sdpa_error(seed=0, d=32, Hq=8, Hk=2, lens=(1, 7, 40)):
    q, ks, vs = _random_case(seed, S=len(lens), Hq=Hq, Hk=Hk, d=d, lens=lens)
    scale = 1.0 / math.sqrt(d)
    got = oracle.decode(q, ks, vs, scale)
    ref = _sdpa_reference(q, ks, vs, scale)
    return float(np.max(np.abs(got - ref)))


def pin_single_row_error():
    q, ks, vs = _random_case(1, S=2, lens=(1, 1))
    got = oracle.decode(q, ks, vs, 0.3)
    g = q.shape[1] // ks[0].shape[1]
    want = np.stack([np.repeat(_bf16_values(v[0]), g, axis=0) for v in vs])
    return float(np.max(np.abs(got - want)))


def pin_zero_query_error():
    q, ks, vs = _random_case(2, S=2, lens=(5, 33))
    q[:] = 0
    got = oracle.decode(q, ks, vs, 0.125)
    g = q.shape[1] // ks[0].shape[1]
    want = np.stack([np.repeat(_bf16_values(v).mean(axis=0), g, axis=0) for v in vs])
    return float(np.max(np.abs(got - want)))


def pin_dominant_logit_error():
    """Key row t0 equals 8x the query of its heads' first query; with a large
    scale the softmax puts all weight on t0 (others are exp(-huge) = 0)."""
    d, Hq, Hk, T, t0 = 16, 4, 1, 9, 5
    q = np.zeros((1, Hq, d), dtype=np.uint16)
    one = _bf16_bits(torch.ones(1))[0]
    q[0, :, 0] = one                     # every query = e_0
    k = np.zeros((T, Hk, d), dtype=np.uint16)
    k[t0, 0, 0] = _bf16_bits(torch.tensor([8.0]))[0]
    gen = torch.Generator().manual_seed(3)
    v = _bf16_bits(torch.randn(T, Hk, d, generator=gen))
    got = oracle.decode(q, [k], [v], 1000.0)
    want = np.repeat(_bf16_values(v[t0]), Hq, axis=0)
    return float(np.max(np.abs(got[0] - want)))


def pin_gqa_grouping_error():
    """Query head j must read KV head j // g: give each KV head a distinct
    constant V row so the output names the head that was read."""
    d, Hq, Hk, T = 8, 6, 3, 4
    gen = torch.Generator().manual_seed(4)
    q = _bf16_bits(torch.randn(1, Hq, d, generator=gen))
    k = _bf16_bits(torch.randn(T, Hk, d, generator=gen))
    v = np.zeros((T, Hk, d), dtype=np.uint16)
    for h in range(Hk):
        v[:, h, :] = _bf16_bits(torch.full((1,), float(h + 1)))[0]
    got = oracle.decode(q, [k], [v], 0.5)
    want = np.array([[float(j // (Hq // Hk) + 1)] * d for j in range(Hq)])
    return float(np.max(np.abs(got[0] - want)))


def pin_partials_merge_error(P=16):
    q, ks, vs = _random_case(5, S=3, lens=(3, 40, 17))
    scale = 0.2
    full = oracle.decode(q, ks, vs, scale)
    npmax = -(-40 // P)
    m, l, o = oracle.decode_partials(q, ks, vs, scale, P, npmax)
    err = 0.0
    for s, T in enumerate((3, 40, 17)):
        n = -(-T // P)
        M = np.max(m[s, :, :n], axis=1, keepdims=True)
        w = l[s, :, :n] * np.exp(m[s, :, :n] - M)
        merged = np.einsum("jp,jpc->jc", w / w.sum(axis=1, keepdims=True), o[s, :, :n])
        err = max(err, float(np.max(np.abs(merged - full[s]))))
    return err


def pin_e4m3_decode_mismatches():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    return int(np.sum(~both_nan & (ours != ref)))


def pin_e4m3_encode_mismatches(scales=(1.0, 0.0089, 0.37, 3.0)):
    """All finite bf16 values divided (fp32) by several scales: the oracle must
    agree with torch's float8_e4m3fn cast wherever that cast is in range, and
    saturate to +-448 above it."""
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x)]
    bad = 0
    for sc in scales:
        with np.errstate(over="ignore"):
            y = (x / np.float32(sc)).astype(np.float32)
        y = y[np.isfinite(y)]
        ours = oracle.e4m3_encode(y)
        inr = np.abs(y) <= 448.0
        ref = torch.from_numpy(y[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        bad += int(np.sum(ours[inr] != ref))
        sat = ours[~inr]
        want = np.where(y[~inr] > 0, 0x7E, 0xFE).astype(np.uint8)
        bad += int(np.sum(sat != want))
    return bad


# ---------------------------------------------------------------- tests
def test_oracle_matches_torch_sdpa_float64():
    assert pin_sdpa_error() < 1e-12
    assert pin_sdpa_error(seed=9, d=128, Hq=8, Hk=8, lens=(64, 3)) < 1e-12
    assert pin_sdpa_error(seed=10, d=256, Hq=24, Hk=4, lens=(70,)) < 1e-12


def test_oracle_large_logits_stable():
    """q x 30 drives logits far beyond exp's range without max subtraction;
    torch's float64 attention is the reference."""
    q, ks, vs = _random_case(11, S=2, d=64, lens=(50, 9), qmul=30.0)
    got = oracle.decode(q, ks, vs, 1.0)
    assert np.all(np.isfinite(got))
    ref = _sdpa_reference(q, ks, vs, 1.0)
    assert np.max(np.abs(got - ref)) < 1e-9


def test_oracle_closed_forms():
    assert pin_single_row_error() == 0.0
    assert pin_zero_query_error() < 1e-14
    assert pin_dominant_logit_error() == 0.0
    assert pin_gqa_grouping_error() == 0.0


def test_oracle_equal_keys_give_mean():
    q, ks, vs = _random_case(6, S=1, lens=(12,))
    ks[0][:] = ks[0][0:1]  # every key row identical -> uniform softmax
    got = oracle.decode(q, ks, vs, 0.7)
    g = q.shape[1] // ks[0].shape[1]
    want = np.repeat(_bf16_values(vs[0]).mean(axis=0), g, axis=0)
    assert np.max(np.abs(got[0] - want)) < 1e-14


def test_oracle_empty_sequence_gives_zero():
    q, ks, vs = _random_case(7, S=2, lens=(0, 5))
    got = oracle.decode(q, ks, vs, 0.5)
    assert np.all(got[0] == 0.0)
    assert np.max(np.abs(got[1] - _sdpa_reference(q[1:], ks[1:], vs[1:], 0.5)[0])) < 1e-12


def test_oracle_partials_merge_to_full_softmax():
    assert pin_partials_merge_error(16) < 1e-13
    assert pin_partials_merge_error(8) < 1e-13


def test_oracle_partials_single_partition_is_full():
    q, ks, vs = _random_case(8, S=2, lens=(30, 31))
    full = oracle.decode(q, ks, vs, 0.3)
    m, l, o = oracle.decode_partials(q, ks, vs, 0.3, 32, 1)
    assert np.max(np.abs(o[:, :, 0, :] - full)) < 1e-14
    # m is the largest logit; recompute it with an einsum
    qv = _bf16_values(q)
    for s in range(2):
        K = _bf16_values(ks[s])
        g = qv.shape[1] // K.shape[1]
        z = 0.3 * np.einsum("jc,tjc->jt", qv[s], np.repeat(K, g, axis=1))
        assert np.max(np.abs(m[s, :, 0] - z.max(axis=1))) < 1e-13
        assert np.max(np.abs(l[s, :, 0] - np.exp(z - z.max(axis=1, keepdims=True)).sum(1))) < 1e-12


def test_oracle_fp8_attention_matches_sdpa_on_dequantised_values():
    gen = torch.Generator().manual_seed(12)
    S, Hq, Hk, d, T = 2, 8, 2, 64, 37
    q = _bf16_bits(torch.randn(S, Hq, d, generator=gen))
    kc = [np.random.default_rng(s).integers(0, 256, (T, Hk, d)).astype(np.uint8) for s in range(S)]
    vc = [np.random.default_rng(10 + s).integers(0, 256, (T, Hk, d)).astype(np.uint8) for s in range(S)]
    for a in kc + vc:  # no NaN codes
        a[(a & 0x7F) == 0x7F] = 0x7E
    k_scale = np.array([0.01, 0.02])
    v_scale = np.array([0.5, 0.25])
    got = oracle.decode(q, kc, vc, 0.1, k_scale, v_scale)
    qv = torch.from_numpy(_bf16_values(q))
    for s in range(S):
        K = torch.from_numpy(kc[s]).view(torch.float8_e4m3fn).to(torch.float64) * torch.tensor(k_scale)[None, :, None]
        V = torch.from_numpy(vc[s]).view(torch.float8_e4m3fn).to(torch.float64) * torch.tensor(v_scale)[None, :, None]
        Kq = K.permute(1, 0, 2).repeat_interleave(Hq // Hk, dim=0)
        Vq = V.permute(1, 0, 2).repeat_interleave(Hq // Hk, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qv[s].unsqueeze(1), Kq, Vq, scale=0.1)
        assert np.max(np.abs(got[s] - o[:, 0, :].numpy())) < 1e-12


def test_e4m3_decode_exhaustive_vs_torch():
    assert pin_e4m3_decode_mismatches() == 0


def test_e4m3_encode_exhaustive_vs_torch_and_saturation():
    assert pin_e4m3_encode_mismatches() == 0


def test_e4m3_ocp_points():
    gold = json.load(open(os.path.join(GOLD, "ocp_e4m3_points.json")))
    xs = np.array([p["x"] for p in gold["points"]], dtype=np.float32)
    codes = oracle.e4m3_encode(xs)
    assert codes.tolist() == [p["code"] for p in gold["points"]]
    for p in gold["decode_points"]:
        v = oracle.e4m3_decode(np.array([p["code"]], dtype=np.uint8))[0]
        if p["value"] == "nan":
            assert math.isnan(v)
        else:
            assert v == p["value"]


def test_kv_footprint_closed_form():
    gold = json.load(open(os.path.join(GOLD, "kv_footprint.json")))
    b = oracle.kv_bytes(gold["layers"], gold["kv_heads"], gold["head_dim"],
                        gold["tokens"], gold["bytes_per_elem"])
    assert b == gold["bytes"] == 536870912
    assert b == 2 ** 29                      # exactly 0.5 GiB
    assert round(b / 1e9, 2) == 0.54         # the printed "0.54" is in GB


def test_figure_1_2_allocation_example():
    gold = json.load(open(os.path.join(GOLD, "figure_1_2_allocation.json")))
    r = oracle.contiguous_vs_paged(gold["lengths"], gold["max_len"], gold["block_size"])
    assert r["contiguous_reserved"] == gold["contiguous_reserved"]
    assert r["used"] == gold["used"]
    assert r["contiguous_unused"] == gold["contiguous_unused"]
    assert round(100 * r["contiguous_wasted_frac"]) == gold["contiguous_wasted_percent_printed"]
    assert r["paged_reserved"] == gold["paged_reserved"]
    assert r["paged_unused"] == gold["paged_unused"]
    assert r["freed_vs_contiguous"] == gold["freed_vs_contiguous"]


def test_pool_image_roundtrip_and_permutation_invariance():
    """Scatter logical rows into a pool at a random physical placement, walk
    the block table back: the rows come back bit for bit, so any attention
    over them is unchanged by the placement."""
    rng = np.random.default_rng(13)
    B, Hk, d, NB = 4, 2, 8, 40
    lens = [5, 13, 1, 8]
    gen0 = torch.Generator().manual_seed(16)
    rows = [_bf16_bits(torch.randn(T, Hk, d, generator=gen0)) for T in lens]
    outs = []
    for perm_seed in (0, 1):
        perm = list(np.random.default_rng(perm_seed).permutation(NB))
        pool = np.zeros((NB, Hk, B, d), dtype=np.uint16)
        pool_fast = np.zeros_like(pool)
        tables = []
        for T, r in zip(lens, rows):
            nb = -(-T // B)
            table = [perm.pop() for _ in range(nb)]
            tables.append(table)
            slots = [table[t // B] * B + t % B for t in range(T)]
            oracle.scatter_rows(pool, r, slots)
            oracle.scatter_rows_fast(pool_fast, r, slots)
        assert np.array_equal(pool, pool_fast)
        back = [oracle.gather_rows(pool, tb, T) for tb, T in zip(tables, lens)]
        for a, b in zip(back, rows):
            assert np.array_equal(a, b)
        gen = torch.Generator().manual_seed(14)
        q = _bf16_bits(torch.randn(len(lens), 4, d, generator=gen))
        outs.append(oracle.decode(q, back, back, 0.5))
    assert np.array_equal(outs[0], outs[1])


def test_shared_prefix_aliasing_equals_private_copies():
    """Two sequences whose tables point at the same prefix blocks read the
    same rows as two sequences holding private copies; copy_blocks of a
    shared block reproduces it byte for byte."""
    rng = np.random.default_rng(15)
    B, Hk, d = 4, 1, 8
    prefix = rng.integers(0, 65536, (6, Hk, d)).astype(np.uint16)
    tails = [rng.integers(0, 65536, (3, Hk, d)).astype(np.uint16) for _ in range(2)]
    pool = np.zeros((12, Hk, B, d), dtype=np.uint16)
    oracle.scatter_rows(pool, prefix, [0, 1, 2, 3, 4 * B + 0, 4 * B + 1])   # blocks 0, 4
    # sequence a appends in place in block 4; sequence b clones block 4 -> 7
    oracle.copy_blocks(pool, [(4, 7)])
    assert np.array_equal(pool[7], pool[4])
    oracle.scatter_rows(pool, tails[0], [4 * B + 2, 4 * B + 3, 9 * B])
    oracle.scatter_rows(pool, tails[1], [7 * B + 2, 7 * B + 3, 10 * B])
    a = oracle.gather_rows(pool, [0, 4, 9], 9)
    b = oracle.gather_rows(pool, [0, 7, 10], 9)
    assert np.array_equal(a, np.concatenate([prefix, tails[0]]))
    assert np.array_equal(b, np.concatenate([prefix, tails[1]]))


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5])
def test_planted_oracle_mistakes_are_caught(mutation):
    oracle.set_mutation(mutation)
    try:
        caught = [
            pin_sdpa_error() > 1e-12,
            pin_single_row_error() != 0.0,
            pin_zero_query_error() > 1e-14,
            pin_dominant_logit_error() != 0.0,
            pin_gqa_grouping_error() != 0.0,
            pin_e4m3_encode_mismatches(scales=(1.0,)) != 0,
        ]
    finally:
        oracle.set_mutation(0)
    assert any(caught), "planted mistake %d slipped through every pin" % mutation


def test_e4m3_table_encoder_equals_direct_encoder():
    """The per-head lookup form of the encoder is the same function."""
    rng = np.random.default_rng(21)
    bits = rng.integers(0, 65536, (50, 3, 16)).astype(np.uint16)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    bits[~np.isfinite(x)] = 0
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    sc = np.array([0.013, 1.0, 7.5], dtype=np.float32)
    with np.errstate(over="ignore"):
        direct = oracle.e4m3_encode((x / sc[None, :, None]).astype(np.float32))
    assert np.array_equal(oracle.e4m3_encode_bf16(bits, sc), direct)
