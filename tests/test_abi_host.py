"""The C-ABI library loads without a GPU, exports every function the header
declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_cache_220_gb300 as pkv
from paged_kv_cache_220_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pkv.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pkv.SIGNATURES), set(names) ^ set(pkv.SIGNATURES)


def test_device_error_codes_match_the_header():
    src = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    codes = dict(re.findall(r"#define PKV_(DEVERR_[A-Z_]+)\s+(\d+)", src))
    assert len(codes) >= 6
    for name, value in codes.items():
        assert getattr(pkv, name) == int(value), name


def test_version_and_status_strings(lib):
    assert lib.pkv_version() >= 100
    for code in range(-6, 1):
        assert pkv.status_string(code) not in ("", "unknown status")
    assert pkv.status_string(-99) == "unknown status"


def _desc(nb=8, bs=16, hk=2, d=128, dt=0):
    return pkv.CacheDesc(nb, bs, hk, d, dt)


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first


def test_cache_write_validation(lib):
    f = lib.pkv_kv_cache_write
    assert f(FAKE, FAKE, FAKE, 0, FAKE, FAKE, _desc(), None, None, None) == pkv.PKV_OK
    assert f(FAKE, FAKE, FAKE, -1, FAKE, FAKE, _desc(), None, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(None, FAKE, FAKE, 4, FAKE, FAKE, _desc(), None, None, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, _desc(bs=8), None, None, None) == pkv.PKV_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, _desc(d=64), None, None, None) == pkv.PKV_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, _desc(dt=1), None, None, None) == pkv.PKV_ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x10008)
    assert f(odd, FAKE, FAKE, 4, FAKE, FAKE, _desc(), None, None, None) == pkv.PKV_ERR_INVALID_ARG


def test_decode_validation(lib):
    f = lib.pkv_paged_attention_decode
    args = lambda **kw: [kw.get("out", FAKE), FAKE, FAKE, FAKE, kw.get("desc", _desc()), None, None,
                         FAKE, kw.get("mb", 64), FAKE, kw.get("S", 4), kw.get("Hq", 8),
                         kw.get("maxc", 1024), kw.get("scale", 0.088), kw.get("P", 0),
                         kw.get("ws", None), kw.get("wsb", 0), None, None]
    assert f(*args(S=0)) == pkv.PKV_OK
    assert f(*args(Hq=7)) == pkv.PKV_ERR_INVALID_ARG           # not a multiple of Hk
    assert f(*args(Hq=18)) == pkv.PKV_ERR_UNSUPPORTED          # group 9
    assert f(*args(maxc=1025)) == pkv.PKV_ERR_INVALID_ARG      # beyond the table
    assert f(*args(P=24)) == pkv.PKV_ERR_INVALID_ARG           # not a multiple of B
    assert f(*args(P=512)) == pkv.PKV_ERR_INVALID_ARG          # no workspace
    assert f(*args(P=512, ws=FAKE, wsb=16)) == pkv.PKV_ERR_INVALID_ARG  # too small
    assert f(*args(out=None)) == pkv.PKV_ERR_INVALID_ARG
    assert f(*args(scale=float("nan"))) == pkv.PKV_ERR_INVALID_ARG
    assert f(*args(desc=_desc(dt=1))) == pkv.PKV_ERR_INVALID_ARG  # fp8 without scales


def test_one_call_and_shared_prefix_validation(lib):
    """pkv_paged_attention returns the decode's error without launching the
    merge; the shared-prefix call checks its own-part bound and groups."""
    f = lib.pkv_paged_attention
    args = lambda **kw: [FAKE, FAKE, FAKE, FAKE, _desc(), None, None, FAKE, 64, FAKE,
                         kw.get("S", 4), 8, kw.get("maxc", 1024), 0.088, kw.get("P", 512),
                         kw.get("ws", None), kw.get("wsb", 0), None, None]
    assert f(*args(S=0)) == pkv.PKV_OK
    assert f(*args()) == pkv.PKV_ERR_INVALID_ARG                 # no workspace
    assert f(*args(P=24)) == pkv.PKV_ERR_INVALID_ARG             # not a multiple of B
    assert f(*args(maxc=1025)) == pkv.PKV_ERR_INVALID_ARG        # beyond the table
    g = lib.pkv_paged_attention_decode_shared_prefix
    sp = lambda **kw: [FAKE, FAKE, FAKE, FAKE, kw.get("desc", _desc()), kw.get("ks", None),
                       kw.get("vs", None), FAKE, 64, FAKE, kw.get("S", 4), 8,
                       kw.get("own", 100), 0.088, FAKE, kw.get("G", 1), kw.get("mm", 4), FAKE,
                       kw.get("mp", 2), kw.get("P", 64), kw.get("ws", None), 0, None, None]
    assert g(*sp(S=0)) == pkv.PKV_OK
    assert g(*sp(desc=_desc(dt=1))) == pkv.PKV_ERR_INVALID_ARG      # E4M3 without scales
    assert g(*sp(mm=0)) == pkv.PKV_ERR_INVALID_ARG               # groups need a member bound
    assert g(*sp(mm=5)) == pkv.PKV_ERR_INVALID_ARG               # more members than sequences
    assert g(*sp(own=64 * 16 + 1)) == pkv.PKV_ERR_INVALID_ARG    # own part beyond the table
    assert g(*sp(mp=65)) == pkv.PKV_ERR_INVALID_ARG              # prefix beyond the table
    assert g(*sp(P=24)) == pkv.PKV_ERR_INVALID_ARG
    assert g(*sp()) == pkv.PKV_ERR_INVALID_ARG                   # no workspace
    assert g(*sp(own=-1)) == pkv.PKV_ERR_INVALID_ARG
    n_own = lib.pkv_shared_prefix_workspace_bytes(4, 8, 128, 100, 32, 64)
    n_all = lib.pkv_shared_prefix_workspace_bytes(4, 8, 128, 1000, 32, 64)
    assert n_own == 4 * 8 * (1 + 2) * (128 + 2) * 4 and n_all > n_own
    q = lib.pkv_shared_prefix_partition_size
    assert q(1, 0, 2, 8, 16, 4, 64) == pkv.PKV_ERR_INVALID_ARG    # no member bound
    assert q(1, 4, 2, 8, 16, 4, 24) == pkv.PKV_ERR_INVALID_ARG    # P not a multiple of B
    assert q(1, 4, 2, 18, 16, 4, 64) == pkv.PKV_ERR_UNSUPPORTED   # group 9


def test_longest_first_order(lib):
    """Indices sorted by length, longest first, equal lengths in index order
    (stable): checked against a brute-force stable sort and a hand case."""
    assert pkv.longest_first_order([3, 9, 1, 9, 5]).tolist() == [1, 3, 4, 0, 2]
    assert pkv.longest_first_order([]).tolist() == []
    rng = np.random.default_rng(5)
    for n in (1, 2, 17, 512):
        lens = rng.integers(0, 8, size=n)            # many ties
        got = pkv.longest_first_order(lens)
        want = sorted(range(n), key=lambda i: (-int(lens[i]), i))
        assert got.dtype == np.int32 and got.tolist() == want
    f = lib.pkv_longest_first_order
    assert f(None, 0, None) == pkv.PKV_OK
    assert f(None, 3, None) == pkv.PKV_ERR_INVALID_ARG
    assert f(None, -1, None) == pkv.PKV_ERR_INVALID_ARG


def test_scheduler_pair_export_validation(lib):
    a = pkv.BlockAllocator(16, 4, seed=1)
    s = pkv.Scheduler(a, 4)
    s.add_request(0, 6, 3, n=3)                # 6 tokens: the last prompt block half full
    s.step()
    n = ctypes.c_int()
    assert lib.pkv_sched_cow_pairs(s._h, None, 0, ctypes.byref(n)) == pkv.PKV_ERR_INVALID_ARG
    assert n.value == 2                         # two samples copy, the last writes in place
    pairs = s.cow_pairs()
    assert pairs.shape == (2, 2) and len(set(pairs[:, 0].tolist())) == 1
    assert lib.pkv_sched_cow_pairs(None, None, 0, ctypes.byref(n)) == pkv.PKV_ERR_INVALID_ARG


def test_workspace_size(lib):
    # [S][Hq][NP] partial outputs of D floats plus max and sum
    n = pkv.decode_workspace_bytes(8, 24, 256, 131072, 512)
    assert n == 8 * 24 * 256 * (256 + 2) * 4
    assert pkv.decode_workspace_bytes(8, 24, 256, 131072, 0) == 0


def test_reduce_and_copy_validation(lib):
    r = lib.pkv_paged_attention_reduce
    assert r(FAKE, None, 0, FAKE, 4, 8, 128, 100, 0, None) == pkv.PKV_ERR_INVALID_ARG
    assert r(FAKE, None, 0, FAKE, 4, 8, 96, 100, 64, None) == pkv.PKV_ERR_UNSUPPORTED
    assert r(FAKE, None, 0, FAKE, 4, 8, 128, 100, 64, None) == pkv.PKV_ERR_INVALID_ARG
    c = lib.pkv_copy_blocks
    assert c(FAKE, FAKE, _desc(), FAKE, 0, None) == pkv.PKV_OK
    assert c(FAKE, FAKE, _desc(), None, 3, None) == pkv.PKV_ERR_INVALID_ARG
    assert c(FAKE, FAKE, _desc(), FAKE, -1, None) == pkv.PKV_ERR_INVALID_ARG


def test_binding_fails_loudly_without_cuda_tensors(lib):
    import torch
    k = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    cache = torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.kv_cache_write(k, k, torch.zeros(4, dtype=torch.int64), cache, cache)


def test_split_partition_size(lib):
    """Covers the longest context in round(max/P) partitions of equal
    length (a multiple of B); unchanged when P divides the longest context."""
    f = pkv.split_partition_size
    assert f(1033, 16, 512) == 528            # 2 partitions instead of 512 + 512 + 9
    assert f(8192, 16, 1024) == 1024
    assert f(131072, 32, 512) == 512
    assert f(16384, 32, 512) == 512
    assert f(100, 16, 512) == 112             # one partition
    assert f(0, 16, 512) == 512
    assert lib.pkv_split_partition_size(100, 16, 24) == pkv.PKV_ERR_INVALID_ARG
    import random
    rng = random.Random(3)
    for _ in range(2000):
        B = rng.choice([16, 32])
        P = B * rng.randint(1, 128)
        m = rng.randint(1, 200000)
        Q = f(m, B, P)
        n = max(1, (2 * m + P) // (2 * P))
        assert Q % B == 0 and Q >= B
        assert -(-m // Q) <= n                 # at most n partitions
        assert Q < m / n + B                   # the smallest such multiple of B
