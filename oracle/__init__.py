"""CPU oracle for the paged decode path — TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. It shares
no code with the CUDA library; it never sees a block table for attention.

Contents
  decode / decode_partials  fp64 attention on contiguous per-sequence rows
                             (C, oracle.c)
  e4m3_encode / e4m3_decode  OCP FP8 E4M3 by the format's definition (C)
  kv_bytes                   the KV-footprint equation (C)
  scatter_rows / copy_blocks / gather_rows
                             the pool image a cache write, a block copy and a
                             block-table walk must produce: plain index loops
                             written from the block-table definition
  contiguous_vs_paged        the slot accounting of the worked allocation
                             example (three requests, Figures 1 and 2 of
                             "High-Throughput LLM Inference & Training: A Deep
                             Dive into vLLM")
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _SO, _SRC, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P = ctypes.c_void_p
        L.oracle_decode.argtypes = [P, P, P, ctypes.c_int, P, P, P, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_double, P]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode_partials.argtypes = [P, P, P, ctypes.c_int, P, P, P,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_int, P, P, P]
        L.oracle_decode_partials.restype = ctypes.c_int
        L.oracle_e4m3_encode_array.argtypes = [P, P, ctypes.c_int64]
        L.oracle_e4m3_decode_array.argtypes = [P, P, ctypes.c_int64]
        L.oracle_kv_bytes.argtypes = [ctypes.c_longlong] * 5
        L.oracle_kv_bytes.restype = ctypes.c_longlong
        L.oracle_set_mutation.argtypes = [ctypes.c_int]
        L.oracle_get_mutation.restype = ctypes.c_int
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_mutation(k: int) -> None:
    """Plant mistake number k in the oracle (0 = none). Tests only."""
    lib().oracle_set_mutation(int(k))


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def kv_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem) -> int:
    return int(lib().oracle_kv_bytes(layers, kv_heads, head_dim, tokens, bytes_per_elem))


def e4m3_encode(x) -> np.ndarray:
    """float32 array -> uint8 E4M3 codes (nearest, ties to even, saturate)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


_ALL_BF16 = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)


def e4m3_encode_bf16(bits: np.ndarray, scale) -> np.ndarray:
    """E4M3 codes of x / scale[h] (fp32 quotient) for bf16 bit patterns
    bits[..., h, :]. The encoder is a pure function of the bf16 input and the
    head's scale, so it is evaluated once on all 65,536 bf16 patterns per
    head and looked up."""
    bits = np.asarray(bits, dtype=np.uint16)
    scale = np.asarray(scale, dtype=np.float32)
    out = np.empty(bits.shape, dtype=np.uint8)
    for h in range(bits.shape[-2]):
        with np.errstate(over="ignore", invalid="ignore"):
            y = (_ALL_BF16 / np.float32(scale[h])).astype(np.float32)
        lut = e4m3_encode(y)
        out[..., h, :] = lut[bits[..., h, :]]
    return out


def e4m3_decode(codes) -> np.ndarray:
    """uint8 E4M3 codes -> float64 values."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def _rows_arg(rows, kind):
    """List of per-sequence [T, Hk, d] arrays -> (concatenated, row_off)."""
    dt = np.uint16 if kind == 0 else np.uint8
    lens = [int(r.shape[0]) for r in rows]
    off = np.zeros(len(rows) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    if rows and off[-1] > 0:
        cat = np.ascontiguousarray(np.concatenate([np.asarray(r, dtype=dt) for r in rows]))
    else:
        cat = np.zeros(1, dtype=dt)
    return cat, off


def decode(q_bits, k_rows, v_rows, scale, k_scale=None, v_scale=None) -> np.ndarray:
    """fp64 decode attention.

    q_bits : uint16 bf16 bit patterns [S, Hq, d]
    k_rows, v_rows : per-sequence arrays [T_s, Hk, d] of bf16 bits (uint16) or,
        with k_scale/v_scale given, E4M3 codes (uint8)
    scale  : logit scale; k_scale, v_scale : per-KV-head dequantisation scales
    returns float64 [S, Hq, d]
    """
    q = np.ascontiguousarray(np.asarray(q_bits, dtype=np.uint16))
    S, Hq, d = q.shape
    kind = 0 if k_scale is None else 1
    Hk = int(k_rows[0].shape[1]) if len(k_rows) else 1
    kc, off = _rows_arg(k_rows, kind)
    vc, off2 = _rows_arg(v_rows, kind)
    assert np.array_equal(off, off2) and len(k_rows) == S
    ks = vs = None
    if kind == 1:
        ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float64))
        vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float64))
    out = np.zeros((S, Hq, d), dtype=np.float64)
    rc = lib().oracle_decode(_ptr(q), _ptr(kc), _ptr(vc), kind, _ptr(off),
                             _ptr(ks) if ks is not None else None,
                             _ptr(vs) if vs is not None else None,
                             S, Hq, Hk, d, float(scale), _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_decode failed: %d" % rc)
    return out


def decode_partials(q_bits, k_rows, v_rows, scale, partition_size, np_max,
                    k_scale=None, v_scale=None):
    """Per-partition (max logit, exp-sum, normalised output) in fp64.
    Returns m [S,Hq,NP], l [S,Hq,NP], o [S,Hq,NP,d]; unused entries are NaN."""
    q = np.ascontiguousarray(np.asarray(q_bits, dtype=np.uint16))
    S, Hq, d = q.shape
    kind = 0 if k_scale is None else 1
    Hk = int(k_rows[0].shape[1])
    kc, off = _rows_arg(k_rows, kind)
    vc, _ = _rows_arg(v_rows, kind)
    ks = vs = None
    if kind == 1:
        ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float64))
        vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float64))
    m = np.full((S, Hq, np_max), np.nan)
    l = np.full((S, Hq, np_max), np.nan)
    o = np.full((S, Hq, np_max, d), np.nan)
    rc = lib().oracle_decode_partials(_ptr(q), _ptr(kc), _ptr(vc), kind, _ptr(off),
                                      _ptr(ks) if ks is not None else None,
                                      _ptr(vs) if vs is not None else None,
                                      S, Hq, Hk, d, float(scale), int(partition_size),
                                      int(np_max), _ptr(m), _ptr(l), _ptr(o))
    if rc != 0:
        raise RuntimeError("oracle_decode_partials failed: %d" % rc)
    return m, l, o


# ---------------------------------------------------------------------------
# Pool images. Block-table definition ("PagedAttention borrows from operating
# systems" in "How vLLM gets real throughput on H100s ..."; "PagedAttention:
# Virtual Memory for KV Cache" in "Dissecting vLLM ..."): logical token t of a
# sequence lives in physical block table[t // B] at offset t % B. The pool is
# [num_blocks, Hk, B, d]; a slot is block * B + offset.
# ---------------------------------------------------------------------------

def scatter_rows(pool: np.ndarray, rows: np.ndarray, slots) -> None:
    """pool[slot // B, h, slot % B, :] = rows[i, h, :] for every slot >= 0."""
    B = pool.shape[2]
    for i, slot in enumerate(slots):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // B, slot % B
        for h in range(pool.shape[1]):
            pool[blk, h, off, :] = rows[i, h, :]


def scatter_rows_fast(pool: np.ndarray, rows: np.ndarray, slots) -> None:
    """Same assignment as scatter_rows, written with fancy indexing for large
    pools (pinned to scatter_rows by the tests)."""
    slots = np.asarray(slots, dtype=np.int64)
    keep = slots >= 0
    B = pool.shape[2]
    blk, off = slots[keep] // B, slots[keep] % B
    pool[blk, :, off, :] = rows[keep]


def gather_rows(pool: np.ndarray, table, length: int) -> np.ndarray:
    """Logical rows [length, Hk, d] of a sequence with block table `table`."""
    B = pool.shape[2]
    out = np.empty((length, pool.shape[1], pool.shape[3]), dtype=pool.dtype)
    for t in range(length):
        out[t] = pool[int(table[t // B]), :, t % B, :]
    return out


def copy_blocks(pool: np.ndarray, pairs) -> None:
    """pool[dst] = pool[src] for each (src, dst), whole block, in order."""
    for src, dst in pairs:
        pool[int(dst)] = pool[int(src)]


def contiguous_vs_paged(lengths, max_len, block_size):
    """Slot accounting of the worked example: every request reserving
    max_len contiguous slots versus ceil(len/B) blocks of B slots."""
    used = int(sum(lengths))
    contiguous = len(lengths) * int(max_len)
    paged = int(sum(-(-int(n) // block_size) * block_size for n in lengths))
    return {
        "contiguous_reserved": contiguous,
        "contiguous_unused": contiguous - used,
        "contiguous_wasted_frac": (contiguous - used) / contiguous,
        "paged_reserved": paged,
        "paged_unused": paged - used,
        "freed_vs_contiguous": contiguous - paged,
        "used": used,
    }
