"""Paged KV-cache decode attention for GB300 (sm_103a).

Python binding of ``libpagedkv.so`` (the C ABI in ``include/pagedkv.h``).
Every call marshals tensors into raw pointers and sizes and calls the
library; all arithmetic runs in the library's CUDA kernels. There is no
fallback: without the built library or a CUDA device the calls raise.

Tensors (caller-owned device memory):
  k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim],
                     torch.bfloat16, or torch.uint8 / torch.float8_e4m3fn
                     holding OCP E4M3 codes
  q, out           : [num_seqs, num_heads, head_dim] torch.bfloat16
  block_tables     : [num_seqs, max_blocks_per_seq] torch.int32
  context_lens     : [num_seqs] torch.int32
  slot_mapping     : [num_tokens] torch.int64 (-1 = skip)
  k_scale, v_scale : [num_kv_heads] torch.float32 (FP8 pools)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_CUDA = -3
PKV_ERR_OUT_OF_BLOCKS = -4
PKV_ERR_NOT_FOUND = -5
PKV_ERR_DEVICE_CHECK = -6
PKV_DTYPE_BF16 = 0
PKV_DTYPE_FP8_E4M3 = 1
PKV_PREEMPT_RECOMPUTE = 0
PKV_PREEMPT_SWAP = 1
PKV_BATCH_ADMISSION = 0
PKV_BATCH_LONGEST_FIRST = 1

DEVERR_NONE = 0
DEVERR_BLOCK_ID = 1
DEVERR_SLOT = 2
DEVERR_WAIT_TIMEOUT = 3
DEVERR_CONTEXT = 4
DEVERR_ORDER = 5


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (%d)" % (what or "pagedkv", status_string(status), status))


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_lib = None

# name -> (restype, argtypes); mirrors include/pagedkv.h
SIGNATURES = {
    "pkv_kv_cache_write": (_I, [_P, _P, _P, _I, _P, _P, CacheDesc, _P, _P, _P]),
    "pkv_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "pkv_split_partition_size": (_I, [_I, _I, _I]),
    "pkv_longest_first_order": (_I, [_P, _I, _P]),
    "pkv_paged_attention_decode": (_I, [_P, _P, _P, _P, CacheDesc, _P, _P, _P, _I, _P, _I, _I,
                                        _I, ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_paged_attention_reduce": (_I, [_P, _P, ctypes.c_size_t, _P, _I, _I, _I, _I, _I, _P]),
    "pkv_paged_attention": (_I, [_P, _P, _P, _P, CacheDesc, _P, _P, _P, _I, _P, _I, _I, _I,
                                 ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, CacheDesc, _P, _P, _P, _I, _P,
                                                _I, _I, _I, ctypes.c_float, _I, _P]),
    "pkv_shared_prefix_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "pkv_shared_prefix_partition_size": (_I, [_I, _I, _I, _I, _I, _I, _I]),
    "pkv_paged_attention_decode_shared_prefix": (_I, [_P, _P, _P, _P, CacheDesc, _P, _P, _P, _I,
                                                      _P, _I,
                                                      _I, _I, ctypes.c_float, _P, _I, _I, _P,
                                                      _I, _I, _P, ctypes.c_size_t, _P, _P]),
    "pkv_copy_blocks": (_I, [_P, _P, CacheDesc, _P, _I, _P]),
    "pkv_swap_out": (_I, [_P, _P, CacheDesc, _P, _I, _P, _P, _P]),
    "pkv_swap_in": (_I, [_P, _P, CacheDesc, _P, _I, _P, _P, _P]),
    "pkv_set_device_check": (_I, [_P]),
    "pkv_selftest_wait_timeout": (_I, [_P, _I, _P]),
    "pkv_status_string": (ctypes.c_char_p, [_I]),
    "pkv_version": (_I, []),
    "pkv_alloc_create": (_I, [_I, _I, ctypes.c_uint64, ctypes.POINTER(_P)]),
    "pkv_alloc_destroy": (None, [_P]),
    "pkv_seq_new": (_I, [_P, ctypes.POINTER(_I)]),
    "pkv_seq_fork": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "pkv_seq_append": (_I, [_P, _I, _I, _P, _P, ctypes.POINTER(_I)]),
    "pkv_seq_free": (_I, [_P, _I]),
    "pkv_seq_block_table": (_I, [_P, _I, _P, _I, ctypes.POINTER(_I)]),
    "pkv_seq_len": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "pkv_block_refcount": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "pkv_alloc_stats": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I),
                             ctypes.POINTER(ctypes.c_longlong)]),
    "pkv_alloc_save": (_I, [_P, _P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
    "pkv_alloc_load": (_I, [_P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "pkv_sched_create": (_I, [_P, _I, _I, ctypes.POINTER(_P)]),
    "pkv_sched_destroy": (None, [_P]),
    "pkv_sched_add_request": (_I, [_P, ctypes.c_int64, _I, _I]),
    "pkv_sched_add_request_n": (_I, [_P, ctypes.c_int64, _I, _I, _I]),
    "pkv_sched_cow_pairs": (_I, [_P, _P, _I, ctypes.POINTER(_I)]),
    "pkv_sched_step": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "pkv_sched_running": (_I, [_P, _P, _P, _P, _I]),
    "pkv_sched_block_tables": (_I, [_P, _P, _I, _I]),
    "pkv_sched_prompt_slots": (_I, [_P, ctypes.c_int64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_sched_events": (_I, [_P, _I, _P, _I, ctypes.POINTER(_I)]),
    "pkv_sched_set_preemption": (_I, [_P, _I]),
    "pkv_sched_set_batch_order": (_I, [_P, _I]),
    "pkv_sched_swap_blocks": (_I, [_P, ctypes.c_int64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_sched_counts": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I),
                              ctypes.POINTER(ctypes.c_longlong)]),
}


def lib() -> ctypes.CDLL:
    """Load libpagedkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libpagedkv.so is not built: run "
                               "`python -m paged_kv_cache_220_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pkv_status_string(int(status)).decode()
    except Exception:  # library missing
        return "status %d" % status


def _check(rc: int, what: str) -> None:
    if rc != PKV_OK:
        raise PagedKVError(rc, what)


def _dev_ptr(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


_FP8_DTYPES = (torch.uint8,) + ((torch.float8_e4m3fn,) if hasattr(torch, "float8_e4m3fn") else ())


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Geometry of a [num_blocks, Hk, B, D] pool tensor."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hk, bs, d = k_cache.shape
    if k_cache.dtype == torch.bfloat16:
        dt = PKV_DTYPE_BF16
    elif k_cache.dtype in _FP8_DTYPES:
        dt = PKV_DTYPE_FP8_E4M3
    else:
        raise ValueError("cache dtype must be bfloat16 or uint8/float8_e4m3fn (E4M3)")
    return CacheDesc(nb, bs, hk, d, dt)


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None,
                   stream=None) -> None:
    """Scatter k, v [T, Hk, D] bf16 into their slots (bit-exact for bf16;
    E4M3 round-to-nearest-even with saturation of x / scale[h] for FP8)."""
    desc = cache_desc(k_cache)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    n = int(slot_mapping.shape[0])
    if k.shape != (n, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim]")
    rc = lib().pkv_kv_cache_write(
        _dev_ptr(k, "k", torch.bfloat16), _dev_ptr(v, "v", torch.bfloat16),
        _dev_ptr(slot_mapping, "slot_mapping", torch.int64), n,
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
        _dev_ptr(k_scale, "k_scale", torch.float32), _dev_ptr(v_scale, "v_scale", torch.float32),
        _stream(stream))
    _check(rc, "kv_cache_write")


def decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context, partition_size) -> int:
    return int(lib().pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context,
                                                partition_size))


def split_partition_size(max_context, block_size, partition_size) -> int:
    """A split size near partition_size without a nearly empty last
    partition (see pkv_split_partition_size)."""
    rc = lib().pkv_split_partition_size(int(max_context), int(block_size), int(partition_size))
    if rc < 0:
        _check(rc, "split_partition_size")
    return int(rc)


def alloc_workspace(num_seqs, num_heads, head_dim, max_context, partition_size,
                    device=None) -> torch.Tensor:
    n = decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context, partition_size)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def longest_first_order(lengths) -> np.ndarray:
    """The indices of `lengths` sorted longest first, ties in index order
    (int32, host): the seq_order that starts the long sequences first."""
    a = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32).reshape(-1))
    order = np.empty(a.shape[0], dtype=np.int32)
    rc = lib().pkv_longest_first_order(a.ctypes.data_as(_P), int(a.shape[0]),
                                       order.ctypes.data_as(_P))
    _check(rc, "longest_first_order")
    return order


def _order_ptr(seq_order, num_seqs):
    if seq_order is None:
        return None
    if tuple(seq_order.shape) != (num_seqs,):
        raise ValueError("seq_order must be [num_seqs]")
    return _dev_ptr(seq_order, "seq_order", torch.int32)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           max_context, partition_size=0, workspace=None, k_scale=None,
                           v_scale=None, stream=None, seq_order=None) -> None:
    """One launch of the decode kernel (see pkv_paged_attention_decode).
    seq_order: None or a device int32 [S] permutation, the order in which the
    CTAs take the sequences (see longest_first_order)."""
    desc = cache_desc(k_cache)
    S, Hq, D = q.shape
    if D != desc.head_dim:
        raise ValueError("q head_dim does not match the cache")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pkv_paged_attention_decode(
        _dev_ptr(out, "out", torch.bfloat16) if partition_size == 0 else None,
        _dev_ptr(q, "q", torch.bfloat16), _dev_ptr(k_cache, "k_cache"),
        _dev_ptr(v_cache, "v_cache"), desc,
        _dev_ptr(k_scale, "k_scale", torch.float32), _dev_ptr(v_scale, "v_scale", torch.float32),
        _dev_ptr(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev_ptr(context_lens, "context_lens", torch.int32), S, Hq, int(max_context),
        float(scale), int(partition_size), _dev_ptr(workspace, "workspace"), ws_bytes,
        _order_ptr(seq_order, S), _stream(stream))
    _check(rc, "paged_attention_decode")


def paged_attention_reduce(out, workspace, context_lens, max_context, partition_size,
                           stream=None) -> None:
    S, Hq, D = out.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pkv_paged_attention_reduce(
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(workspace, "workspace"), ws_bytes,
        _dev_ptr(context_lens, "context_lens", torch.int32), S, Hq, D, int(max_context),
        int(partition_size), _stream(stream))
    _check(rc, "paged_attention_reduce")


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale, max_context,
                    partition_size=0, k_scale=None, v_scale=None, out=None, workspace=None,
                    stream=None, seq_order=None) -> torch.Tensor:
    """Decode attention in one C call: the one-pass decode, or the split
    decode followed by the merge of its partitions. Returns out [S, Hq, D]
    bf16. seq_order as for paged_attention_decode."""
    desc = cache_desc(k_cache)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if partition_size > 0 and workspace is None:
        workspace = alloc_workspace(S, Hq, D, max(int(max_context), 1), partition_size,
                                    device=q.device)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().pkv_paged_attention(
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(q, "q", torch.bfloat16),
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
        _dev_ptr(k_scale, "k_scale", torch.float32), _dev_ptr(v_scale, "v_scale", torch.float32),
        _dev_ptr(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev_ptr(context_lens, "context_lens", torch.int32), S, Hq, int(max_context),
        float(scale), int(partition_size), _dev_ptr(workspace, "workspace"), wsb,
        _order_ptr(seq_order, S), _stream(stream))
    _check(rc, "paged_attention")
    return out


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                   max_context, partition_size, k_scale=None, v_scale=None,
                                   stream=None) -> None:
    """Split decode + merge into `out` with the library's own fixed scratch
    (no workspace, no allocation). For callers that cannot allocate device
    memory; calls that may overlap on the GPU share the scratch and race."""
    desc = cache_desc(k_cache)
    S, Hq, D = q.shape
    rc = lib().pkv_paged_attention_decode_noalloc(
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(q, "q", torch.bfloat16),
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
        _dev_ptr(k_scale, "k_scale", torch.float32), _dev_ptr(v_scale, "v_scale", torch.float32),
        _dev_ptr(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev_ptr(context_lens, "context_lens", torch.int32), S, Hq, int(max_context),
        float(scale), int(partition_size), _stream(stream))
    _check(rc, "paged_attention_decode_noalloc")


def shared_prefix_workspace(num_seqs, num_heads, head_dim, max_own_context, max_prefix_tokens,
                            partition_size, device=None) -> torch.Tensor:
    n = int(lib().pkv_shared_prefix_workspace_bytes(num_seqs, num_heads, head_dim,
                                                    max_own_context, max_prefix_tokens,
                                                    partition_size))
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def shared_prefix_partition_size(num_groups, max_group_members, num_kv_heads, num_heads,
                                 block_size, max_prefix_blocks, partition_size) -> int:
    """Pp, the shared part's partition size on the current device."""
    rc = lib().pkv_shared_prefix_partition_size(int(num_groups), int(max_group_members),
                                                int(num_kv_heads), int(num_heads),
                                                int(block_size), int(max_prefix_blocks),
                                                int(partition_size))
    if rc < 0:
        _check(rc, "shared_prefix_partition_size")
    return int(rc)


def paged_attention_shared_prefix(q, k_cache, v_cache, block_tables, context_lens, scale,
                                  max_own_context, group_start, prefix_blocks, max_prefix_blocks,
                                  partition_size, max_group_members, out=None, workspace=None,
                                  k_scale=None, v_scale=None, stream=None,
                                  seq_order=None) -> torch.Tensor:
    """Decode of groups sharing prompt blocks (see the C header): shared pages
    are read once per group. group_start int32 [G+1], prefix_blocks int32 [S];
    max_own_context bounds context_lens[s] - prefix_blocks[s] * block_size;
    max_group_members bounds the members of a group; seq_order, the order of
    the members' own-block decode (longest own part first pays)."""
    desc = cache_desc(k_cache)
    S, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = shared_prefix_workspace(S, Hq, D, max(int(max_own_context), 1),
                                            int(max_prefix_blocks) * desc.block_size,
                                            partition_size, q.device)
    G = int(group_start.shape[0]) - 1
    rc = lib().pkv_paged_attention_decode_shared_prefix(
        _dev_ptr(out, "out", torch.bfloat16), _dev_ptr(q, "q", torch.bfloat16),
        _dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
        _dev_ptr(k_scale, "k_scale", torch.float32), _dev_ptr(v_scale, "v_scale", torch.float32),
        _dev_ptr(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev_ptr(context_lens, "context_lens", torch.int32), S, Hq, int(max_own_context),
        float(scale), _dev_ptr(group_start, "group_start", torch.int32), G,
        int(max_group_members), _dev_ptr(prefix_blocks, "prefix_blocks", torch.int32),
        int(max_prefix_blocks), int(partition_size), _dev_ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _order_ptr(seq_order, S), _stream(stream))
    _check(rc, "paged_attention_decode_shared_prefix")
    return out


def copy_blocks(k_cache, v_cache, block_pairs, stream=None) -> None:
    """k_cache[dst] = k_cache[src] (same for v) for each row (src, dst) of
    block_pairs [n, 2] int32."""
    desc = cache_desc(k_cache)
    n = int(block_pairs.shape[0]) if block_pairs is not None else 0
    if n == 0:
        return
    rc = lib().pkv_copy_blocks(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
                               _dev_ptr(block_pairs, "block_pairs", torch.int32), n,
                               _stream(stream))
    _check(rc, "copy_blocks")


def _any_ptr(t, name):
    """Pointer of a device tensor or of pinned host memory the device can address."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise ValueError("%s must be a contiguous tensor" % name)
    if not t.is_cuda and not t.is_pinned():
        raise ValueError("%s must be a CUDA tensor or pinned host memory" % name)
    return ctypes.c_void_p(t.data_ptr())


def swap_out(k_cache, v_cache, blocks, k_buf, v_buf, stream=None) -> None:
    """k_buf[i] = k_cache[blocks[i]] (and V); buffers device or pinned host,
    [n, Hk, B, D] like the pool."""
    desc = cache_desc(k_cache)
    n = int(blocks.shape[0])
    if n == 0:
        return
    if blocks.dtype != torch.int32 or k_buf.shape[0] < n or k_buf.shape[1:] != k_cache.shape[1:]:
        raise ValueError("blocks int32 [n]; buffers [>=n, Hk, B, D]")
    rc = lib().pkv_swap_out(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
                            _any_ptr(blocks, "blocks"), n, _any_ptr(k_buf, "k_buf"),
                            _any_ptr(v_buf, "v_buf"), _stream(stream))
    _check(rc, "swap_out")


def swap_in(k_cache, v_cache, blocks, k_buf, v_buf, stream=None) -> None:
    """k_cache[blocks[i]] = k_buf[i] (and V)."""
    desc = cache_desc(k_cache)
    n = int(blocks.shape[0])
    if n == 0:
        return
    if blocks.dtype != torch.int32 or k_buf.shape[0] < n or k_buf.shape[1:] != k_cache.shape[1:]:
        raise ValueError("blocks int32 [n]; buffers [>=n, Hk, B, D]")
    rc = lib().pkv_swap_in(_dev_ptr(k_cache, "k_cache"), _dev_ptr(v_cache, "v_cache"), desc,
                           _any_ptr(blocks, "blocks"), n, _any_ptr(k_buf, "k_buf"),
                           _any_ptr(v_buf, "v_buf"), _stream(stream))
    _check(rc, "swap_in")


def selftest_wait_timeout(flag, limit_us: int = 50000, stream=None) -> None:
    """Run the bounded-wait self-test; `flag` (int32 CUDA tensor) receives
    DEVERR_WAIT_TIMEOUT."""
    _check(lib().pkv_selftest_wait_timeout(_dev_ptr(flag, "flag", torch.int32), int(limit_us),
                                           _stream(stream)), "selftest_wait_timeout")


def set_device_check(flag) -> None:
    """Register a 1-element int32 CUDA tensor as the device error word
    (None switches reporting off). Keep the tensor alive while registered."""
    ptr = None if flag is None else _dev_ptr(flag, "flag", torch.int32)
    lib().pkv_set_device_check(ptr)


class BlockAllocator:
    """Host block allocator (free list, refcounts, fork, copy-on-write)."""

    def __init__(self, num_blocks: int, block_size: int, seed: int = 0):
        h = ctypes.c_void_p()
        _check(lib().pkv_alloc_create(int(num_blocks), int(block_size), int(seed),
                                      ctypes.byref(h)), "alloc_create")
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def save(self) -> bytes:
        """The allocator's complete state as a flat record (pkv_alloc_save)."""
        n = ctypes.c_size_t()
        _check(lib().pkv_alloc_save(self._h, None, 0, ctypes.byref(n)), "alloc_save")
        buf = ctypes.create_string_buffer(n.value)
        _check(lib().pkv_alloc_save(self._h, buf, n, ctypes.byref(n)), "alloc_save")
        return buf.raw[:n.value]

    @classmethod
    def load(cls, record: bytes) -> "BlockAllocator":
        """An allocator restored from a record of save() (pkv_alloc_load)."""
        h = ctypes.c_void_p()
        buf = ctypes.create_string_buffer(bytes(record), len(record))
        _check(lib().pkv_alloc_load(buf, len(record), ctypes.byref(h)), "alloc_load")
        self = cls.__new__(cls)
        self._h = h
        words = np.frombuffer(bytes(record), dtype="<i8")
        self.num_blocks = int(words[2])
        self.block_size = int(words[3])
        return self

    def new_seq(self) -> int:
        sid = ctypes.c_int()
        _check(lib().pkv_seq_new(self._h, ctypes.byref(sid)), "seq_new")
        return sid.value

    def fork(self, parent: int) -> int:
        sid = ctypes.c_int()
        _check(lib().pkv_seq_fork(self._h, int(parent), ctypes.byref(sid)), "seq_fork")
        return sid.value

    def append(self, seq: int, n_tokens: int = 1):
        """Returns (slots int64 [n], cow_pairs int32 [k, 2])."""
        slots = np.empty(max(n_tokens, 1), dtype=np.int64)
        pairs = np.empty((max(n_tokens, 1), 2), dtype=np.int32)
        ncow = ctypes.c_int()
        rc = lib().pkv_seq_append(self._h, int(seq), int(n_tokens),
                                  slots.ctypes.data_as(ctypes.c_void_p),
                                  pairs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(ncow))
        _check(rc, "seq_append")
        return slots[:n_tokens], pairs[:ncow.value]

    def free(self, seq: int) -> None:
        _check(lib().pkv_seq_free(self._h, int(seq)), "seq_free")

    def block_table(self, seq: int) -> np.ndarray:
        n = ctypes.c_int()
        rc = lib().pkv_seq_block_table(self._h, int(seq), None, 0, ctypes.byref(n))
        if rc not in (PKV_OK, PKV_ERR_INVALID_ARG):
            _check(rc, "seq_block_table")
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(lib().pkv_seq_block_table(self._h, int(seq), out.ctypes.data_as(ctypes.c_void_p),
                                         out.size, ctypes.byref(n)), "seq_block_table")
        return out[:n.value]

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int()
        _check(lib().pkv_seq_len(self._h, int(seq), ctypes.byref(n)), "seq_len")
        return n.value

    def refcount(self, block: int) -> int:
        n = ctypes.c_int()
        _check(lib().pkv_block_refcount(self._h, int(block), ctypes.byref(n)), "block_refcount")
        return n.value

    def stats(self):
        f, u, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
        _check(lib().pkv_alloc_stats(self._h, ctypes.byref(f), ctypes.byref(u), ctypes.byref(s)),
               "alloc_stats")
        return {"free_blocks": f.value, "used_blocks": u.value, "used_slots": s.value}

    def block_tables(self, seqs, max_blocks: int) -> np.ndarray:
        """int32 [len(seqs), max_blocks] padded with -1."""
        out = np.full((len(seqs), max_blocks), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = self.block_table(s)
            out[i, :len(t)] = t
        return out


class Scheduler:
    """Iteration-level batching over a BlockAllocator (see pkv_sched_step)."""

    def __init__(self, alloc: "BlockAllocator", max_num_seqs: int):
        h = ctypes.c_void_p()
        _check(lib().pkv_sched_create(alloc._h, alloc.block_size, int(max_num_seqs),
                                      ctypes.byref(h)), "sched_create")
        self._h = h
        self.alloc = alloc  # keeps the allocator alive

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().pkv_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_request(self, request_id: int, prompt_len: int, max_new_tokens: int,
                    n: int = 1) -> None:
        """n > 1: n samples of one prompt, as requests request_id ..
        request_id + n - 1 sharing the prompt's blocks."""
        _check(lib().pkv_sched_add_request_n(self._h, int(request_id), int(prompt_len),
                                             int(max_new_tokens), int(n)), "sched_add_request")

    def cow_pairs(self) -> np.ndarray:
        """Copy-on-write pairs (src, dst) of the last step, int32 [k, 2]; apply
        them with copy_blocks after the admitted prompts' K/V and before this
        iteration's K/V."""
        n = ctypes.c_int()
        rc = lib().pkv_sched_cow_pairs(self._h, None, 0, ctypes.byref(n))
        if rc not in (PKV_OK, PKV_ERR_INVALID_ARG):
            _check(rc, "sched_cow_pairs")
        out = np.empty((max(n.value, 1), 2), np.int32)
        _check(lib().pkv_sched_cow_pairs(self._h, out.ctypes.data_as(ctypes.c_void_p),
                                         out.shape[0], ctypes.byref(n)), "sched_cow_pairs")
        return out[:n.value]

    def step(self):
        """One iteration; returns (num_running, num_admitted, num_finished)."""
        r, a, f = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(lib().pkv_sched_step(self._h, ctypes.byref(r), ctypes.byref(a), ctypes.byref(f)),
               "sched_step")
        return r.value, a.value, f.value

    def running(self):
        """(request_ids int64, context_lens int32, new_slots int64) of the batch."""
        n = self.counts()["running"]
        ids = np.empty(max(n, 1), np.int64)
        cl = np.empty(max(n, 1), np.int32)
        sl = np.empty(max(n, 1), np.int64)
        _check(lib().pkv_sched_running(self._h, ids.ctypes.data_as(ctypes.c_void_p),
                                       cl.ctypes.data_as(ctypes.c_void_p),
                                       sl.ctypes.data_as(ctypes.c_void_p), max(n, 1)),
               "sched_running")
        return ids[:n], cl[:n], sl[:n]

    def block_tables(self, max_blocks: int) -> np.ndarray:
        n = self.counts()["running"]
        t = np.empty((max(n, 1), max_blocks), np.int32)
        _check(lib().pkv_sched_block_tables(self._h, t.ctypes.data_as(ctypes.c_void_p),
                                            int(max_blocks), max(n, 1)), "sched_block_tables")
        return t[:n]

    def prompt_slots(self, request_id: int) -> np.ndarray:
        n = ctypes.c_int()
        rc = lib().pkv_sched_prompt_slots(self._h, int(request_id), None, 0, ctypes.byref(n))
        if rc not in (PKV_OK, PKV_ERR_INVALID_ARG):
            _check(rc, "sched_prompt_slots")
        out = np.empty(max(n.value, 1), np.int64)
        _check(lib().pkv_sched_prompt_slots(self._h, int(request_id),
                                            out.ctypes.data_as(ctypes.c_void_p), out.size,
                                            ctypes.byref(n)), "sched_prompt_slots")
        return out[:n.value]

    def set_batch_order(self, order: int) -> None:
        """Row order of running() / block_tables(): PKV_BATCH_ADMISSION
        (default) or PKV_BATCH_LONGEST_FIRST."""
        _check(lib().pkv_sched_set_batch_order(self._h, int(order)), "sched_set_batch_order")

    def set_preemption(self, mode: int) -> None:
        """PKV_PREEMPT_RECOMPUTE (default) or PKV_PREEMPT_SWAP."""
        _check(lib().pkv_sched_set_preemption(self._h, int(mode)), "sched_set_preemption")

    def swap_blocks(self, request_id: int) -> np.ndarray:
        """Block list of a request swapped out (blocks to save) or in (blocks
        to restore) in the last step, int32, logical order."""
        n = ctypes.c_int()
        rc = lib().pkv_sched_swap_blocks(self._h, int(request_id), None, 0, ctypes.byref(n))
        if rc not in (PKV_OK, PKV_ERR_INVALID_ARG):
            _check(rc, "sched_swap_blocks")
        out = np.empty(max(n.value, 1), np.int32)
        _check(lib().pkv_sched_swap_blocks(self._h, int(request_id),
                                           out.ctypes.data_as(ctypes.c_void_p), out.size,
                                           ctypes.byref(n)), "sched_swap_blocks")
        return out[:n.value]

    def events(self, kind: int) -> np.ndarray:
        """kind 0: admitted, 1: finished, 2: preempted, 3: swapped out,
        4: swapped in (in the last step)."""
        n = ctypes.c_int()
        buf = np.empty(4096, np.int64)
        _check(lib().pkv_sched_events(self._h, int(kind), buf.ctypes.data_as(ctypes.c_void_p),
                                      buf.size, ctypes.byref(n)), "sched_events")
        return buf[:n.value].copy()

    def counts(self):
        w, r, s = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
        _check(lib().pkv_sched_counts(self._h, ctypes.byref(w), ctypes.byref(r), ctypes.byref(s)),
               "sched_counts")
        return {"waiting": w.value, "running": r.value, "steps": s.value}
