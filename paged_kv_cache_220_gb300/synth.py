"""Seeded synthetic inputs for the paged decode path.

This module is the only thing the CUDA path and the CPU oracle share. It holds
none of the attention arithmetic: it turns (seed, tensor, layer, sequence,
element index) into a bf16 number that is distributed like N(0, 1), and it
describes the workload shapes.

Generator. Every element has a 64-bit counter ``key + index``; the counter is
mixed with the SplitMix64 output function (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014: add the golden gamma
0x9E3779B97F4A7C15, then xor-shift-multiply by 0xBF58476D1CE4E5B9 and
0x94D049BB133111EB, shifts 30/27/31). The top 16 bits of the result index a
table of the 65,536 standard-normal quantiles at (i + 1/2) / 65536, rounded to
bf16 (round to nearest even). Only integer operations and a table lookup are
involved, so the same element comes out bit-identical on the host and on the
GPU, whichever side generates it.

Workloads. The five shapes the decode path is measured and checked on; every
shape's numbers are repeated in the test and benchmark output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB

# tensor kinds inside one stream key
KIND_Q = 1
KIND_K = 2
KIND_V = 3
KIND_LEN = 4


def mix64_int(x: int) -> int:
    """SplitMix64 output function on a Python int (exact, unsigned)."""
    z = (x + _GAMMA) & _M64
    z = ((z ^ (z >> 30)) * _C1) & _M64
    z = ((z ^ (z >> 27)) * _C2) & _M64
    return z ^ (z >> 31)


def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _lsr(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def mix64_tensor(x: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function on int64 tensors (two's-complement wrap)."""
    z = x + _signed(_GAMMA)
    z = (z ^ _lsr(z, 30)) * _signed(_C1)
    z = (z ^ _lsr(z, 27)) * _signed(_C2)
    return z ^ _lsr(z, 31)


def stream_key(seed: int, kind: int, layer: int, ident: int) -> int:
    """64-bit key of one tensor stream; elements use key + index."""
    assert 0 <= seed < (1 << 23) and 0 <= kind < 256 and 0 <= layer < 4096
    assert 0 <= ident < (1 << 20)
    packed = (seed << 40) | (kind << 32) | (layer << 20) | ident
    return mix64_int(mix64_int(packed)) & ((1 << 62) - 1)


_TABLES = {}


def normal_table(device="cpu") -> torch.Tensor:
    """bf16 [65536]: N(0,1) quantiles at (i + 1/2)/65536, rounded to bf16."""
    dev = torch.device(device)
    key = (dev.type, dev.index)
    if key not in _TABLES:
        p = (torch.arange(65536, dtype=torch.float64) + 0.5) / 65536.0
        tab = torch.special.ndtri(p).to(torch.bfloat16)
        _TABLES[key] = tab.to(dev)
    return _TABLES[key]


def mix64_inplace_(z: torch.Tensor) -> torch.Tensor:
    """mix64_tensor without the gamma step, computed in place on z (one
    scratch tensor instead of a temporary per operation; used for the large
    host-side streams of the parity tests)."""
    t = torch.empty_like(z)
    for sh, c in ((30, _C1), (27, _C2)):
        torch.bitwise_right_shift(z, sh, out=t)
        t.bitwise_and_((1 << (64 - sh)) - 1)
        z.bitwise_xor_(t)
        z.mul_(_signed(c))
    torch.bitwise_right_shift(z, 31, out=t)
    t.bitwise_and_((1 << 33) - 1)
    return z.bitwise_xor_(t)


def normal_bf16(key: int, n: int, offset: int = 0, device="cpu") -> torch.Tensor:
    """n bf16 values of stream `key`, elements offset .. offset+n-1."""
    # counter + gamma: key < 2^62 and the signed gamma is negative, so the
    # sum stays inside int64 without wrapping
    z = torch.arange(n, dtype=torch.int64, device=device)
    z.add_(key + offset + _signed(_GAMMA))
    mix64_inplace_(z)
    z.bitwise_right_shift_(48)
    z.bitwise_and_(0xFFFF)
    return normal_table(device)[z]


def uniform01(key: int, i: int) -> float:
    """One uniform double in [0, 1) from stream `key`, element i (host only)."""
    return (mix64_int(key + i) >> 11) * (1.0 / (1 << 53))


@dataclass
class Workload:
    """One decode workload: shapes, lengths and seeds.

    ctx[s] counts the cached tokens sequence s attends to, the token written
    this step included (it sits at logical position ctx[s] - 1).
    prefix_len / group: when > 0, sequences s = p*group + r share logical rows
    [0, prefix_len) with the other rollouts of prompt p (a shared prefix).
    """
    name: str
    seed: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    ctx: List[int]
    layers: int = 1
    fp8: bool = False
    partition_size: int = 0
    num_blocks: Optional[int] = None      # pool size; None = exact fit + slack
    slack_blocks: int = 0
    prefix_len: int = 0
    group: int = 1
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.ctx)

    @property
    def scale(self) -> float:
        """Logit scale 1/sqrt(head_dim) as the fp32 number both sides get."""
        return float(torch.tensor(1.0 / math.sqrt(self.head_dim), dtype=torch.float32))

    @property
    def max_context(self) -> int:
        return max(self.ctx) if self.ctx else 0

    # ---- element streams -------------------------------------------------
    def q(self, layer: int, device="cpu") -> torch.Tensor:
        """bf16 [S, Hq, d]."""
        S, Hq, d = self.num_seqs, self.num_heads, self.head_dim
        key = stream_key(self.seed, KIND_Q, layer, 0)
        return normal_bf16(key, S * Hq * d, 0, device).view(S, Hq, d)

    def rows(self, kind: int, layer: int, seq: int, t0: int, t1: int,
             device="cpu") -> torch.Tensor:
        """Logical K (kind=KIND_K) or V rows [t0, t1) of sequence `seq`,
        bf16 [t1 - t0, Hk, d]. Shared-prefix rows come from the prompt's
        stream, the rest from the sequence's own stream."""
        Hk, d = self.num_kv_heads, self.head_dim
        per = Hk * d
        parts = []
        if self.prefix_len > 0:
            p = seq // self.group
            a, b = t0, min(t1, self.prefix_len)
            if a < b:
                key = stream_key(self.seed, kind, layer, p)
                parts.append(normal_bf16(key, (b - a) * per, a * per, device))
            a, b = max(t0, self.prefix_len), t1
            if a < b:
                key = stream_key(self.seed, kind, layer, (1 << 19) + seq)
                parts.append(normal_bf16(key, (b - a) * per,
                                         (a - self.prefix_len) * per, device))
        else:
            key = stream_key(self.seed, kind, layer, seq)
            parts.append(normal_bf16(key, (t1 - t0) * per, t0 * per, device))
        if not parts:
            return torch.empty(0, Hk, d, dtype=torch.bfloat16, device=device)
        return torch.cat(parts).view(t1 - t0, Hk, d)

    def pool_blocks(self) -> int:
        if self.num_blocks is not None:
            return self.num_blocks
        B = self.block_size
        if self.prefix_len > 0:
            n_prompt = len(self.ctx) // self.group
            shared = n_prompt * ((self.prefix_len + B - 1) // B)
            own = sum((c - self.prefix_len) // B + 2 for c in self.ctx)
            return shared + own + self.slack_blocks
        return sum((c + B - 1) // B for c in self.ctx) + self.slack_blocks


def _loguniform_lengths(seed: int, n: int, lo: int, hi: int) -> List[int]:
    key = stream_key(seed, KIND_LEN, 0, 0)
    out = []
    for i in range(n):
        u = uniform01(key, i)
        c = int(math.floor(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
        out.append(min(max(c, lo), hi))
    return out


def _uniform_ints(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """n integers uniform in [lo, hi] (inclusive)."""
    key = stream_key(seed, KIND_LEN, 0, 1)
    return [lo + int(uniform01(key, i) * (hi - lo + 1)) for i in range(n)]


def tiny(seed: int = 1001) -> Workload:
    """Four sequences of 50/120/240/1024 tokens, 8 query / 2 KV heads, d=128,
    B=16, a 128-block pool with seeded random placement."""
    return Workload("tiny_paged_decode", seed, 8, 2, 128, 16, [50, 120, 240, 1024],
                    num_blocks=128)


def qwen_like(seed: int = 1002, layers: int = 16, num_seqs: int = 64,
              ctx: int = 8192, partition_size: int = 1024) -> Workload:
    """16 layers back to back, 64 sequences at 8192 tokens, 24 query / 4 KV
    heads, d=256, B=16, pool exactly fits (0.5 GiB of KV per sequence).
    Split decode in 1024-token partitions (2048 CTAs per layer)."""
    return Workload("qwen_like_gqa_decode", seed, 24, 4, 256, 16, [ctx] * num_seqs,
                    layers=layers, partition_size=partition_size)


def mixed(seed: int = 1003, num_seqs: int = 256) -> Workload:
    """256 sequences, lengths log-uniform in [16, 16384], 24/4 heads, d=256,
    B=32, free list in seeded random order, 256 slack blocks. Split decode in
    1536-token partitions with the sequences taken longest first (GB300, one
    box, step: 768 / 1024 / 1536 / 1664 tokens -> 0.3195 / 0.3160 / 0.3138 /
    0.3133 ms; 1280 and 1408 tokens 0.335 ms, 2048 0.339 ms; 1536 in batch
    order 0.3465 ms)."""
    ctx = _loguniform_lengths(seed, num_seqs, 16, 16384)
    return Workload("mixed_lengths_continuous_batching", seed, 24, 4, 256, 32, ctx,
                    slack_blocks=256, partition_size=1536)


def cow(seed: int = 1004, prompt_len: int = 2048, prompts: int = 32,
        rollouts: int = 16) -> Workload:
    """32 prompts x 16 rollouts sharing the prompt's blocks; completion
    lengths uniform in [0, 1024]; 24/4 heads, d=256, B=16. A prompt of 2048
    tokens fills its last block (no copy on divergence); 2040 leaves it half
    full so every diverging rollout but the last clones it. Split size 1024:
    with the shared-prefix decode each rollout's own part (at most 1033
    tokens) is one partition (GB300, own parts longest first: 0.2095 ms per
    step against 0.2140 in two 528-token partitions; over an E4M3 cache the
    two partitions win, 0.1540 against 0.1555 ms)."""
    comp = _uniform_ints(seed, prompts * rollouts, 0, 1024)
    ctx = [prompt_len + c + 1 for c in comp]
    name = "cow_shared_prefix_%d" % prompt_len
    return Workload(name, seed, 24, 4, 256, 16, ctx, prefix_len=prompt_len,
                    group=rollouts, slack_blocks=64, partition_size=1024,
                    extra={"completion": comp})


def long_fp8(seed: int = 1005, num_seqs: int = 8, ctx: int = 131072) -> Workload:
    """8 sequences at 131072 tokens, FP8-E4M3 K/V with per-head fp32 scales,
    24/4 heads, d=256, B=32, 512-token partitions merged by the reduce."""
    return Workload("long_context_fp8_splitk", seed, 24, 4, 256, 32, [ctx] * num_seqs,
                    fp8=True, partition_size=512)


ALL = {"tiny": tiny, "qwen_like": qwen_like, "mixed": mixed, "cow": cow,
       "long_fp8": long_fp8}


# ---- request streams (continuous batching): a request's K/V row at position
# t and its query at position t are fixed by (seed, layer, request id, t), so
# any iteration can be regenerated on the host.
def request_rows(seed: int, kind: int, layer: int, request_id: int, t0: int, t1: int,
                 num_kv_heads: int, head_dim: int, device="cpu") -> torch.Tensor:
    per = num_kv_heads * head_dim
    key = stream_key(seed, kind, layer, (1 << 18) + request_id)
    return normal_bf16(key, (t1 - t0) * per, t0 * per, device).view(t1 - t0, num_kv_heads,
                                                                    head_dim)


def request_query(seed: int, layer: int, request_id: int, pos: int, num_heads: int,
                  head_dim: int, device="cpu") -> torch.Tensor:
    per = num_heads * head_dim
    key = stream_key(seed, KIND_Q, layer, (1 << 18) + request_id)
    return normal_bf16(key, per, pos * per, device).view(num_heads, head_dim)


def request_mix(seed: int, n: int, prompt_lo: int = 16, prompt_hi: int = 4096,
                gen_lo: int = 8, gen_hi: int = 512):
    """n requests (id, prompt length log-uniform, token budget log-uniform)."""
    p = _loguniform_lengths(seed, n, prompt_lo, prompt_hi)
    g = _loguniform_lengths(seed + 1, n, gen_lo, gen_hi)
    return [(i, p[i], g[i]) for i in range(n)]
