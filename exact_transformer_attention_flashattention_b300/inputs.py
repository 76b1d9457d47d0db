"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: only random draws and tensor layouts.
Every draw uses a CPU ``torch.Generator`` so that the same seed gives the same
bf16 values on any machine; callers move the tensors to the device themselves.

Layouts (d contiguous everywhere):
  prefill  q [B, N, Hq, d], k/v [B, N, Hkv, d]                      bf16
  decode   q [B, Hq, d], k/v cache [B, Lmax, Hkv, d], kv_len [B]     bf16 / int32

Values are i.i.d. N(0, 1) drawn in float32 and rounded to bf16 (round to
nearest even), in the order q, k, v.  For ragged decode the per-sequence
lengths are drawn first, uniform on [lo, hi] inclusive.  Cache rows at or
beyond kv_len[b] are filled with NaN, so a kernel that reads a padded row into
its result shows it at once.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "LayerStack",
    "LAYER_WORKLOADS",
    "layer_stack_inputs",
    "prefill_inputs",
    "decode_inputs",
    "prefill_flops",
    "visible_pairs",
    "decode_kv_bytes",
]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, mask and the seed its inputs come from."""

    name: str
    kind: str  # "prefill" or "decode"
    B: int
    Hq: int
    Hkv: int
    N: int  # sequence length (prefill) or cache capacity Lmax (decode)
    d: int
    seed: int
    causal: bool = False
    window: int = -1  # -1: no window; w >= 0: keys with |i - j| <= w
    o_fp32: bool = False
    kv_len_lo: int = 0  # decode: ragged lengths drawn on [lo, hi]; 0 = all full
    kv_len_hi: int = 0
    num_splits: int = 1  # decode: number of sequence chunks per row

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five synthetic workloads (shapes of long-context prefill, local
# sliding-window encoder attention, batched GQA decode and million-token
# decode).  Seeds 0..4 in this order.
WORKLOADS = {
    "tiny_noncausal": Workload("tiny_noncausal", "prefill", B=1, Hq=2, Hkv=2, N=256, d=64,
                               seed=0, o_fp32=True),
    "causal_prefill_4k": Workload("causal_prefill_4k", "prefill", B=4, Hq=16, Hkv=16, N=4096,
                                  d=128, seed=1, causal=True),
    "window_encoder_8k": Workload("window_encoder_8k", "prefill", B=8, Hq=12, Hkv=12, N=8192,
                                  d=64, seed=2, window=128),
    "gqa_decode_batch32": Workload("gqa_decode_batch32", "decode", B=32, Hq=32, Hkv=8, N=8192,
                                   d=128, seed=3, kv_len_lo=1024, kv_len_hi=8192,
                                   num_splits=16),
    "decode_1m": Workload("decode_1m", "decode", B=1, Hq=32, Hkv=8, N=1 << 20, d=128, seed=4,
                          num_splits=2048),
}


@dataclass(frozen=True)
class LayerStack:
    """A stack of L attention layers whose global / local pattern alternates
    (layer l global when l % global_every == 0, local window otherwise)."""

    name: str
    L: int
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    seed: int
    global_every: int = 3
    local_window: int = 64

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# ModernBERT-style encoder stack (12 heads of d=64, an 8192-token context):
# two groups of one global and two local layers.  Seed 5 follows the five
# workloads above.
LAYER_WORKLOADS = {
    "modernbert_alternating_8k": LayerStack("modernbert_alternating_8k", L=6, B=4, Hq=12, Hkv=12,
                                            N=8192, d=64, seed=5),
}


def _randn_bf16(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int):
    """q [B,N,Hq,d], k [B,N,Hkv,d], v [B,N,Hkv,d], bf16 on the CPU."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = _randn_bf16((B, N, Hq, d), g)
    k = _randn_bf16((B, N, Hkv, d), g)
    v = _randn_bf16((B, N, Hkv, d), g)
    return q, k, v


def layer_stack_inputs(L: int, B: int, Hq: int, Hkv: int, N: int, d: int, seed: int):
    """q [L,B,N,Hq,d], k [L,B,N,Hkv,d], v [L,B,N,Hkv,d], bf16 on the CPU (layers stacked)."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = _randn_bf16((L, B, N, Hq, d), g)
    k = _randn_bf16((L, B, N, Hkv, d), g)
    v = _randn_bf16((L, B, N, Hkv, d), g)
    return q, k, v


def decode_inputs(B: int, Hq: int, Hkv: int, Lmax: int, d: int, seed: int,
                  kv_len_lo: int = 0, kv_len_hi: int = 0):
    """q [B,Hq,d], k/v cache [B,Lmax,Hkv,d] (bf16), kv_len int32 [B], on the CPU.

    With kv_len_lo > 0 the lengths are drawn uniform on [kv_len_lo, kv_len_hi]
    before q, k, v; otherwise every sequence fills the cache.  Rows at or beyond
    kv_len[b] hold NaN.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    if kv_len_lo > 0:
        kv_len = torch.randint(kv_len_lo, kv_len_hi + 1, (B,), generator=g, dtype=torch.int64)
        kv_len = kv_len.to(torch.int32)
    else:
        kv_len = torch.full((B,), Lmax, dtype=torch.int32)
    q = _randn_bf16((B, Hq, d), g)
    k = _randn_bf16((B, Lmax, Hkv, d), g)
    v = _randn_bf16((B, Lmax, Hkv, d), g)
    for b in range(B):
        n = int(kv_len[b])
        if n < Lmax:
            k[b, n:] = float("nan")
            v[b, n:] = float("nan")
    return q, k, v, kv_len


def workload_inputs(w: Workload):
    if w.kind == "prefill":
        return prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    return decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.kv_len_lo, w.kv_len_hi)


def visible_pairs(N: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs left unmasked in one N x N head (a counting
    identity used for the algorithmic work of a launch, not attention maths)."""
    total = 0
    for i in range(N):
        lo, hi = 0, N - 1
        if causal:
            hi = i
        if window >= 0:
            lo = max(lo, i - window)
            if not causal:
                hi = min(hi, i + window)
        total += max(0, hi - lo + 1)
    return total


def prefill_flops(B: int, Hq: int, N: int, d: int, causal: bool, window: int) -> float:
    """Algorithmic flops of one prefill launch: 2*d for S = Q K^T and 2*d for
    O = P V per unmasked (query, key) pair."""
    return 4.0 * d * visible_pairs(N, causal, window) * B * Hq


def decode_kv_bytes(kv_len, Hkv: int, d: int) -> float:
    """Algorithmic bytes of one decode launch: every unmasked K and V row of
    every kv head read once (bf16)."""
    return float(sum(int(n) for n in kv_len)) * Hkv * d * 2 * 2
