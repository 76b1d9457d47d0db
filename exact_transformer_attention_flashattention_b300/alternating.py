"""Alternating global / local attention over a stack of layers, run as a
two-call workload per group of layers.

Source: the Arabic thread on extending context length (web3.ouzhyi.biz),
ModernBERT paragraph: full global attention in every third layer and local
attention over a 128-token window in the others, which lets the model take
far longer sequences.  Layer l is global when l % global_every == 0.  The
128-token window is read as 64 tokens on each side of the query (keys with
|i - j| <= 64), the symmetric window that spans 128 neighbours.

Layers are stacked in one tensor, q/k/v [L, B, N, H, d], so the local layers
of a group (adjacent in memory) form one [n_local * B, N, H, d] view and run
as a single call: each group costs exactly two launches, one global and one
local.  Every step of the computation runs in the library's prefill kernel;
this module only slices views and calls the C ABI through the binding.
"""

from __future__ import annotations

import torch

from . import binding

MODERNBERT_GLOBAL_EVERY = 3
MODERNBERT_LOCAL_WINDOW = 64  # keys with |i - j| <= 64: a 128-token neighbourhood


def layer_groups(L: int, global_every: int = MODERNBERT_GLOBAL_EVERY):
    """[(global layer, first local layer, end of the group's local layers)] for L layers."""
    if global_every < 1:
        raise ValueError("global_every must be >= 1")
    return [(g, g + 1, min(g + global_every, L)) for g in range(0, L, global_every)]


def alternating_attention(q, k, v, global_every: int = MODERNBERT_GLOBAL_EVERY,
                          local_window: int = MODERNBERT_LOCAL_WINDOW, scale: float | None = None,
                          out=None, lse=None, out_dtype=torch.bfloat16, stream=None):
    """q [L, B, N, Hq, d], k/v [L, B, N, Hkv, d] bf16 (contiguous) ->
    (O [L, B, N, Hq, d], LSE [L, B, Hq, N]); global layers attend to every key,
    local layers to keys within ``local_window`` on either side (non-causal)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dim() != 5 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 5-d tensor [L, B, N, H, d]")
    L, B, N, Hq, d = q.shape
    Hkv = k.shape[3]
    if out is None:
        out = torch.empty((L, B, N, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((L, B, Hq, N), dtype=torch.float32, device=q.device)

    def stack(t, a, e):  # layers [a, e) as one batch of (e - a) * B sequences
        return t[a:e].view((e - a) * B, *t.shape[2:])

    for g, a, e in layer_groups(L, global_every):
        binding.attn_fwd(q[g], k[g], v[g], causal=False, window=-1, scale=scale, out=out[g],
                         lse=lse[g], stream=stream)
        if e > a:
            binding.attn_fwd(stack(q, a, e), stack(k, a, e), stack(v, a, e), causal=False,
                             window=local_window, scale=scale, out=stack(out, a, e),
                             lse=stack(lse, a, e), stream=stream)
    return out, lse
