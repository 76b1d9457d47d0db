"""Tree decoding across devices: the sequence axis of the KV cache is sharded,
every device decodes its own shard, and the per-device results are merged by
the associative logsumexp reduction.

Source: "Tree Attention: Topology-aware Decoding for Long-Context Attention on
GPU Clusters" (express24.ir), abstract: the reduction across the sequence axis
can be computed in parallel as a tree, which takes less communication and less
peak memory than Ring Attention.

A device's decode result (O_r, LSE_r) over its shard is itself a partial
triple of the split definition: m = LSE_r, l = 1, o = O_r (because o / l = O_r
and m + ln l = LSE_r).  Merging the world's triples with lse_tree_combine
gives exactly the unsplit result.  The only exchange is one all-gather of
(O_r, LSE_r): B * Hq * (d + 1) floats per device, independent of the sequence
length; Ring Attention instead moves every K/V shard around the ring.

On one GPU the devices are emulated one after another
(``tree_decode_emulated``); ``gather_rank_outputs`` is the real exchange for
one process per device (NCCL on GPUs, gloo on CPU ranks).  All compute runs in
the library's CUDA kernels; this module only slices, gathers and marshals.
"""

from __future__ import annotations

import torch

__all__ = [
    "shard_bounds",
    "shard_kv_len",
    "shard_cache",
    "gather_rank_outputs",
    "merge_rank_outputs",
    "tree_decode_emulated",
    "comm_bytes_tree",
    "comm_bytes_ring",
]


def shard_bounds(L: int, world: int):
    """Contiguous key ranges [lo, hi) of the `world` shards of a length-L axis
    (the first L % world shards get one extra key)."""
    if L < 0 or world < 1:
        raise ValueError("L must be >= 0 and world >= 1")
    base, extra = divmod(L, world)
    out, lo = [], 0
    for r in range(world):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def shard_kv_len(kv_len: torch.Tensor, lo: int, hi: int) -> torch.Tensor:
    """Keys of each sequence that fall in shard [lo, hi): clamp(kv_len - lo, 0, hi - lo)."""
    return (kv_len.to(torch.int64) - lo).clamp(min=0, max=hi - lo).to(torch.int32)


def shard_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, lo: int, hi: int):
    """The shard's own contiguous copy of rows [lo, hi) of the caches, as a
    device holding only that shard would store it."""
    return k_cache[:, lo:hi].contiguous(), v_cache[:, lo:hi].contiguous()


def gather_rank_outputs(O: torch.Tensor, LSE: torch.Tensor, group=None):
    """All-gather every rank's decode output.  O [B, Hq, d] and LSE [B, Hq]
    (float32) -> O_all [B*Hq, world, d], LSE_all [B*Hq, world], ordered by rank."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    B, Hq, d = O.shape
    Os = [torch.empty_like(O) for _ in range(world)]
    Ls = [torch.empty_like(LSE) for _ in range(world)]
    dist.all_gather(Os, O.contiguous(), group=group)
    dist.all_gather(Ls, LSE.contiguous(), group=group)
    O_all = torch.stack(Os, dim=2).reshape(B * Hq, world, d)
    L_all = torch.stack(Ls, dim=2).reshape(B * Hq, world)
    return O_all, L_all


def merge_rank_outputs(O_all: torch.Tensor, LSE_all: torch.Tensor, out_dtype=torch.float32):
    """Merge per-rank (O_r, LSE_r) with the logsumexp tree kernel: the triples
    (m = LSE_r, l = 1, o = O_r).  O_all [R, world, d], LSE_all [R, world] f32 on
    the GPU -> (O [R, d], LSE [R])."""
    from . import binding
    part_l = torch.ones_like(LSE_all)
    return binding.lse_tree_combine(LSE_all.contiguous(), part_l, O_all.contiguous(),
                                    out_dtype=out_dtype)


def tree_decode_emulated(q, shards, num_splits: int, scale: float | None = None,
                         out_dtype=torch.bfloat16):
    """Decode over `shards` = [(k_shard, v_shard, kv_len_shard), ...] as if each
    lived on its own device: one split-KV decode per shard (f32 outputs), then
    one logsumexp tree merge of the per-shard results.  Returns (O [B, Hq, d],
    LSE [B, Hq])."""
    from . import binding
    B, Hq, d = q.shape
    Os, Ls = [], []
    for k_s, v_s, len_s in shards:
        O_r, L_r = binding.attn_decode_splitkv(q, k_s, v_s, len_s, num_splits, scale=scale,
                                               out_dtype=torch.float32)
        Os.append(O_r)
        Ls.append(L_r)
    O_all = torch.stack(Os, dim=2).reshape(B * Hq, len(shards), d)
    L_all = torch.stack(Ls, dim=2).reshape(B * Hq, len(shards))
    O, L = merge_rank_outputs(O_all, L_all, out_dtype=out_dtype)
    return O.view(B, Hq, d), L.view(B, Hq)


def comm_bytes_tree(B: int, Hq: int, d: int, world: int) -> int:
    """Bytes each device receives in the tree scheme: the other devices'
    (O, LSE) in float32 (one all-gather)."""
    return (world - 1) * B * Hq * (d + 1) * 4


def comm_bytes_ring(B: int, L: int, Hkv: int, d: int, world: int, elem_bytes: int = 2) -> int:
    """Bytes each device receives when the K/V shards circulate around a ring
    (Ring Attention): every other device's K and V shard once."""
    per_shard = B * (L // world) * Hkv * d * 2 * elem_bytes
    return (world - 1) * per_shard
