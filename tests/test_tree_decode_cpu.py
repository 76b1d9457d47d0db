"""Cross-device tree decoding, host side, on CPU ranks (gloo).

Every rank holds one contiguous shard of the KV sequence axis, decodes it (the
float64 oracle stands in for a device's decode here; the GPU test runs the
library's kernels), and the ranks all-gather their (O_r, LSE_r) with the
library's exchange; the logsumexp merge of the gathered triples must equal the
unsplit decode.  Also checks the shard bounds and the communication counts of
the tree scheme against Ring Attention ("Tree Attention" page, abstract).
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_bounds_cover_the_axis():
    from exact_transformer_attention_flashattention_b300 import tree_decode as td
    for L, world in [(0, 1), (1, 3), (10, 3), (1 << 20, 8), (1000, 7)]:
        b = td.shard_bounds(L, world)
        assert len(b) == world and b[0][0] == 0 and b[-1][1] == L
        assert all(b[i][1] == b[i + 1][0] for i in range(world - 1))
        sizes = [hi - lo for lo, hi in b]
        assert max(sizes) - min(sizes) <= 1
    kv = torch.tensor([0, 5, 10, 13], dtype=torch.int32)
    assert td.shard_kv_len(kv, 5, 10).tolist() == [0, 0, 5, 5]
    assert td.shard_kv_len(kv, 10, 15).tolist() == [0, 0, 0, 3]


def test_tree_moves_far_less_than_the_ring_at_long_context():
    from exact_transformer_attention_flashattention_b300 import tree_decode as td
    # the million-token decode shape over 8 devices
    tree = td.comm_bytes_tree(B=1, Hq=32, d=128, world=8)
    ring = td.comm_bytes_ring(B=1, L=1 << 20, Hkv=8, d=128, world=8)
    assert tree == 7 * 32 * 129 * 4
    assert ring == 7 * (1 << 17) * 8 * 128 * 2 * 2
    assert ring > 1000 * tree
    assert td.comm_bytes_tree(1, 32, 128, 1) == 0 == td.comm_bytes_ring(1, 1024, 8, 128, 1)


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    import oracle
    from exact_transformer_attention_flashattention_b300 import tree_decode as td
    from exact_transformer_attention_flashattention_b300.inputs import decode_inputs
    dist.init_process_group("gloo")
    try:
        B, Hq, Hkv, L, d = 3, 8, 2, 700, 64
        q, kc, vc, kv_len = decode_inputs(B, Hq, Hkv, L, d, seed=31, kv_len_lo=1, kv_len_hi=L)
        lo, hi = td.shard_bounds(L, world)[rank]
        k_s, v_s = td.shard_cache(kc, vc, lo, hi)
        len_s = td.shard_kv_len(kv_len, lo, hi)
        O_r, L_r = oracle.decode(q, k_s, v_s, len_s, scale=d ** -0.5)  # this rank's decode
        O_all, L_all = td.gather_rank_outputs(torch.tensor(O_r, dtype=torch.float32),
                                              torch.tensor(L_r, dtype=torch.float32))
        # merge the gathered triples (m = LSE_r, l = 1, o = O_r) on the host
        m = L_all.double().numpy()
        O_m, L_m = oracle.combine_rows(m, np.where(np.isneginf(m), 0.0, 1.0), O_all.double().numpy())
        O_ref, L_ref = oracle.decode(q, kc, vc, kv_len, scale=d ** -0.5)
        err_o = float(np.abs(O_m.reshape(B, Hq, d) - O_ref).max())
        err_l = float(np.abs(L_m.reshape(B, Hq) - L_ref).max())
        out.put((rank, tuple(O_all.shape), err_o, err_l))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_gather_and_merge_to_the_unsplit_decode(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0] * world, codes
    res = sorted(out.get(timeout=5) for _ in range(world))
    for rank, shape, err_o, err_l in res:
        assert shape == (3 * 8, world, 64)
        # f32 exchange of f64 results: agreement to f32 rounding
        assert err_o < 1e-5 and err_l < 1e-5, (rank, err_o, err_l)
