"""Head-grouped Ulysses around the sparse attention, on CPU with gloo.

"HeyGen x Google Cloud: Avatar IV on TPU", "Hiding the Collective", Fig. 2:
heads are split into groups, each running all-to-all -> attention ->
all-to-all, pipelined against the others; the token order inside a group is
the unsplit order, so the sparse mask is unchanged.

Two (and four) gloo ranks on 127.0.0.1 run ``ulysses_attention`` with the
fp64 oracle as the attention function, and the result must equal the
single-process oracle on the whole sequence.  The attention function also
checks that every group arrives with all N tokens of its heads in the
original order.  (On the GPU the attention function is the library's
kernels; a one-GPU machine gives a one-rank group, covered by the GPU test in
test_gpu_parity.py.)
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _full_inputs(H, N, d, seed):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
    k += 3.0 * rng.standard_normal((H, 1, d))
    return q, k, v


def _rank_main(rank, world, port, geo, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from frame_aligned_sparse_gb300 import ulysses
    from oracle import reference as ref
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H, d, R0, spans, r, G, seed = geo
        N = sum(spans)
        n = N // world
        q, k, v = _full_inputs(H, N, d, seed)
        # This rank's token shard, plain [n, H, d], then the all-to-all layout.
        shard = [torch.from_numpy(np.ascontiguousarray(x[:, rank * n:(rank + 1) * n].transpose(1, 0, 2)))
                 for x in (q, k, v)]
        a2a = [ulysses.to_a2a_layout(t, G, world) for t in shard]
        hp = H // (G * world)
        calls = []

        def attn(qg, kg, vg):
            g = len(calls)
            heads = [g * (H // G) + rank * hp + j for j in range(hp)]
            # Whole sequence, original token order, this rank's heads of group g.
            for got, full in ((qg, q), (kg, k), (vg, v)):
                assert got.shape == (N, hp, d)
                assert np.array_equal(got.numpy(), full[heads].transpose(1, 0, 2))
            calls.append(g)
            res = ref.masked_attention(qg.numpy().transpose(1, 0, 2), kg.numpy().transpose(1, 0, 2),
                                       vg.numpy().transpose(1, 0, 2), spans, R0, r)
            return torch.from_numpy(np.ascontiguousarray(res["out"].transpose(1, 0, 2))), torch.from_numpy(res["lse"])

        out, lse = ulysses.ulysses_attention(*a2a, attn)
        results[rank] = (ulysses.from_a2a_layout(out).numpy(), lse.numpy(), calls)
    finally:
        dist.destroy_process_group()


GEOMETRIES = [
    # H, d, R0, spans, r, G, seed
    (4, 8, 1, [8] * 6, 1, 2, 61),
    (8, 8, 1, [16, 8, 24, 8, 16, 8], 2, 2, 62),
    (8, 4, 2, [8] * 8, 0, 4, 63),
]


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("geo", GEOMETRIES, ids=["uniform", "ragged", "four_groups"])
def test_ulysses_matches_single_rank_oracle(geo, world):
    from oracle import reference as ref
    H, d, R0, spans, r, G, seed = geo
    if H % (G * world):
        pytest.skip("heads do not split into these groups and ranks")
    N = sum(spans)
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), geo, results), nprocs=world, join=True,
                           start_method="spawn")
        results = dict(results)
    q, k, v = _full_inputs(H, N, d, seed)
    want = ref.masked_attention(q, k, v, spans, R0, r)
    n = N // world
    hp = H // (G * world)
    for rank in range(world):
        out, lse, calls = results[rank]
        assert calls == list(range(G))
        np.testing.assert_allclose(out, want["out"][:, rank * n:(rank + 1) * n].transpose(1, 0, 2),
                                   rtol=1e-13, atol=1e-14)
        for g in range(G):
            heads = [g * (H // G) + rank * hp + j for j in range(hp)]
            np.testing.assert_allclose(lse[g], want["lse"][heads], rtol=1e-13, atol=1e-13)


def test_schedule_overlaps_each_transfer_with_the_previous_groups_attention():
    from frame_aligned_sparse_gb300 import ulysses
    for G in (1, 2, 3, 6):
        ops = ulysses.schedule(G)
        pos = {op: i for i, op in enumerate(ops)}
        assert sorted(ops) == sorted([(s, g) for g in range(G) for s in ("in", "attn", "out")])
        for g in range(G):
            assert pos[("in", g)] < pos[("attn", g)] < pos[("out", g)]
            if g + 1 < G:
                # Group g+1's transfer is in flight while group g computes.
                assert pos[("in", g + 1)] < pos[("attn", g)]
                # Group g's return is issued before group g+1's attention.
                assert pos[("out", g)] < pos[("attn", g + 1)]
        assert ops[0] == ("in", 0) and ops[-1] == ("out", G - 1)


def test_a2a_layout_round_trip_and_slices():
    from frame_aligned_sparse_gb300 import ulysses
    n, H, d, G, P = 5, 12, 3, 2, 3
    x = torch.arange(n * H * d, dtype=torch.float64).reshape(n, H, d)
    y = ulysses.to_a2a_layout(x, G, P)
    assert y.shape == (G, P, n, H // (G * P), d) and y.is_contiguous()
    assert torch.equal(ulysses.from_a2a_layout(y), x)
    hp = H // (G * P)
    for g in range(G):
        for r in range(P):
            for j in range(hp):
                assert torch.equal(y[g, r, :, j], x[:, g * (H // G) + r * hp + j])
    with pytest.raises(ValueError):
        ulysses.to_a2a_layout(torch.zeros(n, 10, d), G, P)
