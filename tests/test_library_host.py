"""Host-side tests of the C-ABI library (no GPU needed).

The library must load, export every function include/fas.h declares, and
its planner must cover exactly the oracle's mask with full, non-overlapping,
frame-aligned key blocks ("HeyGen x Google Cloud: Avatar IV on TPU",
"Deleting the Mask", Fig. 3).
"""
import ctypes
import os
import re

import numpy as np
import pytest

import frame_aligned_sparse_gb300 as fas
import workloads
from oracle import reference as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from frame_aligned_sparse_gb300 import build
    build.build()
    return fas.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fas.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fas_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_function(built_library):
    names = header_functions()
    assert {"fas_plan", "fas_prepass", "fas_forward", "fas_free"} <= set(names)
    for name in names:
        assert hasattr(built_library, name), name
        assert ctypes.cast(getattr(built_library, name), ctypes.c_void_p).value


def test_library_is_built_for_sm_103a():
    """The build compiles every translation unit for sm_103a and nothing
    else, and the built library is the one those flags produced."""
    from frame_aligned_sparse_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    stamp = os.path.join(build.BUILD, "stamp")
    assert open(stamp).read() == build._fingerprint()


GEOMETRIES = [
    # (T, F, R0, r, H, d)
    (48, 8, 1, 1, 2, 64),
    (880, 16, 1, 2, 16, 128),
    (3600, 21, 1, 2, 24, 128),
    (8160, 13, 1, 1, 24, 128),
    (3600, 21, 1, 21, 24, 128),
    (64, 5, 2, 1, 1, 128),
    (32, 6, 0, 1, 1, 64),
    (16, 3, 1, 0, 3, 64),
]


def expand_blocks(table_row, Bk):
    blocks = []
    for start, length in ((table_row[0], table_row[1]), (table_row[2], table_row[3])):
        assert length % Bk == 0 and start % Bk == 0
        blocks += list(range(start, start + length, Bk))
    return blocks


@pytest.mark.parametrize("geo", GEOMETRIES, ids=lambda g: "T%d_F%d_R%d_r%d" % g[:4])
def test_plan_covers_mask_exactly(geo):
    T, F, R0, r, H, d = geo
    info, table, work = fas.fas_plan_describe(T, F, R0, r, H, d)
    Bk = info.block_k
    nf = R0 + F
    N = nf * T
    assert Bk % 16 == 0 and T % Bk == 0 and 16 <= Bk <= 160
    assert info.tokens == N and info.total_frames == nf
    for f in range(nf):
        blocks = expand_blocks(table[f], Bk)
        assert len(blocks) == len(set(blocks)), "duplicate block"
        covered = np.zeros(N, dtype=bool)
        for b in blocks:
            assert b // T == (b + Bk - 1) // T, "block straddles a frame boundary"
            covered[b:b + Bk] = True
        # Every row of the frame has the same visible keys: compare with the
        # explicit oracle mask of the frame's first and last row.
        rows = np.array([f * T, f * T + T - 1])
        mask = ref.token_mask(rows, N, T, R0, r)
        assert np.array_equal(covered, mask[0]) and np.array_equal(covered, mask[1])
    assert info.visible_flops == ref.visible_flops(H, d, T, F, R0, r)
    tiles = -(-T // 128)
    assert info.n_work == H * nf * tiles == len(work)
    # Each (head, frame, tile) exactly once; block counts match the table;
    # heaviest items first.
    keys = {(int(a), int(b), int(c)) for a, b, c, _ in work}
    assert len(keys) == info.n_work
    for h, f, t, nblk in work:
        assert nblk == (table[f][1] + table[f][3]) // Bk
    assert np.all(np.diff(work[:, 3]) <= 0)
    assert info.key_blocks == int(work[:, 3].sum())


RAGGED_GEOMETRIES = [
    # (spans, R0, r, H, d)
    ([48, 32, 64, 16, 48], 1, 1, 2, 64),
    ([3600, 3520, 3600, 3680, 3600, 3440, 3600], 1, 2, 3, 128),
    ([160, 320, 480, 160, 640], 2, 0, 1, 128),
    ([96, 144, 48, 240, 192, 96], 0, 1, 2, 64),
    ([880, 880, 704, 1056, 880], 1, 9, 1, 128),
]


@pytest.mark.parametrize("geo", RAGGED_GEOMETRIES, ids=lambda g: "Nf%d_R%d_r%d" % (len(g[0]), g[1], g[2]))
def test_ragged_plan_covers_mask_exactly(geo):
    """Frames of different spans: the block divides every span, no block
    straddles a frame, every query frame's blocks cover exactly the oracle's
    explicit mask, and the FLOP count is the oracle's."""
    spans, R0, r, H, d = geo
    F = len(spans) - R0
    info, table, work = fas.fas_plan_describe(spans, F, R0, r, H, d)
    Bk = info.block_k
    assert all(t % Bk == 0 for t in spans) and Bk % 16 == 0 and Bk <= 160
    assert all(any(t % b for t in spans) for b in range(Bk + 16, 161, 16)), "a larger block divides every span"
    N = sum(spans)
    starts = np.concatenate([[0], np.cumsum(spans)])
    assert info.tokens == N and info.total_frames == len(spans)
    for f in range(len(spans)):
        covered = np.zeros(N, dtype=bool)
        for b in expand_blocks(table[f], Bk):
            g = np.searchsorted(starts, b, side="right") - 1
            assert b + Bk <= starts[g + 1], "block straddles a frame boundary"
            assert not covered[b:b + Bk].any(), "duplicate block"
            covered[b:b + Bk] = True
        rows = np.array([starts[f], starts[f + 1] - 1])
        mask = ref.token_mask(rows, N, spans, R0, r)
        assert np.array_equal(covered, mask[0]) and np.array_equal(covered, mask[1])
    assert info.visible_flops == ref.visible_flops(H, d, spans, F, R0, r)
    tiles = sum(-(-t // 128) for t in spans)
    assert info.n_work == H * tiles == len(work)
    assert len({(int(a), int(b), int(c)) for a, b, c, _ in work}) == info.n_work
    for h, f, t, nblk in work:
        assert t < -(-spans[f] // 128) and nblk == (table[f][1] + table[f][3]) // Bk
    assert np.all(np.diff(work[:, 3]) <= 0)


def test_ragged_plan_equal_spans_is_the_uniform_plan():
    a = fas.fas_plan_describe(880, 16, 1, 2, 16, 128)
    b = fas.fas_plan_describe([880] * 17, 16, 1, 2, 16, 128)
    assert a[0].block_k == b[0].block_k and a[0].visible_flops == b[0].visible_flops
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


@pytest.mark.parametrize("spans,R0,bk", [([48, 40, 64], 1, 0), ([48, 0, 64], 1, 0), ([48, 64], 2, 0),
                                         ([48, 96, 64], 1, 32), ([48, 96, 64], 1, 48)])
def test_bad_ragged_arguments_are_rejected(spans, R0, bk):
    lib = fas.load()
    info = fas._PlanInfoC()
    arr = np.array(spans, dtype=np.int32)
    F = len(spans) - R0
    if F < 1:
        F = 1  # the span count then does not match R0 + F
        with pytest.raises(ValueError):
            fas.fas_plan_describe(spans, F, R0, 1, 1, 64)
        return
    assert lib.fas_plan_describe_ragged(arr.ctypes.data, F, R0, 1, 1, 64, bk, ctypes.byref(info), None,
                                        None) == fas.FAS_ERR_ARG


def test_noalloc_wrapper_rejects_a_geometry_that_does_not_match_q():
    """fas_prepass_noalloc has no plan to check its buffers against; the
    binding refuses a geometry whose token count differs from q's before
    anything reaches the device."""
    import torch
    q = torch.zeros(2, 9 * 48, 64, dtype=torch.bfloat16)
    rb, stat, elig = torch.zeros(2, 9 * 48), torch.zeros(2), torch.zeros(2, dtype=torch.uint8)
    with pytest.raises(ValueError, match="rows per head"):
        fas.fas_prepass_noalloc(q, q, 48, 9, 1, 1, rb, stat, elig)  # needs 10 * 48 rows
    with pytest.raises(ValueError, match="rows per head"):
        fas.fas_prepass_noalloc(q, q, 64, 8, 1, 1, rb, stat, elig)


def test_key_sums_calls_check_their_arguments_before_any_device_work():
    """The prologue's key-sums output and the prepass that takes it refuse
    bad arguments before touching memory (the pointers below are never
    dereferenced)."""
    lib = fas.load()
    lib.fas_free()
    p = 256
    assert lib.fas_prepass_with_key_sums(p, p, None, None, None) == fas.FAS_ERR_ARG
    assert lib.fas_prepass_with_key_sums(p, p, p, None, None) == fas.FAS_ERR_STATE  # no plan
    four = (p, p, p, p)
    assert lib.fas_prologue_with_key_sums(*four, 120, 128, 2, 64, 1e-6, p, p, p, 0, 1, 1, p,
                                          None) == fas.FAS_ERR_ARG  # tokens not a multiple of 16
    assert lib.fas_prologue_with_key_sums(*four, 128, 128, 2, 64, 1e-6, p, p, p, 0, 1, 1, p + 8,
                                          None) == fas.FAS_ERR_ALIGN
    assert fas.key_sums_shape(24, 79200, 128) == (24, 4950, 128)
    with pytest.raises(ValueError):
        fas.key_sums_shape(2, 120, 64)


def test_block_size_choice_matches_frame_spans():
    # Largest multiple of 16 dividing T within the on-chip budget (<= 160).
    for T, want in ((48, 48), (880, 80), (3600, 144), (8160, 160), (16, 16), (4096, 128), (192, 96), (352, 32), (320, 160), (400, 80)):
        info, _, _ = fas.fas_plan_describe(T, 3, 1, 1, 1, 128)
        assert info.block_k == want, (T, info.block_k)
    info, _, _ = fas.fas_plan_describe(3600, 3, 1, 1, 1, 128, block_k=48)
    assert info.block_k == 48


@pytest.mark.parametrize("args", [
    (0, 8, 1, 1, 2, 64, 0), (40, 8, 1, 1, 2, 64, 0), (48, 0, 1, 1, 2, 64, 0), (48, 8, -1, 1, 2, 64, 0),
    (48, 8, 1, -1, 2, 64, 0), (48, 8, 1, 1, 0, 64, 0), (48, 8, 1, 1, 2, 96, 0), (48, 8, 1, 1, 2, 64, 32),
    (48, 8, 1, 1, 2, 64, 8), (3840, 8, 1, 1, 2, 64, 240), (384, 8, 1, 1, 2, 64, 192), (352, 8, 1, 1, 2, 64, 176),
])
def test_bad_arguments_are_rejected(args):
    lib = fas.load()
    info = fas._PlanInfoC()
    assert lib.fas_plan_describe(*args, ctypes.byref(info), None, None) == fas.FAS_ERR_ARG


def test_calls_out_of_order_return_state_error():
    lib = fas.load()
    lib.fas_free()
    assert lib.fas_prepass(None, None, None, None) == fas.FAS_ERR_STATE
    assert lib.fas_forward(None, None, None, None, None, 0, None) == fas.FAS_ERR_STATE
    assert lib.fas_forward_host(None, None, None, None, None, 0, 0, None) == fas.FAS_ERR_STATE
    assert lib.fas_set_layout(1) == fas.FAS_ERR_STATE
    assert lib.fas_set_layout(5) == fas.FAS_ERR_ARG
    assert lib.fas_status(None) == fas.FAS_ERR_STATE
    assert lib.fas_prepass_readback(None, None, None, None, None, None) == fas.FAS_ERR_STATE
    assert lib.fas_selftest_wait_timeout(0, None) == fas.FAS_ERR_ARG
    assert b"q or k changed" in lib.fas_error_string(fas.FAS_ERR_BOUND)
    assert lib.fas_error_string(fas.FAS_ERR_TIMEOUT).decode().startswith("device-side wait")


def test_partial_block_statistic_for_128_tiling():
    """With 128-multiple tiling, blocks straddle frame boundaries ("Deleting
    the Mask": roughly one in five live blocks came out partial on the
    pages' shapes).  With frame-aligned blocks none does.  This records the
    fraction for our shapes as a planner statistic."""
    for name, want in (("mid", 0.104), ("720p", 0.027)):
        w = workloads.get(name)
        T, nf = w.frame_tokens, w.total_frames
        N = nf * T
        vis = ref.frame_visibility(nf, w.ref_frames, w.window_radius)
        live = partial = 0
        for qb in range(0, N, 128):
            qfr = np.unique(np.arange(qb, min(qb + 128, N)) // T)
            for kb in range(0, N, 128):
                kfr = np.unique(np.arange(kb, min(kb + 128, N)) // T)
                sub = vis[np.ix_(qfr, kfr)]
                if sub.any():
                    live += 1
                    # Partial: the block mixes visible and hidden entries.
                    partial += not sub.all()
        assert abs(partial / live - want) < 0.01, (name, partial, live)
