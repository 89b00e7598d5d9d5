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
    # The fatbin must carry sm_103a code; check the ELF note nvcc embeds.
    data = open(fas.library_path(), "rb").read()
    assert b"sm_103a" in data


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
