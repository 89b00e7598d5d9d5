"""fas_prepass_noalloc: the prepass for callers that cannot allocate.

Some users of this library own all device memory themselves — for example a
serving process that reserves the GPU's memory in its own pool at start-up,
or a per-chunk streaming loop that must not stall on cudaMalloc/cudaFree —
and can only hand the library buffers they sized in advance.  For them the
library offers a prepass whose scratch is a fixed array in device memory, so
it allocates nothing.  These tests call it through the C ABI and check that
two calls in a row give what the allocating fas_prepass gives, within the
tolerances the prepass parity tests use.

This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import frame_aligned_sparse_gb300 as fas
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frame_aligned_sparse_gb300 import build
    build.build()
    return fas.load()


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("name", ["tiny", "mid", "720p"])
def test_noalloc_prepass_matches_allocating_prepass(lib, name):
    w = workloads.get(name)
    x = workloads.generate(w, tensors=("q", "k"))
    q, k = to_dev(x["q"]), to_dev(x["k"])
    H, N = w.heads, w.tokens
    fas.fas_plan(w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius, H, w.head_dim)
    fas.fas_prepass(q, k)
    want = fas.fas_prepass_readback(row_bound=True)
    stream = torch.cuda.current_stream().cuda_stream
    results = []
    for _ in range(2):
        row_bound = torch.full((H, N), float("nan"), device="cuda")
        stat = torch.full((H,), float("nan"), device="cuda")
        elig = torch.full((H,), 255, dtype=torch.uint8, device="cuda")
        rc = lib.fas_prepass_noalloc(q.data_ptr(), k.data_ptr(), w.frame_tokens, w.n_frames, w.ref_frames,
                                     w.window_radius, H, w.head_dim, row_bound.data_ptr(), stat.data_ptr(),
                                     elig.data_ptr(), stream)
        assert rc == fas.FAS_OK, lib.fas_error_string(rc)
        torch.cuda.synchronize()
        got = {"row_bound": row_bound.cpu().numpy(), "stat": stat.cpu().numpy(), "elig": elig.cpu().numpy()}
        np.testing.assert_allclose(got["row_bound"], want["row_bound"], rtol=1e-4, atol=1e-3)
        np.testing.assert_allclose(got["stat"], want["stat"], rtol=1e-4, atol=1e-3)
        assert np.array_equal(got["elig"], want["elig"])
        results.append(got)
    # The second call starts from the first call's leftovers in the shared
    # scratch and must give the same bits.
    for key in results[0]:
        assert np.array_equal(results[0][key], results[1][key]), key


# Geometries where the call's own frame rule (it has no block table) is most
# likely to differ from the planner's: no reference frame, two reference
# frames, a single video frame, a window wider than the clip.
EDGE = [
    # name, H, d, R0, F, T, r, sigma, seed
    ("no_reference", 2, 128, 0, 5, 144, 1, 3.0, 32),
    ("two_references", 1, 128, 2, 4, 208, 1, 3.0, 33),
    ("single_frame", 1, 64, 1, 1, 256, 3, 2.0, 34),
    ("d64_wide_window", 2, 64, 1, 9, 240, 9, 2.0, 38),
]


@pytest.mark.parametrize("spec", EDGE, ids=[e[0] for e in EDGE])
def test_noalloc_prepass_edge_geometries(lib, spec):
    name, H, d, R0, F, T, r, sigma, seed = spec
    w = workloads.Workload(name, H, d, R0, F, T, r, sigma, seed)
    x = workloads.generate(w, tensors=("q", "k"))
    q, k = to_dev(x["q"]), to_dev(x["k"])
    N = w.tokens
    fas.fas_plan(T, F, R0, r, H, d)
    fas.fas_prepass(q, k)
    want = fas.fas_prepass_readback(row_bound=True)
    for _ in range(2):
        row_bound = torch.full((H, N), float("nan"), device="cuda")
        stat = torch.full((H,), float("nan"), device="cuda")
        elig = torch.full((H,), 255, dtype=torch.uint8, device="cuda")
        fas.fas_prepass_noalloc(q, k, T, F, R0, r, row_bound, stat, elig)
        torch.cuda.synchronize()
        np.testing.assert_allclose(row_bound.cpu().numpy(), want["row_bound"], rtol=1e-4, atol=1e-3)
        np.testing.assert_allclose(stat.cpu().numpy(), want["stat"], rtol=1e-4, atol=1e-3)
        assert np.array_equal(elig.cpu().numpy(), want["elig"])


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    # 96 heads of the 720p geometry need about 5.6 MB of scratch (> 4 MiB).
    q = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(16, device="cuda")
    elig = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = lib.fas_prepass_noalloc(q.data_ptr(), q.data_ptr(), 3600, 21, 1, 2, 96, 128, out.data_ptr(),
                                 out.data_ptr(), elig.data_ptr(), None)
    assert rc == fas.FAS_ERR_SCRATCH
    assert "fixed scratch" in lib.fas_error_string(rc).decode()
