"""GPU parity: the CUDA path against the fp64 oracle, through the C ABI.

Tolerances (bf16 inputs, fp32 accumulation, bf16 P in P.V as in "Proving the
Pixels Didn't Change", bf16 output): max |out - oracle| <= 2e-2 and
max |lse - oracle| <= 1e-3; eligibility bits bit-exact.  Small workloads are
compared on every row; the full-size workloads on stratified sampled rows
(every head, every query frame, frame edges, the ragged last query tile,
reference rows, random interior rows), in the launch configuration the
benchmark times.
"""
import ctypes

import numpy as np
import pytest
import torch

import frame_aligned_sparse_gb300 as fas
import workloads
from oracle import reference as ref

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frame_aligned_sparse_gb300 import build
    build.build()
    yield fas.load()
    fas.fas_free()


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def sample_rows(w, per_head_min=512, seed=0):
    T, nf = w.frame_tokens, w.total_frames
    rng = np.random.default_rng(seed)
    rows = set()
    last_tile = ((T - 1) // 128) * 128
    for f in range(nf):
        base = f * T
        for r in (0, 1, 127, 128, T // 2, last_tile - 1, last_tile, T - 2, T - 1):
            if 0 <= r < T:
                rows.add(base + r)
        rows.update((base + rng.choice(T, 8, replace=False)).tolist())
    extra = per_head_min - len(rows)
    if extra > 0:
        rows.update(rng.choice(nf * T, extra + 64, replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


class Case:
    """Inputs on host and device, the plan, and oracle results (cached)."""

    def __init__(self, w, rows=None, x=None):
        self.w = w
        self.x = workloads.generate(w) if x is None else x
        self.q, self.k, self.v = (to_dev(self.x[t]) for t in "qkv")
        self.rows = rows
        self._ref = None
        self._st = None

    def plan(self, block_k=0):
        w = self.w
        return fas.fas_plan(w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius, w.heads, w.head_dim,
                            block_k=block_k)

    @property
    def oracle(self):
        if self._ref is None:
            w = self.w
            self._ref = ref.masked_attention(self.x["q"], self.x["k"], self.x["v"], w.frame_tokens, w.ref_frames,
                                             w.window_radius, rows=self.rows)
        return self._ref

    @property
    def stats(self):
        if self._st is None:
            w = self.w
            self._st = ref.bound_statistics(self.x["q"], self.x["k"], w.frame_tokens, w.ref_frames,
                                            w.window_radius)
        return self._st

    def run(self, mode, block_k=0):
        self.plan(block_k)
        elig = fas.fas_prepass(self.q, self.k, want_elig=True)
        out, lse = fas.fas_forward(self.q, self.k, self.v, mode=mode)
        assert fas.fas_status() == fas.FAS_OK
        return elig, out, lse

    def check(self, out, lse, label=""):
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        if self.rows is not None:
            o, l = o[:, self.rows], l[:, self.rows]
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), label
        d_out = np.abs(o - self.oracle["out"]).max()
        d_lse = np.abs(l - self.oracle["lse"]).max()
        assert d_out <= OUT_TOL, (label, "max |dout|", d_out)
        assert d_lse <= LSE_TOL, (label, "max |dlse|", d_lse)
        return d_out, d_lse


_CASES = {}


def case(name):
    if name not in _CASES:
        w = workloads.get(name)
        rows = None if name in ("tiny", "mid") else sample_rows(w)
        _CASES.clear()  # keep one large workload resident at a time
        _CASES[name] = Case(w, rows)
    return _CASES[name]


def test_bounded_wait_selftest_reports_timeout():
    assert fas.fas_selftest_wait_timeout(2000) == fas.FAS_ERR_TIMEOUT
    # The context is still usable afterwards.
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_prepass_statistics(name):
    c = case(name)
    c.plan()
    elig = fas.fas_prepass(c.q, c.k, want_elig=True)
    got = fas.fas_prepass_readback(row_bound=True)
    st = c.stats
    np.testing.assert_allclose(got["mu"], st["mu"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["frame_max"], st["M"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["row_bound"], st["m"], rtol=1e-4, atol=1e-3)
    np.testing.assert_allclose(got["stat"], st["stat"], rtol=1e-4, atol=1e-3)
    assert np.array_equal(elig.astype(bool), st["elig"])
    assert np.array_equal(got["elig"].astype(bool), st["elig"])


def test_prepass_statistics_720p():
    """The fused prepass on the full 720p SR chunk (its queue interleaves
    24 heads over three phases) against the oracle on every head."""
    c = case("720p")
    c.plan()
    elig = fas.fas_prepass(c.q, c.k, want_elig=True)
    got = fas.fas_prepass_readback(row_bound=True)
    st = c.stats
    np.testing.assert_allclose(got["mu"], st["mu"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["frame_max"], st["M"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["stat"], st["stat"], rtol=1e-4, atol=1e-3)
    rows = c.rows
    np.testing.assert_allclose(got["row_bound"][:, rows], st["m"][:, rows], rtol=1e-4, atol=2e-3)
    assert np.array_equal(elig.astype(bool), st["elig"])


def key_sums_of(k_bits):
    """Column sums of every 16 keys of each head, [H, N/16, d] fp32 on the
    device, from the seeded bf16 keys [H, N, d] (fp64 sums rounded once):
    the input fas_prepass_with_key_sums takes."""
    H, N, d = k_bits.shape
    out = np.empty((H, N // 16, d), np.float32)
    for h in range(H):
        out[h] = ref.bf16_bits_to_f64(k_bits[h]).reshape(N // 16, 16, d).sum(axis=1)
    return torch.from_numpy(out).cuda()


def check_key_sums_statistics(c, got, elig, row_atol=1e-3, rows=None):
    st = c.stats
    np.testing.assert_allclose(got["mu"], st["mu"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["frame_max"], st["M"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["stat"], st["stat"], rtol=1e-4, atol=1e-3)
    sel = slice(None) if rows is None else rows
    np.testing.assert_allclose(got["row_bound"][:, sel], st["m"][:, sel], rtol=1e-4, atol=row_atol)
    assert np.array_equal(elig.astype(bool), st["elig"])
    assert np.array_equal(got["elig"].astype(bool), st["elig"])


def test_prepass_with_key_sums_720p():
    """The prepass fed the 16-token key sums (its key phase adds them
    instead of reading k) on the full 720p SR chunk, against the oracle."""
    c = case("720p")
    c.plan()
    elig = fas.fas_prepass_with_key_sums(c.q, c.k, key_sums_of(c.x["k"]), want_elig=True)
    got = fas.fas_prepass_readback(row_bound=True)
    check_key_sums_statistics(c, got, elig, row_atol=2e-3, rows=c.rows)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_prepass_with_key_sums(name):
    """Statistics against the oracle; against fas_prepass's to fp32
    rounding (the sums are added in another order); bit-reproducible; the
    attention on its bounds against the oracle."""
    c = case(name)
    c.plan()
    ks = key_sums_of(c.x["k"])
    runs = []
    for _ in range(2):
        elig = fas.fas_prepass_with_key_sums(c.q, c.k, ks, want_elig=True)
        runs.append(fas.fas_prepass_readback(row_bound=True))
    check_key_sums_statistics(c, runs[0], elig)
    for key in runs[0]:
        assert np.array_equal(runs[0][key], runs[1][key]), key
    for mode in ("auto", "bounded"):
        out, lse = fas.fas_forward(c.q, c.k, c.v, mode=mode)
        assert fas.fas_status() == fas.FAS_OK
        c.check(out, lse, f"{name}/{mode}/key sums")
    fas.fas_prepass(c.q, c.k)
    plain = fas.fas_prepass_readback(row_bound=True)
    np.testing.assert_allclose(runs[0]["mu"], plain["mu"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(runs[0]["frame_max"], plain["frame_max"], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(runs[0]["row_bound"], plain["row_bound"], rtol=1e-5, atol=1e-4)
    assert np.array_equal(runs[0]["elig"], plain["elig"])


def test_prepass_with_key_sums_errors():
    c = case("tiny")
    c.plan()
    lib = fas.load()
    ks = key_sums_of(c.x["k"])
    st = torch.cuda.current_stream().cuda_stream
    assert lib.fas_prepass_with_key_sums(c.q.data_ptr(), c.k.data_ptr(), None, st, None) == fas.FAS_ERR_ARG
    assert lib.fas_prepass_with_key_sums(c.q.data_ptr(), c.k.data_ptr(), ks.data_ptr() + 4, st,
                                         None) == fas.FAS_ERR_ALIGN
    with pytest.raises((ValueError, TypeError)):
        fas.fas_prepass_with_key_sums(c.q, c.k, ks[:, 1:])
    fas.fas_free()
    assert lib.fas_prepass_with_key_sums(c.q.data_ptr(), c.k.data_ptr(), ks.data_ptr(), st,
                                         None) == fas.FAS_ERR_STATE


def test_prepass_is_bit_reproducible():
    """Whichever CTA finishes a phase reduces in a fixed order: two runs give
    the same bits."""
    c = case("mid")
    c.plan()
    outs = []
    for _ in range(2):
        fas.fas_prepass(c.q, c.k)
        outs.append(fas.fas_prepass_readback(row_bound=True))
    for key in outs[0]:
        assert np.array_equal(outs[0][key], outs[1][key]), key


@pytest.mark.parametrize("mode", ["auto", "online", "bounded"])
@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_forward_full_rows(name, mode):
    c = case(name)
    _, out, lse = c.run(mode)
    c.check(out, lse, f"{name}/{mode}")


@pytest.mark.parametrize("name", ["720p", "1080p", "stress", "dense"])
def test_forward_sampled_rows(name):
    c = case(name)
    results = {}
    for mode in ("auto", "online"):
        elig, out, lse = c.run(mode)
        want = np.ones(c.w.heads, dtype=bool)
        want[c.x["modified_heads"]] = False
        assert np.array_equal(elig.astype(bool), want), (name, elig)
        c.check(out, lse, f"{name}/{mode}")
        results[mode] = (out.float(), lse.clone())
    # Bounded and online softmax agree on the same (eligible) heads.
    eligible = [h for h in range(c.w.heads) if h not in set(c.x["modified_heads"].tolist())]
    a, b = results["auto"], results["online"]
    assert (a[0][eligible] - b[0][eligible]).abs().max().item() <= OUT_TOL
    assert (a[1][eligible] - b[1][eligible]).abs().max().item() <= LSE_TOL


EDGE = [
    # name, H, d, R0, F, T, r, sigma, seed, block_k
    ("T16_r0", 2, 64, 1, 3, 16, 0, 2.0, 31, 0),
    ("no_reference", 2, 128, 0, 5, 144, 1, 3.0, 32, 0),
    ("two_references", 1, 128, 2, 4, 208, 1, 3.0, 33, 0),
    ("single_frame", 1, 64, 1, 1, 256, 3, 2.0, 34, 0),
    ("bk16_many_blocks", 1, 128, 1, 6, 400, 2, 3.0, 35, 16),
    ("bk48_ragged", 3, 128, 1, 5, 336, 1, 3.0, 36, 48),
    ("bk160", 1, 128, 1, 3, 320, 1, 3.0, 37, 160),
    ("d64_wide_window", 2, 64, 1, 9, 240, 9, 2.0, 38, 0),
]


@pytest.mark.parametrize("spec", EDGE, ids=[e[0] for e in EDGE])
def test_edge_geometries(spec):
    name, H, d, R0, F, T, r, sigma, seed, bk = spec
    c = Case(workloads.Workload(name, H, d, R0, F, T, r, sigma, seed))
    for mode in ("auto", "online"):
        _, out, lse = c.run(mode, block_k=bk)
        c.check(out, lse, f"{name}/{mode}")
    # The prepass fed the 16-token key sums (key items cut at 16-row
    # boundaries of frames as short as 16 tokens), then the attention on
    # its bounds.
    elig = fas.fas_prepass_with_key_sums(c.q, c.k, key_sums_of(c.x["k"]), want_elig=True)
    got = fas.fas_prepass_readback(row_bound=True)
    check_key_sums_statistics(c, got, elig)
    out, lse = fas.fas_forward(c.q, c.k, c.v, mode="auto")
    assert fas.fas_status() == fas.FAS_OK
    c.check(out, lse, f"{name}/auto/key sums")


def test_outputs_are_bit_reproducible():
    """Dual baseline ("Proving the Pixels Didn't Change"): two runs of the
    same build on the same inputs must be identical."""
    c = case("mid")
    for mode in ("auto", "online"):
        _, o1, l1 = c.run(mode)
        o1, l1 = o1.clone(), l1.clone()
        _, o2, l2 = c.run(mode)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_argument_and_order_errors():
    c = case("tiny")
    c.plan()
    lib = fas.load()
    st = torch.cuda.current_stream().cuda_stream
    lse = torch.empty(c.w.heads, c.w.tokens, device="cuda")
    out = torch.empty_like(c.q)
    # A different q than the one the prepass saw: state error.
    fas.fas_prepass(c.q, c.k)
    q2 = c.q.clone()
    assert lib.fas_forward(q2.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(), lse.data_ptr(), 0,
                           st) == fas.FAS_ERR_STATE
    # Online mode needs no prepass.
    assert lib.fas_forward(q2.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(), lse.data_ptr(), 1,
                           st) == fas.FAS_OK
    # Misaligned pointers.
    assert lib.fas_prepass(c.q.data_ptr() + 2, c.k.data_ptr(), st, None) == fas.FAS_ERR_ALIGN
    assert lib.fas_forward(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr() + 2, out.data_ptr(), lse.data_ptr(), 1,
                           st) == fas.FAS_ERR_ALIGN
    # Bad mode.
    assert lib.fas_forward(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(), lse.data_ptr(), 7,
                           st) == fas.FAS_ERR_ARG
    assert fas.fas_status() == fas.FAS_OK



def test_stale_bounds_are_reported():
    """q overwritten in place after the prepass (x32, exact in bf16): the
    pointer check cannot see it, the bounded rows' sums overflow and the next
    fas_status reports FAS_ERR_BOUND; a fresh prepass clears it, and AUTO
    then agrees with ONLINE on the new inputs."""
    c = case("mid")
    c.plan()
    q, k = c.q.clone(), c.k.clone()
    fas.fas_prepass(q, k)
    out, lse = fas.fas_forward(q, k, c.v, mode="auto")
    assert fas.fas_status() == fas.FAS_OK
    q.mul_(32)
    fas.fas_forward(q, k, c.v, mode="auto")
    assert fas.fas_status() == fas.FAS_ERR_BOUND
    assert fas.fas_status() == fas.FAS_OK  # the flag was cleared
    elig = fas.fas_prepass(q, k, want_elig=True)
    a_out, a_lse = fas.fas_forward(q, k, c.v, mode="auto")
    a_out, a_lse = a_out.float(), a_lse.clone()
    assert fas.fas_status() == fas.FAS_OK
    o_out, o_lse = fas.fas_forward(q, k, c.v, mode="online")
    assert fas.fas_status() == fas.FAS_OK
    assert elig.sum() < c.w.heads  # the scaled heads lost their eligibility
    assert (a_out - o_out.float()).abs().max().item() <= OUT_TOL
    assert (a_lse - o_lse).abs().max().item() <= LSE_TOL

def host_bf16(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("name,groups", [("tiny", [0, 1, 2]), ("mid", [0, 1, 5, 16])])
def test_forward_host_matches_device_path(name, groups):
    """fas_forward_host (host buffers, head groups pipelined over copy and
    compute streams) runs the same kernels per head as fas_prepass +
    fas_forward, so its outputs must be bit-identical, for any group size,
    and within tolerance of the oracle."""
    c = case(name)
    hq, hk, hv = (host_bf16(c.x[t]) for t in "qkv")
    for mode in ("auto", "online"):
        _, out_d, lse_d = c.run(mode)
        out_d, lse_d = out_d.cpu(), lse_d.cpu()
        for hg in groups:
            out_h, lse_h = fas.fas_forward_host(hq, hk, hv, mode=mode, heads_per_group=hg)
            torch.cuda.current_stream().synchronize()
            assert fas.fas_status() == fas.FAS_OK
            assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16)), (name, mode, hg)
            assert torch.equal(lse_h.view(torch.int32), lse_d.view(torch.int32)), (name, mode, hg)
        c.check(out_h, lse_h, f"{name}/{mode}/host")


def test_forward_host_720p_sampled_rows():
    """The host-buffer path on the full 720p SR chunk, as the benchmark's
    end-to-end measurement runs it (default head groups), against the
    oracle on sampled rows; eligibility read back afterwards."""
    c = case("720p")
    c.plan()
    hq, hk, hv = (host_bf16(c.x[t]) for t in "qkv")
    out_h, lse_h = fas.fas_forward_host(hq, hk, hv, mode="auto")
    torch.cuda.current_stream().synchronize()
    assert fas.fas_status() == fas.FAS_OK
    c.check(out_h, lse_h, "720p/host")
    want = np.ones(c.w.heads, dtype=bool)
    want[c.x["modified_heads"]] = False
    assert np.array_equal(fas.fas_prepass_readback()["elig"].astype(bool), want)


def test_forward_host_argument_errors():
    c = case("tiny")
    c.plan()
    lib = fas.load()
    st = torch.cuda.current_stream().cuda_stream
    hq = host_bf16(c.x["q"])
    out = torch.empty(hq.shape, dtype=torch.bfloat16, pin_memory=True)
    lse = torch.empty(c.w.heads, c.w.tokens, dtype=torch.float32, pin_memory=True)
    p = [hq.data_ptr()] * 3 + [out.data_ptr(), lse.data_ptr()]
    assert lib.fas_forward_host(*p, 0, c.w.heads + 1, st) == fas.FAS_ERR_ARG
    assert lib.fas_forward_host(*p, 0, -1, st) == fas.FAS_ERR_ARG
    assert lib.fas_forward_host(*p, 9, 0, st) == fas.FAS_ERR_ARG
    assert lib.fas_forward_host(None, *p[1:], 0, 0, st) == fas.FAS_ERR_ARG
    with pytest.raises(TypeError):
        fas.fas_forward_host(c.q, c.k, c.v)  # device tensors are refused


def to_nhd(bits):
    """[H, N, d] bf16 bits -> contiguous [N, H, d]."""
    return np.ascontiguousarray(bits.transpose(1, 0, 2))


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_token_major_layout_matches_head_major(name):
    """q, k, v, out as [N, H, d] (fas_set_layout nhd): the kernels read and
    write the strided layout directly, so the results must be bit-identical
    to the head-major path on the same data, through both the device and
    the host-buffer entry points."""
    c = case(name)
    qn, kn, vn = (to_dev(to_nhd(c.x[t])) for t in "qkv")
    for mode in ("auto", "online"):
        elig_h, out_h, lse_h = c.run(mode)
        out_h, lse_h = out_h.cpu(), lse_h.cpu()
        fas.fas_set_layout("nhd")
        elig_n = fas.fas_prepass(qn, kn, want_elig=True)
        out_n, lse_n = fas.fas_forward(qn, kn, vn, mode=mode)
        assert fas.fas_status() == fas.FAS_OK
        assert out_n.shape == (c.w.tokens, c.w.heads, c.w.head_dim)
        assert np.array_equal(elig_n, elig_h)
        assert torch.equal(out_n.cpu().transpose(0, 1).contiguous().view(torch.int16), out_h.view(torch.int16))
        assert torch.equal(lse_n.cpu().view(torch.int32), lse_h.view(torch.int32))
        hq, hk, hv = (host_bf16(to_nhd(c.x[t])) for t in "qkv")
        for hg in (0, 1):
            o2, l2 = fas.fas_forward_host(hq, hk, hv, mode=mode, heads_per_group=hg)
            torch.cuda.current_stream().synchronize()
            assert fas.fas_status() == fas.FAS_OK
            assert torch.equal(o2.transpose(0, 1).contiguous().view(torch.int16), out_h.view(torch.int16)), hg
            assert torch.equal(l2.view(torch.int32), lse_h.view(torch.int32)), hg
        fas.fas_set_layout("hnd")
    c.check(out_n.cpu().transpose(0, 1).contiguous(), lse_n, f"{name}/nhd")


def test_token_major_layout_720p_sampled_rows():
    """The token-major layout on the full 720p SR chunk against the oracle."""
    c = case("720p")
    c.plan()
    fas.fas_set_layout("nhd")
    try:
        qn, kn, vn = (to_dev(to_nhd(c.x[t])) for t in "qkv")
        elig = fas.fas_prepass(qn, kn, want_elig=True)
        want = np.ones(c.w.heads, dtype=bool)
        want[c.x["modified_heads"]] = False
        assert np.array_equal(elig.astype(bool), want)
        out, lse = fas.fas_forward(qn, kn, vn, mode="auto")
        assert fas.fas_status() == fas.FAS_OK
        c.check(out.transpose(0, 1).contiguous(), lse, "720p/nhd")
    finally:
        fas.fas_set_layout("hnd")


def test_layout_errors():
    c = case("tiny")
    c.plan()
    lib = fas.load()
    assert lib.fas_set_layout(2) == fas.FAS_ERR_ARG
    fas.fas_prepass(c.q, c.k)
    assert lib.fas_set_layout(1) == fas.FAS_OK
    st = torch.cuda.current_stream().cuda_stream
    out = torch.empty_like(c.q)
    lse = torch.empty(c.w.heads, c.w.tokens, device="cuda")
    # A layout change invalidates the prepass: AUTO needs a new one.
    assert lib.fas_forward(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(), lse.data_ptr(), 0,
                           st) == fas.FAS_ERR_STATE
    assert lib.fas_set_layout(0) == fas.FAS_OK
    fas.fas_set_layout("hnd")


def test_forward_host_back_to_back_calls():
    """Consecutive fas_forward_host calls overlap on the library's streams
    (one call's copy-in under the previous call's last head groups), with
    per-group ordering on the shared device copies.  Three calls on two
    different inputs, with no synchronisation in between, must each give
    the device path's result for their own inputs."""
    c = case("mid")
    c.plan()
    xa = c.x
    xb = {t: xa[t][::-1].copy() for t in "qkv"}  # heads in reverse order: other data per head
    ha = [host_bf16(xa[t]) for t in "qkv"]
    hb = [host_bf16(xb[t]) for t in "qkv"]
    outs = []
    for h in (ha, hb, ha):
        outs.append(fas.fas_forward_host(*h, mode="auto"))
    torch.cuda.current_stream().synchronize()
    assert fas.fas_status() == fas.FAS_OK
    for x, (o, l) in zip((xa, xb, xa), outs):
        q, k, v = (to_dev(x[t]) for t in "qkv")
        fas.fas_prepass(q, k)
        od, ld = fas.fas_forward(q, k, v, mode="auto")
        assert fas.fas_status() == fas.FAS_OK
        assert torch.equal(o.view(torch.int16), od.cpu().view(torch.int16))
        assert torch.equal(l.view(torch.int32), ld.cpu().view(torch.int32))


# Frames of different spans (a ragged block table): per-frame spans that
# share a block size, query tiles clipped at each frame's own end.
RAGGED = [
    # name, H, d, R0, spans, r, sigma, seed
    ("ragged_small", 2, 64, 1, [48, 32, 64, 16, 48, 80], 1, 2.0, 51),
    ("ragged_mid", 3, 128, 1, [880, 720, 1040, 880, 560, 880, 1200], 2, 3.0, 52),
    ("ragged_two_refs", 2, 128, 2, [208, 144, 272, 208, 336, 160], 1, 3.0, 53),
    ("ragged_no_reference", 2, 128, 0, [288, 144, 432, 288, 96], 1, 3.0, 54),
]


def ragged_inputs(H, d, spans, sigma, seed):
    """Seeded bf16 q, k, v for a ragged geometry: draw as for a uniform
    workload with the same total token count."""
    N = sum(spans)
    w = workloads.Workload("ragged", H, d, 0, 1, N, 0, sigma, seed)  # one frame of N tokens: only the draws
    return workloads.generate(w)


@pytest.mark.parametrize("spec", RAGGED, ids=[e[0] for e in RAGGED])
def test_ragged_frames_full_rows(spec):
    name, H, d, R0, spans, r, sigma, seed = spec
    F = len(spans) - R0
    x = ragged_inputs(H, d, spans, sigma, seed)
    q, k, v = (to_dev(x[t]) for t in "qkv")
    info = fas.fas_plan(spans, F, R0, r, H, d)
    assert info.visible_flops == ref.visible_flops(H, d, spans, F, R0, r)
    want = ref.masked_attention(x["q"], x["k"], x["v"], spans, R0, r)
    st = ref.bound_statistics(x["q"], x["k"], spans, R0, r)
    elig = fas.fas_prepass(q, k, want_elig=True)
    assert np.array_equal(elig.astype(bool), st["elig"])
    got = fas.fas_prepass_readback(row_bound=True)
    np.testing.assert_allclose(got["frame_max"], st["M"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["row_bound"], st["m"], rtol=1e-4, atol=1e-3)
    for mode in ("auto", "online", "bounded"):
        out, lse = fas.fas_forward(q, k, v, mode=mode)
        assert fas.fas_status() == fas.FAS_OK
        o, l = out.float().cpu().numpy(), lse.cpu().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), (name, mode)
        assert np.abs(o - want["out"]).max() <= OUT_TOL, (name, mode)
        assert np.abs(l - want["lse"]).max() <= LSE_TOL, (name, mode)
    fas.fas_free()


def test_ragged_frames_key_sums_token_major():
    """The prepass fed the key sums on ragged frames (its key items cut at
    16-token boundaries of every frame) with q, k token-major."""
    name, H, d, R0, spans, r, sigma, seed = RAGGED[1]
    F = len(spans) - R0
    x = ragged_inputs(H, d, spans, sigma, seed)
    st = ref.bound_statistics(x["q"], x["k"], spans, R0, r)
    fas.fas_plan(spans, F, R0, r, H, d)
    fas.fas_set_layout("nhd")
    try:
        q, k = (to_dev(to_nhd(x[t])) for t in "qk")
        elig = fas.fas_prepass_with_key_sums(q, k, key_sums_of(x["k"]), want_elig=True)
        got = fas.fas_prepass_readback(row_bound=True)
    finally:
        fas.fas_set_layout("hnd")
        fas.fas_free()
    assert np.array_equal(elig.astype(bool), st["elig"])
    np.testing.assert_allclose(got["mu"], st["mu"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["frame_max"], st["M"], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(got["row_bound"], st["m"], rtol=1e-4, atol=1e-3)


def test_ragged_frames_token_major_and_host_path():
    """A ragged plan through the token-major layout and the host-buffer
    entry point gives the head-major device path's bits."""
    name, H, d, R0, spans, r, sigma, seed = RAGGED[1]
    F = len(spans) - R0
    x = ragged_inputs(H, d, spans, sigma, seed)
    fas.fas_plan(spans, F, R0, r, H, d)
    q, k, v = (to_dev(x[t]) for t in "qkv")
    fas.fas_prepass(q, k)
    out_h, lse_h = fas.fas_forward(q, k, v, mode="auto")
    out_h, lse_h = out_h.cpu(), lse_h.cpu()
    fas.fas_set_layout("nhd")
    qn, kn, vn = (to_dev(to_nhd(x[t])) for t in "qkv")
    fas.fas_prepass(qn, kn)
    out_n, lse_n = fas.fas_forward(qn, kn, vn, mode="auto")
    assert fas.fas_status() == fas.FAS_OK
    assert torch.equal(out_n.cpu().transpose(0, 1).contiguous().view(torch.int16), out_h.view(torch.int16))
    assert torch.equal(lse_n.cpu().view(torch.int32), lse_h.view(torch.int32))
    fas.fas_set_layout("hnd")
    o2, l2 = fas.fas_forward_host(*(host_bf16(x[t]) for t in "qkv"), mode="auto")
    torch.cuda.current_stream().synchronize()
    assert fas.fas_status() == fas.FAS_OK
    assert torch.equal(o2.view(torch.int16), out_h.view(torch.int16))
    assert torch.equal(l2.view(torch.int32), lse_h.view(torch.int32))
    fas.fas_free()


@pytest.mark.parametrize("name", ["tiny", "mid", "720p"])
def test_splash_ablation_matches_oracle(name):
    """The splash-style ablation (128-multiple tiles over the padded
    sequence, mask predicates, window and reference passes merged from fp32
    intermediates) computes the same attention: within tolerance of the
    oracle, and of the frame-aligned kernel's online path."""
    c = case(name)
    c.plan()
    out, lse = fas.fas_forward_ablation(c.q, c.k, c.v)
    assert fas.fas_status() == fas.FAS_OK
    assert fas.fas_last_launch_count() == 3
    c.check(out, lse, f"{name}/ablation")
    # Every row (the oracle check samples the large workloads): each kernel
    # is within the tolerance of the exact result, so the two are within
    # twice it of each other.
    _, out_o, lse_o = c.run("online")
    assert (out.float() - out_o.float()).abs().max().item() <= 2 * OUT_TOL
    assert (lse - lse_o).abs().max().item() <= 2 * LSE_TOL


@pytest.mark.parametrize("spec", [e for e in EDGE if e[0] in ("no_reference", "two_references", "T16_r0",
                                                             "d64_wide_window")], ids=lambda e: e[0])
def test_splash_ablation_edge_geometries(spec):
    name, H, d, R0, F, T, r, sigma, seed, bk = spec
    c = Case(workloads.Workload(name, H, d, R0, F, T, r, sigma, seed))
    c.plan()
    out, lse = fas.fas_forward_ablation(c.q, c.k, c.v)
    assert fas.fas_status() == fas.FAS_OK
    assert fas.fas_last_launch_count() == (2 if R0 == 0 else 3)
    c.check(out, lse, f"{name}/ablation")


def test_splash_ablation_refuses_what_it_does_not_cover():
    c = case("tiny")
    c.plan()
    lib = fas.load()
    st = torch.cuda.current_stream().cuda_stream
    out = torch.empty_like(c.q)
    lse = torch.empty(c.w.heads, c.w.tokens, device="cuda")
    fas.fas_set_layout("nhd")
    assert lib.fas_forward_ablation(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), st) == fas.FAS_ERR_UNSUPPORTED
    fas.fas_set_layout("hnd")
    fas.fas_plan([48, 32, 64], 2, 1, 1, 1, 64)
    assert lib.fas_forward_ablation(c.q.data_ptr(), c.k.data_ptr(), c.v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), st) == fas.FAS_ERR_UNSUPPORTED
    fas.fas_free()
