"""GPU parity of the attention prologue ("Layout Is the ABI", Fig. 5).

fas_prologue fuses RMSNorm, the QKV projection (tcgen05), the rotary
embedding and head packing; fas_prologue_fold_weights folds the norm scale
into the weight once.  Checks, all against CPU definitions:

* the folded weight is bit-exact against bf16(W * gamma) computed on the CPU;
* q, k, v against the fp64 oracle (unfolded weight) within a bound derived
  from the arithmetic: the folded weight's bf16 rounding (at most 2^-8
  relative per element, about 2^-8/sqrt(3) x sqrt(sum_c (xh_c W_oc)^2) per
  output, ~2.3e-3 for these N(0, 1/C) weights; 8 sigma over 1e8 outputs is
  below 0.02) plus the output's own bf16 rounding (2^-8 relative);
* q, k, v against the oracle fed the CPU-folded weight (so only fp32
  accumulation and the output rounding remain): 2^-8 relative + 1e-3;
* the token-major and all-to-all layouts are the head-major result moved;
* the key sums (column sums of k over each 16 tokens) against the same
  sums of the oracle's k (per element the folded-weight bound above, added
  over the 16 rows, plus the fp32 addition's 2^-20 of their absolute sum),
  and against the k the kernel wrote (within that 2^-20);
* the chain prologue -> prepass -> attention on the Mid geometry, with the
  prepass reading k or taking the prologue's key sums, against the fp64
  oracle run on the oracle prologue's own q, k, v (CPU-folded weight,
  rounded to bf16).  The kernel's fp32 accumulation rounds an element to
  the neighbouring bf16 value now and then (an fp32 emulation of it on this
  workload: 1.7e-4 of the elements, moving the oracle's LSE by 2.7e-4 and
  out by 1.4e-4 on the rows checked), so LSE gets 1e-3 on top of the
  attention's own 1e-3; out keeps 2e-2; eligibility bit-exact.
"""
import numpy as np
import pytest
import torch

import frame_aligned_sparse_gb300 as fas
import workloads
from oracle import prologue as opro
from oracle import reference as ref

pytestmark = pytest.mark.gpu

REL = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from frame_aligned_sparse_gb300 import build
    build.build()
    yield fas.load()
    fas.fas_free()


def bf16_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def cpu_fold(w_bits, gamma):
    w = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).float()
    return (w * torch.from_numpy(gamma)[None, :]).to(torch.bfloat16)


class Inputs:
    def __init__(self, name):
        self.w = workloads.get(name)
        self.p = workloads.prologue_inputs(self.w)
        self.x = bf16_dev(self.p["x"])
        self.wt = bf16_dev(self.p["w"])
        self.gamma = torch.from_numpy(self.p["gamma"]).cuda()
        self.cos = torch.from_numpy(self.p["cos"]).cuda()
        self.sin = torch.from_numpy(self.p["sin"]).cuda()

    def run(self, layout="hnd", groups=1, ranks=1):
        wf = fas.fas_prologue_fold_weights(self.wt, self.gamma)
        out = fas.fas_prologue(self.x, wf, self.cos, self.sin, self.w.heads, self.w.head_dim, layout=layout,
                               groups=groups, ranks=ranks)
        torch.cuda.synchronize()
        return wf, out

    def run_sums(self, layout="hnd", groups=1, ranks=1):
        wf = fas.fas_prologue_fold_weights(self.wt, self.gamma)
        out = fas.fas_prologue_with_key_sums(self.x, wf, self.cos, self.sin, self.w.heads, self.w.head_dim,
                                             layout=layout, groups=groups, ranks=ranks)
        torch.cuda.synchronize()
        return out

    def oracle_folded(self, rows=None):
        """The oracle prologue with the CPU-folded weight (fp64 q, k, v)."""
        H, d = self.w.heads, self.w.head_dim
        folded = cpu_fold(self.p["w"], self.p["gamma"]).view(torch.int16).numpy().view(np.uint16)
        x, c, s = self.p["x"], self.p["cos"], self.p["sin"]
        if rows is not None:
            x, c, s = x[rows], c[rows], s[rows]
        return opro.qkv_prologue(x, np.ones_like(self.p["gamma"]), folded, c, s, H, d)


def check_close(got, want, atol, label):
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    bound = REL * np.abs(want) + atol
    assert np.all(np.isfinite(got)), label
    worst = np.max(err - bound)
    assert worst <= 0, (label, float(np.max(err)), float(worst))


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_prologue_matches_oracle_all_rows(name):
    c = Inputs(name)
    wf, (q, k, v) = c.run()
    # The fold kernel against the CPU definition, bit for bit.
    assert torch.equal(wf.cpu().view(torch.int16), cpu_fold(c.p["w"], c.p["gamma"]).view(torch.int16))
    H, d = c.w.heads, c.w.head_dim
    want = opro.qkv_prologue(c.p["x"], c.p["gamma"], c.p["w"], c.p["cos"], c.p["sin"], H, d)
    for t, r, label in zip((q, k, v), want, "qkv"):
        check_close(t, r, 0.02, f"{name}/{label}")
    folded = cpu_fold(c.p["w"], c.p["gamma"]).view(torch.int16).numpy().view(np.uint16)
    want_f = opro.qkv_prologue(c.p["x"], np.ones_like(c.p["gamma"]), folded, c.p["cos"], c.p["sin"], H, d)
    for t, r, label in zip((q, k, v), want_f, "qkv"):
        check_close(t, r, 1e-3, f"{name}/{label}/folded")


def test_prologue_720p_sampled_rows():
    """The full 720p geometry (79,200 tokens, C = 3072, 9216 output
    features), checked on sampled rows: every frame's first and last tokens,
    each 128-token panel's edges around frame boundaries, random rows."""
    c = Inputs("720p")
    _, (q, k, v) = c.run()
    T, N = c.w.frame_tokens, c.w.tokens
    rng = np.random.default_rng(0)
    rows = set(rng.choice(N, 600, replace=False).tolist())
    for f in range(c.w.total_frames):
        rows.update([f * T, f * T + T - 1])
    rows.update([127, 128, N - 1, N - 128])
    rows = np.array(sorted(rows))
    H, d = c.w.heads, c.w.head_dim
    want = opro.qkv_prologue(c.p["x"][rows], c.p["gamma"], c.p["w"], c.p["cos"][rows], c.p["sin"][rows], H, d)
    for t, r, label in zip((q, k, v), want, "qkv"):
        check_close(t[:, rows], r, 0.02, f"720p/{label}")


def test_prologue_layouts_move_the_same_values():
    c = Inputs("mid")
    _, ref_out = c.run("hnd")
    H, d, N = c.w.heads, c.w.head_dim, c.w.tokens
    _, nhd = c.run("nhd")
    for a, b in zip(ref_out, nhd):
        assert torch.equal(a.transpose(0, 1).contiguous().view(torch.int16), b.view(torch.int16))
    G, P = 2, 4
    _, a2a = c.run("a2a", groups=G, ranks=P)
    hp = H // (G * P)
    for a, b in zip(ref_out, a2a):
        assert b.shape == (G, P, N, hp, d)
        want = a.view(G, P, hp, N, d).permute(0, 1, 3, 2, 4)
        assert torch.equal(b.view(torch.int16), want.contiguous().view(torch.int16))


def sums16(t):
    """[H, N, d] -> column sums over each 16 tokens [H, N/16, d] (fp64)."""
    H, N, d = t.shape
    return t.reshape(H, N // 16, 16, d).sum(axis=2)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_prologue_key_sums(name):
    c = Inputs(name)
    H, d, N = c.w.heads, c.w.head_dim, c.w.tokens
    q, k, v, ks = c.run_sums()
    assert ks.shape == (H, N // 16, d)
    # q, k, v are those of the plain prologue, bit for bit.
    _, plain = c.run()
    for a, b in zip((q, k, v), plain):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    got = ks.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    # Against the oracle's k: each element within 2^-8 |k| + 1e-3.
    ko = c.oracle_folded()[1]
    bound = (REL + 2.0 ** -20) * sums16(np.abs(ko)) + 16 * 1e-3
    assert np.max(np.abs(got - sums16(ko)) - bound) <= 0
    # Against the k the kernel wrote: 16 values added in fp32.
    kw = k.float().cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - sums16(kw)) - 2.0 ** -20 * sums16(np.abs(kw))) <= 0
    # The sums do not depend on the layout q, k, v are written in.
    for layout, g, r in (("nhd", 1, 1), ("a2a", 2, 2)):
        if H % (g * r):
            continue
        ks2 = c.run_sums(layout, g, r)[3]
        assert torch.equal(ks2.view(torch.int32), ks.view(torch.int32)), layout


def test_prologue_key_sums_720p_sampled_groups():
    """The full 720p geometry: every group of two heads against the written k,
    and sampled 16-token groups (frame edges and random ones) of every head
    against the oracle."""
    c = Inputs("720p")
    H, d, N, T = c.w.heads, c.w.head_dim, c.w.tokens, c.w.frame_tokens
    q, k, v, ks = c.run_sums()
    got = ks.cpu().numpy().astype(np.float64)
    for h in (0, H - 1):
        kw = k[h].float().cpu().numpy().astype(np.float64)[None]
        assert np.max(np.abs(got[h:h + 1] - sums16(kw)) - 2.0 ** -20 * sums16(np.abs(kw))) <= 0, h
    rng = np.random.default_rng(1)
    groups = set(rng.choice(N // 16, 20, replace=False).tolist())
    for f in range(c.w.total_frames):
        groups.update([f * T // 16, (f + 1) * T // 16 - 1])
    groups = np.array(sorted(groups))
    rows = (groups[:, None] * 16 + np.arange(16)[None, :]).reshape(-1)
    ko = c.oracle_folded(rows)[1]  # [H, 16 * len(groups), d]
    bound = (REL + 2.0 ** -20) * sums16(np.abs(ko)) + 16 * 1e-3
    assert np.max(np.abs(got[:, groups] - sums16(ko)) - bound) <= 0


@pytest.mark.parametrize("sums", [False, True], ids=["prepass_reads_k", "key_sums_from_prologue"])
def test_prologue_then_attention_chain(sums):
    """x -> prologue -> prepass -> attention, token-major, against the
    oracle on the oracle prologue's q, k, v (see the module docstring for
    the tolerances)."""
    c = Inputs("mid")
    w = c.w
    if sums:
        q, k, v, ks = c.run_sums("nhd")
    else:
        _, (q, k, v) = c.run("nhd")
    fas.fas_plan(w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius, w.heads, w.head_dim)
    fas.fas_set_layout("nhd")
    if sums:
        elig = fas.fas_prepass_with_key_sums(q, k, ks, want_elig=True)
    else:
        elig = fas.fas_prepass(q, k, want_elig=True)
    out, lse = fas.fas_forward(q, k, v, mode="auto")
    assert fas.fas_status() == fas.FAS_OK
    fas.fas_set_layout("hnd")
    bits = {n: workloads.round_to_bf16_bits(t) for n, t in zip("qkv", c.oracle_folded())}
    st = ref.bound_statistics(bits["q"], bits["k"], w.frame_tokens, w.ref_frames, w.window_radius)
    assert np.array_equal(elig.astype(bool), st["elig"])
    rows = np.unique(np.concatenate([np.arange(0, w.tokens, 97), [w.tokens - 1]]))
    want = ref.masked_attention(bits["q"], bits["k"], bits["v"], w.frame_tokens, w.ref_frames, w.window_radius,
                                rows=rows)
    o = out.transpose(0, 1).float().cpu().numpy()[:, rows]
    assert np.abs(o - want["out"]).max() <= 2e-2
    assert np.abs(lse.cpu().numpy()[:, rows] - want["lse"]).max() <= 2e-3
    fas.fas_free()


def test_prologue_argument_errors():
    lib = fas.load()
    x = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(128, 32, dtype=torch.float32, device="cuda")
    w = torch.zeros(384, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(2 * 128 * 64, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    args = [x.data_ptr(), w.data_ptr(), t.data_ptr(), t.data_ptr()]
    o3 = [out.data_ptr()] * 3
    assert lib.fas_prologue(*args, 128, 96, 2, 64, 1e-6, *o3, 0, 1, 1, st) == fas.FAS_ERR_ARG   # width % 64
    assert lib.fas_prologue(*args, 128, 128, 1, 64, 1e-6, *o3, 0, 1, 1, st) == fas.FAS_ERR_ARG  # H*d % 128
    assert lib.fas_prologue(*args, 128, 128, 2, 96, 1e-6, *o3, 0, 1, 1, st) == fas.FAS_ERR_ARG  # d
    assert lib.fas_prologue(*args, 128, 128, 2, 64, 1e-6, *o3, 2, 1, 4, st) == fas.FAS_ERR_ARG  # a2a split
    assert lib.fas_prologue(*args, 128, 128, 2, 64, 1e-6, *o3, 7, 1, 1, st) == fas.FAS_ERR_ARG  # layout
    assert lib.fas_prologue(x.data_ptr() + 2, *args[1:], 128, 128, 2, 64, 1e-6, *o3, 0, 1, 1,
                            st) == fas.FAS_ERR_ALIGN
    ks = torch.zeros(2 * 8 * 64 + 4, dtype=torch.float32, device="cuda")
    assert lib.fas_prologue_with_key_sums(*args, 120, 128, 2, 64, 1e-6, *o3, 0, 1, 1, ks.data_ptr(),
                                          st) == fas.FAS_ERR_ARG  # tokens % 16
    assert lib.fas_prologue_with_key_sums(*args, 128, 128, 2, 64, 1e-6, *o3, 0, 1, 1, ks.data_ptr() + 8,
                                          st) == fas.FAS_ERR_ALIGN
    assert lib.fas_prologue_with_key_sums(*args, 128, 96, 2, 64, 1e-6, *o3, 0, 1, 1, ks.data_ptr(),
                                          st) == fas.FAS_ERR_ARG  # as fas_prologue


def test_ulysses_one_rank_with_the_library_kernels():
    """The head-grouped Ulysses schedule with the library's kernels as the
    attention, on a one-rank NCCL group (each box has one GPU): the prologue
    writes q, k, v in the all-to-all layout, every group's slab goes through
    NCCL's all-to-all, and the per-group attention (token-major, hp heads)
    gives bit for bit what one call over all heads gives."""
    import os
    import socket
    import torch.distributed as dist
    from frame_aligned_sparse_gb300 import ulysses

    c = Inputs("mid")
    w = c.w
    G = 4
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        _, (qa, ka, va) = c.run("a2a", groups=G, ranks=1)
        fn = ulysses.fas_attention_fn(w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius, w.heads // G,
                                      w.head_dim)
        out, lse = ulysses.ulysses_attention(qa, ka, va, fn)
        torch.cuda.synchronize()
        assert fas.fas_status() == fas.FAS_OK
        got = ulysses.from_a2a_layout(out)  # [N, H, d]
        _, (q, k, v) = c.run("nhd")
        fas.fas_plan(w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius, w.heads, w.head_dim)
        fas.fas_set_layout("nhd")
        fas.fas_prepass(q, k)
        want, want_lse = fas.fas_forward(q, k, v, mode="auto")
        assert fas.fas_status() == fas.FAS_OK
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        assert torch.equal(lse.reshape(w.heads, -1).view(torch.int32), want_lse.view(torch.int32))
    finally:
        fas.fas_set_layout("hnd")
        fas.fas_free()
        dist.destroy_process_group()
