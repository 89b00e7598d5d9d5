"""Pins for the fp64 oracle (CPU only).

Every check ties the oracle to something other than itself: a pure-Python
brute force written from the English rule, a closed form, an invariant that
holds in exact arithmetic, or a library routine (torch's
scaled_dot_product_attention in fp64).  The mutation tests at the end plant
plausible mistakes in the oracle (on the CPU) and show that a pin catches
each of them.

Passages: "HeyGen x Google Cloud: Avatar IV on TPU", sections "Deleting the
Mask" (window plus global reference, frame-aligned full blocks, single pass)
and "Unchaining the Softmax" (Cauchy-Schwarz bound, centring invariance,
per-row visible slices).
"""
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import reference as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent formulations (pure Python, written from the English rule).
# ---------------------------------------------------------------------------

def brute_sees(fi, fj, ref_frames, radius):
    """Frame fi sees frame fj: reference frames are global both ways, video
    frames see video frames within the radius."""
    reference = set(range(ref_frames))
    if fi in reference or fj in reference:
        return True
    return abs(fi - fj) <= radius


def brute_attention(q, k, v, T, R0, r, rows):
    """Triple loop with math.exp; q, k, v float64 [N, d] for one head."""
    N, d = len(q), len(q[0])
    s = 1.0 / math.sqrt(d)
    outs, lses, zmaxs = [], [], []
    for i in rows:
        logits = []
        for j in range(N):
            if brute_sees(i // T, j // T, R0, r):
                logits.append((j, s * sum(q[i][c] * k[j][c] for c in range(d))))
        zmax = max(z for _, z in logits)
        tot = sum(math.exp(z - zmax) for _, z in logits)
        out = [0.0] * d
        for j, z in logits:
            w = math.exp(z - zmax) / tot
            for c in range(d):
                out[c] += w * v[j][c]
        outs.append(out)
        lses.append(zmax + math.log(tot))
        zmaxs.append(zmax)
    return np.array(outs), np.array(lses), np.array(zmaxs)


def closed_form_frame_pairs(F, R0, r):
    """Visible (query frame, key frame) pairs in closed form.

    Reference rows see all R0+F frames; video rows see the R0 reference
    frames plus a window of 2r+1 video frames, shortened by 1..r frames at
    each end of the clip (r(r+1) in total) unless it covers every frame.
    """
    window = F * F if r >= F - 1 else F * (2 * r + 1) - r * (r + 1)
    return R0 * (R0 + F) + F * R0 + window


MICRO = [
    dict(H=2, d=4, R0=1, F=5, T=3, r=1, seed=11),
    dict(H=1, d=8, R0=2, F=4, T=2, r=0, seed=12),
    dict(H=1, d=4, R0=1, F=3, T=4, r=5, seed=13),
]


def micro_inputs(c, key_shift=0.0):
    rng = np.random.default_rng(c["seed"])
    N = (c["R0"] + c["F"]) * c["T"]
    q = rng.standard_normal((c["H"], N, c["d"]))
    k = rng.standard_normal((c["H"], N, c["d"])) + key_shift * rng.standard_normal((c["H"], 1, c["d"]))
    v = rng.standard_normal((c["H"], N, c["d"]))
    return q, k, v


# ---------------------------------------------------------------------------
# Checks (each takes the oracle module so mutation tests can re-run them).
# ---------------------------------------------------------------------------

def check_golden_frame_visibility(o):
    rows = [list(map(int, line.split())) for line in open(os.path.join(GOLDEN, "tiny_frame_visibility.txt"))
            if line.strip() and not line.startswith("#")]
    want = np.array(rows, dtype=bool)
    got = o.frame_visibility(9, 1, 1)
    assert np.array_equal(got, want)


def check_pair_counts(o):
    geos = [(w.n_frames, w.ref_frames, w.window_radius) for w in workloads.WORKLOADS.values()]
    geos += [(F, R0, r) for F in (1, 2, 3, 7) for R0 in (1, 2) for r in (0, 1, 2, 3, 9)]
    for F, R0, r in geos:
        assert o.visible_pairs(5, F, R0, r) == closed_form_frame_pairs(F, R0, r) * 25, (F, R0, r)
    # Explicit token mask agrees with the count.
    for F, R0, r in [(8, 1, 1), (4, 2, 0), (5, 1, 7)]:
        T = 4
        N = (R0 + F) * T
        assert o.token_mask(np.arange(N), N, T, R0, r).sum() == o.visible_pairs(T, F, R0, r)


def check_token_mask(o):
    for F, R0, r, T in [(8, 1, 1, 3), (4, 2, 0, 2), (5, 1, 2, 2), (3, 1, 9, 2), (6, 3, 1, 1)]:
        N = (R0 + F) * T
        got = o.token_mask(np.arange(N), N, T, R0, r)
        for i in range(N):
            for j in range(N):
                assert got[i, j] == brute_sees(i // T, j // T, R0, r), (F, R0, r, T, i, j)


def check_attention_brute(o):
    for c in MICRO:
        q, k, v = micro_inputs(c, key_shift=2.0)
        res = o.masked_attention(q, k, v, c["T"], c["R0"], c["r"])
        for h in range(c["H"]):
            out, lse, zmax = brute_attention(q[h].tolist(), k[h].tolist(), v[h].tolist(),
                                             c["T"], c["R0"], c["r"], range(q.shape[1]))
            np.testing.assert_allclose(res["out"][h], out, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(res["lse"][h], lse, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(res["zmax"][h], zmax, rtol=1e-12, atol=1e-12)
    # Tiny workload (bf16 inputs), a handful of rows spread over the frames.
    w = workloads.get("tiny")
    x = workloads.generate(w)
    rows = np.array([0, 47, 48, 95, 100, 150, 200, 239, 288, 335, 384, 431])
    res = o.masked_attention(x["q"], x["k"], x["v"], w.frame_tokens, w.ref_frames, w.window_radius,
                             rows=rows, heads=[1])
    q, k, v = (o.bf16_bits_to_f64(x[t][1]) for t in "qkv")
    out, lse, _ = brute_attention(q.tolist(), k.tolist(), v.tolist(), w.frame_tokens, w.ref_frames,
                                  w.window_radius, rows)
    np.testing.assert_allclose(res["out"][0], out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["lse"][0], lse, rtol=1e-12, atol=1e-12)


def check_full_window_is_sdpa(o):
    rng = np.random.default_rng(5)
    H, d, R0, F, T = 3, 16, 1, 6, 10
    N = (R0 + F) * T
    q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
    k += 3.0 * rng.standard_normal((H, 1, d))
    for r in (F - 1, F, 40):
        res = o.masked_attention(q, k, v, T, R0, r)
        tq, tk, tv = (torch.from_numpy(a)[None] for a in (q, k, v))
        want = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)[0].numpy()
        scores = torch.einsum("hnd,hmd->hnm", tq[0], tk[0]) / math.sqrt(d)
        want_lse = torch.logsumexp(scores, dim=-1).numpy()
        np.testing.assert_allclose(res["out"], want, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(res["lse"], want_lse, rtol=1e-12, atol=1e-12)


def check_centring_invariance(o):
    rng = np.random.default_rng(6)
    H, d, R0, F, T, r = 2, 8, 1, 6, 5, 1
    N = (R0 + F) * T
    q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
    shift = 4.0 * rng.standard_normal((H, 1, d))
    a = o.masked_attention(q, k, v, T, R0, r)
    b = o.masked_attention(q, k + shift, v, T, R0, r)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-11, atol=1e-12)
    delta = np.einsum("hnd,hd->hn", q, shift[:, 0]) / math.sqrt(d)
    np.testing.assert_allclose(b["lse"] - a["lse"], delta, rtol=1e-10, atol=1e-11)


def check_q_zero_closed_form(o):
    rng = np.random.default_rng(7)
    H, d, R0, F, T, r = 2, 8, 1, 7, 4, 2
    N = (R0 + F) * T
    q = np.zeros((H, N, d))
    k, v = (rng.standard_normal((H, N, d)) for _ in range(2))
    res = o.masked_attention(q, k, v, T, R0, r)
    for i in range(N):
        keys = [j for j in range(N) if brute_sees(i // T, j // T, R0, r)]
        np.testing.assert_allclose(res["lse"][:, i], math.log(len(keys)), rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["out"][:, i], v[:, keys].mean(axis=1), rtol=1e-12, atol=1e-13)


def check_invariants(o):
    rng = np.random.default_rng(8)
    H, d, R0, F, T, r = 2, 8, 1, 6, 6, 1
    N = (R0 + F) * T
    q, k, v = (2.0 * rng.standard_normal((H, N, d)) for _ in range(3))
    # V constant -> output constant.
    cv = np.broadcast_to(rng.standard_normal((H, 1, d)), (H, N, d)).copy()
    res = o.masked_attention(q, k, cv, T, R0, r)
    np.testing.assert_allclose(res["out"], np.broadcast_to(cv[:, :1], res["out"].shape), rtol=1e-12, atol=1e-12)
    # max z <= lse <= max z + ln(#visible keys).
    mask = o.token_mask(np.arange(N), N, T, R0, r)
    nvis = mask.sum(axis=1)
    assert np.all(res["lse"] >= res["zmax"] - 1e-12)
    assert np.all(res["lse"] <= res["zmax"] + np.log(nvis)[None, :] + 1e-12)
    # Permuting keys (with their values) inside a frame changes nothing.
    perm = np.arange(N)
    for g in range(R0 + F):
        perm[g * T:(g + 1) * T] = g * T + rng.permutation(T)
    a = o.masked_attention(q, k, v, T, R0, r)
    b = o.masked_attention(q, k[:, perm], v[:, perm], T, R0, r)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-12, atol=1e-12)


def check_block_sparse(o):
    """An fp64 online-softmax loop over frame-aligned key blocks (block size
    dividing the frame span, every block fully inside the live region) gives
    the dense masked result."""
    for (H, d, R0, F, T, r, B) in [(2, 8, 1, 8, 12, 1, 4), (1, 16, 1, 5, 48, 2, 16), (1, 4, 2, 4, 6, 0, 3)]:
        rng = np.random.default_rng(9 + T)
        N = (R0 + F) * T
        q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
        k += 2.0 * rng.standard_normal((H, 1, d))
        res = o.masked_attention(q, k, v, T, R0, r)
        s = 1.0 / math.sqrt(d)
        for h in range(H):
            for f in range(R0 + F):
                frames = [g for g in range(R0 + F) if brute_sees(f, g, R0, r)]
                rows = np.arange(f * T, (f + 1) * T)
                m = np.full(T, -np.inf)
                l = np.zeros(T)
                acc = np.zeros((T, d))
                for g in frames:
                    for b0 in range(g * T, (g + 1) * T, B):
                        z = s * q[h, rows] @ k[h, b0:b0 + B].T
                        m_new = np.maximum(m, z.max(axis=1))
                        alpha = np.exp(m - m_new)
                        p = np.exp(z - m_new[:, None])
                        l = alpha * l + p.sum(axis=1)
                        acc = alpha[:, None] * acc + p @ v[h, b0:b0 + B]
                        m = m_new
                np.testing.assert_allclose(acc / l[:, None], res["out"][h, rows], rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(m + np.log(l), res["lse"][h, rows], rtol=1e-12, atol=1e-12)


def check_two_pass_merge(o):
    """Window pass and reference pass merged by their LSEs equal one pass."""
    rng = np.random.default_rng(10)
    H, d, R0, F, T, r = 2, 8, 1, 7, 5, 2
    N = (R0 + F) * T
    q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
    res = o.masked_attention(q, k, v, T, R0, r)
    s = 1.0 / math.sqrt(d)

    def one_pass(h, i, keys):
        z = s * (k[h, keys] @ q[h, i])
        lse = np.log(np.exp(z - z.max()).sum()) + z.max()
        return np.exp(z - lse) @ v[h, keys], lse

    for h in range(H):
        for i in range(R0 * T, N):
            f = i // T
            win = [j for j in range(R0 * T, N) if abs(j // T - f) <= r]
            refk = list(range(R0 * T))
            oa, la = one_pass(h, i, win)
            ob, lb = one_pass(h, i, refk)
            lse = np.logaddexp(la, lb)
            out = np.exp(la - lse) * oa + np.exp(lb - lse) * ob
            np.testing.assert_allclose(out, res["out"][h, i], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse, res["lse"][h, i], rtol=1e-12, atol=1e-12)


def check_bound_stats_brute(o):
    for c in MICRO:
        q, k, _ = micro_inputs(c, key_shift=3.0)
        T, R0, r = c["T"], c["R0"], c["r"]
        N, d = q.shape[1], q.shape[2]
        nf = N // T
        s = 1.0 / math.sqrt(d)
        st = o.bound_statistics(q, k, T, R0, r)
        for h in range(c["H"]):
            kk = k[h].tolist()
            mu = [sum(kk[j][cc] for j in range(N)) / N for cc in range(d)]
            cnorm = [math.sqrt(sum((kk[j][cc] - mu[cc]) ** 2 for cc in range(d))) for j in range(N)]
            M = [max(cnorm[g * T:(g + 1) * T]) for g in range(nf)]
            np.testing.assert_allclose(st["mu"][h], mu, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(st["M"][h], M, rtol=1e-12, atol=1e-13)
            for i in range(N):
                f = i // T
                keys = [j for j in range(N) if brute_sees(f, j // T, R0, r)]
                mvis = max(cnorm[j] for j in keys)
                kbar = [sum(kk[j][cc] for j in keys) / len(keys) - mu[cc] for cc in range(d)]
                qi = q[h, i].tolist()
                qn = math.sqrt(sum(x * x for x in qi))
                b = s * qn * mvis
                G = b - s * sum(qi[cc] * kbar[cc] for cc in range(d))
                cshift = s * sum(qi[cc] * mu[cc] for cc in range(d))
                assert abs(st["b"][h, i] - b) < 1e-11
                assert abs(st["G"][h, i] - G) < 1e-11
                assert abs(st["m"][h, i] - (cshift + b)) < 1e-11
            assert abs(st["stat"][h] - st["G"][h].max()) == 0.0
            assert st["elig"][h] == (st["stat"][h] <= 32.0)


def check_bound_holds(o, st=None, res=None, q=None, k=None, T=None, R0=None, r=None):
    """Cauchy-Schwarz: m_i >= true row max; G_i >= b_i - true centred max >= 0."""
    if st is None:
        st = o.bound_statistics(q, k, T, R0, r)
    if res is None:
        res = o.masked_attention(q, k, k, T, R0, r)
    zc = res["zmax"] - st["c"]          # true centred row maximum
    assert np.all(st["m"] >= res["zmax"] - 1e-9)
    assert np.all(st["b"] >= zc - 1e-9)
    assert np.all(st["G"] >= st["b"] - zc - 1e-9)
    assert np.all(st["G"] >= -1e-9)


def check_bound_on_inputs(o):
    for c in MICRO:
        q, k, _ = micro_inputs(c, key_shift=3.0)
        check_bound_holds(o, q=q, k=k, T=c["T"], R0=c["R0"], r=c["r"])
    w = workloads.get("tiny")
    x = workloads.generate(w, tensors=("q", "k"))
    check_bound_holds(o, q=x["q"], k=x["k"], T=w.frame_tokens, R0=w.ref_frames, r=w.window_radius)
    # Heavy-tailed keys with outliers (small synthetic case).
    rng = np.random.default_rng(21)
    H, d, R0, F, T, r = 2, 16, 1, 6, 20, 1
    N = (R0 + F) * T
    q = 8.0 * rng.standard_normal((H, N, d))
    k = rng.standard_t(3, (H, N, d)) + 3.0 * rng.standard_normal((H, 1, d))
    k[:, ::17] *= 4.0
    check_bound_holds(o, q=q, k=k, T=T, R0=R0, r=r)


# ---------------------------------------------------------------------------
# Frames of different spans (a ragged block table): the same rule over
# frames, with token j in the frame whose token range holds it.
# ---------------------------------------------------------------------------

def brute_frame(j, spans):
    """Frame of token j, by walking the frames' token ranges."""
    start = 0
    for g, t in enumerate(spans):
        if start <= j < start + t:
            return g
        start += t
    raise IndexError(j)


RAGGED = [
    dict(H=2, d=4, R0=1, spans=[3, 2, 5, 1, 4, 2], r=1, seed=41),
    dict(H=1, d=8, R0=2, spans=[2, 4, 1, 3, 3, 2], r=0, seed=42),
    dict(H=1, d=4, R0=0, spans=[4, 1, 2, 6, 3], r=2, seed=43),
    dict(H=1, d=4, R0=1, spans=[5, 2, 3, 1], r=9, seed=44),
]


def ragged_inputs(c, key_shift=3.0):
    rng = np.random.default_rng(c["seed"])
    N = sum(c["spans"])
    q = rng.standard_normal((c["H"], N, c["d"]))
    k = rng.standard_normal((c["H"], N, c["d"])) + key_shift * rng.standard_normal((c["H"], 1, c["d"]))
    v = rng.standard_normal((c["H"], N, c["d"]))
    return q, k, v


def brute_attention_ragged(q, k, v, spans, R0, r):
    N, d = len(q), len(q[0])
    s = 1.0 / math.sqrt(d)
    outs, lses = [], []
    for i in range(N):
        logits = [(j, s * sum(q[i][c] * k[j][c] for c in range(d))) for j in range(N)
                  if brute_sees(brute_frame(i, spans), brute_frame(j, spans), R0, r)]
        zmax = max(z for _, z in logits)
        tot = sum(math.exp(z - zmax) for _, z in logits)
        out = [sum(math.exp(z - zmax) / tot * v[j][c] for j, z in logits) for c in range(d)]
        outs.append(out)
        lses.append(zmax + math.log(tot))
    return np.array(outs), np.array(lses)


def check_ragged_token_mask(o):
    for c in RAGGED:
        spans, N = c["spans"], sum(c["spans"])
        F = len(spans) - c["R0"]
        got = o.token_mask(np.arange(N), N, spans, c["R0"], c["r"])
        for i in range(N):
            for j in range(N):
                want = brute_sees(brute_frame(i, spans), brute_frame(j, spans), c["R0"], c["r"])
                assert got[i, j] == want, (c, i, j)
        assert got.sum() == o.visible_pairs(spans, F, c["R0"], c["r"])


def check_ragged_attention_brute(o):
    for c in RAGGED:
        q, k, v = ragged_inputs(c)
        res = o.masked_attention(q, k, v, c["spans"], c["R0"], c["r"])
        for h in range(c["H"]):
            out, lse = brute_attention_ragged(q[h].tolist(), k[h].tolist(), v[h].tolist(), c["spans"], c["R0"],
                                              c["r"])
            np.testing.assert_allclose(res["out"][h], out, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(res["lse"][h], lse, rtol=1e-12, atol=1e-12)


def check_ragged_bound_stats_brute(o):
    for c in RAGGED:
        q, k, _ = ragged_inputs(c)
        spans, R0, r = c["spans"], c["R0"], c["r"]
        N, d = q.shape[1], q.shape[2]
        s = 1.0 / math.sqrt(d)
        st = o.bound_statistics(q, k, spans, R0, r)
        for h in range(c["H"]):
            kk = k[h].tolist()
            mu = [sum(kk[j][cc] for j in range(N)) / N for cc in range(d)]
            cnorm = [math.sqrt(sum((kk[j][cc] - mu[cc]) ** 2 for cc in range(d))) for j in range(N)]
            M = [max(cnorm[j] for j in range(N) if brute_frame(j, spans) == g) for g in range(len(spans))]
            np.testing.assert_allclose(st["M"][h], M, rtol=1e-12, atol=1e-13)
            for i in range(N):
                f = brute_frame(i, spans)
                keys = [j for j in range(N) if brute_sees(f, brute_frame(j, spans), R0, r)]
                kbar = [sum(kk[j][cc] for j in keys) / len(keys) - mu[cc] for cc in range(d)]
                qi = q[h, i].tolist()
                b = s * math.sqrt(sum(x * x for x in qi)) * max(cnorm[j] for j in keys)
                G = b - s * sum(qi[cc] * kbar[cc] for cc in range(d))
                assert abs(st["b"][h, i] - b) < 1e-11
                assert abs(st["G"][h, i] - G) < 1e-11
        check_bound_holds(o, st=st, res=o.masked_attention(q, k, k, spans, R0, r))


def check_ragged_equal_spans_reduce_to_uniform(o):
    """A list of equal spans is the uniform geometry: same mask, same
    attention, same bound statistics, and the closed-form pair count."""
    rng = np.random.default_rng(45)
    H, d, R0, F, T, r = 2, 8, 1, 6, 5, 1
    N = (R0 + F) * T
    q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
    spans = [T] * (R0 + F)
    a = o.masked_attention(q, k, v, T, R0, r)
    b = o.masked_attention(q, k, v, spans, R0, r)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["lse"], b["lse"])
    sa, sb = o.bound_statistics(q, k, T, R0, r), o.bound_statistics(q, k, spans, R0, r)
    for name in ("M", "m", "G", "stat"):
        np.testing.assert_allclose(sa[name], sb[name], rtol=1e-14, atol=1e-14)
    assert o.visible_pairs(spans, F, R0, r) == closed_form_frame_pairs(F, R0, r) * T * T


def check_ragged_block_sparse(o):
    """Blocks of a size dividing every frame's span never straddle a frame:
    an fp64 online-softmax loop over the visible frames' blocks gives the
    dense masked result."""
    for spans, R0, r, B in [([12, 4, 8, 16, 4, 8], 1, 1, 4), ([6, 9, 3, 12], 1, 0, 3)]:
        rng = np.random.default_rng(46 + B)
        H, d = 1, 8
        N = sum(spans)
        q, k, v = (rng.standard_normal((H, N, d)) for _ in range(3))
        res = o.masked_attention(q, k, v, spans, R0, r)
        s = 1.0 / math.sqrt(d)
        starts = np.concatenate([[0], np.cumsum(spans)])
        for f in range(len(spans)):
            rows = np.arange(starts[f], starts[f + 1])
            m, l, acc = np.full(len(rows), -np.inf), np.zeros(len(rows)), np.zeros((len(rows), d))
            for g in range(len(spans)):
                if not brute_sees(f, g, R0, r):
                    continue
                for b0 in range(starts[g], starts[g + 1], B):
                    z = s * q[0, rows] @ k[0, b0:b0 + B].T
                    m_new = np.maximum(m, z.max(axis=1))
                    alpha = np.exp(m - m_new)
                    p = np.exp(z - m_new[:, None])
                    l = alpha * l + p.sum(axis=1)
                    acc = alpha[:, None] * acc + p @ v[0, b0:b0 + B]
                    m = m_new
            np.testing.assert_allclose(acc / l[:, None], res["out"][0, rows], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(m + np.log(l), res["lse"][0, rows], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# The pins.
# ---------------------------------------------------------------------------

CHECKS = [check_golden_frame_visibility, check_pair_counts, check_token_mask, check_attention_brute,
          check_full_window_is_sdpa, check_centring_invariance, check_q_zero_closed_form, check_invariants,
          check_block_sparse, check_two_pass_merge, check_bound_stats_brute, check_bound_on_inputs,
          check_ragged_token_mask, check_ragged_attention_brute, check_ragged_bound_stats_brute,
          check_ragged_equal_spans_reduce_to_uniform, check_ragged_block_sparse]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ref)


def test_bound_on_mid_sampled_rows():
    w = workloads.get("mid")
    x = workloads.generate(w, tensors=("q", "k"), heads=[0, 7])
    T = w.frame_tokens
    rows = np.concatenate([f * T + np.array([0, 1, T // 2, T - 1]) for f in range(w.total_frames)])
    st = ref.bound_statistics(x["q"], x["k"], T, w.ref_frames, w.window_radius)
    res = ref.masked_attention(x["q"], x["k"], x["k"], T, w.ref_frames, w.window_radius, rows=rows)
    sub = {name: st[name][:, rows] for name in ("c", "b", "m", "G")}
    check_bound_holds(ref, st=sub, res=res)


VISIBLE_FLOPS_TFLOP = {"tiny": 4.6e-5, "mid": 0.679, "720p": 22.61, "1080p": 52.37, "stress": 22.61, "dense": 77.08,
                       "720p_h4": 22.61 * 4 / 24, "720p_f5": 4.778}


def test_visible_flops_per_workload():
    for name, w in workloads.WORKLOADS.items():
        pairs = closed_form_frame_pairs(w.n_frames, w.ref_frames, w.window_radius)
        want = 4.0 * w.head_dim * w.heads * pairs * w.frame_tokens ** 2
        got = ref.visible_flops(w.heads, w.head_dim, w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius)
        assert got == want
        assert abs(got / 1e12 - VISIBLE_FLOPS_TFLOP[name]) / VISIBLE_FLOPS_TFLOP[name] < 0.01


# Eligibility: the workloads are built so that exactly the modified heads
# have a loose bound ("Unchaining the Softmax": heads whose bound is too loose
# fall back to the online path).  Margins of at least one nat on both sides
# of the threshold keep float32 and float64 decisions identical.
@pytest.mark.parametrize("name", ["tiny", "mid", "720p", "1080p", "stress", "dense"])
def test_eligibility_pattern(name):
    w = workloads.get(name)
    x = workloads.generate(w, tensors=("q", "k"))
    st = ref.bound_statistics(x["q"], x["k"], w.frame_tokens, w.ref_frames, w.window_radius)
    want = np.ones(w.heads, dtype=bool)
    want[x["modified_heads"]] = False
    assert np.array_equal(st["elig"], want)
    assert np.min(np.abs(st["stat"] - ref.ELIG_SLACK_NATS)) >= 1.0


def test_workload_generator_is_deterministic_per_head():
    w = workloads.get("720p")
    a = workloads.generate(w, tensors=("k",), heads=[5])
    b = workloads.generate(w, tensors=("q", "k"), heads=[3, 5])
    assert np.array_equal(a["k"][0], b["k"][1])
    assert list(a["modified_heads"]) == [5, 13]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3], dtype=np.float32)
    bits = workloads.round_to_bf16_bits(x)
    back = ref.bf16_bits_to_f64(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even mantissa (1.0);
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6 -> 1 + 2^-6.
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2 ** -6 and back[3] == 1.0
    assert back[4] == -2.5
    assert abs(back[5] - 3.0e-3) <= 3.0e-3 * 2 ** -8
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


# ---------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail.
# ---------------------------------------------------------------------------

def _fails(check):
    try:
        check(ref)
    except AssertionError:
        return True
    return False


def test_planted_window_off_by_one(monkeypatch):
    orig = ref.token_mask

    def bad(rows, n_tokens, frame_tokens, ref_frames, radius):
        return orig(rows, n_tokens, frame_tokens, ref_frames, max(radius - 1, 0) if radius else 1)

    monkeypatch.setattr(ref, "token_mask", bad)
    assert _fails(check_attention_brute)


def test_planted_reference_not_global_for_its_rows(monkeypatch):
    orig = ref.visible_frames

    def bad(f, total_frames, ref_frames, radius):
        if f < ref_frames:
            return list(range(ref_frames)) + list(range(ref_frames, min(total_frames, ref_frames + radius + 1)))
        return orig(f, total_frames, ref_frames, radius)

    monkeypatch.setattr(ref, "visible_frames", bad)
    assert _fails(check_golden_frame_visibility)
    assert _fails(check_pair_counts)


def test_planted_dropped_reference_keys(monkeypatch):
    def bad(rows, n_tokens, frame_tokens, ref_frames, radius):
        fi = (np.asarray(rows) // frame_tokens)[:, None]
        fj = (np.arange(n_tokens) // frame_tokens)[None, :]
        return (fi < ref_frames) | ((fi >= ref_frames) & (fj >= ref_frames) & (np.abs(fi - fj) <= radius))

    monkeypatch.setattr(ref, "token_mask", bad)
    assert _fails(check_attention_brute)
    assert _fails(check_two_pass_merge)


def test_planted_wrong_scale(monkeypatch):
    class FakeMath:
        sqrt = staticmethod(lambda x: x)  # scale 1/d instead of 1/sqrt(d)
        log = staticmethod(math.log)
        exp = staticmethod(math.exp)

    monkeypatch.setattr(ref, "math", FakeMath)
    assert _fails(check_attention_brute)
    assert _fails(check_bound_stats_brute)


def test_planted_transposed_operand(monkeypatch):
    orig = ref.masked_attention

    def bad(q, k, v, *a, **kw):
        return orig(k, q, v, *a, **kw)  # roles of q and k swapped

    monkeypatch.setattr(ref, "masked_attention", bad)
    assert _fails(check_attention_brute)


def test_planted_bound_sign_error():
    c = MICRO[0]
    q, k, _ = micro_inputs(c, key_shift=3.0)
    st = ref.bound_statistics(q, k, c["T"], c["R0"], c["r"])
    res = ref.masked_attention(q, k, k, c["T"], c["R0"], c["r"])
    st_bad = dict(st, m=st["b"] - st["c"])  # centring shift with the wrong sign
    with pytest.raises(AssertionError):
        check_bound_holds(ref, st=st_bad, res=res)


def test_planted_uncentred_key_norms(monkeypatch):
    orig = ref.bound_statistics

    def bad(q, k, T, R0, r, heads=None):
        st = orig(q, k, T, R0, r, heads)
        kk = ref._as_f64(k)
        nf = kk.shape[1] // T
        st["M"] = np.sqrt((kk * kk).sum(axis=2)).reshape(kk.shape[0], nf, T).max(axis=2)
        return st

    monkeypatch.setattr(ref, "bound_statistics", bad)
    assert _fails(check_bound_stats_brute)


def test_planted_ragged_spans_taken_as_uniform(monkeypatch):
    """A ragged oracle that treats every frame as having the first frame's
    span (a plausible slip) fails the ragged pins."""
    orig = ref.frame_spans

    def bad(frame_tokens, n_tokens):
        spans = orig(frame_tokens, n_tokens)
        if len(spans) > 1 and not np.all(spans == spans[0]):
            t0 = int(spans[0])
            spans = np.full(len(spans), t0, dtype=np.int64)
            spans[-1] = n_tokens - t0 * (len(spans) - 1)
        return spans

    monkeypatch.setattr(ref, "frame_spans", bad)
    assert _fails(check_ragged_token_mask)
    assert _fails(check_ragged_attention_brute)
    assert _fails(check_ragged_bound_stats_brute)
