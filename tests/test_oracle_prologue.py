"""Pins for the fp64 prologue oracle (CPU only).

"HeyGen x Google Cloud: Avatar IV on TPU", section "Layout Is the ABI",
Fig. 5: attention's inputs come from normalization, rotary embeddings,
projections and head packing, fused into one kernel that writes the
consumer's layout.  The oracle's readings (RMSNorm of the hidden state, one
[out, in] projection to q|k|v, rotate-half rotary embedding of q and k,
[H, N, d] packing) are pinned here against a pure-Python brute force written
from those words, torch's fp64 rms_norm and linear, and the closed-form
properties of a rotation; planted mistakes show each pin bites.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import prologue as pro


def brute_prologue(x, gamma, w, cos, sin, H, d, eps):
    """Loops only: RMSNorm, the projection as sums, the rotation pair by pair."""
    N, C = len(x), len(x[0])
    q = [[[0.0] * d for _ in range(N)] for _ in range(H)]
    k = [[[0.0] * d for _ in range(N)] for _ in range(H)]
    v = [[[0.0] * d for _ in range(N)] for _ in range(H)]
    for n in range(N):
        ms = sum(x[n][c] ** 2 for c in range(C)) / C
        xh = [x[n][c] / math.sqrt(ms + eps) * gamma[c] for c in range(C)]
        y = [sum(xh[c] * w[o][c] for c in range(C)) for o in range(3 * H * d)]
        for h in range(H):
            for part, dst in enumerate((q, k, v)):
                vals = y[part * H * d + h * d: part * H * d + (h + 1) * d]
                if part < 2:  # rotate q and k: pair i with i + d/2
                    half = d // 2
                    rot = list(vals)
                    for i in range(half):
                        a, b = vals[i], vals[i + half]
                        rot[i] = a * cos[n][i] - b * sin[n][i]
                        rot[i + half] = a * sin[n][i] + b * cos[n][i]
                    vals = rot
                dst[h][n] = list(vals)
    return np.array(q), np.array(k), np.array(v)


def small_case(seed=3, N=5, C=8, H=2, d=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, C)) * 2.0
    gamma = 1.0 + 0.3 * rng.standard_normal(C)
    w = rng.standard_normal((3 * H * d, C)) / math.sqrt(C)
    ang = rng.uniform(-math.pi, math.pi, (N, d // 2))
    return x, gamma, w, np.cos(ang), np.sin(ang), H, d


def check_brute(o):
    for seed, (N, C, H, d) in ((3, (5, 8, 2, 4)), (4, (3, 6, 1, 8)), (5, (4, 16, 3, 2))):
        x, gamma, w, cos, sin, H, d = small_case(seed, N, C, H, d)
        got = o.qkv_prologue(x, gamma, w, cos, sin, H, d)
        want = brute_prologue(x.tolist(), gamma.tolist(), w.tolist(), cos.tolist(), sin.tolist(), H, d, o.RMS_EPS)
        for g, t in zip(got, want):
            np.testing.assert_allclose(g, t, rtol=1e-12, atol=1e-13)


def check_library_routines(o):
    """RMSNorm against torch's rms_norm; with unit scale and zero angles the
    prologue is the plain projection (torch's linear), heads split in order."""
    rng = np.random.default_rng(7)
    N, C, H, d = 9, 32, 2, 8
    x = rng.standard_normal((N, C))
    gamma = 1.0 + 0.2 * rng.standard_normal(C)
    w = rng.standard_normal((3 * H * d, C)) / math.sqrt(C)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (C,), torch.from_numpy(gamma), eps=o.RMS_EPS)
    np.testing.assert_allclose(o.rms_norm(x, gamma), want.numpy(), rtol=1e-13, atol=1e-14)
    ones = np.ones(C)
    q, k, v = o.qkv_prologue(x, ones, w, np.ones((N, d // 2)), np.zeros((N, d // 2)), H, d)
    xn = torch.nn.functional.rms_norm(torch.from_numpy(x), (C,), eps=o.RMS_EPS)
    y = torch.nn.functional.linear(xn, torch.from_numpy(w)).numpy().reshape(N, 3, H, d)
    for part, t in enumerate((q, k, v)):
        np.testing.assert_allclose(t, y[:, part].transpose(1, 0, 2), rtol=1e-12, atol=1e-13)


def check_rotation_properties(o):
    """The rotary step is a rotation of each (i, i + d/2) pair: it keeps
    every head's norm, leaves v alone, composes by adding angles, and makes
    q.k depend only on the difference of positions."""
    x, gamma, w, cos, sin, H, d = small_case(11, N=6, C=12, H=2, d=8)
    q, k, v = o.qkv_prologue(x, gamma, w, cos, sin, H, d)
    q0, k0, v0 = o.qkv_prologue(x, gamma, w, np.ones_like(cos), np.zeros_like(sin), H, d)
    np.testing.assert_allclose(np.linalg.norm(q, axis=2), np.linalg.norm(q0, axis=2), rtol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(k, axis=2), np.linalg.norm(k0, axis=2), rtol=1e-12)
    np.testing.assert_array_equal(v, v0)
    rng = np.random.default_rng(12)
    a1, a2 = rng.uniform(-3, 3, (6, d // 2)), rng.uniform(-3, 3, (6, d // 2))
    y = rng.standard_normal((6, H, d))
    twice = o.rotate(o.rotate(y, np.cos(a1), np.sin(a1)), np.cos(a2), np.sin(a2))
    once = o.rotate(y, np.cos(a1 + a2), np.sin(a1 + a2))
    np.testing.assert_allclose(twice, once, rtol=1e-12, atol=1e-12)
    # Relative positions: angles pos * omega for 1D positions; shifting every
    # position by the same amount leaves all q.k products unchanged.
    omega = 10000.0 ** (-np.arange(d // 2) / (d // 2))
    pos = np.arange(6)[:, None].astype(np.float64)
    qa, ka = (o.rotate(t, np.cos(pos * omega), np.sin(pos * omega)) for t in (y, y[::-1].copy()))
    qb, kb = (o.rotate(t, np.cos((pos + 5) * omega), np.sin((pos + 5) * omega)) for t in (y, y[::-1].copy()))
    np.testing.assert_allclose(np.einsum("nhd,mhd->hnm", qa, ka), np.einsum("nhd,mhd->hnm", qb, kb),
                               rtol=1e-11, atol=1e-11)


def check_rms_scale_invariance(o):
    """RMSNorm divides out the hidden state's scale (up to eps)."""
    x, gamma, w, cos, sin, H, d = small_case(13, N=4, C=16, H=1, d=8)
    a = o.qkv_prologue(x, gamma, w, cos, sin, H, d, eps=0.0)
    b = o.qkv_prologue(x * 37.5, gamma, w, cos, sin, H, d, eps=0.0)
    for s, t in zip(a, b):
        np.testing.assert_allclose(s, t, rtol=1e-12, atol=1e-13)


CHECKS = [check_brute, check_library_routines, check_rotation_properties, check_rms_scale_invariance]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_prologue_pin(check):
    check(pro)


def test_rotary_tables_are_unit_rotations():
    w = workloads.get("mid")
    cos, sin = workloads.rotary_tables(w)
    assert cos.shape == (w.tokens, w.head_dim // 2)
    np.testing.assert_allclose(cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2, 1.0, atol=1e-6)
    # Token 0 of every frame sits at row 0, column 0: only the frame pairs turn.
    n_t = w.head_dim // 8
    f0 = np.arange(w.total_frames) * w.frame_tokens
    np.testing.assert_array_equal(cos[f0][:, n_t:], 1.0)


def _fails(check):
    try:
        check(pro)
    except AssertionError:
        return True
    return False


def test_planted_rotation_sign(monkeypatch):
    def bad(x, cos, sin):
        half = x.shape[-1] // 2
        c, s = cos[:, None, :], sin[:, None, :]
        a, b = x[..., :half], x[..., half:]
        return np.concatenate([a * c + b * s, -a * s + b * c], axis=-1)  # turns the other way

    monkeypatch.setattr(pro, "rotate", bad)
    assert _fails(check_brute)


def test_planted_qk_swap_and_pairing(monkeypatch):
    orig = pro.qkv_prologue

    def swapped(x, gamma, w, cos, sin, heads, head_dim, eps=pro.RMS_EPS):
        q, k, v = orig(x, gamma, w, cos, sin, heads, head_dim, eps)
        return k, q, v

    monkeypatch.setattr(pro, "qkv_prologue", swapped)
    assert _fails(check_brute)
    monkeypatch.undo()

    def adjacent_pairs(x, cos, sin):
        a, b = x[..., 0::2], x[..., 1::2]  # pairs (2i, 2i+1) instead of (i, i + d/2)
        out = np.empty_like(x)
        out[..., 0::2] = a * cos[:, None, :] - b * sin[:, None, :]
        out[..., 1::2] = a * sin[:, None, :] + b * cos[:, None, :]
        return out

    monkeypatch.setattr(pro, "rotate", adjacent_pairs)
    assert _fails(check_brute)


def test_planted_norm_over_tokens(monkeypatch):
    def bad(x, gamma, eps=pro.RMS_EPS):
        x = np.asarray(x, dtype=np.float64)
        return x / np.sqrt((x * x).mean(axis=0, keepdims=True) + eps) * gamma

    monkeypatch.setattr(pro, "rms_norm", bad)
    assert _fails(check_brute)
    assert _fails(check_library_routines)
