"""fp64 definitions of frame-aligned sparse attention (test infrastructure only).

Notation (all integers are token or frame indices):

* ``T`` tokens per frame; frames ``0 .. R0-1`` are reference frames, frames
  ``R0 .. Nf-1`` are video frames; token ``j`` lies in frame ``j // T``.
  Wherever a function takes ``frame_tokens`` it also accepts a sequence of
  per-frame token counts ``T_0 .. T_{Nf-1}`` (frames of different spans,
  still contiguous and in the same order); token ``j`` then lies in the
  frame ``g`` with ``T_0 + .. + T_{g-1} <= j < T_0 + .. + T_g``.
* ``r`` window radius; ``s = 1 / sqrt(d)``.

Readings where the pages are silent (each listed in the design notes):

* token order is frame-contiguous, reference frame(s) first;
* the reference frame is global both ways: every row sees it, and its own
  rows see every frame;
* the window is clipped to the video frames ``[R0, Nf-1]`` (no wrap, no
  shift);
* one mean key per head over all ``N`` keys (a per-row constant shift of the
  logits, hence softmax-invariant);
* the bound of row ``i`` uses the largest centred key norm over the frames
  that row sees; the eligibility statistic is the slack
  ``G_i = b_i - s q_i . kbar_c`` (an upper bound on ``b_i`` minus the true
  centred row maximum, because a maximum is at least a mean), and a head is
  eligible when ``max_i G_i <= 32``;
* LSE is the natural log over the uncentred scaled logits of visible keys.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

#: Largest guaranteed gap (nats) between a row's bound and its true maximum
#: for which a head keeps the bounded softmax.  e^-32 ~ 1.3e-14 is far above
#: the float32 underflow threshold e^-87, so every row keeps a term that
#: survives.  ("Unchaining the Softmax": a bound far above the true maximum
#: pushes the exponentials toward underflow.)
ELIG_SLACK_NATS = 32.0


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _as_f64(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:
        return bf16_bits_to_f64(x)
    return np.asarray(x, dtype=np.float64)


def frame_spans(frame_tokens, n_tokens: int) -> np.ndarray:
    """Per-frame token counts: ``frame_tokens`` itself when it is a
    sequence, else ``n_tokens // frame_tokens`` copies of it."""
    if np.ndim(frame_tokens) == 0:
        return np.full(n_tokens // int(frame_tokens), int(frame_tokens), dtype=np.int64)
    spans = np.asarray(frame_tokens, dtype=np.int64)
    assert spans.sum() == n_tokens, "frame spans must add up to the sequence length"
    return spans


def frame_of(tokens, frame_tokens, n_tokens: int) -> np.ndarray:
    """Frame index of each token."""
    spans = frame_spans(frame_tokens, n_tokens)
    starts = np.cumsum(spans) - spans
    return np.searchsorted(starts, np.asarray(tokens, dtype=np.int64), side="right") - 1


# ---------------------------------------------------------------------------
# The mask ("Deleting the Mask": window of nearby frames plus one global
# reference frame; live regions snap to frame boundaries).
# ---------------------------------------------------------------------------

def visible_frames(f: int, total_frames: int, ref_frames: int, radius: int) -> list:
    """Key frames visible from query frame ``f``, ascending."""
    if f < ref_frames:
        return list(range(total_frames))
    lo = max(ref_frames, f - radius)
    hi = min(total_frames - 1, f + radius)
    return list(range(ref_frames)) + list(range(lo, hi + 1))


def frame_visibility(total_frames: int, ref_frames: int, radius: int) -> np.ndarray:
    """``[Nf, Nf]`` boolean: entry ``[f, g]`` is True when frame ``f`` sees ``g``."""
    vis = np.zeros((total_frames, total_frames), dtype=bool)
    for f in range(total_frames):
        vis[f, visible_frames(f, total_frames, ref_frames, radius)] = True
    return vis


def token_mask(rows: np.ndarray, n_tokens: int, frame_tokens: int,
               ref_frames: int, radius: int) -> np.ndarray:
    """Explicit ``[len(rows), N]`` boolean mask written from the token rule.

    ``vis(i, j) = fr(j) < R0  or  fr(i) < R0  or  |fr(i) - fr(j)| <= r``
    (the last clause only between video frames).
    """
    fi = frame_of(rows, frame_tokens, n_tokens)[:, None]
    fj = frame_of(np.arange(n_tokens), frame_tokens, n_tokens)[None, :]
    ref_key = fj < ref_frames
    ref_row = fi < ref_frames
    window = (fi >= ref_frames) & (fj >= ref_frames) & (np.abs(fi - fj) <= radius)
    return ref_key | ref_row | window


def visible_pairs(frame_tokens, n_frames: int, ref_frames: int, radius: int) -> int:
    """Number of visible (query, key) pairs for one head (valid rows only)."""
    nf = ref_frames + n_frames
    if np.ndim(frame_tokens) == 0:
        frames = sum(len(visible_frames(f, nf, ref_frames, radius)) for f in range(nf))
        return frames * frame_tokens * frame_tokens
    spans = [int(t) for t in frame_tokens]
    assert len(spans) == nf
    return sum(spans[f] * sum(spans[g] for g in visible_frames(f, nf, ref_frames, radius)) for f in range(nf))


def visible_flops(heads: int, head_dim: int, frame_tokens, n_frames: int,
                  ref_frames: int, radius: int) -> float:
    """4*d FLOPs per visible pair (2*d for q.k, 2*d for p*v)."""
    return 4.0 * head_dim * heads * visible_pairs(frame_tokens, n_frames, ref_frames, radius)


# ---------------------------------------------------------------------------
# Dense masked attention, the definition the single-pass kernel reaches.
# ---------------------------------------------------------------------------

def masked_attention(q, k, v, frame_tokens, ref_frames: int, radius: int,
                     rows: Optional[np.ndarray] = None,
                     heads: Optional[Sequence[int]] = None,
                     slab: int = 256) -> Dict[str, np.ndarray]:
    """fp64 softmax attention under the explicit frame mask.

    ``q, k, v``: ``[H, N, d]`` (bf16 bit patterns or floats).  ``rows``
    restricts the query rows (same rows for every head); ``heads`` restricts
    the heads.  Returns ``out [h, R, d]``, ``lse [h, R]`` (natural log of the
    sum of ``exp(s q.k)`` over visible keys) and ``zmax [h, R]`` (largest
    visible scaled logit).
    """
    H, N, d = q.shape
    hs = list(range(H)) if heads is None else list(heads)
    rs = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    s = 1.0 / math.sqrt(d)
    out = np.zeros((len(hs), len(rs), d))
    lse = np.zeros((len(hs), len(rs)))
    zmax = np.zeros((len(hs), len(rs)))
    for a, h in enumerate(hs):
        kh = _as_f64(k[h])
        vh = _as_f64(v[h])
        for lo in range(0, len(rs), slab):
            rr = rs[lo:lo + slab]
            qh = _as_f64(q[h][rr])
            z = s * (qh @ kh.T)
            z[~token_mask(rr, N, frame_tokens, ref_frames, radius)] = -np.inf
            mx = z.max(axis=1)
            e = np.exp(z - mx[:, None])
            tot = e.sum(axis=1)
            lse[a, lo:lo + len(rr)] = mx + np.log(tot)
            out[a, lo:lo + len(rr)] = (e @ vh) / tot[:, None]
            zmax[a, lo:lo + len(rr)] = mx
    return {"out": out, "lse": lse, "zmax": zmax}


# ---------------------------------------------------------------------------
# Cauchy-Schwarz bound and per-head eligibility ("Unchaining the Softmax").
# ---------------------------------------------------------------------------

def bound_statistics(q, k, frame_tokens, ref_frames: int, radius: int,
                     heads: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Bound quantities in fp64 for every row of the selected heads.

    Per head ``h``:

    * ``mu[h]``       mean of all ``N`` keys;
    * ``M[h, g]``     ``max_{j in frame g} |k_j - mu_h|``;
    * ``fsum[h, g]``  ``sum_{j in frame g} k_j``;
    * ``Mvis[h, f]``  ``max_{g visible from f} M[h, g]``;
    * ``kbar_c[h,f]`` mean over the keys visible from ``f`` of ``k_j - mu_h``.

    Per row ``i`` (frame ``f = i // T``):

    * ``c = s q_i . mu_h``  (the per-row shift that centring removes);
    * ``b = s |q_i| Mvis[h, f]`` (bound on the centred row maximum);
    * ``m = c + b``  (bound on the uncentred row maximum);
    * ``G = b - s q_i . kbar_c[h, f]`` (bound on ``b`` minus the true centred max).

    ``stat[h] = max_i G_i`` and ``elig[h] = stat[h] <= 32``.
    """
    H, N, d = q.shape
    spans = frame_spans(frame_tokens, N)
    nf = len(spans)
    bounds = np.concatenate([[0], np.cumsum(spans)])
    hs = list(range(H)) if heads is None else list(heads)
    s = 1.0 / math.sqrt(d)
    vis = frame_visibility(nf, ref_frames, radius)
    res = {name: [] for name in ("mu", "M", "fsum", "Mvis", "kbar_c", "c", "b", "m", "G", "stat", "elig")}
    for h in hs:
        kh = _as_f64(k[h])
        qh = _as_f64(q[h])
        mu = kh.mean(axis=0)
        kc = kh - mu[None, :]
        norms = np.sqrt((kc * kc).sum(axis=1))
        M = np.array([norms[bounds[g]:bounds[g + 1]].max() for g in range(nf)])
        fsum = np.stack([kh[bounds[g]:bounds[g + 1]].sum(axis=0) for g in range(nf)])
        Mvis = np.array([M[vis[f]].max() for f in range(nf)])
        kbar_c = np.stack([fsum[vis[f]].sum(axis=0) / spans[vis[f]].sum() - mu for f in range(nf)])
        fr = frame_of(np.arange(N), spans, N)
        qn = np.sqrt((qh * qh).sum(axis=1))
        c = s * (qh @ mu)
        b = s * qn * Mvis[fr]
        G = b - s * np.einsum("nd,nd->n", qh, kbar_c[fr])
        stat = G.max()
        for name, val in (("mu", mu), ("M", M), ("fsum", fsum), ("Mvis", Mvis), ("kbar_c", kbar_c),
                          ("c", c), ("b", b), ("m", c + b), ("G", G), ("stat", stat),
                          ("elig", stat <= ELIG_SLACK_NATS)):
            res[name].append(val)
    return {name: np.array(val) for name, val in res.items()}
