"""Seeded synthetic inputs for frame-aligned sparse attention.

This module only draws random tensors and rounds them to bf16.  It holds none
of the attention arithmetic: no mask, no softmax, no bound.  Both the fp64
oracle (``oracle/``) and the CUDA path's tests and benchmark take their inputs
from here, so the two sides see the same bits.

Shapes follow the super-resolution workloads described in "HeyGen x Google
Cloud: Avatar IV on TPU" (news.xcc.im/article/5328), sections "The Workload,
and the Port" (720p / 1080p output, 25 fps) and "Deleting the Mask" (tens of
thousands of tokens per chunk, one reference frame plus a window of frames,
frame spans that are not multiples of 128).

Token order is frame-contiguous: the reference frame(s) first, then the video
frames in time order, ``frame_tokens`` tokens each.  Tensors are ``[H, N, d]``
with ``N = (ref_frames + n_frames) * frame_tokens``.

Recipe (every draw has its own counter-free stream, so any head can be made
alone and in any order):

* stream ``(seed, 0, h)``: ``q[h] ~ N(0, 1)`` as float32 ``[N, d]``
* stream ``(seed, 1, h)``: key noise ``~ N(0, 1)`` float32 ``[N, d]``
* stream ``(seed, 2, h)``: ``v[h] ~ N(0, 1)`` float32 ``[N, d]``
* stream ``(seed, 3, h)``: the common key vector ``mu_h ~ N(0, 1)`` (float64,
  ``[d]``); ``k[h] = noise + float32(sigma * mu_h)``
* stream ``(seed, 4)``: ``permutation(H)``; its first ``n_modified`` entries
  are the modified heads
* ``"qscale"`` modifier: ``q[h] *= 8`` on the modified heads (loose bound)
* ``"heavy"`` modifier: on the modified heads the key noise is instead drawn
  from stream ``(seed, 5, h)`` as Student-t with 3 degrees of freedom, and
  ``N // 100`` rows chosen by stream ``(seed, 6, h)`` (without replacement)
  have that noise multiplied by 4 (norm outliers)
* every tensor is rounded once from float32 to bf16, round-to-nearest-even.

Arrays are returned as raw bf16 bit patterns (``numpy.uint16``).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Iterable, Optional, Sequence

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get", "generate", "round_to_bf16_bits"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    heads: int          # H (batch folded in; B = 1 everywhere)
    head_dim: int       # d
    ref_frames: int     # R0
    n_frames: int       # F (video frames)
    frame_tokens: int   # T
    window_radius: int  # r
    sigma: float        # scale of the common key vector
    seed: int
    modifier: Optional[str] = None  # None | "qscale" | "heavy"
    n_modified: int = 0

    @property
    def total_frames(self) -> int:
        return self.ref_frames + self.n_frames

    @property
    def tokens(self) -> int:
        return self.total_frames * self.frame_tokens

    def describe(self) -> str:
        return (f"{self.name}: H={self.heads} d={self.head_dim} "
                f"{self.ref_frames} ref + {self.n_frames} frames x "
                f"{self.frame_tokens} tokens (N={self.tokens}), "
                f"window radius {self.window_radius}, sigma={self.sigma}, "
                f"seed={self.seed}, modifier={self.modifier}"
                f"{'x' + str(self.n_modified) if self.modifier else ''}")


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 2, 64, 1, 8, 48, 1, 2.0, 0),
        Workload("mid", 16, 128, 1, 16, 880, 2, 3.0, 1),
        Workload("720p", 24, 128, 1, 21, 3600, 2, 3.0, 2, "qscale", 2),
        Workload("1080p", 24, 128, 1, 13, 8160, 1, 3.0, 3),
        Workload("stress", 24, 128, 1, 21, 3600, 2, 3.0, 4, "heavy", 12),
        # Same tensors as "stress" (same seed and modifier); every frame visible.
        Workload("dense", 24, 128, 1, 21, 3600, 21, 3.0, 4, "heavy", 12),
        # The 720p geometry with 4 heads (0.24 GB of Q/K/V, still larger than
        # L2): small enough for multi-pass profiler captures.
        Workload("720p_h4", 4, 128, 1, 21, 3600, 2, 3.0, 5),
        # The 720p heads and frames with 5 video frames (21,600 tokens): the
        # prologue's full 3072-wide projection over ~3.4 waves of CTAs in a
        # few GB, for multi-pass profiler captures.
        Workload("720p_f5", 24, 128, 1, 5, 3600, 2, 3.0, 6),
    ]
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _stream(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(list(key)))


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even.

    Inputs here are finite and far from the float32 range limits.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def modified_heads(w: Workload) -> np.ndarray:
    """Sorted indices of the heads that the workload's modifier touches."""
    if not w.modifier:
        return np.zeros(0, dtype=np.int64)
    perm = _stream(w.seed, 4).permutation(w.heads)
    return np.sort(perm[: w.n_modified])


def _make_head(w: Workload, tensor: str, h: int, modified: bool) -> np.ndarray:
    n, d = w.tokens, w.head_dim
    if tensor == "q":
        x = _stream(w.seed, 0, h).standard_normal((n, d), dtype=np.float32)
        if modified and w.modifier == "qscale":
            x *= np.float32(8.0)
    elif tensor == "k":
        if modified and w.modifier == "heavy":
            x = _stream(w.seed, 5, h).standard_t(3, (n, d)).astype(np.float32)
            rows = _stream(w.seed, 6, h).choice(n, n // 100, replace=False)
            x[rows] *= np.float32(4.0)
        else:
            x = _stream(w.seed, 1, h).standard_normal((n, d), dtype=np.float32)
        mu = _stream(w.seed, 3, h).standard_normal(d)
        x += (w.sigma * mu).astype(np.float32)[None, :]
    elif tensor == "v":
        x = _stream(w.seed, 2, h).standard_normal((n, d), dtype=np.float32)
    else:
        raise ValueError(tensor)
    return round_to_bf16_bits(x)


def generate(w: Workload | str,
             tensors: Sequence[str] = ("q", "k", "v"),
             heads: Optional[Iterable[int]] = None,
             workers: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw the workload's tensors as bf16 bits, ``[len(heads), N, d]`` each.

    ``heads`` defaults to all heads.  The result also carries
    ``"modified_heads"`` (indices into the full head range).
    """
    if isinstance(w, str):
        w = get(w)
    hs = list(range(w.heads)) if heads is None else [int(h) for h in heads]
    mod = set(modified_heads(w).tolist())
    out: Dict[str, np.ndarray] = {}
    jobs = []
    for t in tensors:
        arr = np.empty((len(hs), w.tokens, w.head_dim), dtype=np.uint16)
        out[t] = arr
        for i, h in enumerate(hs):
            jobs.append((arr, i, t, h))

    def run(job):
        arr, i, t, h = job
        arr[i] = _make_head(w, t, h, h in mod)

    nw = workers or min(len(jobs), os.cpu_count() or 1, 16)
    if nw <= 1 or len(jobs) <= 1:
        for j in jobs:
            run(j)
    else:
        with ThreadPoolExecutor(max_workers=nw) as ex:
            list(ex.map(run, jobs))
    out["modified_heads"] = modified_heads(w)
    return out


# ---------------------------------------------------------------------------
# Inputs of the attention prologue (normalization, projection, rotary
# embedding, head packing): hidden states, norm scale, projection weight and
# the rotary angle tables a caller supplies.  Random draws and position
# tables only; the prologue's arithmetic is the oracle's and the library's.
# ---------------------------------------------------------------------------

#: Latent grid width (patches per row) of each workload's frames: the frame
#: span T is grid_w x (T / grid_w) patches.
GRID_W = {"tiny": 8, "mid": 40, "720p": 80, "1080p": 120, "stress": 80, "dense": 80, "720p_h4": 80, "720p_f5": 80}


def rotary_tables(w: Workload, grid_w: Optional[int] = None, base: float = 10000.0):
    """cos, sin [N, d/2] float32 for 3D rotary positions (frame, row, column).

    Token j of frame f = j // T sits at row (j % T) // grid_w and column
    (j % T) % grid_w.  The d/2 rotation pairs are split over the three axes
    (d/8 pairs for the frame index, the rest shared equally by row and
    column); pair k of an axis with n pairs turns at base^(-k/n) radians per
    unit of that axis's position.
    """
    d = w.head_dim
    gw = grid_w or GRID_W.get(w.name, 1)
    n_t = d // 8
    n_y = (d // 2 - n_t) // 2
    n_x = d // 2 - n_t - n_y
    j = np.arange(w.tokens, dtype=np.int64)
    pos = [j // w.frame_tokens, (j % w.frame_tokens) // gw, (j % w.frame_tokens) % gw]
    angles = [p[:, None].astype(np.float64) * base ** (-np.arange(n, dtype=np.float64) / n)[None, :]
              for p, n in zip(pos, (n_t, n_y, n_x))]
    ang = np.concatenate(angles, axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def prologue_inputs(w: Workload | str, width: Optional[int] = None, workers: Optional[int] = None):
    """Hidden states x [N, C] (bf16 bits, N(0,1)), norm scale gamma [C]
    (float32, 1 + 0.1 N(0,1)), projection weight [3*H*d, C] (bf16 bits,
    N(0, 1/C)) and the rotary tables; C defaults to H*d.  Streams:
    (seed, 10, row block) for x, (seed, 11) gamma, (seed, 12, row block)
    for the weight."""
    if isinstance(w, str):
        w = get(w)
    C = width or w.heads * w.head_dim
    out_f = 3 * w.heads * w.head_dim
    x = np.empty((w.tokens, C), dtype=np.uint16)
    wt = np.empty((out_f, C), dtype=np.uint16)
    rows = 4096
    jobs = [(x, i, 10, 1.0) for i in range(0, w.tokens, rows)] + \
           [(wt, i, 12, 1.0 / np.sqrt(C)) for i in range(0, out_f, rows)]

    def run(job):
        arr, i0, tag, scale = job
        n = min(rows, arr.shape[0] - i0)
        vals = _stream(w.seed, tag, i0 // rows).standard_normal((n, C), dtype=np.float32)
        arr[i0:i0 + n] = round_to_bf16_bits(vals * np.float32(scale))

    nw = workers or min(len(jobs), os.cpu_count() or 1, 16)
    with ThreadPoolExecutor(max_workers=nw) as ex:
        list(ex.map(run, jobs))
    gamma = (1.0 + 0.1 * _stream(w.seed, 11).standard_normal(C)).astype(np.float32)
    cos, sin = rotary_tables(w)
    return {"x": x, "gamma": gamma, "w": wt, "cos": cos, "sin": sin}
