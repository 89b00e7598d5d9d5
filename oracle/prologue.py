"""fp64 definition of the attention prologue (test infrastructure only).

"HeyGen x Google Cloud: Avatar IV on TPU", section "Layout Is the ABI" and
Fig. 5: attention's inputs come from a chain of small operations —
normalization, rotary embeddings, projections, head packing — that was
fused into one kernel writing its output in exactly the layout its
consumer wants.  The pages name the operations but not their order or
conventions; the readings taken here:

* the normalization is an RMSNorm of each token's hidden state
  ``x [C]``: ``xh = x / sqrt(mean(x^2) + eps) * gamma`` (``eps = 1e-6``);
* the projection is one matrix ``w [3*H*d, C]`` (the ``[out, in]``
  convention of a linear layer's weight) giving q, k and v side by side:
  output features ``[0, H*d)`` are q, then k, then v; head ``h`` of each is
  the ``d`` features starting at ``h*d``; no bias;
* rotary embeddings apply to q and k, per head, pairing element ``i`` with
  element ``i + d/2`` (the rotate-half form): with ``c = cos[n, i]`` and
  ``s = sin[n, i]`` for token ``n``, ``(a, b) -> (a c - b s, a s + b c)``;
  the angle tables ``cos, sin [N, d/2]`` are inputs (positions and
  frequencies are the caller's, e.g. a frame/row/column split for video);
* head packing writes q, k, v as ``[H, N, d]`` here (the consumer's layout;
  the product also writes ``[N, H, d]`` and the all-to-all layout).
"""
from __future__ import annotations

import numpy as np

from .reference import _as_f64

RMS_EPS = 1e-6


def rms_norm(x, gamma, eps: float = RMS_EPS) -> np.ndarray:
    """``x / sqrt(mean(x^2) + eps) * gamma`` over the last axis, fp64."""
    x = _as_f64(x)
    g = _as_f64(gamma)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * g


def rotate(x, cos, sin) -> np.ndarray:
    """Rotary embedding of ``x [N, H, d]`` with tables ``[N, d/2]``."""
    half = x.shape[-1] // 2
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def qkv_prologue(x, gamma, w, cos, sin, heads: int, head_dim: int, eps: float = RMS_EPS):
    """RMSNorm -> projection -> rotary (q, k) -> [H, N, d] packing.

    ``x [N, C]``, ``gamma [C]``, ``w [3*H*d, C]`` (bf16 bit patterns or
    floats), ``cos, sin [N, d/2]``.  Returns fp64 ``q, k, v`` of shape
    ``[H, N, d]``.
    """
    xh = rms_norm(x, gamma, eps)
    y = xh @ _as_f64(w).T
    N = y.shape[0]
    y = y.reshape(N, 3, heads, head_dim)
    q = rotate(y[:, 0], cos, sin)
    k = rotate(y[:, 1], cos, sin)
    v = y[:, 2]
    return tuple(np.ascontiguousarray(t.transpose(1, 0, 2)) for t in (q, k, v))


def prologue_flops(tokens: int, width: int, heads: int, head_dim: int) -> float:
    """FLOPs of the projection (2 per multiply-add), the prologue's
    contraction: ``2 * N * C * 3*H*d``."""
    return 2.0 * tokens * width * 3 * heads * head_dim

