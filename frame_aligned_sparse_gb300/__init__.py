"""Frame-aligned sparse attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/fas.h`` (``libfas.so``).  It
only marshals arguments: every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  If the library is
not built, every call raises: there is no CPU fallback.

The operation ("HeyGen x Google Cloud: Avatar IV on TPU", sections "Deleting
the Mask" and "Unchaining the Softmax"): queries of each video frame attend
to a window of neighbouring frames plus the global reference frame(s), in one
pass over frame-aligned full key blocks; eligible heads use a precomputed
Cauchy-Schwarz row bound instead of a running maximum.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Tuple

import numpy as np

__all__ = [
    "FasError", "PlanInfo", "MODES", "library_path", "load",
    "fas_plan", "fas_plan_describe", "fas_prepass", "fas_forward", "fas_free",
    "fas_status", "fas_prepass_readback", "fas_selftest_wait_timeout", "fas_last_launch_count",
    "fas_prepass_noalloc", "fas_forward_host", "fas_set_layout", "LAYOUTS", "fas_forward_ablation",
    "fas_prologue", "fas_prologue_fold_weights", "PROLOGUE_LAYOUTS",
    "fas_prologue_with_key_sums", "fas_prepass_with_key_sums", "key_sums_shape",
]

FAS_OK, FAS_ERR_ARG, FAS_ERR_STATE, FAS_ERR_ALIGN, FAS_ERR_CUDA, FAS_ERR_TIMEOUT, FAS_ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5, -6
FAS_ERR_SCRATCH = -7
FAS_ERR_BOUND = -8
FAS_NOALLOC_SCRATCH_BYTES = 4 << 20
MODES = {"auto": 0, "online": 1, "bounded": 2}
LAYOUTS = {"hnd": 0, "nhd": 1}  # q, k, v, out as [H, N, d] or [N, H, d]
PROLOGUE_LAYOUTS = {"hnd": 0, "nhd": 1, "a2a": 2}  # fas_prologue's outputs (a2a: [G, P, n, H/(G*P), d])
RMS_EPS = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "libfas.so")


class FasError(RuntimeError):
    def __init__(self, call: str, code: int, message: str):
        super().__init__(f"{call} failed: {message} (status {code})")
        self.code = code


class _PlanInfoC(ctypes.Structure):
    _fields_ = [
        ("block_k", ctypes.c_int32),
        ("q_tile", ctypes.c_int32),
        ("n_work", ctypes.c_int32),
        ("total_frames", ctypes.c_int32),
        ("tokens", ctypes.c_int64),
        ("key_blocks", ctypes.c_int64),
        ("visible_flops", ctypes.c_double),
        ("host_table", ctypes.POINTER(ctypes.c_int32)),
    ]


@dataclasses.dataclass
class PlanInfo:
    block_k: int
    q_tile: int
    n_work: int
    total_frames: int
    tokens: int
    key_blocks: int
    visible_flops: float
    table: np.ndarray  # [Nf, 4] int32: start0, len0, start1, len1


_LIB: Optional[ctypes.CDLL] = None

_SIGS = {
    "fas_plan": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.POINTER(_PlanInfoC)]),
    "fas_plan_ex": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(_PlanInfoC)]),
    "fas_plan_describe": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(_PlanInfoC), ctypes.c_void_p,
                                                              ctypes.c_void_p]),
    "fas_plan_ragged": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_int] * 6 + [ctypes.POINTER(_PlanInfoC)]),
    "fas_plan_describe_ragged": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_int] * 6 +
                                 [ctypes.POINTER(_PlanInfoC), ctypes.c_void_p, ctypes.c_void_p]),
    "fas_prepass": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "fas_prepass_with_key_sums": (ctypes.c_int, [ctypes.c_void_p] * 5),
    "fas_forward": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_void_p]),
    "fas_forward_host": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fas_forward_ablation": (ctypes.c_int, [ctypes.c_void_p] * 6),
    "fas_prologue": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_float] +
                     [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]),
    "fas_prologue_with_key_sums": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_float] +
                                   [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 2),
    "fas_prologue_fold_weights": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int] * 2 + [ctypes.c_void_p]),
    "fas_free": (ctypes.c_int, []),
    "fas_status": (ctypes.c_int, [ctypes.c_void_p]),
    "fas_prepass_readback": (ctypes.c_int, [ctypes.c_void_p] * 6),
    "fas_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p]),
    "fas_last_launch_count": (ctypes.c_int, []),
    "fas_prepass_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 6 +
                            [ctypes.c_void_p] * 4),
    "fas_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fas_set_layout": (ctypes.c_int, [ctypes.c_int]),
}


def load() -> ctypes.CDLL:
    """Loads libfas.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m frame_aligned_sparse_gb300.build` "
                "(nvcc, sm_103a). There is no CPU fallback.")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(call: str, rc: int) -> None:
    if rc != FAS_OK:
        msg = load().fas_error_string(rc).decode()
        raise FasError(call, rc, msg)


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _info(c: _PlanInfoC, table: Optional[np.ndarray] = None) -> PlanInfo:
    if table is None:
        table = np.ctypeslib.as_array(c.host_table, shape=(c.total_frames * 4,)).reshape(-1, 4).copy()
    return PlanInfo(c.block_k, c.q_tile, c.n_work, c.total_frames, c.tokens, c.key_blocks, c.visible_flops, table)


_PLAN: dict = {}


def _spans_arg(frame_tokens, n_frames: int, ref_frames: int):
    """(int32 array of per-frame spans, or None for uniform frames)."""
    if np.ndim(frame_tokens) == 0:
        return None
    spans = np.ascontiguousarray(frame_tokens, dtype=np.int32)
    if spans.ndim != 1 or len(spans) != ref_frames + n_frames:
        raise ValueError(f"frame_tokens must hold ref_frames + n_frames = {ref_frames + n_frames} spans")
    return spans


def fas_plan(frame_tokens, n_frames: int, ref_frames: int, window_radius: int, heads: int, head_dim: int,
             block_k: int = 0) -> PlanInfo:
    """Builds (or reuses) the library's plan; see ``fas_plan`` in fas.h.
    ``frame_tokens``: one span for every frame, or a sequence of
    ref_frames + n_frames per-frame spans (``fas_plan_ragged``)."""
    c = _PlanInfoC()
    spans = _spans_arg(frame_tokens, n_frames, ref_frames)
    if spans is None:
        rc = load().fas_plan_ex(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim, block_k,
                                ctypes.byref(c))
    else:
        rc = load().fas_plan_ragged(spans.ctypes.data, n_frames, ref_frames, window_radius, heads, head_dim,
                                    block_k, ctypes.byref(c))
    _check("fas_plan", rc)
    info = _info(c)
    geometry = (tuple(spans.tolist()) if spans is not None else frame_tokens, n_frames, ref_frames, window_radius,
                heads, head_dim, info.block_k)
    if _PLAN.get("geometry") != geometry:
        _PLAN["layout"] = "hnd"  # a new plan starts head-major (the library resets it too)
    _PLAN.update(heads=heads, head_dim=head_dim, tokens=info.tokens, info=info, geometry=geometry)
    return info


def fas_set_layout(layout: str) -> None:
    """Layout of q, k, v and out for the following calls: "hnd" ([H, N, d])
    or "nhd" ([N, H, d]); lse stays [H, N].  See ``fas_set_layout`` in fas.h."""
    _check("fas_set_layout", load().fas_set_layout(LAYOUTS[layout]))
    _PLAN["layout"] = layout


def fas_plan_describe(frame_tokens, n_frames: int, ref_frames: int, window_radius: int, heads: int,
                      head_dim: int, block_k: int = 0) -> Tuple[PlanInfo, np.ndarray, np.ndarray]:
    """Host-only plan: (info, table [Nf, 4], work [n_work, 4]).  frame_tokens
    as in ``fas_plan``."""
    lib = load()
    spans = _spans_arg(frame_tokens, n_frames, ref_frames)

    def call(c, table, work):
        if spans is None:
            return lib.fas_plan_describe(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim,
                                         block_k, ctypes.byref(c), table, work)
        return lib.fas_plan_describe_ragged(spans.ctypes.data, n_frames, ref_frames, window_radius, heads,
                                            head_dim, block_k, ctypes.byref(c), table, work)

    c = _PlanInfoC()
    _check("fas_plan_describe", call(c, None, None))
    table = np.zeros((c.total_frames, 4), dtype=np.int32)
    work = np.zeros((c.n_work, 4), dtype=np.int32)
    _check("fas_plan_describe", call(c, table.ctypes.data, work.ctypes.data))
    return _info(c, table), table, work


def _check_tensor(name, t, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, the plan needs {tuple(shape)}")


def _qkv_shape():
    """Shape of q, k, v and out in the current layout."""
    if not _PLAN:
        raise FasError("fas_plan", FAS_ERR_STATE, "no plan")
    if _PLAN.get("layout", "hnd") == "nhd":
        return (_PLAN["tokens"], _PLAN["heads"], _PLAN["head_dim"])
    return (_PLAN["heads"], _PLAN["tokens"], _PLAN["head_dim"])


def _lse_shape():
    return (_PLAN["heads"], _PLAN["tokens"])


def fas_prepass(q, k, stream=None, want_elig: bool = False) -> Optional[np.ndarray]:
    """Mean-centred key norms, row bounds and head eligibility (bf16 q, k [H, N, d])."""
    import torch
    shape = _qkv_shape()
    _check_tensor("q", q, shape, torch.bfloat16)
    _check_tensor("k", k, shape, torch.bfloat16)
    elig = np.zeros(_PLAN["heads"], dtype=np.uint8) if want_elig else None
    rc = load().fas_prepass(q.data_ptr(), k.data_ptr(), _stream_handle(stream),
                            elig.ctypes.data if want_elig else None)
    _check("fas_prepass", rc)
    return elig


def key_sums_shape(heads: int, tokens: int, head_dim: int) -> tuple:
    """Shape of the 16-token key column sums: [H, N/16, d] (fp32)."""
    if tokens % 16:
        raise ValueError(f"tokens ({tokens}) must be a multiple of 16 for key sums")
    return (heads, tokens // 16, head_dim)


def fas_prepass_with_key_sums(q, k, key_sums, stream=None, want_elig: bool = False) -> Optional[np.ndarray]:
    """fas_prepass with the key column sums per 16 tokens given (fp32
    [H, N/16, d], e.g. from fas_prologue_with_key_sums): k is read once."""
    import torch
    shape = _qkv_shape()
    _check_tensor("q", q, shape, torch.bfloat16)
    _check_tensor("k", k, shape, torch.bfloat16)
    _check_tensor("key_sums", key_sums, key_sums_shape(_PLAN["heads"], _PLAN["tokens"], _PLAN["head_dim"]),
                  torch.float32)
    elig = np.zeros(_PLAN["heads"], dtype=np.uint8) if want_elig else None
    rc = load().fas_prepass_with_key_sums(q.data_ptr(), k.data_ptr(), key_sums.data_ptr(), _stream_handle(stream),
                                          elig.ctypes.data if want_elig else None)
    _check("fas_prepass_with_key_sums", rc)
    return elig


def fas_forward(q, k, v, out=None, lse=None, mode: str = "auto", stream=None):
    """Attention; returns (out bf16 [H, N, d], lse fp32 [H, N])."""
    import torch
    shape = _qkv_shape()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, shape, torch.bfloat16)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(_lse_shape(), dtype=torch.float32, device=q.device)
    _check_tensor("out", out, shape, torch.bfloat16)
    _check_tensor("lse", lse, _lse_shape(), torch.float32)
    rc = load().fas_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                            MODES[mode], _stream_handle(stream))
    _check("fas_forward", rc)
    return out, lse


def fas_forward_ablation(q, k, v, out=None, lse=None, stream=None):
    """The splash-style ablation (128-multiple tiles, padding, mask
    predicates, two passes and a merge; see ``fas_forward_ablation`` in
    fas.h); head-major [H, N, d] only.  Returns (out, lse)."""
    import torch
    shape = _qkv_shape()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, shape, torch.bfloat16)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(_lse_shape(), dtype=torch.float32, device=q.device)
    _check_tensor("out", out, shape, torch.bfloat16)
    _check_tensor("lse", lse, _lse_shape(), torch.float32)
    rc = load().fas_forward_ablation(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                     _stream_handle(stream))
    _check("fas_forward_ablation", rc)
    return out, lse


def fas_prologue_fold_weights(w, gamma, out=None, stream=None):
    """W' = bf16(W * gamma) per input feature (see fas.h): w bf16
    [3*H*d, C], gamma fp32 [C] (CUDA tensors)."""
    import torch
    O, C = w.shape
    _check_tensor("w", w, (O, C), torch.bfloat16)
    _check_tensor("gamma", gamma, (C,), torch.float32)
    if out is None:
        out = torch.empty_like(w)
    _check_tensor("out", out, (O, C), torch.bfloat16)
    _check("fas_prologue_fold_weights",
           load().fas_prologue_fold_weights(w.data_ptr(), gamma.data_ptr(), out.data_ptr(), C, O,
                                            _stream_handle(stream)))
    return out


def fas_prologue(x, w_folded, cos, sin, heads: int, head_dim: int, layout: str = "hnd", groups: int = 1,
                 ranks: int = 1, q=None, k=None, v=None, eps: float = RMS_EPS, stream=None):
    """RMSNorm -> QKV projection -> rotary -> head packing in one kernel
    (see ``fas_prologue`` in fas.h).  x bf16 [N, C]; w_folded bf16
    [3*H*d, C]; cos, sin fp32 [N, d/2].  Returns (q, k, v) bf16 in
    ``layout``: "hnd" [H, N, d], "nhd" [N, H, d] or "a2a" [G, P, N, H/(G*P), d]."""
    return _prologue(x, w_folded, cos, sin, heads, head_dim, layout, groups, ranks, q, k, v, False, None, eps,
                     stream)


def fas_prologue_with_key_sums(x, w_folded, cos, sin, heads: int, head_dim: int, layout: str = "hnd",
                               groups: int = 1, ranks: int = 1, q=None, k=None, v=None, key_sums=None,
                               eps: float = RMS_EPS, stream=None):
    """fas_prologue that also writes the column sums of the written k over
    each 16 tokens (fp32 [H, N/16, d], the input of
    fas_prepass_with_key_sums).  Returns (q, k, v, key_sums)."""
    return _prologue(x, w_folded, cos, sin, heads, head_dim, layout, groups, ranks, q, k, v, True, key_sums, eps,
                     stream)


def _prologue(x, w_folded, cos, sin, heads, head_dim, layout, groups, ranks, q, k, v, sums, key_sums, eps, stream):
    import torch
    N, C = x.shape
    _check_tensor("x", x, (N, C), torch.bfloat16)
    _check_tensor("w_folded", w_folded, (3 * heads * head_dim, C), torch.bfloat16)
    _check_tensor("cos", cos, (N, head_dim // 2), torch.float32)
    _check_tensor("sin", sin, (N, head_dim // 2), torch.float32)
    if layout == "hnd":
        shape = (heads, N, head_dim)
    elif layout == "nhd":
        shape = (N, heads, head_dim)
    elif layout == "a2a":
        if heads % (groups * ranks):
            raise ValueError(f"heads ({heads}) must divide into {groups} groups x {ranks} ranks")
        shape = (groups, ranks, N, heads // (groups * ranks), head_dim)
    else:
        raise ValueError(layout)
    outs = []
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t is None:
            t = torch.empty(shape, dtype=torch.bfloat16, device=x.device)
        _check_tensor(name, t, shape, torch.bfloat16)
        outs.append(t)
    if not sums:
        rc = load().fas_prologue(x.data_ptr(), w_folded.data_ptr(), cos.data_ptr(), sin.data_ptr(), N, C, heads,
                                 head_dim, float(eps), outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                 PROLOGUE_LAYOUTS[layout], groups, ranks, _stream_handle(stream))
        _check("fas_prologue", rc)
        return tuple(outs)
    ks_shape = key_sums_shape(heads, N, head_dim)
    if key_sums is None:
        key_sums = torch.empty(ks_shape, dtype=torch.float32, device=x.device)
    _check_tensor("key_sums", key_sums, ks_shape, torch.float32)
    rc = load().fas_prologue_with_key_sums(x.data_ptr(), w_folded.data_ptr(), cos.data_ptr(), sin.data_ptr(), N, C,
                                           heads, head_dim, float(eps), outs[0].data_ptr(), outs[1].data_ptr(),
                                           outs[2].data_ptr(), PROLOGUE_LAYOUTS[layout], groups, ranks,
                                           key_sums.data_ptr(), _stream_handle(stream))
    _check("fas_prologue_with_key_sums", rc)
    return (*outs, key_sums)


def _check_host_tensor(name, t, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, the plan needs {tuple(shape)}")


def fas_forward_host(q, k, v, out=None, lse=None, mode: str = "auto", heads_per_group: int = 0, stream=None):
    """Prepass + attention on HOST tensors (bf16 [H, N, d]; page-locked for
    copy/compute overlap), pipelined over head groups on the library's own
    streams; see ``fas_forward_host`` in fas.h.  Returns (out, lse) host
    tensors, complete once ``stream`` (default: the current CUDA stream) has
    reached this point."""
    import torch
    shape = _qkv_shape()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_host_tensor(name, t, shape, torch.bfloat16)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)
    if lse is None:
        lse = torch.empty(_lse_shape(), dtype=torch.float32, pin_memory=True)
    _check_host_tensor("out", out, shape, torch.bfloat16)
    _check_host_tensor("lse", lse, _lse_shape(), torch.float32)
    rc = load().fas_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 MODES[mode], int(heads_per_group), _stream_handle(stream))
    _check("fas_forward_host", rc)
    return out, lse


def fas_free() -> None:
    _PLAN.clear()
    _check("fas_free", load().fas_free())


def fas_status(stream=None) -> int:
    """Synchronises the stream; returns FAS_OK, FAS_ERR_TIMEOUT (a device wait
    gave up) or FAS_ERR_BOUND (a bounded row's softmax sum left its safe
    range: q or k changed since the prepass); raises on other errors."""
    rc = load().fas_status(_stream_handle(stream))
    if rc not in (FAS_OK, FAS_ERR_TIMEOUT, FAS_ERR_BOUND):
        _check("fas_status", rc)
    return rc


def fas_prepass_readback(stream=None, row_bound: bool = False) -> dict:
    H, N, d = _PLAN["heads"], _PLAN["tokens"], _PLAN["head_dim"]
    nf = _PLAN["info"].total_frames
    res = {"mu": np.zeros((H, d), np.float32), "frame_max": np.zeros((H, nf), np.float32),
           "stat": np.zeros(H, np.float32), "elig": np.zeros(H, np.uint8)}
    rb = np.zeros((H, N), np.float32) if row_bound else None
    rc = load().fas_prepass_readback(res["mu"].ctypes.data, res["frame_max"].ctypes.data, res["stat"].ctypes.data,
                                     res["elig"].ctypes.data, rb.ctypes.data if row_bound else None,
                                     _stream_handle(stream))
    _check("fas_prepass_readback", rc)
    if row_bound:
        res["row_bound"] = rb
    return res


def fas_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return load().fas_selftest_wait_timeout(limit_us, _stream_handle(stream))


def fas_prepass_noalloc(q, k, frame_tokens: int, n_frames: int, ref_frames: int, window_radius: int,
                        row_bound, stat, elig, stream=None) -> None:
    """The prepass without any allocation (see ``fas_prepass_noalloc`` in
    fas.h): the caller provides every output buffer; the library uses a fixed
    device array as scratch.  q, k: bf16 [H, N, d]; row_bound: fp32 [H, N];
    stat: fp32 [H]; elig: uint8 [H] (all CUDA tensors)."""
    import torch
    H, N, d = q.shape
    if N != (ref_frames + n_frames) * frame_tokens:
        # The C call has no plan to check the buffers against: a geometry
        # that does not match q would read past the ends of q and k.
        raise ValueError(f"q has {N} rows per head; the geometry needs (ref_frames + n_frames) * frame_tokens = "
                         f"{(ref_frames + n_frames) * frame_tokens}")
    _check_tensor("q", q, (H, N, d), torch.bfloat16)
    _check_tensor("k", k, (H, N, d), torch.bfloat16)
    _check_tensor("row_bound", row_bound, (H, N), torch.float32)
    _check_tensor("stat", stat, (H,), torch.float32)
    _check_tensor("elig", elig, (H,), torch.uint8)
    rc = load().fas_prepass_noalloc(q.data_ptr(), k.data_ptr(), frame_tokens, n_frames, ref_frames, window_radius,
                                    H, d, row_bound.data_ptr(), stat.data_ptr(), elig.data_ptr(),
                                    _stream_handle(stream))
    _check("fas_prepass_noalloc", rc)


def fas_last_launch_count() -> int:
    return load().fas_last_launch_count()
