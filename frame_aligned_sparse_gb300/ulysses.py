"""Head-grouped Ulysses sequence parallelism around the sparse attention.

"HeyGen x Google Cloud: Avatar IV on TPU", section "Hiding the Collective"
and Fig. 2: under Ulysses sequence parallelism each self-attention trades
sequence shards for head shards with an all-to-all, runs the attention on
whole sequences of a subset of heads, and trades back.  Splitting the heads
into independent groups turns the monolithic all-to-all into a pipeline:
each group's transfer hides behind another group's attention, leaving only
the first entry and the last return exposed.  The sparse mask is defined
over a token order, and the head grouping leaves that order untouched, so
every group sees exactly the mask it would see unsplit.

Layout ("Layout Is the ABI", Fig. 5: the producer writes the collective's
operand layout, so nothing is repacked).  With P ranks, G head groups and
H heads, every rank holds its contiguous token shard of n = N / P tokens
(rank p: tokens p*n .. p*n + n - 1) in the all-to-all layout

    [G, P, n, hp, d],   hp = H / (G * P),

element [g, r, t, j] being token p*n + t of head g*(H/G) + r*hp + j.  For
group g the slab x[g] ([P, n, hp, d], contiguous) is the all-to-all's input
as it stands: slice r goes to rank r.  Rank r receives [P, n, hp, d] with
the source ranks in order, which is the token-major [N, hp, d] tensor of its
hp heads of group g with the tokens in their original order: the input the
attention reads (``fas_set_layout("nhd")``), again with no copy.  The
attention's output [N, hp, d] goes back through the same all-to-all and
lands in the same [G, P, n, hp, d] layout on the token shard's owner.
``to_a2a_layout`` and ``from_a2a_layout`` convert from and to a plain
[n, H, d] shard for callers whose producer does not write this layout.

Every rank runs the same schedule; the collectives are NCCL's all-to-all
(gloo on CPU) through ``torch.distributed``, and the attention is the
library's kernels on the rank's own GPU.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

__all__ = ["a2a_heads_per_rank", "to_a2a_layout", "from_a2a_layout", "schedule", "ulysses_attention",
           "fas_attention_fn"]


def a2a_heads_per_rank(heads: int, groups: int, world: int) -> int:
    """Heads of one group that one rank attends to (hp)."""
    if heads % (groups * world) != 0:
        raise ValueError(f"heads ({heads}) must divide into {groups} groups x {world} ranks")
    return heads // (groups * world)


def to_a2a_layout(x, groups: int, world: int):
    """Plain token shard [n, H, d] -> all-to-all layout [G, P, n, hp, d]."""
    n, H, d = x.shape
    hp = a2a_heads_per_rank(H, groups, world)
    return x.reshape(n, groups, world, hp, d).permute(1, 2, 0, 3, 4).contiguous()


def from_a2a_layout(y):
    """All-to-all layout [G, P, n, hp, d] -> plain token shard [n, H, d]."""
    G, P, n, hp, d = y.shape
    return y.permute(2, 0, 1, 3, 4).reshape(n, G * P * hp, d)


def schedule(groups: int) -> List[Tuple[str, int]]:
    """Issue order of the per-group steps: ("in", g) all-to-all of group g's
    q, k, v to head shards; ("attn", g) its attention; ("out", g) the
    all-to-all of its output back to token shards.  Group g+1's transfer is
    issued before group g's attention, so it runs while that attention
    computes; group g's return is issued right after its attention."""
    ops = [("in", 0)]
    for g in range(groups):
        if g + 1 < groups:
            ops.append(("in", g + 1))
        ops.append(("attn", g))
        ops.append(("out", g))
    return ops


AttentionFn = Callable[[object, object, object], Tuple[object, object]]


def ulysses_attention(q, k, v, attn_fn: AttentionFn, group=None):
    """Sequence-parallel attention, pipelined over head groups.

    q, k, v: this rank's token shard in the all-to-all layout
    [G, P, n, hp, d] (see the module docstring).  attn_fn(q, k, v) takes
    token-major [N, hp, d] tensors of whole sequences (tokens in their
    original order) and returns (out [N, hp, d], lse [hp, N]).

    Returns (out, lse): out in the same [G, P, n, hp, d] layout (this rank's
    tokens, all heads), lse [G, hp, N] for the heads this rank attended to
    (group g, heads g*(H/G) + rank*hp + j).
    """
    import torch
    import torch.distributed as dist

    G, P, n, hp, d = q.shape
    world = dist.get_world_size(group)
    if P != world:
        raise ValueError(f"q has {P} rank slices, the process group has {world} ranks")
    for name, t in (("k", k), ("v", v)):
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, q has {tuple(q.shape)}")
    N = P * n
    recv = [[torch.empty((P, n, hp, d), dtype=x.dtype, device=x.device) for x in (q, k, v)] for _ in range(G)]
    outs: List[Optional[object]] = [None] * G
    lses: List[Optional[object]] = [None] * G
    result = torch.empty_like(q)
    pending_in = {}
    pending_out = []
    for op, g in schedule(G):
        if op == "in":
            pending_in[g] = [dist.all_to_all_single(recv[g][i], x[g], group=group, async_op=True)
                             for i, x in enumerate((q, k, v))]
        elif op == "attn":
            for w in pending_in.pop(g):
                w.wait()
            qg, kg, vg = (t.view(N, hp, d) for t in recv[g])
            out, lse = attn_fn(qg, kg, vg)
            outs[g] = out.reshape(P, n, hp, d).contiguous()
            lses[g] = lse
        else:
            pending_out.append(dist.all_to_all_single(result[g], outs[g], group=group, async_op=True))
    for w in pending_out:
        w.wait()
    return result, torch.stack(lses)


def fas_attention_fn(frame_tokens, n_frames: int, ref_frames: int, window_radius: int, heads: int,
                     head_dim: int, mode: str = "auto", stream=None) -> AttentionFn:
    """attn_fn for ``ulysses_attention`` on the library's kernels: a plan for
    hp heads, the token-major layout, prepass and attention on the rank's
    GPU.  frame_tokens as in ``fas_plan`` (one span, or per-frame spans)."""
    import frame_aligned_sparse_gb300 as fas

    def fn(q, k, v):
        fas.fas_plan(frame_tokens, n_frames, ref_frames, window_radius, heads, head_dim)
        fas.fas_set_layout("nhd")
        fas.fas_prepass(q, k, stream=stream)
        return fas.fas_forward(q, k, v, mode=mode, stream=stream)

    return fn
