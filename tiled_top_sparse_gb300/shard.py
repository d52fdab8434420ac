"""Partition of one hot-path step over ranks (one process per GPU, no exchange).

The step splits into independent units that need nothing from one another while they
compute: dense attention by (sequence, KV-head group) -- every query head of a group reads
only that group's keys and values, and every sequence only its own tokens; top-k by rows;
sparse attention by queries, each rank holding the whole paged KV cache (a few MB). The
pages run their engine on several GPUs ("DeepSeek V4.1 上 4×RTX 3090", 一、部署, and
"从 SGLang Kernel源码到 GPU Trace", section 1: `--tp 2`); which units each GPU owns is
this module's choice, not theirs.

Everything here is host-side planning and data movement (slicing, packing, scattering
results back); no arithmetic of the method happens here. A rank packs its units into one
call per part, runs it, and `scatter_*` puts its rows back at their places in the
single-rank layout, so the union over ranks of the scattered results is exactly the
single-rank result (a final all-gather, if wanted, is the only collective).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


# ---------------------------------------------------------------------------- planning
def dense_units(lengths_q, lengths_k, hq: int, hkv: int, causal: bool):
    """Units (sequence b, KV-head group g) with their attention work in (query, key) pairs
    per head times the group's hq / hkv query heads (the FLOPs up to a constant)."""
    if hq % hkv:
        raise ValueError("hq must be a multiple of hkv")
    r = hq // hkv
    units = []
    for b, (lq, lk) in enumerate(zip(lengths_q, lengths_k)):
        if causal:  # bottom-right aligned: row i sees keys j <= i + lk - lq
            pairs = sum(max(0, min(lk, i + lk - lq + 1)) for i in range(lq))
        else:
            pairs = lq * lk
        for g in range(hkv):
            units.append((b, g, pairs * r))
    return units


def plan_lpt(works, world: int):
    """Longest-processing-time-first assignment of units (by index) to `world` ranks.

    Units are taken heaviest first (ties: lower index first) and each goes to the rank
    with the least work so far (ties: lower rank). Deterministic; the result lists every
    unit exactly once, each rank's units in ascending index order. The heaviest rank
    carries at most mean + max unit work (the greedy bound)."""
    order = sorted(range(len(works)), key=lambda i: (-works[i], i))
    load = [0] * world
    owned = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda q: (load[q], q))
        owned[r].append(i)
        load[r] += works[i]
    return [sorted(o) for o in owned], load


def split_range(n: int, world: int, rank: int):
    """Contiguous [start, end) share of n items for `rank` (sizes differ by at most 1)."""
    return n * rank // world, n * (rank + 1) // world


# ---------------------------------------------------------------------------- dense
@dataclass
class DenseShard:
    """One rank's dense-attention units packed as one varlen batch.

    `pieces` lists (b, g0, g1): the query rows of sequence b with KV-head groups
    [g0, g1) (and their (g1 - g0) * r query heads). Units of one sequence with
    consecutive groups form a single piece (the vision encoder's head split: one
    sequence, hq' = (g1 - g0) * r heads); otherwise every (b, g) unit is its own piece
    with r query heads and one KV head. q [sum Lq, hq', d], k / v [sum Lk, hkv', d]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_q: torch.Tensor
    cu_k: torch.Tensor
    max_q: int
    max_k: int
    hq: int
    hkv: int
    pieces: list
    q_rows: list   # per piece: (token start, token end) in the full q / out
    r: int


def pack_dense(q, k, v, cu_q, cu_k, units, hq: int, hkv: int) -> DenseShard:
    """Gather the units' tokens and heads into one packed batch (on q's device)."""
    r = hq // hkv
    cq = [int(x) for x in cu_q.tolist()]
    ck = [int(x) for x in cu_k.tolist()]
    units = sorted(units)
    by_seq = {}
    for (b, g) in units:
        by_seq.setdefault(b, []).append(g)
    ranges = {b: (gs[0], gs[-1] + 1) for b, gs in by_seq.items()
              if gs == list(range(gs[0], gs[-1] + 1))}
    if len(ranges) == len(by_seq) and len(set(ranges.values())) == 1:
        # every sequence with the same contiguous groups: one piece per sequence
        pieces = [(b, g0, g1) for b, (g0, g1) in sorted(ranges.items())]
    else:
        pieces = [(b, g, g + 1) for (b, g) in units]
    qs, ks, vs, rows = [], [], [], []
    lq_list, lk_list = [0], [0]
    for (b, g0, g1) in pieces:
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        qs.append(q[q0:q1, g0 * r:g1 * r])
        ks.append(k[k0:k1, g0:g1])
        vs.append(v[k0:k1, g0:g1])
        rows.append((q0, q1))
        lq_list.append(lq_list[-1] + (q1 - q0))
        lk_list.append(lk_list[-1] + (k1 - k0))
    groups = (pieces[0][2] - pieces[0][1]) if pieces else 1
    d = q.shape[2]
    dev = q.device

    def cat(xs, heads, like):
        if xs:
            return torch.cat(xs).contiguous()
        return torch.empty((0, heads, d), dtype=like.dtype, device=dev)

    lens_q = [lq_list[i + 1] - lq_list[i] for i in range(len(pieces))]
    lens_k = [lk_list[i + 1] - lk_list[i] for i in range(len(pieces))]
    return DenseShard(cat(qs, groups * r, q), cat(ks, groups, k), cat(vs, groups, v),
                      torch.tensor(lq_list, dtype=torch.int32, device=dev),
                      torch.tensor(lk_list, dtype=torch.int32, device=dev),
                      max(lens_q + [0]), max(lens_k + [0]), groups * r, groups, pieces, rows,
                      r)


def scatter_dense(shard: DenseShard, out, lse, out_full, lse_full):
    """Put a shard's outputs (out [sum Lq, hq', d], lse [sum Lq, hq']) back in place in
    the full [T, hq, d] / [T, hq] tensors."""
    cu = [int(x) for x in shard.cu_q.tolist()]
    r = shard.r
    for i, ((b, g0, g1), (q0, q1)) in enumerate(zip(shard.pieces, shard.q_rows)):
        out_full[q0:q1, g0 * r:g1 * r] = out[cu[i]:cu[i + 1]]
        if lse is not None and lse_full is not None:
            lse_full[q0:q1, g0 * r:g1 * r] = lse[cu[i]:cu[i + 1]]


def plan_dense(lengths_q, lengths_k, hq, hkv, causal, world):
    """Per rank, the (b, g) units it owns, and every rank's load (work as in dense_units).

    When the rank count divides the KV-head count, rank r takes the same contiguous range
    of groups in every sequence: exact balance, and the rank's units pack into one call
    with hq / world query heads. Otherwise the units are assigned by plan_lpt."""
    units = dense_units(lengths_q, lengths_k, hq, hkv, causal)
    works = {(b, g): w for (b, g, w) in units}
    if hkv % world == 0:
        owned = []
        for rank in range(world):
            g0, g1 = split_range(hkv, world, rank)
            owned.append([(b, g) for b in range(len(lengths_q)) for g in range(g0, g1)])
    else:
        idx, _ = plan_lpt([w for (_, _, w) in units], world)
        owned = [[(units[i][0], units[i][1]) for i in o] for o in idx]
    return owned, [sum(works[u] for u in o) for o in owned]
