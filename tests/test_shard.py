"""The partition of one step over ranks (host logic; CPU, gloo, world size 2).

Each rank plans its share of a small step, packs its units, runs the float64 oracle on
its pack alone and scatters the rows back into the single-rank layout; summing the
ranks' scattered results (gloo all-reduce) must give exactly the oracle's result on the
whole step, with every output row written by exactly one rank. Dense attention is split
by (sequence, KV-head group), the vision-shaped batch by heads, top-k by rows and sparse
attention by queries.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as W
from tiled_top_sparse_gb300 import shard as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _dense_oracle(inp_q, inp_k, inp_v, cq, ck, causal, scale):
    return oracle.attn_varlen(inp_q.float().numpy(), inp_k.float().numpy(),
                              inp_v.float().numpy(), cq.numpy(), ck.numpy(), causal, scale)


def _step_inputs():
    var = W.dense_inputs([70, 1, 130, 0, 45, 200], hq=6, hkv=3, d=32, causal=True, seed=90)
    vis = W.vision(n=150, heads=4, d=16, seed=91)
    tk = W.topk_inputs(rows=9, cols=300, k=64, seed=92)
    sp = W.sparse_inputs(nq=5, kv_len=260, topk=96, seed=93)
    return var, vis, tk, sp


def _rank_results(rank, world):
    """This rank's share of the step, scattered into full-size tensors (zeros elsewhere),
    plus a count of how many times each output row was written."""
    var, vis, tk, sp = _step_inputs()
    res = {}
    # varlen causal GQA: (sequence, KV-head group) units, LPT-balanced (3 groups, 2 ranks)
    owned, _ = S.plan_dense(var.lengths_q, var.lengths_k, 6, 3, True, world)
    sh = S.pack_dense(var.q, var.k, var.v, var.cu_seqlens_q, var.cu_seqlens_k, owned[rank],
                      6, 3)
    out = torch.zeros(var.q.shape, dtype=torch.float64)
    lse = torch.zeros(var.q.shape[:2], dtype=torch.float64)
    cnt = torch.zeros(var.q.shape[:2], dtype=torch.float64)
    if sh.pieces:
        o, l = _dense_oracle(sh.q, sh.k, sh.v, sh.cu_q, sh.cu_k, True, var.scale)
        S.scatter_dense(sh, torch.from_numpy(o), torch.from_numpy(l), out, lse)
        S.scatter_dense(sh, torch.ones(o.shape), torch.ones(l.shape), torch.zeros_like(out),
                        cnt)
    res["varlen"] = (out, lse, cnt)
    # vision-shaped: contiguous heads of one sequence
    units = S.plan_dense(vis.lengths_q, vis.lengths_k, 4, 4, False, world)[0][rank]
    sh = S.pack_dense(vis.q, vis.k, vis.v, vis.cu_seqlens_q, vis.cu_seqlens_k, units, 4, 4)
    assert len(sh.pieces) <= 1  # one packed sequence with this rank's heads
    out = torch.zeros(vis.q.shape, dtype=torch.float64)
    lse = torch.zeros(vis.q.shape[:2], dtype=torch.float64)
    cnt = torch.zeros(vis.q.shape[:2], dtype=torch.float64)
    if sh.pieces:
        o, l = _dense_oracle(sh.q, sh.k, sh.v, sh.cu_q, sh.cu_k, False, vis.scale)
        S.scatter_dense(sh, torch.from_numpy(o), torch.from_numpy(l), out, lse)
        S.scatter_dense(sh, torch.ones(o.shape), torch.ones(l.shape), torch.zeros_like(out),
                        cnt)
    res["vision"] = (out, lse, cnt)
    # top-k: rows
    r0, r1 = S.split_range(tk.logits.shape[0], world, rank)
    idx = torch.zeros((tk.logits.shape[0], tk.k), dtype=torch.float64)
    cnt = torch.zeros(tk.logits.shape[0], dtype=torch.float64)
    if r1 > r0:
        got, _ = oracle.topk(tk.logits[r0:r1].numpy(), tk.row_starts[r0:r1].numpy(),
                             tk.row_lens[r0:r1].numpy(), tk.k)
        idx[r0:r1] = torch.from_numpy(got.astype(np.float64))
        cnt[r0:r1] = 1
    res["topk"] = (idx, cnt)
    # sparse: queries (the paged cache is whole on every rank)
    n0, n1 = S.split_range(sp.q.shape[0], world, rank)
    out = torch.zeros((sp.q.shape[0], sp.q.shape[1], sp.dv), dtype=torch.float64)
    cnt = torch.zeros(sp.q.shape[0], dtype=torch.float64)
    if n1 > n0:
        o, _, _ = oracle.sparse_paged(sp.q[n0:n1].float().numpy(), sp.kv_cache.float().numpy(),
                                      sp.page_table.numpy(), sp.idx[n0:n1].numpy(), sp.kv_len,
                                      sp.dv, sp.scale)
        out[n0:n1] = torch.from_numpy(o)
        cnt[n0:n1] = 1
    res["sparse"] = (out, cnt)
    return res


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = _rank_results(rank, world)
        for key in sorted(res):
            for t in res[key]:
                dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            q.put({k: [t.numpy() for t in v] for k, v in res.items()})
    finally:
        dist.destroy_process_group()


def test_two_rank_partition_reassembles_the_single_rank_step():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    var, vis, tk, sp = _step_inputs()
    ro, rl = _dense_oracle(var.q, var.k, var.v, var.cu_seqlens_q, var.cu_seqlens_k, True,
                           var.scale)
    out, lse, cnt = got["varlen"]
    assert np.all(cnt == 1)           # every (token, head) row written by exactly one rank
    assert np.array_equal(out, ro)    # same float64 arithmetic per row: bitwise equal
    assert np.array_equal(lse, rl)
    ro, rl = _dense_oracle(vis.q, vis.k, vis.v, vis.cu_seqlens_q, vis.cu_seqlens_k, False,
                           vis.scale)
    out, lse, cnt = got["vision"]
    assert np.all(cnt == 1)
    assert np.array_equal(out, ro) and np.array_equal(lse, rl)
    ref, _ = oracle.topk(tk.logits.numpy(), tk.row_starts.numpy(), tk.row_lens.numpy(), tk.k)
    idx, cnt = got["topk"]
    assert np.all(cnt == 1) and np.array_equal(idx, ref.astype(np.float64))
    ro, _, _ = oracle.sparse_paged(sp.q.float().numpy(), sp.kv_cache.float().numpy(),
                                   sp.page_table.numpy(), sp.idx.numpy(), sp.kv_len, sp.dv,
                                   sp.scale)
    out, cnt = got["sparse"]
    assert np.all(cnt == 1) and np.array_equal(out, ro)


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_varlen_plan_covers_every_unit_once_and_is_balanced(world):
    lengths = W.varlen_lengths(2)  # the benchmark's accepted batch
    units = S.dense_units(lengths, lengths, 32, 8, True)
    owned, load = S.plan_dense(lengths, lengths, 32, 8, True, world)
    flat = [u for o in owned for u in o]
    assert sorted(flat) == sorted((b, g) for (b, g, _) in units) and len(flat) == len(set(flat))
    works = {(b, g): w for (b, g, w) in units}
    assert load == [sum(works[u] for u in o) for o in owned]
    mean = sum(load) / world
    assert max(load) <= mean + max(works.values())  # the greedy bound
    if world <= 8:  # 64 units of unequal work: within 10 % of perfect at these sizes
        assert max(load) <= 1.10 * mean, (world, max(load) / mean)


def test_causal_unit_work_counts_visible_pairs():
    # bottom-right alignment: Lq = 3, Lk = 5 -> rows see 3, 4, 5 keys
    assert S.dense_units([3], [5], 2, 1, True) == [(0, 0, (3 + 4 + 5) * 2)]
    assert S.dense_units([4], [4], 1, 1, True) == [(0, 0, 10)]
    assert S.dense_units([4], [2], 1, 1, True) == [(0, 0, 0 + 0 + 1 + 2)]
    assert S.dense_units([3], [5], 1, 1, False) == [(0, 0, 15)]


def test_split_range_and_heads_cover_exactly():
    for n in (0, 1, 7, 16, 323):
        for world in (1, 2, 3, 8):
            spans = [S.split_range(n, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            assert max(b - a for a, b in spans) - min(b - a for a, b in spans) <= 1
    owned, load = S.plan_dense([8547], [8547], 16, 16, False, 2)  # vision: heads split
    assert owned == [[(0, g) for g in range(8)], [(0, g) for g in range(8, 16)]]
    assert load[0] == load[1]


def test_pack_makes_one_call_per_rank():
    var = W.dense_inputs([70, 1, 130, 0, 45, 200], hq=8, hkv=4, d=16, causal=True, seed=94)
    owned, _ = S.plan_dense(var.lengths_q, var.lengths_k, 8, 4, True, 2)  # groups split
    sh = S.pack_dense(var.q, var.k, var.v, var.cu_seqlens_q, var.cu_seqlens_k, owned[1], 8, 4)
    assert (sh.hq, sh.hkv) == (4, 2) and [p[1:] for p in sh.pieces] == [(2, 4)] * 6
    assert torch.equal(sh.q[:70], var.q[:70, 4:8]) and torch.equal(sh.k[:70], var.k[:70, 2:4])
    owned, _ = S.plan_dense(var.lengths_q, var.lengths_k, 8, 4, True, 3)  # LPT units
    for o in owned:
        sh = S.pack_dense(var.q, var.k, var.v, var.cu_seqlens_q, var.cu_seqlens_k, o, 8, 4)
        assert (sh.hq, sh.hkv) == (2, 1) and len(sh.pieces) == len(o)
