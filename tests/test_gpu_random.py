"""Seeded random sweeps of every entry point against the float64 oracle.

Each test draws a handful of configurations from a fixed seed (shapes, value
distributions, ties, windows, index lists) at sizes the oracle finishes in seconds, and
holds the results to the same bars as the targeted tests: indices bit-exact, attention
within the stated tolerances, sparse outputs bitwise invariant under index permutations.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close_attn, assert_lse_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts():
    import tiled_top_sparse_gb300 as m
    m.lib()
    return m


def _logits(rng, rows, cols):
    """One of several value distributions, chosen per row."""
    x = np.empty((rows, cols), np.float32)
    for r in range(rows):
        kind = rng.integers(0, 6)
        if kind == 0:    # normal on the bf16 grid (ties)
            v = torch.from_numpy(rng.standard_normal(cols).astype(np.float32))
            x[r] = v.to(torch.bfloat16).float().numpy()
        elif kind == 1:  # plain fp32 normal (few ties)
            x[r] = rng.standard_normal(cols)
        elif kind == 2:  # few distinct integers (heavy ties)
            x[r] = rng.integers(-3, 4, cols)
        elif kind == 3:  # one-signed, wide dynamic range
            x[r] = np.exp(rng.uniform(-30, 30, cols)).astype(np.float32)
        elif kind == 4:  # mostly equal with signed zeros and infinities sprinkled in
            v = np.full(cols, 0.5, np.float32)
            m = rng.integers(0, cols, max(1, cols // 50))
            v[m] = rng.choice(np.array([0.0, -0.0, np.inf, -np.inf, 7.0], np.float32), m.size)
            x[r] = v
        else:            # a sorted ramp, ascending or descending
            v = np.linspace(-2, 2, cols, dtype=np.float32)
            x[r] = v if rng.integers(0, 2) else v[::-1]
    return x


@pytest.mark.parametrize("seed", range(6))
def test_random_topk_windows(tts, seed):
    rng = np.random.default_rng(1000 + seed)
    rows = int(rng.integers(1, 40))
    cols = int(rng.choice([7, 300, 2590, 4096, 5000, 16384]))
    k = int(rng.integers(1, min(4096, 2 * cols) + 1))
    x = _logits(rng, rows, cols)
    starts = rng.integers(0, cols, rows).astype(np.int32) // 3
    lens = np.minimum(rng.integers(0, cols + 1, rows), cols - starts).astype(np.int32)
    if rows > 2:
        starts[0], lens[0] = 0, cols          # whole row
        starts[1], lens[1] = cols - 1, 2      # a window past the row's end: flagged, all -1
    inp = W.TopkInputs(torch.from_numpy(x), torch.from_numpy(starts), torch.from_numpy(lens), k)
    ref, bad = oracle.topk(x, starts, lens, k)
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = tts.topk_select(inp.logits.to(dev), inp.row_starts.to(dev), inp.row_lens.to(dev), k,
                          status=st)
    assert np.array_equal(got.cpu().numpy(), ref), f"seed {seed}: rows {rows} cols {cols} k {k}"
    assert bool(int(st.item()) & tts.TTS_DEV_INDEX_RANGE) == (bad > 0)
    got_l = tts.topk_select_long(inp.logits.to(dev), inp.row_starts.to(dev),
                                 inp.row_lens.to(dev), k)
    assert np.array_equal(got_l.cpu().numpy(), ref), f"seed {seed} (long-row path)"


@pytest.mark.parametrize("seed", range(3))
def test_random_long_rows(tts, seed):
    rng = np.random.default_rng(2000 + seed)
    rows = int(rng.integers(1, 6))
    cols = int(rng.choice([16385, 50000, 131072]))
    k = int(rng.choice([1, 100, 2048, 4096]))
    x = _logits(rng, rows, cols)
    starts = np.zeros(rows, np.int32)
    lens = rng.integers(cols // 2, cols + 1, rows).astype(np.int32)
    ref, _ = oracle.topk(x, starts, lens, k)
    dev = torch.device("cuda")
    got = tts.topk_select_long(torch.from_numpy(x).to(dev), torch.from_numpy(starts).to(dev),
                               torch.from_numpy(lens).to(dev), k)
    assert np.array_equal(got.cpu().numpy(), ref), f"seed {seed}: rows {rows} cols {cols} k {k}"


@pytest.mark.parametrize("seed", range(6))
def test_random_dense_batches(tts, seed):
    rng = np.random.default_rng(3000 + seed)
    d = int(rng.choice([64, 80, 128]))
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    causal = bool(rng.integers(0, 2))
    batch = int(rng.integers(1, 6))
    lq = [int(v) for v in rng.integers(0, 700, batch)]
    lk = lq if rng.integers(0, 2) else [int(v) for v in rng.integers(0, 700, batch)]
    dtype = torch.float32 if rng.integers(0, 4) == 0 else torch.bfloat16
    inp = W.dense_inputs(lq, lk, hq=hq, hkv=hkv, d=d, causal=causal, dtype=dtype, seed=seed)
    if max(lq) == 0:
        return
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = tts.attn_fwd_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                                   inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev),
                                   inp.max_seqlen_q, inp.max_seqlen_k, causal, inp.scale,
                                   status=st)
    tts.check_status(st)
    q, k, v = (t.float().numpy() for t in (inp.q, inp.k, inp.v))
    if dtype == torch.float32:  # the CUDA path rounds fp32 inputs to bf16 first
        q, k, v = oracle.round_bf16(q), oracle.round_bf16(k), oracle.round_bf16(v)
    ro, rl = oracle.attn_varlen(q, k, v, inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(),
                                causal, inp.scale)
    what = f"seed {seed}: d {d} {hq}/{hkv} causal {causal} lq {lq} lk {lk} {dtype}"
    assert_close_attn(out.cpu().numpy(), ro, what)
    assert_lse_close(lse.cpu().numpy(), rl, what)


@pytest.mark.parametrize("seed", range(5))
def test_random_sparse_lists(tts, seed):
    rng = np.random.default_rng(4000 + seed)
    nq = int(rng.integers(1, 9))
    kv_len = int(rng.integers(1, 6000))
    page_size = int(rng.choice([1, 16, 64, 100]))
    topk = int(rng.integers(1, 2049))
    inp = W.sparse_inputs(nq=nq, kv_len=kv_len, page_size=page_size, topk=topk, seed=seed,
                          causal_windows=False)
    idx = inp.idx.clone()
    for n in range(nq):                      # holes and duplicates
        holes = rng.integers(0, topk, topk // 4)
        idx[n, holes] = -1
        if topk > 2:
            idx[n, 1] = idx[n, 0]
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    args = [inp.q.to(dev), inp.kv_cache.to(dev), inp.page_table.to(dev)]
    out, lse = tts.sparse_attn_paged(*args, idx.to(dev), inp.kv_len, inp.scale, status=st)
    tts.check_status(st)
    ro, rl, bad = oracle.sparse_paged(inp.q.float().numpy(), inp.kv_cache.float().numpy(),
                                      inp.page_table.numpy(), idx.numpy(), inp.kv_len, inp.dv,
                                      inp.scale)
    assert bad == 0
    what = f"seed {seed}: nq {nq} kv_len {kv_len} page {page_size} topk {topk}"
    empty = (idx < 0).all(dim=1).numpy()
    if not empty.all():
        assert_close_attn(out.cpu().numpy()[~empty], ro[~empty], what)
    assert_lse_close(lse.cpu().numpy(), rl, what)
    p_out, p_lse = tts.sparse_attn_paged(*args, W.permute_rows(idx, seed).to(dev), inp.kv_len,
                                         inp.scale)
    assert torch.equal(p_out, out) and torch.equal(p_lse, lse)


@pytest.mark.parametrize("seed", range(3))
def test_random_decode_requests(tts, seed):
    rng = np.random.default_rng(5000 + seed)
    lens = [int(v) for v in rng.integers(1, 9000, int(rng.integers(1, 7)))]
    inp = W.sparse_decode_inputs(kv_lens=lens, topk=int(rng.integers(1, 2049)), seed=seed,
                                 page_size=int(rng.choice([16, 64])))
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = tts.sparse_attn_decode(inp.q.to(dev), inp.kv_cache.to(dev),
                                      inp.page_tables.to(dev), inp.kv_lens.to(dev),
                                      inp.idx.to(dev), inp.scale, dv=inp.dv, status=st)
    tts.check_status(st)
    q, kv, ix = inp.q.float().numpy(), inp.kv_cache.float().numpy(), inp.idx.numpy()
    for n, L in enumerate(lens):
        ro, rl, bad = oracle.sparse_paged(q[n:n + 1], kv, inp.page_tables[n].numpy(),
                                          ix[n:n + 1], L, inp.dv, inp.scale)
        assert bad == 0
        assert_close_attn(out[n:n + 1].cpu().numpy(), ro, f"seed {seed} request {n} len {L}")
        assert_lse_close(lse[n:n + 1].cpu().numpy(), rl, f"seed {seed} request {n}")
