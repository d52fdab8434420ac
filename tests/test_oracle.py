"""Pins for the float64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: a closed form, an
invariant, a library routine the oracle does not call (torch SDPA in float64,
numpy's stable argsort, torch's bf16 cast), brute force on tiny inputs, or a
worked example printed in the pages. Together they are chosen so that a dropped
term, a wrong sign or index, or a transposed operand anywhere in the oracle
fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.float().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


# --------------------------------------------------------------------- bf16 rounding
def test_round_bf16_matches_torch_cast():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 4)
    # exact halfway cases: 1 + 2^-8 (ties to even -> 1), 1 + 3*2^-8 (-> 1 + 2^-6 ... even)
    extra = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0, 3.0e38, 1e-40])
    x = torch.cat([x, extra]).float()
    ref = x.to(torch.bfloat16).float().numpy()
    got = oracle.round_bf16(x.numpy())
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------- O1 dense attention
def _attn_all(inp: W.DenseInputs):
    return oracle.attn_varlen(_np(inp.q), _np(inp.k), _np(inp.v), inp.cu_seqlens_q.numpy(),
                              inp.cu_seqlens_k.numpy(), inp.causal, inp.scale)


def test_attn_q_zero_is_mean_of_visible_v_bottom_right_causal():
    # Lq = 3, Lk = 5, causal with bottom-right alignment: row i sees keys 0..i+2.
    inp = W.dense_inputs([3, 4], [5, 2], hq=2, hkv=1, d=8, causal=True, dtype=torch.float32,
                         seed=11)
    q = np.zeros_like(_np(inp.q))
    out, lse = oracle.attn_varlen(q, _np(inp.k), _np(inp.v), inp.cu_seqlens_q.numpy(),
                                  inp.cu_seqlens_k.numpy(), True, 0.3)
    v = _np(inp.v).astype(np.float64)
    for i in range(3):  # sequence 0: keys 0..i+2 of 5
        n = i + 3
        np.testing.assert_allclose(out[i, :, :], np.broadcast_to(v[:n, 0].mean(0), (2, 8)),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[i], math.log(n), rtol=0, atol=1e-13)
    # sequence 1: Lq = 4 > Lk = 2: rows 0, 1 see nothing; row 2 sees key 0; row 3 sees 0..1
    base = 3
    assert np.all(out[base + 0] == 0) and np.all(out[base + 1] == 0)
    assert np.all(np.isneginf(lse[base:base + 2]))
    np.testing.assert_allclose(out[base + 2, 0], v[5, 0], atol=1e-14)
    np.testing.assert_allclose(out[base + 3, 1], v[5:7, 0].mean(0), atol=1e-14)
    np.testing.assert_allclose(lse[base + 3], math.log(2), atol=1e-14)


def test_attn_huge_scale_is_argmax_row():
    inp = W.dense_inputs([17], hq=2, hkv=2, d=16, causal=False, dtype=torch.float32, seed=12)
    scale = 1e4
    out, lse = oracle.attn_varlen(_np(inp.q), _np(inp.k), _np(inp.v), inp.cu_seqlens_q.numpy(),
                                  inp.cu_seqlens_k.numpy(), False, scale)
    q, k, v = (_np(t).astype(np.float64) for t in (inp.q, inp.k, inp.v))
    for h in range(2):
        s = q[:, h] @ k[:, h].T
        j = s.argmax(1)
        np.testing.assert_allclose(out[:, h], v[j, h], atol=1e-9)
        np.testing.assert_allclose(lse[:, h], scale * s.max(1), rtol=1e-12)


def test_attn_causal_row0_is_v0():
    inp = W.dense_inputs([9, 5, 1], hq=4, hkv=2, d=8, causal=True, dtype=torch.float32, seed=13)
    out, lse = _attn_all(inp)
    q, k, v = (_np(t).astype(np.float64) for t in (inp.q, inp.k, inp.v))
    for b in range(3):
        t0 = int(inp.cu_seqlens_q[b])
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(out[t0, h], v[t0, g], atol=1e-15)
            np.testing.assert_allclose(lse[t0, h], inp.scale * q[t0, h] @ k[t0, g], rtol=1e-13)


def test_attn_identical_keys_give_uniform_weights():
    inp = W.dense_inputs([12], hq=1, hkv=1, d=4, causal=False, dtype=torch.float32, seed=14)
    k = np.repeat(_np(inp.k)[:1], 12, axis=0)
    out, lse = oracle.attn_varlen(_np(inp.q), k, _np(inp.v), inp.cu_seqlens_q.numpy(),
                                  inp.cu_seqlens_k.numpy(), False, 0.5)
    v = _np(inp.v).astype(np.float64)
    np.testing.assert_allclose(out[:, 0], np.broadcast_to(v[:, 0].mean(0), (12, 4)), atol=1e-14)


def test_attn_rows_of_p_sum_to_one():
    # V = identity (Lk <= d) turns each output row into the probability row itself.
    L = 24
    inp = W.dense_inputs([L], hq=1, hkv=1, d=32, causal=True, dtype=torch.float32, seed=15)
    v = np.zeros((L, 1, 32), np.float32)
    for j in range(L):
        v[j, 0, j] = 1.0
    out, lse = oracle.attn_varlen(_np(inp.q), _np(inp.k), v, inp.cu_seqlens_q.numpy(),
                                  inp.cu_seqlens_k.numpy(), True, 1.0)
    p = out[:, 0, :L]
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-12)
    assert np.all(np.triu(p, 1) == 0)  # causal: no weight above the diagonal
    # p_j = exp(s_j - lse) exactly (the definition of lse)
    q, k = _np(inp.q).astype(np.float64), _np(inp.k).astype(np.float64)
    s = q[:, 0] @ k[:, 0].T
    ref = np.tril(np.exp(s - lse[:, 0:1]))
    np.testing.assert_allclose(p, ref, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("causal", [False, True])
def test_attn_matches_torch_sdpa_float64_with_gqa(causal):
    lens = [33, 7, 64]
    inp = W.dense_inputs(lens, hq=6, hkv=2, d=16, causal=causal, dtype=torch.float32, seed=16)
    out, lse = _attn_all(inp)
    for b, L in enumerate(lens):
        t0 = int(inp.cu_seqlens_q[b])
        q = inp.q[t0:t0 + L].double().transpose(0, 1)[None]
        k = inp.k[t0:t0 + L].double().transpose(0, 1)[None]
        v = inp.v[t0:t0 + L].double().transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=causal, scale=inp.scale, enable_gqa=True)[0].transpose(0, 1)
        np.testing.assert_allclose(out[t0:t0 + L], ref.numpy(), rtol=0, atol=1e-12)


def test_attn_brute_force_tiny():
    # per-element loops, no matrix products: a different algorithm from the oracle's
    inp = W.dense_inputs([5], hq=2, hkv=1, d=3, causal=True, dtype=torch.float32, seed=17)
    out, lse = _attn_all(inp)
    q, k, v = (_np(t).astype(np.float64) for t in (inp.q, inp.k, inp.v))
    for h in range(2):
        for i in range(5):
            w = [math.exp(inp.scale * sum(q[i, h, t] * k[j, 0, t] for t in range(3)))
                 for j in range(i + 1)]
            z = sum(w)
            for t in range(3):
                assert abs(out[i, h, t] - sum(w[j] * v[j, 0, t] for j in range(i + 1)) / z) < 1e-13
            assert abs(lse[i, h] - math.log(z)) < 1e-13


def test_attn_online_merge_equations_reproduce_full_row():
    # Equations 1-2 of the V32 write-up (进一步探索): merging the (m, s) statistics of two
    # key blocks gives the statistics of the union. In log form: lse = logaddexp(lse_A, lse_B)
    # and out = (e^{lse_A} out_A + e^{lse_B} out_B) / e^{lse}.
    L, half = 40, 17
    inp = W.dense_inputs([L], hq=2, hkv=2, d=8, causal=False, dtype=torch.float32, seed=18)
    q, k, v = _np(inp.q), _np(inp.k), _np(inp.v)
    cq = np.array([0, L], np.int32)
    full_o, full_l = oracle.attn_varlen(q, k, v, cq, cq, False, inp.scale)
    oa, la = oracle.attn_varlen(q, k[:half], v[:half], cq, np.array([0, half], np.int32), False,
                                inp.scale)
    ob, lb = oracle.attn_varlen(q, k[half:], v[half:], cq, np.array([0, L - half], np.int32),
                                False, inp.scale)
    m = np.maximum(la, lb)  # eq. 1 on the per-block log-sums
    s = np.exp(la - m) + np.exp(lb - m)  # eq. 2
    np.testing.assert_allclose(full_l, m + np.log(s), rtol=1e-13)
    merged = (np.exp(la - full_l)[..., None] * oa + np.exp(lb - full_l)[..., None] * ob)
    np.testing.assert_allclose(full_o, merged, atol=1e-13)


def test_attn_sampled_rows_equal_full():
    inp = W.dense_inputs([50, 70], hq=4, hkv=2, d=16, causal=True, dtype=torch.float32, seed=19)
    out, lse = _attn_all(inp)
    tok = np.array([0, 49, 50, 119, 77], np.int32)
    head = np.array([0, 3, 1, 2, 3], np.int32)
    o2, l2 = oracle.attn_varlen(_np(inp.q), _np(inp.k), _np(inp.v), inp.cu_seqlens_q.numpy(),
                                inp.cu_seqlens_k.numpy(), True, inp.scale, rows=(tok, head))
    assert np.array_equal(o2, out[tok, head]) and np.array_equal(l2, lse[tok, head])


def test_attn_rejects_bad_cu_seqlens():
    inp = W.dense_inputs([4, 4], hq=1, hkv=1, d=4, dtype=torch.float32, seed=20)
    bad = np.array([0, 5, 3], np.int32)
    with pytest.raises(ValueError):
        oracle.attn_varlen(_np(inp.q), _np(inp.k), _np(inp.v), bad, bad, False, 1.0)


# --------------------------------------------------------------------- O2 top-k
def test_topk_matches_numpy_stable_argsort_with_ties():
    inp = W.topk_inputs(rows=40, cols=700, k=256, seed=21)
    x = inp.logits.numpy()
    idx, bad = oracle.topk(x, inp.row_starts.numpy(), inp.row_lens.numpy(), inp.k)
    assert bad == 0
    for r in range(40):
        L = int(inp.row_lens[r])
        ref = np.argsort(-x[r, :L], kind="stable")[:inp.k]
        assert np.array_equal(idx[r, :len(ref)], ref)
    # the bf16 grid really produced boundary ties
    vals = np.sort(x[0, :int(inp.row_lens[0])])[::-1]
    assert len(np.unique(vals)) < len(vals)


def test_topk_brute_force_repeated_max():
    g = np.random.default_rng(22)
    for trial in range(30):
        n = int(g.integers(1, 64))
        k = int(g.integers(1, 70))
        x = g.integers(-3, 4, size=n).astype(np.float32)  # many ties
        idx, _ = oracle.topk(x[None], [0], [n], k)
        taken, ref = set(), []
        for _ in range(min(k, n)):
            best = None
            for j in range(n):  # first (lowest) position holding the largest remaining value
                if j not in taken and (best is None or x[j] > x[best]):
                    best = j
            taken.add(best)
            ref.append(best)
        assert list(idx[0, :len(ref)]) == ref
        assert np.all(idx[0, len(ref):] == -1)


def test_topk_invariants_full_size():
    inp = W.topk_inputs()
    x = inp.logits.numpy()
    idx, bad = oracle.topk(x, inp.row_starts.numpy(), inp.row_lens.numpy(), inp.k)
    assert bad == 0 and idx.shape == (323, 2048)
    for r in range(0, 323, 17):
        L = int(inp.row_lens[r])
        sel = idx[r]
        assert np.all((sel >= 0) & (sel < L)) and len(np.unique(sel)) == 2048
        v = x[r, sel]
        assert np.all(np.diff(v) <= 0)  # value descending
        eq = np.diff(v) == 0
        assert np.all(np.diff(sel)[eq] > 0)  # equal values by ascending index
        rest = np.setdiff1d(np.arange(L), sel)
        t = v[-1]
        assert np.all(x[r, rest] <= t)
        # among boundary ties, the selected are the lowest indices
        tied_out = rest[x[r, rest] == t]
        tied_in = sel[v == t]
        if len(tied_out):
            assert tied_in.max() < tied_out.min()


def test_topk_worked_example_boundary_tie():
    fx = {}
    with open(os.path.join(GOLDEN, "topk_boundary_tie.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, *vals = line.split()
                fx[key] = [int(v) for v in vals]
    rows, cols, k, row = fx["rows"][0], fx["cols"][0], fx["k"][0], fx["row"][0]
    inp = W.topk_inputs(rows=rows, cols=cols, k=k, seed=23)
    x = inp.logits.numpy().copy()
    L = int(inp.row_lens[row])
    a, b, c = fx["stable_window"]
    loser = fx["unstable_window"][2]
    col = fx["flat_first"][0] - row * k  # column of the window's first entry
    g = np.random.default_rng(24)
    # Row `row`: `col` selected positions below a, then a, b(tie), c, loser(tie) dropped,
    # the rest of the k selections above the loser; every other position below the tie.
    below = g.permutation(a)[:col]
    above = np.arange(loser + 1, L)
    above = g.permutation(above)[:k - col - 3]
    sel = np.concatenate([below, [a, b, c], above])
    y = g.uniform(-3.0, 0.25, size=cols).astype(np.float32)
    y[sel] = g.uniform(1.0, 2.0, size=len(sel)).astype(np.float32)
    y[b] = y[loser] = 0.5
    x[row] = y
    idx, bad = oracle.topk(x, inp.row_starts.numpy(), inp.row_lens.numpy(), k)
    srt = np.sort(idx, axis=1)
    flat = srt.reshape(-1)
    first = fx["flat_first"][0]
    assert list(flat[first:first + 3]) == fx["stable_window"]
    assert list(flat[first:first + 3]) != fx["unstable_window"]
    assert loser not in idx[row]
    assert idx[row, k - 1] == b  # the tie winner sits at the last selected rank


def test_topk_short_rows_offsets_and_bad_windows():
    x = np.arange(20, dtype=np.float32)[None].repeat(4, 0)
    x[1, 5:9] = [1.0, -0.0, 0.0, 1.0]
    starts = np.array([0, 5, 18, -1], np.int32)
    lens = np.array([3, 4, 5, 2], np.int32)  # row 2: 18+5 > 20, row 3: negative start
    idx, bad = oracle.topk(x, starts, lens, 6)
    assert bad == 2
    assert list(idx[0]) == [2, 1, 0, -1, -1, -1]
    assert list(idx[1]) == [0, 3, 1, 2, -1, -1]  # -0.0 == +0.0: lower index first
    assert np.all(idx[2] == -1) and np.all(idx[3] == -1)


# --------------------------------------------------------------------- O3 sparse attention
def _sparse(inp: W.SparseInputs, idx=None):
    return oracle.sparse_paged(_np(inp.q), _np(inp.kv_cache), inp.page_table.numpy(),
                               (inp.idx if idx is None else idx).numpy(), inp.kv_len, inp.dv,
                               inp.scale)


def test_sparse_all_positions_equals_dense_oracle():
    # Cross-pin: selecting every position through an identity page table is plain
    # non-causal attention with one KV head shared by all query heads.
    L, H, dqk, dv, ps = 100, 4, 24, 16, 16
    inp = W.sparse_inputs(nq=3, heads=H, dqk=dqk, dv=dv, kv_len=L, page_size=ps, topk=L, seed=30,
                          causal_windows=False)
    pages = inp.kv_cache.shape[0]
    inp.page_table = torch.arange(pages, dtype=torch.int32)
    out, lse, bad = _sparse(inp)
    assert bad == 0
    kv = _np(inp.kv_cache).reshape(-1, dqk)[:L][:, None, :]
    q = _np(inp.q)
    for n in range(3):
        cq = np.array([0, 1], np.int32)
        ck = np.array([0, L], np.int32)
        o1, l1 = oracle.attn_varlen(q[n:n + 1], kv, kv, cq, ck, False, inp.scale)
        np.testing.assert_allclose(out[n], o1[0, :, :dv], atol=1e-13)
        np.testing.assert_allclose(lse[n], l1[0], rtol=1e-13)


def test_sparse_matches_torch_sdpa_on_gathered_rows():
    inp = W.sparse_inputs(nq=5, heads=8, dqk=32, dv=24, kv_len=300, page_size=64, topk=50,
                          seed=31)
    out, lse, bad = _sparse(inp)
    assert bad == 0
    kv = inp.kv_cache.double()
    for n in range(5):
        ids = inp.idx[n][inp.idx[n] >= 0].long()
        rows = kv[inp.page_table.long()[ids // 64], ids % 64]  # [cnt, dqk]
        ref = torch.nn.functional.scaled_dot_product_attention(
            inp.q[n].double()[None], rows[None], rows[:, :24][None], scale=inp.scale)[0]
        np.testing.assert_allclose(out[n], ref.numpy(), atol=1e-12)


def test_sparse_closed_forms_and_multiplicity():
    inp = W.sparse_inputs(nq=3, heads=4, dqk=16, dv=8, kv_len=128, page_size=64, topk=4, seed=32)
    q0 = torch.zeros_like(inp.q)
    inp.idx = torch.tensor([[5, 5, 70, -1], [9, -1, -1, -1], [-1, -1, -1, -1]], dtype=torch.int32)
    z = W.SparseInputs(q0, inp.kv_cache, inp.page_table, inp.idx, 128, 8, inp.scale)
    out, lse, bad = _sparse(z)
    kv = _np(inp.kv_cache).astype(np.float64)
    pt = inp.page_table.numpy()
    row = lambda i: kv[pt[i // 64], i % 64]
    np.testing.assert_allclose(out[0], np.broadcast_to((2 * row(5) + row(70))[:8] / 3, (4, 8)),
                               atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(3), atol=1e-14)
    out1, _, _ = _sparse(inp)  # single index with any q: that row's V
    np.testing.assert_allclose(out1[1], np.broadcast_to(row(9)[:8], (4, 8)), atol=1e-15)
    assert np.all(out1[2] == 0) and np.all(np.isneginf(_sparse(inp)[1][2]))


def test_sparse_permutation_invariance_is_bitwise():
    inp = W.sparse_inputs(nq=6, heads=4, dqk=32, dv=16, kv_len=500, page_size=64, topk=200,
                          seed=33)
    out, lse, _ = _sparse(inp)
    for s in W.PERM_SEEDS[:3]:
        o2, l2, _ = _sparse(inp, W.permute_rows(inp.idx, s))
        assert np.array_equal(o2, out) and np.array_equal(l2, lse)


def test_sparse_page_table_indirection():
    # Scatter a logical KV array into shuffled physical pages: with the matching page
    # table the result must equal the identity layout bit for bit.
    L, ps, dqk = 256, 64, 16
    inp = W.sparse_inputs(nq=4, heads=2, dqk=dqk, dv=8, kv_len=L, page_size=ps, topk=60, seed=34)
    logical = inp.kv_cache.clone()  # treat as logical pages 0..3
    ident = W.SparseInputs(inp.q, logical, torch.arange(4, dtype=torch.int32), inp.idx, L, 8,
                           inp.scale)
    perm = torch.tensor([2, 0, 3, 1], dtype=torch.int32)  # logical page p -> physical perm[p]
    phys = torch.empty_like(logical)
    phys[perm.long()] = logical
    paged = W.SparseInputs(inp.q, phys, perm, inp.idx, L, 8, inp.scale)
    o1, l1, _ = _sparse(ident)
    o2, l2, _ = _sparse(paged)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_sparse_skips_and_counts_bad_entries():
    inp = W.sparse_inputs(nq=2, heads=2, dqk=16, dv=8, kv_len=100, page_size=64, topk=6, seed=35)
    good = torch.tensor([[3, 50, 99, -1, -1, -1], [0, 1, -1, -1, -1, -1]], dtype=torch.int32)
    badi = torch.tensor([[3, 50, 99, 100, -7, -1], [0, 1, 2 ** 30, -1, -1, -1]], dtype=torch.int32)
    o1, l1, b1 = _sparse(inp, good)
    o2, l2, b2 = _sparse(inp, badi)
    assert b1 == 0 and b2 == 3
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---- QKV projection + RoPE ------------------------------------------------------------

def _proj(x, w, b):
    """The projection alone, by numpy's float64 matmul (a routine the oracle does not call)."""
    y = x.astype(np.float64) @ w.astype(np.float64).T
    return y if b is None else y + b.astype(np.float64)


def test_qkv_rope_worked_example_and_bias():
    # d = 4, base 10000: pair (0, 2) turns by pos * 1, pair (1, 3) by pos * 0.01
    x = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 0, 0, 0]], np.float32)
    w = np.vstack([np.eye(4)] * 3).astype(np.float32)   # q = k = v = x
    q, k, v = oracle.qkv_rope(x, w, None, [1, 1, 3], heads=1, d=4)
    c1, s1, c2, s2 = math.cos(1.0), math.sin(1.0), math.cos(0.01), math.sin(0.01)
    np.testing.assert_allclose(q[0, 0], [c1, 0, s1, 0], atol=1e-15)
    np.testing.assert_allclose(q[1, 0], [0, c2, 0, s2], atol=1e-15)
    np.testing.assert_allclose(q[2, 0], [math.cos(3.0), 0, math.sin(3.0), 0], atol=1e-15)
    np.testing.assert_array_equal(k, q)
    np.testing.assert_array_equal(v[:, 0], x)            # v is not rotated
    # the bias is added before the rotation: bias e_2 on q turns (1, 0, 1, 0) at pos 1
    b = np.zeros(12, np.float32)
    b[2] = 1.0
    qb, kb, _ = oracle.qkv_rope(x[:1], w, b, [1], heads=1, d=4)
    np.testing.assert_allclose(qb[0, 0], [c1 - s1, 0, s1 + c1, 0], atol=1e-15)
    np.testing.assert_allclose(kb[0, 0], [c1, 0, s1, 0], atol=1e-15)


def test_qkv_rope_position_zero_is_the_projection():
    rng = np.random.default_rng(30)
    heads, d, hidden, n = 3, 80, 96, 17
    x = rng.standard_normal((n, hidden)).astype(np.float32)
    w = rng.standard_normal((3 * heads * d, hidden)).astype(np.float32)
    b = rng.standard_normal(3 * heads * d).astype(np.float32)
    q, k, v = oracle.qkv_rope(x, w, b, np.zeros(n), heads, d)
    y = _proj(x, w, b).reshape(n, 3, heads, d)
    for got, part in ((q, 0), (k, 1), (v, 2)):
        np.testing.assert_allclose(got, y[:, part], rtol=1e-12, atol=1e-10)


def test_qkv_rope_keeps_pair_norms_and_relative_positions():
    rng = np.random.default_rng(31)
    heads, d, hidden, n = 2, 80, 64, 6
    x = rng.standard_normal((n, hidden)).astype(np.float32)
    w = rng.standard_normal((3 * heads * d, hidden)).astype(np.float32)
    pos = rng.integers(0, 8547, n)
    q, k, _ = oracle.qkv_rope(x, w, None, pos, heads, d)
    y = _proj(x, w, None).reshape(n, 3, heads, d)
    h = d // 2
    for got, part in ((q, 0), (k, 1)):
        norm_got = np.hypot(got[..., :h], got[..., h:])
        norm_raw = np.hypot(y[:, part, :, :h], y[:, part, :, h:])
        np.testing.assert_allclose(norm_got, norm_raw, rtol=1e-12)
    # q(m) . k(n) depends on m - n only: shift every position by the same amount
    q2, k2, _ = oracle.qkv_rope(x, w, None, pos + 1234, heads, d)
    dots = np.einsum("ihd,jhd->hij", q, k)
    dots2 = np.einsum("ihd,jhd->hij", q2, k2)
    np.testing.assert_allclose(dots2, dots, rtol=1e-9, atol=1e-8)
    # ... but not on the positions alone: a shift of only the keys changes it
    _, k3, _ = oracle.qkv_rope(x, w, None, pos + 7, heads, d)
    assert np.abs(np.einsum("ihd,jhd->hij", q, k3) - dots).max() > 1e-3


def test_rope_cache_rows_are_powers_of_the_first():
    c = oracle.rope_cache(300, 80)
    z = c[..., 0] + 1j * c[..., 1]                      # [pos, 40] unit complex numbers
    np.testing.assert_allclose(z[0], np.ones(40), atol=0)
    p = np.arange(300)[:, None]
    np.testing.assert_allclose(z, np.power(z[1][None, :], p), atol=1e-11)
    np.testing.assert_allclose(np.abs(z), 1.0, atol=1e-15)


def test_rope_cache_frequencies_closed_form():
    # The angle of position 1, pair j is base^(-2j/d): an exponent of -j/d or a base
    # other than the stated one fails here (every angle is below pi, so atan2 recovers it).
    for d, base in ((80, 10000.0), (64, 10000.0), (128, 500000.0)):
        c = oracle.rope_cache(2, d, base)
        j = np.arange(d // 2)
        np.testing.assert_allclose(np.arctan2(c[1, :, 1], c[1, :, 0]), base ** (-2.0 * j / d),
                                   rtol=1e-13, atol=0)
        np.testing.assert_array_equal(c[0, :, 0], 1.0)
        np.testing.assert_array_equal(c[0, :, 1], 0.0)


def test_rope_cache_equals_qkv_rope_with_identity_projection():
    # With W = I and x = e_j the projected q is e_j, and RoPE turns it into
    # cos(angle) e_j + sin(angle) e_{j+d/2}: the cache and the fused step must agree.
    d = 80
    h = d // 2
    eye = np.eye(3 * d, dtype=np.float32)
    positions = [0, 1, 7, 1000, 8546, 32767]
    cache = oracle.rope_cache(32768, d)
    for pos in positions:
        x = eye[:h]                                   # token j carries e_j in the q part
        q, k, _ = oracle.qkv_rope(x, eye, None, np.full(h, pos), heads=1, d=d)
        j = np.arange(h)
        np.testing.assert_allclose(q[j, 0, j], cache[pos, :, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(q[j, 0, j + h], cache[pos, :, 1], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(k, np.zeros_like(k))  # x has no k part


# ---- FP8 (e4m3) rounding and block quantization ----------------------------------------

def _e4m3_table():
    """Every finite e4m3 value with its code, decoded from the bit layout (sign, 4
    exponent bits with bias 7, 3 mantissa bits; exponent field 0 = subnormal; the code
    with all exponent and mantissa bits set is NaN)."""
    vals, codes = [], []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(-v if s else v)
        codes.append(c)
    return np.array(vals), np.array(codes)


def _nearest_e4m3(x, vals, codes):
    """Brute force: the nearest table value; ties to the even code; beyond 448 -> 448."""
    out = []
    for v in x:
        d = np.abs(vals - v)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if codes[b] % 2 == 0] or best
        out.append(vals[best[0]])
    return np.array(out)


def test_e4m3_rounding_matches_brute_force_nearest():
    vals, codes = _e4m3_table()
    assert vals.max() == 448.0 and np.min(vals[vals > 0]) == 2.0 ** -9
    # every representable value maps to itself
    np.testing.assert_array_equal(oracle.round_e4m3(vals), vals)
    rng = np.random.default_rng(40)
    x = np.concatenate([
        rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 9, 3000),   # all binades
        (vals[:-1] + vals[1:]) / 2,                                       # exact midpoints
        rng.uniform(-448, 448, 500),
    ])
    x = x.astype(np.float32).astype(np.float64)   # the oracle rounds fp32 values
    inside = np.abs(x) <= 448
    np.testing.assert_array_equal(oracle.round_e4m3(x[inside]),
                                  _nearest_e4m3(x[inside], vals, codes))
    # saturation: beyond the largest finite value the magnitude clamps to 448
    big = np.array([448.0, 449.0, 463.9, 464.0, 1e6, -500.0, -1e30])
    np.testing.assert_array_equal(oracle.round_e4m3(big), np.sign(big) * 448.0)


def test_e4m3_rounding_matches_torch_float8():
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(41)
    x = (rng.standard_normal(20000) * 2.0 ** rng.integers(-12, 9, 20000)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    lib = torch.from_numpy(x).to(f8).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_e4m3(x.astype(np.float64)), lib)


def test_block_quantization_scales_and_error_bound():
    rng = np.random.default_rng(42)
    x = (rng.standard_normal((50, 128)) * np.exp(rng.uniform(-6, 4, (50, 1)))).astype(np.float32)
    x[7] = 0.0                                              # an all-zero block
    s, c = oracle.quant_e4m3(x, 128)
    assert s[7] == 1.0 and not c[7].any()
    amax = np.abs(x).max(axis=1)
    nz = amax > 0
    np.testing.assert_array_equal(s[nz], (amax[nz] / np.float32(448)).astype(np.float32))
    # the largest element of every block lands on +-448, and no code exceeds it
    assert np.all(np.abs(c).max(axis=1)[nz] == 448.0) and np.abs(c).max() <= 448.0
    # dequantized values are within half a grid step of x (relative 2^-4 for normal
    # values, 2^-10 of the scale in the subnormal range)
    deq = c.astype(np.float64) * s[:, None]
    bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s[:, None] + 1e-30
    assert np.all(np.abs(deq - x) <= bound * (1 + 1e-6))


def test_fp8_prefill_quantization_blocks():
    rng = np.random.default_rng(43)
    q = rng.standard_normal((37, 4, 128)).astype(np.float32)
    k = (rng.standard_normal((37, 2, 128)) * np.array([1.0, 30.0])[None, :, None]).astype(np.float32)
    qc, qs, kc, ks, qd, kd = oracle.quant_fp8_prefill(q, k)
    assert qs.shape == (37, 4) and ks.shape == (2,)
    # q: one scale per token and head; k: one scale per KV head over every token
    np.testing.assert_array_equal(qs, (np.abs(q).max(axis=2) / np.float32(448)).astype(np.float32))
    np.testing.assert_array_equal(ks, (np.abs(k).max(axis=(0, 2)) / np.float32(448)).astype(np.float32))
    np.testing.assert_allclose(kd[:, 1], kc[:, 1] * ks[1], rtol=1e-7)
    # the dequantized tensors stay within the e4m3 half-step of the inputs
    assert np.all(np.abs(qd - q) <= 2.0 ** -4 * np.abs(q) + 2.0 ** -10 * qs[:, :, None] + 1e-6)
