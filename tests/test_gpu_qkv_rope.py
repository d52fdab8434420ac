"""GPU parity for the vision QKV projection + RoPE (tts_qkv_rope) and its cos/sin table
(tts_rope_cache) against the float64 oracle.

Tolerance, from the arithmetic: the products of bf16 operands are exact in fp32 and
the fp32 sums over `hidden` terms, bias add and rotation add errors of order 1e-6
for unit-scale outputs; the final rounding to bf16 (nearest even) adds at most half
an ulp, 2^-8 of the magnitude. So every element satisfies |gpu - ref| <= 2^-8 |ref|
+ 1e-4, and the block's relative L2 error stays under 2e-3 (the vision write-up calls
block errors below 0.2% healthy)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

REL_ELEM = 2.0 ** -8
ABS_ELEM = 1e-4
MAX_REL_L2 = 2e-3


@pytest.fixture(scope="module")
def tts():
    import tiled_top_sparse_gb300 as m
    m.lib()
    return m


def gpu_run(tts, inp: W.QkvInputs, cs=None, status=None):
    dev = torch.device("cuda")
    if cs is None:
        cs = tts.rope_cache(inp.max_pos, inp.d, inp.base, device=dev)
    b = None if inp.bias is None else inp.bias.to(dev)
    return tts.qkv_rope(inp.x.to(dev), inp.w.to(dev), b, inp.positions.to(dev), cs, inp.heads,
                        status=status)


def oracle_run(inp: W.QkvInputs, rows=None):
    x = inp.x.float().numpy()
    pos = inp.positions.numpy()
    if rows is not None:
        x, pos = x[rows], pos[rows]
    b = None if inp.bias is None else inp.bias.numpy()
    return oracle.qkv_rope(x, inp.w.float().numpy(), b, pos, inp.heads, inp.d, inp.base)


def check(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = REL_ELEM * np.abs(ref) + ABS_ELEM
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"{what}: |err| {err[worst]:.3e} > {bound[worst]:.3e} at {worst}"
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert rel <= MAX_REL_L2, f"{what}: rel L2 {rel:.3e}"
    return rel


def test_rope_cache_matches_oracle(tts):
    for max_pos, rot in ((300, 80), (32768, 80), (1000, 64), (777, 128)):
        got = tts.rope_cache(max_pos, rot, 10000.0, device="cuda").cpu().numpy()
        ref = oracle.rope_cache(max_pos, rot, 10000.0)
        # double-precision angle and sine / cosine, one rounding to fp32: within half an
        # fp32 ulp of values <= 1
        assert np.abs(got - ref).max() <= 2.0 ** -25 + 1e-10, (max_pos, rot)
    got = tts.rope_cache(50, 80, 500000.0, device="cuda").cpu().numpy()
    assert np.abs(got - oracle.rope_cache(50, 80, 500000.0)).max() <= 2.0 ** -25 + 1e-10


@pytest.mark.parametrize("n,heads,d,hidden,bias", [
    (300, 16, 80, 1280, True),    # vision heads; 3 token tiles, ragged last (44 rows)
    (129, 16, 80, 1280, False),   # one row past a tile, no bias
    (77, 4, 64, 200, True),       # d = 64 (4 heads per tile); hidden not a multiple of 64
    (260, 2, 128, 136, True),     # d = 128 (2 heads per tile), three stages
    (1, 1, 80, 8, True),          # smallest: one token, one head, one 8-column K step
    (40, 5, 80, 96, True),        # 15 heads: q / k / v boundaries inside tiles
])
def test_parity_random_positions(tts, n, heads, d, hidden, bias):
    g = torch.Generator().manual_seed(n * 31 + d)
    pos = torch.randint(0, 8547, (n,), generator=g, dtype=torch.int32)
    inp = W.vision_qkv_inputs(n=n, heads=heads, d=d, hidden=hidden, max_pos=8547, bias=bias,
                              positions=pos, seed=n + heads)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v = gpu_run(tts, inp, status=st)
    tts.check_status(st)
    rq, rk, rv = oracle_run(inp)
    for got, ref, name in ((q, rq, "q"), (k, rk, "k"), (v, rv, "v")):
        check(got, ref, f"{name} n={n} H={heads} d={d}")
    q2, k2, v2 = gpu_run(tts, inp)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)


@pytest.mark.parametrize("n,heads,d,hidden", [
    (1100, 16, 80, 256),   # 5 x 16 pair tiles: on a 152-SM GPU some pairs take two
    (3300, 8, 64, 128),    # 13 x 6 pair tiles of 4 heads of 64
])
def test_parity_with_several_tiles_per_pair(tts, n, heads, d, hidden):
    """More pair tiles than CTA pairs, so pairs run several tiles through both TMEM
    accumulators and the stage ring wraps across tiles. Every row and head is compared."""
    g = torch.Generator().manual_seed(n)
    pos = torch.randint(0, 8547, (n,), generator=g, dtype=torch.int32)
    inp = W.vision_qkv_inputs(n=n, heads=heads, d=d, hidden=hidden, max_pos=8547,
                              positions=pos, seed=n + 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v = gpu_run(tts, inp, status=st)
    tts.check_status(st)
    rq, rk, rv = oracle_run(inp)
    for got, ref, name in ((q, rq, "q"), (k, rk, "k"), (v, rv, "v")):
        check(got, ref, f"{name} n={n} H={heads} d={d}")


def test_out_of_range_positions_are_zeroed_and_flagged(tts):
    n, heads, d = 200, 16, 80
    pos = torch.arange(n, dtype=torch.int32)
    pos[[3, 150, 199]] = torch.tensor([-1, 4096, 1 << 30], dtype=torch.int32)
    inp = W.vision_qkv_inputs(n=n, heads=heads, d=d, hidden=256, max_pos=4096,
                              positions=pos, seed=5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v = gpu_run(tts, inp, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    bad = [3, 150, 199]
    good = [i for i in range(n) if i not in bad]
    assert not q[bad].float().abs().any() and not k[bad].float().abs().any()
    rq, rk, rv = oracle_run(inp, rows=good)
    check(q[good], rq, "q (valid rows)")
    check(k[good], rk, "k (valid rows)")
    # v does not depend on the position: every row matches
    inp_all = W.QkvInputs(inp.x, inp.w, inp.bias, torch.zeros(n, dtype=torch.int32), heads, d,
                          inp.max_pos)
    _, _, rv_all = oracle_run(inp_all)
    check(v, rv_all, "v")


def test_empty_input_enqueues_nothing(tts):
    inp = W.vision_qkv_inputs(n=0, heads=16, d=80, hidden=64, max_pos=16)
    q, k, v = gpu_run(tts, inp)
    assert q.shape == (0, 16, 80) and k.shape == v.shape == q.shape


def test_full_vision_size_sampled_rows(tts):
    """The workload the benchmark times: 8547 tokens, hidden 1280, 16 heads of 80,
    positions 0..8546, cos/sin table of 32768 positions. Rows sampled across the
    tiles (first, tile borders, the ragged last tile) are checked against the oracle;
    the whole output is checked for repeatability."""
    inp = W.vision_qkv_inputs()
    n = inp.x.shape[0]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v = gpu_run(tts, inp, status=st)
    tts.check_status(st)
    g = np.random.default_rng(7)
    rows = sorted(set([0, 1, 127, 128, 4095, 4096, n - 100, n - 99, n - 1] +
                      g.choice(n, 55, replace=False).tolist()))
    rq, rk, rv = oracle_run(inp, rows=rows)
    for got, ref, name in ((q, rq, "q"), (k, rk, "k"), (v, rv, "v")):
        check(got[rows], ref, f"{name} (full vision, sampled rows)")
    q2, k2, v2 = gpu_run(tts, inp)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)
    # q . k of a pair of tokens depends on the position difference only: shifting all
    # positions by 1000 keeps every per-head dot product (up to the bf16 rounding)
    shifted = W.QkvInputs(inp.x, inp.w, inp.bias, inp.positions + 1000, inp.heads, inp.d,
                          inp.max_pos)
    qs, ks, _ = gpu_run(tts, shifted)
    sel = torch.tensor(rows[:32], device="cuda")
    d0 = torch.einsum("ihd,jhd->hij", q[sel].float(), k[sel].float())
    d1 = torch.einsum("ihd,jhd->hij", qs[sel].float(), ks[sel].float())
    assert (d0 - d1).abs().max().item() <= 0.05 * d0.abs().max().item()
