"""GPU parity for tts_attn_fwd_varlen against the float64 oracle.

Element-wise over whole outputs at sizes the oracle finishes in seconds (several
tiles and ragged tails), and on sampled rows at the full vision / varlen sizes.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import assert_close_attn, assert_lse_close, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts():
    import tiled_top_sparse_gb300 as m
    m.lib()
    return m


def run(tts, inp: W.DenseInputs, status=None, out=None):
    dev = torch.device("cuda")
    return tts.attn_fwd_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                               inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev),
                               inp.max_seqlen_q, inp.max_seqlen_k, inp.causal, inp.scale,
                               status=status, out=out)


def oracle_full(inp: W.DenseInputs, rows=None):
    q, k, v = (t.float().numpy() for t in (inp.q, inp.k, inp.v))
    if inp.q.dtype == torch.float32:  # the CUDA path rounds fp32 inputs to bf16 first
        q, k, v = oracle.round_bf16(q), oracle.round_bf16(k), oracle.round_bf16(v)
    return oracle.attn_varlen(q, k, v, inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(),
                              inp.causal, inp.scale, rows=rows)


def check(tts, inp, what):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, st)
    tts.check_status(st)
    ref_o, ref_l = oracle_full(inp)
    assert_close_attn(out.cpu().numpy(), ref_o, what)
    assert_lse_close(lse.cpu().numpy(), ref_l, what)
    return out, lse


def test_tiny_fp32_inputs(tts):
    inp = W.tiny()
    out, lse = check(tts, inp, "tiny")
    out2, lse2 = run(tts, inp)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # For information: the same output against the oracle on the unrounded fp32 inputs,
    # i.e. the cost of computing in bf16 at all. Inputs ~ N(0,1) rounded to bf16 carry a
    # relative error of at most 2^-9 each; the scores (64 products, scale 1/8) then move
    # by ~2^-9 in absolute terms, and so do the softmax weights relative to themselves,
    # which bounds the output's relative L2 error by a few 2^-9 ~ 1e-2.
    q, k, v = (t.numpy() for t in (inp.q, inp.k, inp.v))
    uo, ul = oracle.attn_varlen(q, k, v, inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(),
                                inp.causal, inp.scale)
    max_abs, cos, rel = compare(out.cpu().numpy(), uo)
    lse_err = float(np.abs(lse.cpu().numpy() - ul).max())
    print(f"\n[tiny vs unrounded fp32 inputs] max_abs={max_abs:.3e} cos={cos:.7f} "
          f"rel_l2={rel:.3e} lse_err={lse_err:.3e}")
    assert rel <= 1e-2 and cos >= 0.999


@pytest.mark.parametrize("n,d", [(1000, 80), (129, 64), (385, 128), (1, 80), (3536, 80)])
def test_vision_like_noncausal(tts, n, d):
    inp = W.vision(n=n, heads=2, d=d, seed=n + d)
    check(tts, inp, f"vision n={n} d={d}")


def test_varlen_causal_gqa_ragged(tts):
    inp = W.dense_inputs([300, 1, 0, 777, 513, 128, 255, 257], hq=4, hkv=2, d=128, causal=True,
                         seed=40)
    check(tts, inp, "varlen causal")


def test_varlen_noncausal_lq_ne_lk(tts):
    inp = W.dense_inputs([100, 300, 5], [400, 7, 0], hq=2, hkv=1, d=64, causal=False, seed=41)
    check(tts, inp, "varlen lq!=lk")


def test_varlen_causal_lq_ne_lk_bottom_right(tts):
    inp = W.dense_inputs([100, 300, 5], [400, 7, 3], hq=2, hkv=2, d=80, causal=True, seed=42)
    check(tts, inp, "causal lq!=lk")


def test_multi_block_boundary_3535_vs_8547_rows(tts):
    # The vision write-up's overflow appeared only once N needed more than one block
    # (N > 3535 there). Sample rows across every 128-row tile of N = 8547.
    inp = W.vision(n=8547, heads=1, d=80, seed=43)
    out, lse = run(tts, inp)
    tok = np.concatenate([np.arange(0, 8547, 67), [8546, 3534, 3535, 3536]]).astype(np.int32)
    head = np.zeros_like(tok)
    ro, rl = oracle_full(inp, rows=(tok, head))
    assert_close_attn(out[tok, 0].cpu().numpy(), ro, "8547 sampled")
    assert_lse_close(lse[tok, 0].cpu().numpy(), rl, "8547 sampled lse")


def test_full_vision_config_sampled_rows(tts):
    inp = W.vision()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, st)
    out2, lse2 = run(tts, inp, st)
    tts.check_status(st)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)  # bitwise run-to-run
    g = np.random.default_rng(44)
    tok = g.integers(0, 8547, 768).astype(np.int32)
    tok[:4] = [0, 127, 128, 8546]
    head = g.integers(0, 16, 768).astype(np.int32)
    ro, rl = oracle_full(inp, rows=(tok, head))
    assert_close_attn(out[tok, head].cpu().numpy(), ro, "vision sampled")
    assert_lse_close(lse[tok, head].cpu().numpy(), rl, "vision lse")


def test_full_varlen_config_sampled_rows(tts):
    inp = W.varlen()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, st)
    tts.check_status(st)
    g = np.random.default_rng(45)
    T = int(inp.cu_seqlens_q[-1])
    tok = g.integers(0, T, 512).astype(np.int32)
    cu = inp.cu_seqlens_q.numpy()
    nb = len(cu) - 1
    tok[:nb] = cu[:-1]  # every sequence's row 0
    tok[nb:2 * nb] = cu[1:] - 1  # and its last row (last query tile, causal diagonal)
    tok[2 * nb:3 * nb] = np.minimum(cu[:-1] + 128, cu[1:] - 1)  # the second query tile's first
    head = g.integers(0, 32, 512).astype(np.int32)
    ro, rl = oracle_full(inp, rows=(tok, head))
    assert_close_attn(out[tok, head].cpu().numpy(), ro, "varlen sampled")
    assert_lse_close(lse[tok, head].cpu().numpy(), rl, "varlen lse")


def test_uncovered_rows_and_canaries_untouched(tts):
    inp = W.dense_inputs([200, 50], hq=2, hkv=1, d=128, causal=True, seed=46)
    dev = torch.device("cuda")
    total = 250 + 10  # 10 trailing q rows not covered by any sequence
    q = torch.zeros(total, 2, 128, dtype=torch.bfloat16)
    q[:250] = inp.q
    n = total * 2 * 128
    buf = torch.full((n + 2 * 1024,), 7.0, dtype=torch.float32, device=dev)
    out = buf[1024:1024 + n].view(total, 2, 128)
    tts.attn_fwd_varlen(q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens_q.to(dev),
                        inp.cu_seqlens_k.to(dev), 200, 200, True, inp.scale, out=out)
    torch.cuda.synchronize()
    assert bool((buf[:1024] == 7).all()) and bool((buf[-1024:] == 7).all())
    assert bool((out[250:] == 7).all())
    ref_o, _ = oracle_full(inp)
    assert_close_attn(out[:250].cpu().numpy(), ref_o, "canary")


def test_bad_cu_seqlens_flagged_not_faulting(tts):
    dev = torch.device("cuda")
    inp = W.dense_inputs([64, 64], hq=1, hkv=1, d=64, seed=47)
    bad = torch.tensor([0, 100, 50], dtype=torch.int32, device=dev)  # decreasing
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    tts.attn_fwd_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), bad, bad, 128, 128, False,
                        inp.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tts.TTS_DEV_BAD_ARG


def test_persistent_schedule_many_items_workspace_reuse(tts):
    # 32 heads x 11 ragged sequences: ~500 work items on 152 persistent CTAs, items
    # with no key tiles (causal, fewer keys than queries), empty sequences, one workspace
    # reused by consecutive calls (its counter is re-zeroed on the stream by each call).
    inp = W.dense_inputs([0, 1, 700, 2, 0, 900, 3, 129, 257, 64, 1],
                         [0, 1, 700, 2, 5, 900, 1, 129, 257, 64, 0],
                         hq=32, hkv=8, d=128, causal=True, seed=43)
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (inp.q, inp.k, inp.v, inp.cu_seqlens_q, inp.cu_seqlens_k)]
    ws = torch.empty(tts.attn_workspace_bytes(inp.q.shape[0], inp.k.shape[0], 32, 8, 128,
                                              torch.bfloat16), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    outs = [tts.attn_fwd_varlen(*args, inp.max_seqlen_q, inp.max_seqlen_k, True, inp.scale,
                                workspace=ws, status=st) for _ in range(3)]
    tts.check_status(st)
    ref_o, ref_l = oracle_full(inp)
    assert_close_attn(outs[0][0].cpu().numpy(), ref_o, "persistent many items")
    assert_lse_close(outs[0][1].cpu().numpy(), ref_l, "persistent many items")
    for o, l in outs[1:]:  # the item-to-CTA assignment varies; the results may not
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])

