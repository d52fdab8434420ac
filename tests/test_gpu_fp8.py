"""GPU parity for the FP8 prefill path: the e4m3 block quantization
(tts_quantize_fp8_prefill) bit-exact against the oracle's, and attention with e4m3 q / k
(tts_attn_fwd_varlen_fp8) against the float64 attention oracle run on the oracle's own
dequantized q and k (the oracle quantizes the same bf16 inputs itself; nothing it uses
comes from the CUDA path). The attention tolerances are those of the bf16 path: once q
and k are on the e4m3 grid, the products are exact and the GPU's remaining error is the
fp32 accumulation and the bf16 rounding of P."""
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


def gpu_fp8(tts, inp: W.DenseInputs, status=None):
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    q8, qs, k8, ks = tts.quantize_fp8_prefill(q, k)
    out, lse = tts.attn_fwd_varlen_fp8(q8, qs, k8, ks, v, inp.cu_seqlens_q.to(dev),
                                       inp.cu_seqlens_k.to(dev), inp.max_seqlen_q,
                                       inp.max_seqlen_k, inp.causal, inp.scale, status=status)
    return (q8, qs, k8, ks), out, lse


def oracle_fp8(inp: W.DenseInputs, rows=None):
    qc, qs, kc, ks, qd, kd = oracle.quant_fp8_prefill(inp.q.float().numpy(),
                                                      inp.k.float().numpy())
    o, l = oracle.attn_varlen(qd, kd, inp.v.float().numpy(), inp.cu_seqlens_q.numpy(),
                              inp.cu_seqlens_k.numpy(), inp.causal, inp.scale, rows=rows)
    return (qc, qs, kc, ks), o, l


def codes(t):
    return t.view(torch.float8_e4m3fn).float().cpu().numpy()


@pytest.mark.parametrize("d", [128, 64, 132])   # 128: half-warp rows; others: warp rows
def test_quantization_bit_exact(d):
    import tiled_top_sparse_gb300 as tts
    inp = W.dense_inputs([300, 77], hq=6, hkv=3, d=d, seed=50)
    q, k = inp.q.clone(), inp.k.clone()
    g = torch.Generator().manual_seed(51)
    # rows over a wide range of magnitudes (subnormal codes included), an all-zero row,
    # an all-zero KV head, and exact ties on the e4m3 grid after scaling
    q *= torch.exp(torch.empty(q.shape[0], q.shape[1], 1).uniform_(-12, 6, generator=g)).to(q.dtype)
    q[5, 2] = 0
    k[:, 1] = 0
    k[3, 0, :4] = torch.tensor([448.0, 1.0625, 1.1875, -0.001], dtype=k.dtype)
    dev = torch.device("cuda")
    q8, qs, k8, ks = tts.quantize_fp8_prefill(q.to(dev), k.to(dev))
    qc, rqs, kc, rks, _, _ = oracle.quant_fp8_prefill(q.float().numpy(), k.float().numpy())
    np.testing.assert_array_equal(qs.cpu().numpy(), rqs)
    np.testing.assert_array_equal(ks.cpu().numpy(), rks)
    np.testing.assert_array_equal(codes(q8), qc)
    np.testing.assert_array_equal(codes(k8), kc)
    assert rks[1] == 1.0 and not codes(k8)[:, 1].any()


@pytest.mark.parametrize("lq,lk,hq,hkv,causal", [
    ([300, 129, 1, 520], None, 4, 2, True),          # ragged tiles, GQA, causal
    ([100, 257], [300, 129], 2, 1, False),           # Lq != Lk, non-causal
    ([200, 64], [450, 64], 2, 2, True),              # causal, bottom-right with Lq < Lk
])
def test_attention_parity(tts, lq, lk, hq, hkv, causal):
    inp = W.dense_inputs(lq, lk, hq=hq, hkv=hkv, d=128, causal=causal, seed=len(lq) + hq)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, out, lse = gpu_fp8(tts, inp, st)
    tts.check_status(st)
    _, ro, rl = oracle_fp8(inp)
    assert_close_attn(out.cpu().numpy(), ro, f"fp8 {lq} {lk}")
    assert_lse_close(lse.cpu().numpy(), rl, f"fp8 lse {lq} {lk}")
    _, out2, lse2 = gpu_fp8(tts, inp)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_fp8_differs_from_bf16_only_by_the_quantization(tts):
    """Against the unquantized bf16 inputs the FP8 result moves by the e4m3 rounding of q
    and k only: it stays within a loose bound of the bf16 oracle, while the comparison
    with the oracle on the quantized inputs is tight."""
    inp = W.dense_inputs([400], hq=2, hkv=2, d=128, causal=True, seed=52)
    _, out, _ = gpu_fp8(tts, inp)
    ro_bf16, _ = oracle.attn_varlen(inp.q.float().numpy(), inp.k.float().numpy(),
                                    inp.v.float().numpy(), inp.cu_seqlens_q.numpy(),
                                    inp.cu_seqlens_k.numpy(), True, inp.scale)
    _, ro_fp8, _ = oracle_fp8(inp)
    g = out.cpu().numpy().astype(np.float64)
    err_q = np.linalg.norm(g - ro_fp8) / np.linalg.norm(ro_fp8)
    err_b = np.linalg.norm(g - ro_bf16) / np.linalg.norm(ro_bf16)
    assert err_q <= 2e-3 and err_b <= 0.1 and err_b > err_q


def test_full_varlen_config_sampled_rows(tts):
    """The varlen prefill workload (8 sequences, 32 / 8 heads, d 128, causal) through the
    FP8 path, 512 sampled (row, head) outputs against the oracle, every sequence's first,
    last and second-tile rows included."""
    inp = W.varlen()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    (q8, qs, k8, ks), out, lse = gpu_fp8(tts, inp, st)
    tts.check_status(st)
    g = np.random.default_rng(53)
    T = int(inp.cu_seqlens_q[-1])
    tok = g.integers(0, T, 512).astype(np.int32)
    cu = inp.cu_seqlens_q.numpy()
    nb = len(cu) - 1
    tok[:nb] = cu[:-1]
    tok[nb:2 * nb] = cu[1:] - 1
    tok[2 * nb:3 * nb] = np.minimum(cu[:-1] + 128, cu[1:] - 1)
    head = g.integers(0, 32, 512).astype(np.int32)
    (qc, rqs, kc, rks), ro, rl = oracle_fp8(inp, rows=(tok, head))
    np.testing.assert_array_equal(ks.cpu().numpy(), rks)
    np.testing.assert_array_equal(qs.cpu().numpy(), rqs)
    assert_close_attn(out[tok, head].cpu().numpy(), ro, "fp8 varlen sampled")
    assert_lse_close(lse[tok, head].cpu().numpy(), rl, "fp8 varlen lse")
