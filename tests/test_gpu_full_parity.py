"""Every output row of the full-size workloads against the float64 oracle.

One GPU call per workload, in the launch configuration the benchmark times, then the
oracle over every (token, head) row of the whole-image vision attention (8547 patch
tokens, "DeepSeek V4.1 上 4×RTX 3090", section 三), of the varlen causal GQA prefill
batch ("从 SGLang Kernel源码到 GPU Trace", section 2.2), and every (query, head) row of
the paged sparse attention ("推理引擎的蝴蝶效应", 实验方法和结果). Each test asserts the
stated tolerances over the whole output, holds every row's max-abs error to the same
bound, and prints the margins (worst and mean per-row relative L2) so a drift towards
the bound is on record. The top-k workload is compared in full in test_gpu_topk.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import LSE_ABS, MAX_ABS, MAX_REL_L2, MIN_COS, assert_lse_close, compare

@pytest.fixture(scope="module")
def tts():
    import tiled_top_sparse_gb300 as m
    m.lib()
    return m


class RowStats:
    """Accumulates whole-output and per-row error statistics over chunks of rows."""

    def __init__(self):
        self.dd = 0.0    # sum of squared differences
        self.rr = 0.0    # sum of squared reference values
        self.gg = 0.0    # sum of squared outputs
        self.gr = 0.0    # dot product of outputs and references
        self.max_abs = 0.0
        self.row_rel_max = 0.0
        self.row_rel_sum = 0.0
        self.rows = 0
        self.worst = None

    def add(self, got, ref, labels):
        """got / ref [rows, d]; labels[i] names row i."""
        g = np.asarray(got, np.float64)
        r = np.asarray(ref, np.float64)
        diff = g - r
        self.dd += float(np.sum(diff * diff))
        self.rr += float(np.sum(r * r))
        self.gg += float(np.sum(g * g))
        self.gr += float(np.sum(g * r))
        if diff.size:
            self.max_abs = max(self.max_abs, float(np.abs(diff).max()))
        dn = np.linalg.norm(diff, axis=1)
        rn = np.linalg.norm(r, axis=1)
        rel = np.where(rn > 0, dn / np.where(rn > 0, rn, 1.0), dn)
        if rel.size:
            i = int(np.argmax(rel))
            if rel[i] >= self.row_rel_max:
                self.row_rel_max = float(rel[i])
                self.worst = labels[i]
            self.row_rel_sum += float(rel.sum())
            self.rows += rel.size

    def finish(self, what):
        rel = (self.dd ** 0.5) / (self.rr ** 0.5)
        cos = self.gr / ((self.gg ** 0.5) * (self.rr ** 0.5))
        mean_row = self.row_rel_sum / max(self.rows, 1)
        print(f"\n[{what}] rows={self.rows} max_abs={self.max_abs:.3e} cos={cos:.8f} "
              f"rel_l2={rel:.3e} row_rel_l2: max={self.row_rel_max:.3e} "
              f"(row {self.worst}) mean={mean_row:.3e}")
        assert self.max_abs <= MAX_ABS and cos >= MIN_COS and rel <= MAX_REL_L2, (
            f"{what}: max_abs={self.max_abs:.3e} cos={cos:.8f} rel_l2={rel:.3e}")
        return rel


def dense_call(tts, inp):
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = tts.attn_fwd_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                                   inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev),
                                   inp.max_seqlen_q, inp.max_seqlen_k, inp.causal, inp.scale,
                                   status=st)
    tts.check_status(st)
    return out.cpu().numpy(), lse.cpu().numpy()


def dense_every_row(inp, out, lse, what):
    """Runs the oracle sequence by sequence (bounded host memory) over every row."""
    q, k, v = (t.float().numpy() for t in (inp.q, inp.k, inp.v))
    cq = inp.cu_seqlens_q.numpy()
    ck = inp.cu_seqlens_k.numpy()
    hq = q.shape[1]
    stats = RowStats()
    lse_err = 0.0
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        ro, rl = oracle.attn_varlen(q[q0:q1], k[k0:k1], v[k0:k1], [0, q1 - q0], [0, k1 - k0],
                                    inp.causal, inp.scale)
        n = (q1 - q0) * hq
        labels = [(q0 + i // hq, i % hq) for i in range(n)]
        stats.add(out[q0:q1].reshape(n, -1), ro.reshape(n, -1), labels)
        assert_lse_close(lse[q0:q1], rl, f"{what} lse seq {b}")
        lse_err = max(lse_err, float(np.abs(lse[q0:q1] - rl).max()))
    print(f"[{what}] lse max abs err {lse_err:.3e} (bound {LSE_ABS})")
    return stats.finish(what)


@pytest.mark.gpu
@pytest.mark.slow
def test_vision_every_row(tts):
    inp = W.vision()
    out, lse = dense_call(tts, inp)
    dense_every_row(inp, out, lse, "vision 8547x16 d80 every row")


@pytest.mark.gpu
@pytest.mark.slow
def test_varlen_every_row(tts):
    inp = W.varlen()
    out, lse = dense_call(tts, inp)
    dense_every_row(inp, out, lse, f"varlen {inp.lengths_q} every row")


@pytest.mark.gpu
@pytest.mark.slow
def test_sparse_every_query(tts):
    inp = W.sparse_inputs()
    dev = torch.device("cuda")
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = tts.sparse_attn_paged(inp.q.to(dev), inp.kv_cache.to(dev),
                                     inp.page_table.to(dev), inp.idx.to(dev), inp.kv_len,
                                     inp.scale, dv=inp.dv, status=st)
    tts.check_status(st)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    stats = RowStats()
    kv = inp.kv_cache.float().numpy()
    pt = inp.page_table.numpy()
    q = inp.q.float().numpy()
    ix = inp.idx.numpy()
    H = q.shape[1]
    step = 64
    for n0 in range(0, q.shape[0], step):
        n1 = min(n0 + step, q.shape[0])
        ro, rl, bad = oracle.sparse_paged(q[n0:n1], kv, pt, ix[n0:n1], inp.kv_len, inp.dv,
                                          inp.scale)
        assert bad == 0
        n = (n1 - n0) * H
        stats.add(out[n0:n1].reshape(n, -1), ro.reshape(n, -1),
                  [(n0 + i // H, i % H) for i in range(n)])
        assert_lse_close(lse[n0:n1], rl, f"sparse lse queries {n0}..{n1}")
    stats.finish("sparse 323x128 every query")


def test_compare_helper_matches_row_stats():
    # The streaming statistics equal the one-shot comparison on the same data.
    rng = np.random.default_rng(5)
    r = rng.standard_normal((50, 16))
    g = r + 1e-4 * rng.standard_normal((50, 16))
    s = RowStats()
    s.add(g[:20], r[:20], list(range(20)))
    s.add(g[20:], r[20:], list(range(20, 50)))
    max_abs, cos, rel = compare(g, r)
    assert abs(s.max_abs - max_abs) == 0.0
    assert abs((s.dd ** 0.5) / (s.rr ** 0.5) - rel) < 1e-12
    assert abs(s.gr / ((s.gg ** 0.5) * (s.rr ** 0.5)) - cos) < 1e-12
