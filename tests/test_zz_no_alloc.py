"""The allocation-free fp32 attention entry point (tts_attn_fwd_varlen_f32_noalloc).

Some callers cannot allocate device memory at call time (another runtime owns the
device's memory pool, or allocation is forbidden once serving has started). For them
the library offers one entry point whose scratch is a fixed array inside the
library. These tests call it through the C ABI and compare it with the regular
entry point, which gets its scratch from a caller-provided workspace. The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from helpers import assert_close_attn, assert_lse_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20  # TTS_NOALLOC_SCRATCH_BYTES in include/tts.h


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(L, inp, out, lse, status):
    dev = out.device
    q, k, v = (t.to(dev).contiguous() for t in (inp.q, inp.k, inp.v))
    cq, ck = inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    code = L.tts_attn_fwd_varlen_f32_noalloc(
        _p(q), _p(k), _p(v), q.shape[0], k.shape[0], _p(cq), _p(ck), cq.numel() - 1,
        inp.max_seqlen_q, inp.max_seqlen_k, q.shape[1], k.shape[1], q.shape[2],
        int(inp.causal), inp.scale, _p(out), _p(lse), _p(status), stream)
    return code


def run_both(tts, L, inp, dev):
    """The allocation-free call, then the workspace call, on the same inputs."""
    out = torch.full(inp.q.shape, float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full(inp.q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    assert call_noalloc(L, inp, out, lse, st) == tts.TTS_OK
    ref_o, ref_l = tts.attn_fwd_varlen(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                                       inp.cu_seqlens_q.to(dev), inp.cu_seqlens_k.to(dev),
                                       inp.max_seqlen_q, inp.max_seqlen_k, inp.causal, inp.scale)
    torch.cuda.synchronize()
    tts.check_status(st)
    return out, lse, ref_o, ref_l


def test_noalloc_matches_workspace_entry_point_twice():
    import tiled_top_sparse_gb300 as tts
    L = tts.lib()
    dev = torch.device("cuda")
    cases = [W.tiny(),
             W.dense_inputs([300, 77, 129], hq=4, hkv=2, d=128, causal=True,
                            dtype=torch.float32, seed=60)]
    for inp in cases:  # two calls in a row share the one scratch array
        out, lse, ref_o, ref_l = run_both(tts, L, inp, dev)
        # Same kernel on the same bf16-rounded inputs: the results must be bitwise equal,
        # so stale scratch contents cannot hide inside a tolerance.
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        assert_close_attn(out.cpu().numpy(), ref_o.cpu().double().numpy(), "noalloc vs workspace")
        assert_lse_close(lse.cpu().numpy(), ref_l.cpu().double().numpy(), "noalloc lse")


def test_noalloc_at_the_scratch_limit_and_one_step_over():
    import tiled_top_sparse_gb300 as tts
    L = tts.lib()
    dev = torch.device("cuda")
    # 256 (work counter) + 2 * 21846 * 64 (q copy) + 2 * (2 * 21844 * 64) (k, v copies),
    # every part a multiple of 256: exactly the array's size.
    tq, tk = 21846, 21844
    assert 256 + 2 * tq * 64 + 2 * (2 * tk * 64) == SCRATCH_BYTES
    assert tts.attn_workspace_bytes(tq, tk, 1, 1, 64, torch.float32) == SCRATCH_BYTES
    inp = W.dense_inputs([tq], [tk], hq=1, hkv=1, d=64, causal=False, dtype=torch.float32,
                         seed=62)
    out, lse, ref_o, ref_l = run_both(tts, L, inp, dev)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    # two more query rows need 256 bytes more than the array holds
    over = W.dense_inputs([tq + 2], [tk], hq=1, hkv=1, d=64, causal=False, dtype=torch.float32,
                          seed=63)
    assert tts.attn_workspace_bytes(tq + 2, tk, 1, 1, 64, torch.float32) == SCRATCH_BYTES + 256
    o2 = torch.zeros(over.q.shape, dtype=torch.float32, device=dev)
    assert call_noalloc(L, over, o2, None, None) == tts.TTS_ERR_WORKSPACE


def test_noalloc_rejects_inputs_larger_than_scratch():
    import tiled_top_sparse_gb300 as tts
    L = tts.lib()
    dev = torch.device("cuda")
    # bf16 copies of q, k, v would need 3 * 40000 * 1 * 64 * 2 bytes > 8 MiB
    inp = W.dense_inputs([40000], hq=1, hkv=1, d=64, dtype=torch.float32, seed=61)
    out = torch.zeros(inp.q.shape, dtype=torch.float32, device=dev)
    assert 3 * 40000 * 64 * 2 > SCRATCH_BYTES
    assert call_noalloc(L, inp, out, None, None) == tts.TTS_ERR_WORKSPACE
