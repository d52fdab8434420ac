"""CPU checks of the C ABI: the library builds, loads without a GPU, exports every
function tts.h declares, and rejects bad host-side arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from tiled_top_sparse_gb300 import _build
    _build.build()
    import tiled_top_sparse_gb300 as tts
    return tts.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tts.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tts_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(L, n), f"libtts.so does not export {n}"
    import tiled_top_sparse_gb300 as tts
    assert set(names) == set(tts.EXPORTED)


def test_status_strings_and_device_mapping(L):
    import tiled_top_sparse_gb300 as tts
    assert tts.status_string(0) == "ok"
    for c in range(1, 7):
        assert tts.status_string(c) not in ("ok", "unknown status")
    f = L.tts_status_from_device
    assert f(0) == tts.TTS_OK
    assert f(tts.TTS_DEV_INDEX_RANGE) == tts.TTS_ERR_INDEX_RANGE
    assert f(tts.TTS_DEV_TIMEOUT | tts.TTS_DEV_INDEX_RANGE) == tts.TTS_ERR_DEVICE_TIMEOUT
    assert f(tts.TTS_DEV_BAD_ARG) == tts.TTS_ERR_INVALID_ARG
    assert L.tts_version() >= 100


def test_workspace_size(L):
    import tiled_top_sparse_gb300 as tts
    # bf16 inputs: only the work-item counter of the persistent kernel
    assert L.tts_attn_workspace_bytes(256, 256, 1, 1, 64, tts.TTS_BF16) == 256
    n = L.tts_attn_workspace_bytes(256, 256, 1, 1, 64, tts.TTS_F32)
    assert n >= 256 + 3 * 256 * 64 * 2


# Fake, never-dereferenced pointers: host validation must reject before any CUDA call.
P = ctypes.c_void_p(0x1000)
NUL = None


def test_topk_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    f = L.tts_topk_select
    assert f(NUL, 10, 1, P, P, 4, P, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 10, 1, P, P, 0, P, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 0, 1, P, P, 4, P, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 10, -1, P, P, 4, P, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 10, 1, P, P, 4097, P, NUL, NUL) == tts.TTS_ERR_UNSUPPORTED
    assert f(P, 16385, 1, P, P, 16, P, NUL, NUL) == tts.TTS_ERR_UNSUPPORTED
    assert f(P, 10, 0, P, P, 4, P, NUL, NUL) == tts.TTS_OK  # nothing to do


def test_topk_long_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    f = L.tts_topk_select_long
    need = L.tts_topk_long_workspace_bytes(3, 300000, 2048)
    # per row: a 16-byte header (threshold key, candidate count) and room for 16384
    # candidates of 8 bytes, whatever the row's length
    assert need == 3 * (16 + 8 * 16384)
    assert L.tts_topk_long_workspace_bytes(0, 300000, 2048) == 0
    assert L.tts_topk_long_workspace_bytes(3, 300000, 4097) == 0
    A = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced
    assert f(NUL, 300000, 3, P, P, 2048, P, A, need, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 300000, 3, P, P, 0, P, A, need, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 300000, 3, P, P, 4097, P, A, need, NUL, NUL) == tts.TTS_ERR_UNSUPPORTED
    assert f(P, (1 << 30) + 1, 3, P, P, 16, P, A, need, NUL, NUL) == tts.TTS_ERR_UNSUPPORTED
    assert f(P, 300000, 3, P, P, 2048, P, NUL, need, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 300000, 3, P, P, 2048, P, A, need - 1, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(P, 300000, 3, P, P, 2048, P, ctypes.c_void_p(0x10008), need, NUL,
             NUL) == tts.TTS_ERR_INVALID_ARG  # misaligned workspace
    assert f(P, 300000, 0, P, P, 2048, P, NUL, 0, NUL, NUL) == tts.TTS_OK  # nothing to do


def _attn(L, **kw):
    a = dict(q=P, k=P, v=P, dt=0, tq=256, tk=256, cq=P, ck=P, b=1, mq=256, mk=256, hq=2, hkv=1,
             d=64, causal=0, scale=0.125, out=P, lse=NUL, ws=NUL, wsb=0, st=NUL, stream=NUL)
    a.update(kw)
    return L.tts_attn_fwd_varlen(*a.values())


def test_attn_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    assert _attn(L, q=NUL) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, hq=3, hkv=2) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, scale=0.0) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, scale=float("nan")) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, causal=2) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, b=0) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, dt=7) == tts.TTS_ERR_INVALID_ARG
    assert _attn(L, d=96) == tts.TTS_ERR_UNSUPPORTED
    assert _attn(L, q=ctypes.c_void_p(0x1008)) == tts.TTS_ERR_INVALID_ARG  # misaligned
    assert _attn(L, dt=1) == tts.TTS_ERR_WORKSPACE  # fp32 needs a workspace
    assert _attn(L, dt=0) == tts.TTS_ERR_WORKSPACE  # so does bf16 (the work counter)
    assert _attn(L, ws=P, wsb=255) == tts.TTS_ERR_WORKSPACE
    assert _attn(L, tq=0) == tts.TTS_OK


def _sparse(L, **kw):
    a = dict(q=P, nq=4, H=128, dqk=576, dv=512, kv=P, pages=41, ps=64, pt=P, nlp=41, kv_len=2590,
             idx=P, topk=2048, scale=0.04, out=P, lse=NUL, ws=NUL, wsb=0, st=NUL, stream=NUL)
    a.update(kw)
    return L.tts_sparse_attn_paged(*a.values())


def test_sparse_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    assert _sparse(L, q=NUL) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, idx=NUL) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, topk=0) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, dv=600) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, ps=0) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, scale=-1.0) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, H=64) == tts.TTS_ERR_UNSUPPORTED
    assert _sparse(L, topk=2049) == tts.TTS_ERR_UNSUPPORTED
    assert _sparse(L, ws=ctypes.c_void_p(0x1008), wsb=1 << 20) == tts.TTS_ERR_INVALID_ARG
    assert _sparse(L, nq=0) == tts.TTS_OK


def test_decode_and_kv_write_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    f = L.tts_sparse_attn_decode
    F32 = ctypes.c_float

    def dec(**kw):
        a = dict(q=P, n=4, h=128, dqk=576, dv=512, kv=P, pages=64, ps=64, pt=P, maxp=8, lens=P,
                 idx=P, topk=2048, scale=F32(0.05), out=P, lse=NUL, ws=NUL, wsb=0, st=NUL,
                 stream=NUL)
        a.update(kw)
        return f(*a.values())
    assert dec(lens=NUL) == tts.TTS_ERR_INVALID_ARG           # kv_lens is required
    assert dec(pt=NUL) == tts.TTS_ERR_INVALID_ARG
    assert dec(maxp=0) == tts.TTS_ERR_INVALID_ARG
    assert dec(scale=F32(0.0)) == tts.TTS_ERR_INVALID_ARG
    assert dec(h=64) == tts.TTS_ERR_UNSUPPORTED
    assert dec(topk=2049) == tts.TTS_ERR_UNSUPPORTED
    assert dec(q=ctypes.c_void_p(0x1008)) == tts.TTS_ERR_INVALID_ARG  # misaligned
    assert dec(n=0) == tts.TTS_OK
    g = L.tts_paged_kv_write
    #        kv_new ntok dim req pos  pt maxp nreq cache pages ps st stream
    assert g(NUL, 4, 576, NUL, P, P, 8, 4, P, 64, 64, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert g(P, 4, 577, NUL, P, P, 8, 4, P, 64, 64, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert g(P, 4, 576, NUL, NUL, P, 8, 4, P, 64, 64, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert g(P, 4, 576, NUL, P, P, 0, 4, P, 64, 64, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert g(ctypes.c_void_p(0x1004), 4, 576, NUL, P, P, 8, 4, P, 64, 64, NUL,
             NUL) == tts.TTS_ERR_INVALID_ARG
    assert g(P, 0, 576, NUL, P, P, 8, 4, P, 64, 64, NUL, NUL) == tts.TTS_OK


def test_sparse_workspace_bytes_without_device(L):
    # No GPU here: no split is planned; with nq <= 0 never.
    import torch
    assert L.tts_sparse_workspace_bytes(0) == 0
    if not torch.cuda.is_available():
        assert L.tts_sparse_workspace_bytes(323) == 0


def test_product_has_no_cpu_fallback():
    """The binding must not import the oracle or any CPU path."""
    pkg = os.path.join(ROOT, "tiled_top_sparse_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn


def test_qkv_rope_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    f = L.tts_qkv_rope
    A = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced
    ok = (A, 300, 1280, A, A, A, A, 32768, 16, 80, A, A, A, NUL, NUL)

    def call(**kw):
        names = ("x", "n", "hidden", "w", "bias", "pos", "cs", "max_pos", "heads", "d", "q",
                 "k", "v", "st", "stream")
        args = dict(zip(names, ok))
        args.update(kw)
        return f(*[args[n] for n in names])

    for name in ("x", "w", "pos", "cs", "q", "k", "v"):
        assert call(**{name: NUL}) == tts.TTS_ERR_INVALID_ARG, name
    assert call(n=-1) == tts.TTS_ERR_INVALID_ARG
    assert call(hidden=1284) == tts.TTS_ERR_INVALID_ARG       # rows not 16-byte strided
    assert call(hidden=0) == tts.TTS_ERR_INVALID_ARG
    assert call(max_pos=0) == tts.TTS_ERR_INVALID_ARG
    assert call(heads=0) == tts.TTS_ERR_INVALID_ARG
    assert call(x=ctypes.c_void_p(0x10008)) == tts.TTS_ERR_INVALID_ARG  # misaligned
    assert call(bias=ctypes.c_void_p(0x10004)) == tts.TTS_ERR_INVALID_ARG
    assert call(d=96) == tts.TTS_ERR_UNSUPPORTED
    assert call(d=128, heads=3) == tts.TTS_ERR_UNSUPPORTED    # 9 heads: not 2 per tile
    assert call(d=64, heads=3) == tts.TTS_ERR_UNSUPPORTED     # 9 heads: not 4 per tile
    assert call(n=0) == tts.TTS_OK                            # nothing to do
    assert call(n=0, bias=NUL) == tts.TTS_OK


def test_rope_cache_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    f = L.tts_rope_cache
    A = ctypes.c_void_p(0x10000)
    assert f(0, 80, 10000.0, A, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 79, 10000.0, A, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 0, 10000.0, A, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 80, 1.0, A, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 80, float("inf"), A, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 80, 10000.0, NUL, NUL) == tts.TTS_ERR_INVALID_ARG
    assert f(10, 80, 10000.0, ctypes.c_void_p(0x10004), NUL) == tts.TTS_ERR_INVALID_ARG


def test_fp8_prefill_host_validation(L):
    import tiled_top_sparse_gb300 as tts
    A = ctypes.c_void_p(0x10000)
    f = L.tts_attn_fwd_varlen_fp8
    ok = [A, A, A, A, A, 256, 256, A, A, 1, 256, 256, 4, 2, 128, 1, 0.1, A, A, A, 256, NUL, NUL]

    def call(i=None, val=None):
        args = list(ok)
        if i is not None:
            args[i] = val
        return f(*args)

    for i in (0, 1, 2, 3, 4, 7, 8, 17):
        assert call(i, NUL) == tts.TTS_ERR_INVALID_ARG, i
    assert call(14, 64) == tts.TTS_ERR_UNSUPPORTED         # e4m3 path: head_dim 128 only
    assert call(13, 3) == tts.TTS_ERR_INVALID_ARG          # 4 q heads over 3 KV heads
    assert call(16, -1.0) == tts.TTS_ERR_INVALID_ARG
    assert call(15, 2) == tts.TTS_ERR_INVALID_ARG
    assert call(19, NUL) == tts.TTS_ERR_WORKSPACE
    assert call(20, 16) == tts.TTS_ERR_WORKSPACE
    assert call(5, 0) == tts.TTS_OK                        # nothing to compute
    g = L.tts_quantize_fp8_prefill
    okq = [A, 10, 4, A, 10, 2, 128, A, A, A, A, NUL]
    for i, bad in ((1, -1), (2, 0), (5, 0), (6, 126), (10, NUL), (10, ctypes.c_void_p(0x10004)),
                   (0, NUL), (7, NUL), (8, NUL), (3, NUL), (9, NUL)):
        args = list(okq)
        args[i] = bad
        assert g(*args) == tts.TTS_ERR_INVALID_ARG, i
