"""Float64 CPU oracle for the tiled / top-k / sparse attention hot path.

TEST INFRASTRUCTURE ONLY: the plain, slow reference that the CUDA library is
checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. It shares no code with
the CUDA path (``tiled_top_sparse_gb300``) and neither imports the other.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
independent rows); this module only builds it with gcc and marshals numpy
arrays. Each function cites the passage of the pages it follows in that file:

* ``attn_varlen`` -- dense (optionally causal, grouped-KV) attention over packed
  variable-length sequences: the S = Q K^T, row softmax, P V pieces of the
  vision-encoder write-up ("DeepSeek V4.1 上 4×RTX 3090", section 三) and the
  cu_seqlens_q / cu_seqlens_k batch of the SGLang prefill write-up (section 2.2).
* ``topk`` -- stable descending selection, lower index wins on ties
  ("推理引擎的蝴蝶效应", 实验方法和结果; "AMD MI250部署", section 4.2).
* ``sparse_paged`` -- gather through a page table, canonical ascending index
  order, then attention ("推理引擎的蝴蝶效应", 实验方法和结果 / 进一步探索).
* ``qkv_rope`` / ``rope_cache`` -- the vision encoder's QKV projection followed by
  rotary position embedding of q and k ("DeepSeek V4.1 上 4×RTX 3090", 坑 1) and the
  position-indexed cos/sin cache ("从 SGLang Kernel源码到 GPU Trace", section 3.3);
  the RoPE variant is not on the pages: one-dimensional, rotate-half pairs
  (j, j + d/2), angle pos * base^(-2j/d), base 10000 unless given.
* ``round_bf16`` -- round-to-nearest-even of fp32 values to the bf16 grid, the
  rounding the CUDA path applies to fp32 inputs at its boundary.
* ``round_e4m3`` / ``quant_e4m3`` / ``quant_fp8_prefill`` -- FP8 (e4m3) rounding and
  block quantization of the prefill's q (one scale per token and head) and k (one scale
  per KV head) ("从 SGLang Kernel源码到 GPU Trace", section 3.2; "AMD MI250部署", sections
  4.1 and 5.3); the format and blocks are not on the pages: e4m3, scale = max|x| / 448.

Pins (tests/test_oracle.py): closed forms (Q = 0, huge scale, causal row 0,
identical keys, q = 0 / single index for sparse), invariants (rows of P sum to
1, selected >= unselected, permutation invariance), library routines that the
oracle does not itself call (torch SDPA in float64, numpy stable argsort),
brute force on tiny inputs, the boundary-tie worked example of the top-k
write-up, and the cross-pin sparse == dense when every position is selected.
No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP). Returns the path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_round_bf16.argtypes = [P, P, i64]
            lib.oracle_round_bf16.restype = None
            lib.oracle_attn_varlen.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, dbl,
                                               P, P, i64, P, P]
            lib.oracle_attn_varlen.restype = ctypes.c_int
            lib.oracle_topk.argtypes = [P, i64, i64, P, P, i32, P]
            lib.oracle_topk.restype = ctypes.c_int64
            lib.oracle_sparse_paged.argtypes = [P, i64, i32, i32, i32, P, i64, i32, P, i64, i64,
                                                P, i32, dbl, P, P]
            lib.oracle_sparse_paged.restype = ctypes.c_int64
            lib.oracle_qkv_rope.argtypes = [P, i64, i32, P, P, i32, i32, P, dbl, P, P, P]
            lib.oracle_qkv_rope.restype = None
            lib.oracle_rope_cache.argtypes = [i32, i32, dbl, P]
            lib.oracle_rope_cache.restype = None
            lib.oracle_round_e4m3.argtypes = [dbl]
            lib.oracle_round_e4m3.restype = dbl
            lib.oracle_quant_e4m3.argtypes = [P, i64, i64, P, P]
            lib.oracle_quant_e4m3.restype = None
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def round_bf16(x) -> np.ndarray:
    """fp32 -> nearest bf16 value (ties to even), returned as fp32."""
    x = _f32(x)
    out = np.empty_like(x)
    _load().oracle_round_bf16(_p(x), _p(out), x.size)
    return out


def attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, scale: float,
                rows=None):
    """Dense attention. q [Tq, Hq, d], k/v [Tk, Hkv, d] (float values).

    rows=None computes every (token, head); otherwise rows = (tok[], head[]) and
    the result is out [n, d], lse [n]. Returns (out float64, lse float64).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    cq, ck = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    Tq, hq, d = q.shape
    hkv = k.shape[1]
    batch = cq.size - 1
    if rows is None:
        out = np.empty((Tq, hq, d), np.float64)
        lse = np.empty((Tq, hq), np.float64)
        tp = hp = None
        n = 0
    else:
        tok, head = _i32(rows[0]), _i32(rows[1])
        n = tok.size
        out = np.empty((n, d), np.float64)
        lse = np.empty((n,), np.float64)
        tp, hp = _p(tok), _p(head)
    rc = _load().oracle_attn_varlen(_p(q), _p(k), _p(v), _p(cq), _p(ck), batch, hq, hkv, d,
                                    int(bool(causal)), float(scale), tp, hp, n, _p(out), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_varlen: invalid arguments (code {rc})")
    return out, lse


def topk(logits, row_starts, row_lens, k: int):
    """Top-k positions per row. Returns (idx int32 [rows, k], number of bad rows)."""
    x = _f32(logits)
    rows, stride = x.shape
    rs, rl = _i32(row_starts), _i32(row_lens)
    idx = np.empty((rows, k), np.int32)
    bad = _load().oracle_topk(_p(x), stride, rows, _p(rs), _p(rl), int(k), _p(idx))
    return idx, int(bad)


def sparse_paged(q, kv_cache, page_table, idx, kv_len: int, dv: int, scale: float):
    """Sparse attention through a page table.

    q [nq, H, dqk], kv_cache [pages, page_size, dqk], page_table [logical pages],
    idx [nq, topk]. Returns (out float64 [nq, H, dv], lse float64 [nq, H], skipped).
    """
    q, kv = _f32(q), _f32(kv_cache)
    pt, ix = _i32(page_table), _i32(idx)
    nq, H, dqk = q.shape
    pages, page_size, dk2 = kv.shape
    assert dk2 == dqk
    topk_ = ix.shape[1]
    out = np.empty((nq, H, dv), np.float64)
    lse = np.empty((nq, H), np.float64)
    bad = _load().oracle_sparse_paged(_p(q), nq, H, dqk, dv, _p(kv), pages, page_size, _p(pt),
                                      pt.size, int(kv_len), _p(ix), topk_, float(scale),
                                      _p(out), _p(lse))
    return out, lse, int(bad)


def qkv_rope(x, w, bias, positions, heads: int, d: int, base: float = 10000.0):
    """QKV projection + RoPE. x [n, hidden], w [3*heads*d, hidden], bias [3*heads*d] or
    None, positions [n]. Returns (q, k, v) float64 [n, heads, d]."""
    x, w = _f32(x), _f32(w)
    n, hidden = x.shape
    assert w.shape == (3 * heads * d, hidden) and d % 2 == 0
    b = None if bias is None else _f32(bias)
    pos = _i32(positions)
    assert pos.shape == (n,)
    q = np.empty((n, heads, d), np.float64)
    k = np.empty_like(q)
    v = np.empty_like(q)
    _load().oracle_qkv_rope(_p(x), n, hidden, _p(w), None if b is None else _p(b), heads, d,
                            _p(pos), float(base), _p(q), _p(k), _p(v))
    return q, k, v


def rope_cache(max_pos: int, rot_dim: int, base: float = 10000.0):
    """float64 [max_pos, rot_dim/2, 2]: (cos, sin) of pos * base^(-2j/rot_dim)."""
    out = np.empty((max_pos, rot_dim // 2, 2), np.float64)
    _load().oracle_rope_cache(int(max_pos), int(rot_dim), float(base), _p(out))
    return out


def round_e4m3(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even, |x| > 448 clamped to 448), float64."""
    a = np.asarray(x, dtype=np.float64)
    f = _load().oracle_round_e4m3
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.float64).reshape(a.shape)


def quant_e4m3(x, block_len: int):
    """Quantize contiguous blocks of block_len values. Returns (scales float32 [nblocks],
    codes float32 [same shape as x], the e4m3 values)."""
    xf = _f32(x)
    n = xf.size
    assert block_len > 0 and n % block_len == 0
    nb = n // block_len
    scale = np.empty(nb, np.float32)
    codes = np.empty(xf.shape, np.float32)
    _load().oracle_quant_e4m3(_p(xf), nb, block_len, _p(scale), _p(codes))
    return scale, codes


def quant_fp8_prefill(q, k):
    """The FP8 prefill's quantization of q [T, Hq, d] (one block per token and head) and
    k [T, Hkv, d] (one block per KV head, over all tokens). Returns (q_codes, q_scale
    [T, Hq], k_codes, k_scale [Hkv]) and the dequantized q and k (codes * scale, rounded
    to float32 for the attention oracle)."""
    q = _f32(q)
    k = _f32(k)
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    qs, qc = quant_e4m3(q, d)
    kt = np.ascontiguousarray(k.transpose(1, 0, 2))          # [Hkv, T, d]
    ks, kct = quant_e4m3(kt, max(tk, 1) * d) if tk > 0 else (np.ones(hkv, np.float32), kt)
    kc = np.ascontiguousarray(kct.transpose(1, 0, 2))
    qs = qs.reshape(tq, hq)
    qd = (qc.astype(np.float64) * qs[:, :, None]).astype(np.float32)
    kd = (kc.astype(np.float64) * ks[None, :, None]).astype(np.float32)
    return qc, qs, kc, ks, qd, kd
