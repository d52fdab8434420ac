"""Thin Python binding over libtts.so (the C ABI declared in include/tts.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There is
no fallback: if the library is missing or fails to load, calls raise.

    attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                    causal, scale, out=None, lse=None, workspace=None, status=None)
    topk_select(logits, row_starts, row_lens, k, idx=None, status=None)
    sparse_attn_paged(q, kv_cache, page_table, idx, kv_len, scale, dv=512,
                      out=None, lse=None, status=None)
    quantize_fp8_prefill(q, k)
    attn_fwd_varlen_fp8(q8, q_scale, k8, k_scale, v, cu_seqlens_q, cu_seqlens_k,
                        max_seqlen_q, max_seqlen_k, causal, scale, out=None, lse=None,
                        workspace=None, status=None)
    rope_cache(max_pos, rot_dim, base=10000.0, out=None, device=None)
    qkv_rope(x, w, bias, positions, cos_sin, num_heads, q=None, k=None, v=None,
             status=None)

`status`, when given, is a 1-element int32 CUDA tensor the kernels OR their
device-side flags into (see TTS_DEV_* in the header); `check_status(status)`
synchronises and raises on a set flag.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtts.so")

TTS_OK = 0
TTS_ERR_INVALID_ARG = 1
TTS_ERR_UNSUPPORTED = 2
TTS_ERR_CUDA = 3
TTS_ERR_INDEX_RANGE = 4
TTS_ERR_DEVICE_TIMEOUT = 5
TTS_ERR_WORKSPACE = 6
TTS_BF16 = 0
TTS_F32 = 1
TTS_DEV_INDEX_RANGE = 0x1
TTS_DEV_TIMEOUT = 0x2
TTS_DEV_BAD_ARG = 0x4

EXPORTED = (
    "tts_status_string",
    "tts_status_from_device",
    "tts_version",
    "tts_attn_workspace_bytes",
    "tts_attn_fwd_varlen",
    "tts_topk_select",
    "tts_topk_long_workspace_bytes",
    "tts_topk_select_long",
    "tts_sparse_attn_paged",
    "tts_sparse_workspace_bytes",
    "tts_sparse_attn_decode",
    "tts_paged_kv_write",
    "tts_quantize_fp8_prefill",
    "tts_attn_fwd_varlen_fp8",
    "tts_rope_cache",
    "tts_qkv_rope",
    "tts_attn_fwd_varlen_f32_noalloc",
    "tts_debug_wait_timeout",
)


class TTSError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libtts.so (built by tiled_top_sparse_gb300._build). Raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtts.so not built ({LIB_PATH}); run tiled_top_sparse_gb300/_build.py")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    L.tts_status_string.argtypes = [ctypes.c_int]
    L.tts_status_string.restype = ctypes.c_char_p
    L.tts_status_from_device.argtypes = [ctypes.c_uint32]
    L.tts_status_from_device.restype = ctypes.c_int
    L.tts_version.argtypes = []
    L.tts_version.restype = ctypes.c_int
    L.tts_attn_workspace_bytes.argtypes = [i64, i64, i32, i32, i32, ctypes.c_int]
    L.tts_attn_workspace_bytes.restype = ctypes.c_size_t
    L.tts_attn_fwd_varlen.argtypes = [P, P, P, ctypes.c_int, i64, i64, P, P, i32, i32, i32, i32,
                                      i32, i32, i32, f32, P, P, P, ctypes.c_size_t, P, P]
    L.tts_attn_fwd_varlen.restype = ctypes.c_int
    L.tts_topk_select.argtypes = [P, i64, i32, P, P, i32, P, P, P]
    L.tts_topk_select.restype = ctypes.c_int
    L.tts_topk_long_workspace_bytes.argtypes = [i32, i64, i32]
    L.tts_topk_long_workspace_bytes.restype = ctypes.c_size_t
    L.tts_topk_select_long.argtypes = [P, i64, i32, P, P, i32, P, P, ctypes.c_size_t, P, P]
    L.tts_topk_select_long.restype = ctypes.c_int
    L.tts_sparse_attn_paged.argtypes = [P, i32, i32, i32, i32, P, i32, i32, P, i32, i32, P, i32,
                                        f32, P, P, P, ctypes.c_size_t, P, P]
    L.tts_sparse_attn_paged.restype = ctypes.c_int
    L.tts_sparse_attn_decode.argtypes = [P, i32, i32, i32, i32, P, i32, i32, P, i32, P, P, i32,
                                         f32, P, P, P, ctypes.c_size_t, P, P]
    L.tts_sparse_attn_decode.restype = ctypes.c_int
    L.tts_paged_kv_write.argtypes = [P, i64, i32, P, P, P, i32, i32, P, i32, i32, P, P]
    L.tts_paged_kv_write.restype = ctypes.c_int
    L.tts_sparse_workspace_bytes.argtypes = [i32]
    L.tts_sparse_workspace_bytes.restype = ctypes.c_size_t
    L.tts_quantize_fp8_prefill.argtypes = [P, i64, i32, P, i64, i32, i32, P, P, P, P, P]
    L.tts_quantize_fp8_prefill.restype = ctypes.c_int
    L.tts_attn_fwd_varlen_fp8.argtypes = [P, P, P, P, P, i64, i64, P, P, i32, i32, i32, i32,
                                          i32, i32, i32, f32, P, P, P, ctypes.c_size_t, P, P]
    L.tts_attn_fwd_varlen_fp8.restype = ctypes.c_int
    L.tts_rope_cache.argtypes = [i32, i32, f32, P, P]
    L.tts_rope_cache.restype = ctypes.c_int
    L.tts_qkv_rope.argtypes = [P, i64, i32, P, P, P, P, i32, i32, i32, P, P, P, P, P]
    L.tts_qkv_rope.restype = ctypes.c_int
    L.tts_attn_fwd_varlen_f32_noalloc.argtypes = [P, P, P, i64, i64, P, P, i32, i32, i32, i32,
                                                  i32, i32, i32, f32, P, P, P, P]
    L.tts_attn_fwd_varlen_f32_noalloc.restype = ctypes.c_int
    L.tts_debug_wait_timeout.argtypes = [P, P]
    L.tts_debug_wait_timeout.restype = ctypes.c_int
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().tts_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(code: int, what: str):
    if code != TTS_OK:
        raise TTSError(code, what)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda_contig(t: torch.Tensor, name: str, dtype=None):
    _need(isinstance(t, torch.Tensor) and t.is_cuda, f"{name} must be a CUDA tensor")
    _need(t.is_contiguous(), f"{name} must be contiguous")
    if dtype is not None:
        _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")


def check_status(status: torch.Tensor, what: str = "device status"):
    """Synchronise on `status` (1-element int32 CUDA tensor) and raise if a flag is set."""
    v = int(status.item()) & 0xFFFFFFFF
    _check(lib().tts_status_from_device(ctypes.c_uint32(v)), what)


def debug_wait_timeout(status: torch.Tensor):
    """Run the library's bounded-wait self-test kernel (see tts_debug_wait_timeout)."""
    _cuda_contig(status, "status", torch.int32)
    _check(lib().tts_debug_wait_timeout(_ptr(status), _stream(status.device)),
           "tts_debug_wait_timeout")


def attn_workspace_bytes(total_q, total_k, num_heads_q, num_heads_kv, head_dim, dtype) -> int:
    code = TTS_F32 if dtype == torch.float32 else TTS_BF16
    return int(lib().tts_attn_workspace_bytes(int(total_q), int(total_k), int(num_heads_q),
                                              int(num_heads_kv), int(head_dim), code))


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal,
                    scale, out=None, lse=None, workspace=None, status=None, want_lse=True):
    """Dense attention forward over packed varlen sequences (tts_attn_fwd_varlen).

    q [total_q, Hq, d], k/v [total_k, Hkv, d] (bf16 or fp32, same dtype), cu_seqlens_* int32
    [batch+1] on the device. Returns (out fp32 [total_q, Hq, d], lse fp32 [total_q, Hq]).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _cuda_contig(t, n)
        _need(t.dim() == 3, f"{n} must be [tokens, heads, head_dim]")
    _need(q.dtype == k.dtype == v.dtype and q.dtype in (torch.bfloat16, torch.float32),
          "q, k, v must share dtype bf16 or fp32")
    _need(k.shape == v.shape, "k and v must have the same shape")
    _cuda_contig(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _cuda_contig(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    total_q, hq, d = q.shape
    total_k, hkv, d2 = k.shape
    _need(d == d2, "head_dim mismatch")
    batch = cu_seqlens_q.numel() - 1
    _need(batch >= 1 and cu_seqlens_k.numel() == batch + 1, "cu_seqlens sizes must be batch+1")
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=torch.float32, device=q.device)
    _cuda_contig(out, "out", torch.float32)
    _need(tuple(out.shape) == (total_q, hq, d), "out shape")
    if lse is None and want_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _cuda_contig(lse, "lse", torch.float32)
    dt = TTS_F32 if q.dtype == torch.float32 else TTS_BF16
    need = attn_workspace_bytes(total_q, total_k, hq, hkv, d, q.dtype)
    if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib().tts_attn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), dt, total_q, total_k, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        batch, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d, int(bool(causal)), float(scale),
        _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(status), _stream(q.device))
    _check(code, "tts_attn_fwd_varlen")
    return out, lse


def topk_select(logits, row_starts, row_lens, k, idx=None, status=None):
    """Deterministic per-row top-k (tts_topk_select). Returns idx int32 [rows, k]."""
    _cuda_contig(logits, "logits", torch.float32)
    _need(logits.dim() == 2, "logits must be [rows, row_stride]")
    _cuda_contig(row_starts, "row_starts", torch.int32)
    _cuda_contig(row_lens, "row_lens", torch.int32)
    rows, stride = logits.shape
    _need(row_starts.numel() == rows and row_lens.numel() == rows, "row_starts/row_lens size")
    if idx is None:
        idx = torch.empty((rows, int(k)), dtype=torch.int32, device=logits.device)
    _cuda_contig(idx, "idx", torch.int32)
    _need(tuple(idx.shape) == (rows, int(k)), "idx shape")
    code = lib().tts_topk_select(_ptr(logits), stride, rows, _ptr(row_starts), _ptr(row_lens),
                                 int(k), _ptr(idx), _ptr(status), _stream(logits.device))
    _check(code, "tts_topk_select")
    return idx


def topk_long_workspace_bytes(rows, row_stride, k) -> int:
    return int(lib().tts_topk_long_workspace_bytes(int(rows), int(row_stride), int(k)))


def topk_select_long(logits, row_starts, row_lens, k, idx=None, workspace=None, status=None):
    """Deterministic top-k over long rows (tts_topk_select_long): the same result as
    topk_select for rows up to 2^30 values. Returns idx int32 [rows, k]. A workspace of
    topk_long_workspace_bytes(...) bytes is allocated here when `workspace` is missing."""
    _cuda_contig(logits, "logits", torch.float32)
    _need(logits.dim() == 2, "logits must be [rows, row_stride]")
    _cuda_contig(row_starts, "row_starts", torch.int32)
    _cuda_contig(row_lens, "row_lens", torch.int32)
    rows, stride = logits.shape
    _need(row_starts.numel() == rows and row_lens.numel() == rows, "row_starts/row_lens size")
    if idx is None:
        idx = torch.empty((rows, int(k)), dtype=torch.int32, device=logits.device)
    _cuda_contig(idx, "idx", torch.int32)
    _need(tuple(idx.shape) == (rows, int(k)), "idx shape")
    need = topk_long_workspace_bytes(rows, stride, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=logits.device)
    _cuda_contig(workspace, "workspace", torch.uint8)
    code = lib().tts_topk_select_long(_ptr(logits), stride, rows, _ptr(row_starts),
                                      _ptr(row_lens), int(k), _ptr(idx), _ptr(workspace),
                                      workspace.numel(), _ptr(status), _stream(logits.device))
    _check(code, "tts_topk_select_long")
    return idx


def sparse_attn_decode(q, kv_cache, page_tables, kv_lens, idx, scale, dv=512, out=None,
                       lse=None, workspace=None, status=None, want_lse=True, split=True):
    """Decode-shaped sparse attention (tts_sparse_attn_decode): one query per request,
    request n reading through page_tables[n] with length kv_lens[n].

    q bf16 [nreq, H, dqk], kv_cache bf16 [pages, page_size, dqk], page_tables int32
    [nreq, max_pages], kv_lens int32 [nreq], idx int32 [nreq, topk]. Returns (out fp32
    [nreq, H, dv], lse fp32 [nreq, H]); `split` as in sparse_attn_paged."""
    _cuda_contig(q, "q", torch.bfloat16)
    _cuda_contig(kv_cache, "kv_cache", torch.bfloat16)
    _cuda_contig(page_tables, "page_tables", torch.int32)
    _cuda_contig(kv_lens, "kv_lens", torch.int32)
    _cuda_contig(idx, "idx", torch.int32)
    _need(q.dim() == 3 and kv_cache.dim() == 3 and idx.dim() == 2 and page_tables.dim() == 2,
          "ranks")
    nreq, H, dqk = q.shape
    pages, page_size, dk2 = kv_cache.shape
    _need(dk2 == dqk and idx.shape[0] == nreq and page_tables.shape[0] == nreq and
          kv_lens.numel() == nreq, "shapes")
    if out is None:
        out = torch.empty((nreq, H, dv), dtype=torch.float32, device=q.device)
    _cuda_contig(out, "out", torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((nreq, H), dtype=torch.float32, device=q.device)
    ws_bytes = 0
    if split:
        need = sparse_workspace_bytes(nreq)
        if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    else:
        workspace = None
    code = lib().tts_sparse_attn_decode(
        _ptr(q), nreq, H, dqk, int(dv), _ptr(kv_cache), pages, page_size, _ptr(page_tables),
        page_tables.shape[1], _ptr(kv_lens), _ptr(idx), idx.shape[1], float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), ws_bytes, _ptr(status), _stream(q.device))
    _check(code, "tts_sparse_attn_decode")
    return out, lse


def paged_kv_write(kv_cache, page_tables, kv_new, positions, req_ids=None, status=None):
    """Write rows into the paged KV cache (tts_paged_kv_write): token t's row kv_new[t]
    goes to its request's page at logical position positions[t]. In place; returns
    kv_cache."""
    _cuda_contig(kv_cache, "kv_cache", torch.bfloat16)
    _cuda_contig(page_tables, "page_tables", torch.int32)
    _cuda_contig(kv_new, "kv_new", torch.bfloat16)
    _cuda_contig(positions, "positions", torch.int32)
    if req_ids is not None:
        _cuda_contig(req_ids, "req_ids", torch.int32)
    _need(kv_cache.dim() == 3 and kv_new.dim() == 2 and page_tables.dim() == 2, "ranks")
    pages, page_size, dim = kv_cache.shape
    ntok = kv_new.shape[0]
    _need(kv_new.shape[1] == dim and positions.numel() == ntok and
          (req_ids is None or req_ids.numel() == ntok), "shapes")
    code = lib().tts_paged_kv_write(_ptr(kv_new), ntok, dim, _ptr(req_ids), _ptr(positions),
                                    _ptr(page_tables), page_tables.shape[1],
                                    page_tables.shape[0], _ptr(kv_cache), pages, page_size,
                                    _ptr(status), _stream(kv_new.device))
    _check(code, "tts_paged_kv_write")
    return kv_cache


def sparse_workspace_bytes(nq) -> int:
    return int(lib().tts_sparse_workspace_bytes(int(nq)))


def sparse_attn_paged(q, kv_cache, page_table, idx, kv_len, scale, dv=512, out=None, lse=None,
                      workspace=None, status=None, want_lse=True, split=True):
    """Order-invariant sparse attention through a page table (tts_sparse_attn_paged).

    q bf16 [nq, H, dqk], kv_cache bf16 [pages, page_size, dqk], page_table int32 [n_pages],
    idx int32 [nq, topk]. Returns (out fp32 [nq, H, dv], lse fp32 [nq, H]). With split
    (default) a workspace for the split of the last wave is passed (allocated here when
    `workspace` is missing or too small); split=False passes none.
    """
    _cuda_contig(q, "q", torch.bfloat16)
    _cuda_contig(kv_cache, "kv_cache", torch.bfloat16)
    _cuda_contig(page_table, "page_table", torch.int32)
    _cuda_contig(idx, "idx", torch.int32)
    _need(q.dim() == 3 and kv_cache.dim() == 3 and idx.dim() == 2, "ranks")
    nq, H, dqk = q.shape
    pages, page_size, dk2 = kv_cache.shape
    _need(dk2 == dqk and idx.shape[0] == nq, "shapes")
    if out is None:
        out = torch.empty((nq, H, dv), dtype=torch.float32, device=q.device)
    _cuda_contig(out, "out", torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((nq, H), dtype=torch.float32, device=q.device)
    ws_bytes = 0
    if split:
        need = sparse_workspace_bytes(nq)
        if need > 0 and (workspace is None or workspace.numel() * workspace.element_size() < need):
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    else:
        workspace = None
    code = lib().tts_sparse_attn_paged(
        _ptr(q), nq, H, dqk, int(dv), _ptr(kv_cache), pages, page_size, _ptr(page_table),
        page_table.numel(), int(kv_len), _ptr(idx), idx.shape[1], float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), ws_bytes, _ptr(status), _stream(q.device))
    _check(code, "tts_sparse_attn_paged")
    return out, lse


def rope_cache(max_pos, rot_dim, base=10000.0, out=None, device=None):
    """cos/sin table of rotary embedding (tts_rope_cache): fp32 [max_pos, rot_dim/2, 2]
    holding (cos, sin) of p * base^(-2j/rot_dim)."""
    if out is None:
        dev = torch.device("cuda") if device is None else torch.device(device)
        out = torch.empty((int(max_pos), int(rot_dim) // 2, 2), dtype=torch.float32, device=dev)
    _cuda_contig(out, "out", torch.float32)
    _need(tuple(out.shape) == (int(max_pos), int(rot_dim) // 2, 2), "out shape")
    code = lib().tts_rope_cache(int(max_pos), int(rot_dim), float(base), _ptr(out),
                                _stream(out.device))
    _check(code, "tts_rope_cache")
    return out


def qkv_rope(x, w, bias, positions, cos_sin, num_heads, q=None, k=None, v=None, status=None):
    """Vision QKV projection + RoPE (tts_qkv_rope).

    x bf16 [n, hidden], w bf16 [3*H*d, hidden], bias fp32 [3*H*d] or None, positions
    int32 [n], cos_sin fp32 [max_pos, d/2, 2] (rope_cache with rot_dim = d). Returns
    (q, k, v) bf16 [n, H, d]: q and k rotated, v as projected."""
    _cuda_contig(x, "x", torch.bfloat16)
    _cuda_contig(w, "w", torch.bfloat16)
    _cuda_contig(positions, "positions", torch.int32)
    _cuda_contig(cos_sin, "cos_sin", torch.float32)
    _need(x.dim() == 2 and w.dim() == 2 and w.shape[1] == x.shape[1], "x [n, hidden], "
          "w [3*H*d, hidden]")
    n, hidden = x.shape
    H = int(num_heads)
    _need(w.shape[0] % (3 * H) == 0, "w rows must be 3 * num_heads * head_dim")
    d = w.shape[0] // (3 * H)
    _need(positions.numel() == n, "positions size")
    _need(cos_sin.dim() == 3 and cos_sin.shape[1] == d // 2 and cos_sin.shape[2] == 2,
          "cos_sin must be [max_pos, head_dim/2, 2]")
    if bias is not None:
        _cuda_contig(bias, "bias", torch.float32)
        _need(bias.numel() == 3 * H * d, "bias size")
    outs = []
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if t is None:
            t = torch.empty((n, H, d), dtype=torch.bfloat16, device=x.device)
        _cuda_contig(t, name, torch.bfloat16)
        _need(tuple(t.shape) == (n, H, d), f"{name} shape")
        outs.append(t)
    code = lib().tts_qkv_rope(_ptr(x), n, hidden, _ptr(w), _ptr(bias), _ptr(positions),
                              _ptr(cos_sin), cos_sin.shape[0], H, d, _ptr(outs[0]),
                              _ptr(outs[1]), _ptr(outs[2]), _ptr(status), _stream(x.device))
    _check(code, "tts_qkv_rope")
    return tuple(outs)


def quantize_fp8_prefill(q, k, q8=None, q_scale=None, k8=None, k_scale=None):
    """e4m3 block quantization (tts_quantize_fp8_prefill) of q bf16 [Tq, Hq, d] (scale per
    token and head) and k bf16 [Tk, Hkv, d] (scale per KV head). Returns (q8, q_scale, k8,
    k_scale): codes as uint8 tensors of the input shapes (view them as
    torch.float8_e4m3fn to read values), scales fp32 [Tq, Hq] and [Hkv]."""
    _cuda_contig(q, "q", torch.bfloat16)
    _cuda_contig(k, "k", torch.bfloat16)
    _need(q.dim() == 3 and k.dim() == 3 and q.shape[2] == k.shape[2], "q, k [tokens, heads, d]")
    tq, hq, d = q.shape
    tk, hkv, _ = k.shape
    dev = q.device
    q8 = torch.empty((tq, hq, d), dtype=torch.uint8, device=dev) if q8 is None else q8
    k8 = torch.empty((tk, hkv, d), dtype=torch.uint8, device=dev) if k8 is None else k8
    q_scale = torch.empty((tq, hq), dtype=torch.float32, device=dev) if q_scale is None else q_scale
    k_scale = torch.empty((hkv,), dtype=torch.float32, device=dev) if k_scale is None else k_scale
    for t, n, dt in ((q8, "q8", torch.uint8), (k8, "k8", torch.uint8),
                     (q_scale, "q_scale", torch.float32), (k_scale, "k_scale", torch.float32)):
        _cuda_contig(t, n, dt)
    code = lib().tts_quantize_fp8_prefill(_ptr(q), tq, hq, _ptr(k), tk, hkv, d, _ptr(q8),
                                          _ptr(q_scale), _ptr(k8), _ptr(k_scale),
                                          _stream(dev))
    _check(code, "tts_quantize_fp8_prefill")
    return q8, q_scale, k8, k_scale


def attn_fwd_varlen_fp8(q8, q_scale, k8, k_scale, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                        max_seqlen_k, causal, scale, out=None, lse=None, workspace=None,
                        status=None, want_lse=True):
    """Dense attention with e4m3 q / k in Q K^T (tts_attn_fwd_varlen_fp8). q8 / k8 uint8
    codes [T, H, 128] with their scales from quantize_fp8_prefill, v bf16. Returns (out
    fp32 [Tq, Hq, 128], lse fp32 [Tq, Hq])."""
    _cuda_contig(q8, "q8", torch.uint8)
    _cuda_contig(k8, "k8", torch.uint8)
    _cuda_contig(q_scale, "q_scale", torch.float32)
    _cuda_contig(k_scale, "k_scale", torch.float32)
    _cuda_contig(v, "v", torch.bfloat16)
    _cuda_contig(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _cuda_contig(cu_seqlens_k, "cu_seqlens_k", torch.int32)
    _need(q8.dim() == 3 and k8.shape == v.shape, "q8 [Tq, Hq, d]; k8, v [Tk, Hkv, d]")
    total_q, hq, d = q8.shape
    total_k, hkv, _ = k8.shape
    _need(tuple(q_scale.shape) == (total_q, hq) and k_scale.numel() == hkv, "scale shapes")
    batch = cu_seqlens_q.numel() - 1
    _need(batch >= 1 and cu_seqlens_k.numel() == batch + 1, "cu_seqlens sizes must be batch+1")
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=torch.float32, device=q8.device)
    _cuda_contig(out, "out", torch.float32)
    if lse is None and want_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q8.device)
    need = attn_workspace_bytes(total_q, total_k, hq, hkv, d, torch.bfloat16)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q8.device)
    code = lib().tts_attn_fwd_varlen_fp8(
        _ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(v), total_q, total_k,
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, int(max_seqlen_q), int(max_seqlen_k), hq,
        hkv, d, int(bool(causal)), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(q8.device))
    _check(code, "tts_attn_fwd_varlen_fp8")
    return out, lse
