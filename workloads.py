"""Seeded synthetic inputs shaped like the workloads the pages describe.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path's tests/benchmark and the CPU oracle
take their inputs from here. All draws use ``torch.Generator('cpu')`` with a
fixed seed, so a given (config, seed) yields identical tensors on any machine.

Named workloads (sizes from the pages):
  tiny     1 head, N = 256, d = 64, fp32 Q/K/V ~ N(0,1), non-causal, scale 1/8.
  vision   N = 8547 patch tokens (111 x 77 grid), 16 heads, d = 80, bf16, non-causal
           (the image size of the vision-encoder write-up, section 三).
  varlen   8 sequences, lengths ~ U[512, 8192] redrawn until the total <= 32768,
           32 query / 8 KV heads, d = 128, bf16, causal (SGLang prefill write-up,
           section 2.2: cu_seqlens_q / cu_seqlens_k, max_seq_len 32768).
  topk     fp32 logits (323, 2590) ~ N(0,1) rounded to the bf16 grid (so that equal
           values occur), row_lens[i] = 2590 - 323 + 1 + i, row_starts = 0, k = 2048
           (the (323, 2590) -> (323, 2048) shapes of the V32 write-up).
  sparse   323 queries x 128 heads, q/k dim 576 (512 latent + 64 rope), v dim 512,
           bf16 paged KV cache of 2590 tokens in pages of 64 with a shuffled page
           table, 2048 distinct indices per query inside its causal window,
           scale 1/sqrt(576); index permutations drawn with seeds 100..107.
  vision_qkv  the projection in front of the vision attention: N = 8547 tokens,
           hidden = 16 x 80 = 1280, x ~ N(0,1) and W ~ N(0, 1/hidden) in bf16 (so
           q/k/v come out near unit variance), bias ~ N(0, 0.1^2) fp32, positions
           0..N-1, cos/sin table over 32768 positions (the max_seq_len of the
           SGLang write-up's RoPE table).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SEEDS = {"tiny": 0, "vision": 1, "varlen": 2, "topk": 3, "sparse": 4, "topk_long": 5,
         "decode": 6, "vision_qkv": 7}
PERM_SEEDS = tuple(range(100, 108))


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return g


@dataclass
class DenseInputs:
    q: torch.Tensor  # [Tq, Hq, d]   fp32 or bf16, CPU
    k: torch.Tensor  # [Tk, Hkv, d]
    v: torch.Tensor  # [Tk, Hkv, d]
    cu_seqlens_q: torch.Tensor  # int32 [B+1]
    cu_seqlens_k: torch.Tensor  # int32 [B+1]
    max_seqlen_q: int
    max_seqlen_k: int
    causal: bool
    scale: float
    lengths_q: list = field(default_factory=list)
    lengths_k: list = field(default_factory=list)

    def flops(self) -> float:
        """Algorithmic FLOPs: 2 matmuls x 2 flops per multiply-add per visible (q, k) pair."""
        d = self.q.shape[2]
        hq = self.q.shape[1]
        pairs = 0
        for lq, lk in zip(self.lengths_q, self.lengths_k):
            if self.causal:
                # row i sees min(lk, max(0, i + lk - lq + 1)) keys
                for_rows = 0
                off = lk - lq
                # closed-form sum over i of clamp(i + off + 1, 0, lk)
                for i in range(lq):
                    for_rows += min(lk, max(0, i + off + 1))
                pairs += for_rows
            else:
                pairs += lq * lk
        return 4.0 * d * hq * pairs


def dense_inputs(lengths_q, lengths_k=None, hq=1, hkv=1, d=64, causal=False, dtype=torch.bfloat16,
                 seed=0, scale=None) -> DenseInputs:
    """Packed varlen Q/K/V ~ N(0,1) for the given per-sequence lengths."""
    lengths_q = [int(x) for x in lengths_q]
    lengths_k = lengths_q if lengths_k is None else [int(x) for x in lengths_k]
    g = _gen(seed)
    tq, tk = sum(lengths_q), sum(lengths_k)
    q = torch.randn(tq, hq, d, generator=g, dtype=torch.float32)
    k = torch.randn(tk, hkv, d, generator=g, dtype=torch.float32)
    v = torch.randn(tk, hkv, d, generator=g, dtype=torch.float32)
    if dtype != torch.float32:
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    cq = torch.zeros(len(lengths_q) + 1, dtype=torch.int32)
    ck = torch.zeros(len(lengths_k) + 1, dtype=torch.int32)
    cq[1:] = torch.cumsum(torch.tensor(lengths_q, dtype=torch.int64), 0).to(torch.int32)
    ck[1:] = torch.cumsum(torch.tensor(lengths_k, dtype=torch.int64), 0).to(torch.int32)
    return DenseInputs(q, k, v, cq, ck, max(lengths_q + [0]), max(lengths_k + [0]), causal,
                       float(scale if scale is not None else 1.0 / math.sqrt(d)),
                       lengths_q, lengths_k)


def varlen_lengths(seed: int, batch=8, lo=512, hi=8192, total_max=32768) -> list:
    """Draw `batch` lengths ~ U[lo, hi]; redraw the whole batch until sum <= total_max."""
    g = _gen(seed)
    while True:
        lens = torch.randint(lo, hi + 1, (batch,), generator=g).tolist()
        if sum(lens) <= total_max:
            return lens


def tiny() -> DenseInputs:
    return dense_inputs([256], hq=1, hkv=1, d=64, causal=False, dtype=torch.float32,
                        seed=SEEDS["tiny"])


def vision(n=8547, heads=16, d=80, seed=None) -> DenseInputs:
    return dense_inputs([n], hq=heads, hkv=heads, d=d, causal=False, dtype=torch.bfloat16,
                        seed=SEEDS["vision"] if seed is None else seed)


def varlen(seed=None, hq=32, hkv=8, d=128, lengths=None) -> DenseInputs:
    s = SEEDS["varlen"] if seed is None else seed
    lens = varlen_lengths(s) if lengths is None else list(lengths)
    return dense_inputs(lens, hq=hq, hkv=hkv, d=d, causal=True, dtype=torch.bfloat16, seed=s + 1000)


@dataclass
class TopkInputs:
    logits: torch.Tensor  # fp32 [rows, stride]
    row_starts: torch.Tensor  # int32 [rows]
    row_lens: torch.Tensor  # int32 [rows]
    k: int

    def bytes(self) -> int:
        """Algorithmic HBM bytes: the valid windows read once, the index matrix written once."""
        rows = self.logits.shape[0]
        return int(self.row_lens.clamp(min=0).sum().item()) * 4 + rows * self.k * 4 + rows * 8


def topk_inputs(rows=323, cols=2590, k=2048, seed=None, causal=True, bf16_grid=True,
                row_lens=None, row_starts=None) -> TopkInputs:
    g = _gen(SEEDS["topk"] if seed is None else seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    if bf16_grid:
        x = x.to(torch.bfloat16).to(torch.float32)
    if row_lens is None:
        if causal:
            # the last `rows` queries of a `cols`-token context
            row_lens = torch.arange(rows, dtype=torch.int32) + (cols - rows + 1)
        else:
            row_lens = torch.full((rows,), cols, dtype=torch.int32)
    if row_starts is None:
        row_starts = torch.zeros(rows, dtype=torch.int32)
    return TopkInputs(x, torch.as_tensor(row_starts, dtype=torch.int32),
                      torch.as_tensor(row_lens, dtype=torch.int32), int(k))


def topk_long_inputs(rows=64, cols=262144, k=2048, seed=None) -> TopkInputs:
    """Indexer logits of the last `rows` queries of a `cols`-token context (rows longer
    than one CTA can hold: the long-row top-k); same value recipe as topk_inputs."""
    return topk_inputs(rows=rows, cols=cols, k=k,
                       seed=SEEDS["topk_long"] if seed is None else seed, causal=True)


@dataclass
class SparseInputs:
    q: torch.Tensor  # bf16 [nq, H, dqk]
    kv_cache: torch.Tensor  # bf16 [pages, page_size, dqk]
    page_table: torch.Tensor  # int32 [logical pages]
    idx: torch.Tensor  # int32 [nq, topk]
    kv_len: int
    dv: int
    scale: float

    def gathered_bytes(self) -> int:
        """Bytes of KV rows the method gathers: one dqk-wide bf16 row per valid index."""
        valid = int((self.idx >= 0).sum().item())
        return valid * self.kv_cache.shape[2] * 2

    def flops(self) -> float:
        valid = int((self.idx >= 0).sum().item())
        H, dqk = self.q.shape[1], self.q.shape[2]
        return 2.0 * H * valid * (dqk + self.dv)


def sparse_inputs(nq=323, heads=128, dqk=576, dv=512, kv_len=2590, page_size=64, topk=2048,
                  seed=None, causal_windows=True) -> SparseInputs:
    g = _gen(SEEDS["sparse"] if seed is None else seed)
    pages = (kv_len + page_size - 1) // page_size
    q = torch.randn(nq, heads, dqk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.randn(pages, page_size, dqk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    page_table = torch.randperm(pages, generator=g).to(torch.int32)
    idx = torch.full((nq, topk), -1, dtype=torch.int32)
    for n in range(nq):
        # query n sits at position kv_len - nq + n and sees positions 0 .. that position
        win = (kv_len - nq + 1 + n) if causal_windows else kv_len
        win = max(1, min(win, kv_len))
        take = min(topk, win)
        idx[n, :take] = torch.randperm(win, generator=g)[:take].to(torch.int32)
    return SparseInputs(q, kv, page_table, idx, kv_len, dv, 1.0 / math.sqrt(dqk))


@dataclass
class DecodeInputs:
    q: torch.Tensor            # bf16 [nreq, H, dqk]: each request's one new query
    kv_cache: torch.Tensor     # bf16 [pages, page_size, dqk], a pool shared by the requests
    page_tables: torch.Tensor  # int32 [nreq, max_pages]; -1 past a request's pages
    kv_lens: torch.Tensor      # int32 [nreq]
    idx: torch.Tensor          # int32 [nreq, topk] logical positions, -1 = empty slot
    kv_new: torch.Tensor       # bf16 [nreq, dqk]: each request's next KV row
    dv: int
    scale: float

    def gathered_bytes(self) -> int:
        valid = int((self.idx >= 0).sum().item())
        return valid * self.kv_cache.shape[2] * 2

    def flops(self) -> float:
        valid = int((self.idx >= 0).sum().item())
        H, dqk = self.q.shape[1], self.q.shape[2]
        return 2.0 * H * valid * (dqk + self.dv)


def sparse_decode_inputs(kv_lens=(2590,) * 8, heads=128, dqk=576, dv=512, page_size=64,
                         topk=2048, seed=None, spare_pages=3) -> DecodeInputs:
    """Decode step of several requests: request n has kv_lens[n] tokens in its own pages,
    drawn shuffled from one pool (plus room for one more token), and one query whose
    top-k index list is a random subset of its positions (all of them when shorter)."""
    g = _gen(SEEDS["decode"] if seed is None else seed)
    nreq = len(kv_lens)
    need = [(int(L) + 1 + page_size - 1) // page_size for L in kv_lens]  # + the next token
    max_pages = max(need)
    pool = sum(need) + spare_pages
    order = torch.randperm(pool, generator=g).to(torch.int32)
    page_tables = torch.full((nreq, max_pages), -1, dtype=torch.int32)
    at = 0
    for n, c in enumerate(need):
        page_tables[n, :c] = order[at:at + c]
        at += c
    q = torch.randn(nreq, heads, dqk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    kv = torch.randn(pool, page_size, dqk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    idx = torch.full((nreq, topk), -1, dtype=torch.int32)
    for n, L in enumerate(kv_lens):
        take = min(topk, int(L))
        if take > 0:
            idx[n, :take] = torch.randperm(int(L), generator=g)[:take].to(torch.int32)
    kv_new = torch.randn(nreq, dqk, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return DecodeInputs(q, kv, page_tables, torch.tensor(kv_lens, dtype=torch.int32), idx,
                        kv_new, dv, 1.0 / math.sqrt(dqk))


def permute_rows(idx: torch.Tensor, seed: int) -> torch.Tensor:
    """Shuffle the entries of every row of an index matrix (seeded)."""
    g = _gen(seed)
    out = idx.clone()
    for r in range(idx.shape[0]):
        out[r] = idx[r, torch.randperm(idx.shape[1], generator=g)]
    return out


@dataclass
class QkvInputs:
    x: torch.Tensor          # bf16 [n, hidden]
    w: torch.Tensor          # bf16 [3 * heads * d, hidden]
    bias: torch.Tensor       # fp32 [3 * heads * d] or None
    positions: torch.Tensor  # int32 [n]
    heads: int
    d: int
    max_pos: int
    base: float = 10000.0

    def flops(self) -> float:
        """Algorithmic FLOPs of the projection: 2 per multiply-add of x W^T."""
        n, hidden = self.x.shape
        return 2.0 * n * hidden * self.w.shape[0]


def vision_qkv_inputs(n=8547, heads=16, d=80, hidden=None, max_pos=32768, bias=True,
                      positions=None, seed=None) -> QkvInputs:
    g = _gen(SEEDS["vision_qkv"] if seed is None else seed)
    hidden = heads * d if hidden is None else hidden
    x = torch.randn(n, hidden, generator=g).to(torch.bfloat16)
    w = (torch.randn(3 * heads * d, hidden, generator=g) / math.sqrt(hidden)).to(torch.bfloat16)
    b = (0.1 * torch.randn(3 * heads * d, generator=g)) if bias else None
    if positions is None:
        positions = torch.arange(n, dtype=torch.int32)
    return QkvInputs(x, w, b, positions.to(torch.int32), heads, d, max_pos)
