"""GPU parity for the decode-shaped calls: tts_sparse_attn_decode (one query per request,
per-request page tables and lengths) against the float64 oracle applied request by
request, its bitwise invariance under index permutations and its split-KV path, and
tts_paged_kv_write (rows land where the page table says, bad tokens are skipped)."""
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


def dev(t):
    return t.to("cuda")


def run(tts, inp: W.DecodeInputs, idx=None, kv_lens=None, kv_cache=None, status=None,
        split=True):
    return tts.sparse_attn_decode(dev(inp.q), dev(inp.kv_cache if kv_cache is None else kv_cache),
                                  dev(inp.page_tables),
                                  dev(inp.kv_lens if kv_lens is None else kv_lens),
                                  dev(inp.idx if idx is None else idx), inp.scale, dv=inp.dv,
                                  status=status, split=split)


def ref(inp: W.DecodeInputs, idx=None, kv_lens=None, kv_cache=None):
    """The oracle's sparse attention, one request at a time with its own table."""
    ix = (inp.idx if idx is None else idx).numpy()
    lens = (inp.kv_lens if kv_lens is None else kv_lens).numpy()
    kv = (inp.kv_cache if kv_cache is None else kv_cache).float().numpy()
    q = inp.q.float().numpy()
    outs, lses, bad = [], [], 0
    for n in range(q.shape[0]):
        o, l, b = oracle.sparse_paged(q[n:n + 1], kv, inp.page_tables[n].numpy(), ix[n:n + 1],
                                      int(lens[n]), inp.dv, inp.scale)
        outs.append(o)
        lses.append(l)
        bad += b
    return np.concatenate(outs), np.concatenate(lses), bad


@pytest.mark.parametrize("kv_lens", [(1, 63, 64, 65, 2590, 700),
                                     (20000, 3000, 40000, 5)])  # above the counting sort
def test_parity_per_request(tts, kv_lens):
    inp = W.sparse_decode_inputs(kv_lens=kv_lens, seed=sum(kv_lens))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, status=st)
    tts.check_status(st)
    ro, rl, bad = ref(inp)
    assert bad == 0
    assert_close_attn(out.cpu().numpy(), ro, f"decode {kv_lens}")
    assert_lse_close(lse.cpu().numpy(), rl, "decode lse")


def test_permutation_invariance_bitwise(tts):
    inp = W.sparse_decode_inputs(kv_lens=(2590, 5000, 900, 30000), seed=61)
    base = [t.clone() for t in run(tts, inp)]
    for s in W.PERM_SEEDS[:3]:
        out, lse = run(tts, inp, idx=W.permute_rows(inp.idx, s))
        assert torch.equal(out, base[0]) and torch.equal(lse, base[1])


def test_split_kv_small_batch(tts):
    # three requests: six (request, V half) units on the SMs, so each runs as 4 parts
    inp = W.sparse_decode_inputs(kv_lens=(2590, 16000, 65536), seed=62)
    out, lse = run(tts, inp)
    ro, rl, _ = ref(inp)
    assert_close_attn(out.cpu().numpy(), ro, "decode split")
    assert_lse_close(lse.cpu().numpy(), rl, "decode split lse")
    again = run(tts, inp)
    assert torch.equal(again[0], out) and torch.equal(again[1], lse)  # fixed-order combine
    whole, _ = run(tts, inp, split=False)
    scale = float(np.abs(ro).max())
    assert float((whole - out).abs().max()) <= 2 ** -7 * scale  # rounding of the bf16 P only


def test_shared_table_equals_prefill_call(tts):
    # every request with the same table and length: the decode call is the prefill call
    inp = W.sparse_inputs(nq=5, kv_len=3000, topk=2048, seed=63)
    q, kv, pt, ix = dev(inp.q), dev(inp.kv_cache), dev(inp.page_table), dev(inp.idx)
    a = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, dv=inp.dv)
    tables = pt.unsqueeze(0).repeat(5, 1).contiguous()
    lens = torch.full((5,), inp.kv_len, dtype=torch.int32, device="cuda")
    b = tts.sparse_attn_decode(q, kv, tables, lens, ix, inp.scale, dv=inp.dv)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_kv_write_then_attend_to_the_new_token(tts):
    inp = W.sparse_decode_inputs(kv_lens=(100, 2590, 64, 4095), seed=64)
    cache = dev(inp.kv_cache).clone()
    pos = dev(inp.kv_lens)  # each request's next position
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.paged_kv_write(cache, dev(inp.page_tables), dev(inp.kv_new), pos, status=st)
    tts.check_status(st)
    # exactly the addressed rows changed, to the new rows
    want = inp.kv_cache.clone()
    ps = inp.kv_cache.shape[1]
    for n, L in enumerate(inp.kv_lens.tolist()):
        want[inp.page_tables[n, L // ps], L % ps] = inp.kv_new[n]
    assert torch.equal(cache.cpu(), want)
    # the new token joins each request's index list
    idx = inp.idx.clone()
    for n, L in enumerate(inp.kv_lens.tolist()):
        free = (idx[n] < 0).nonzero()
        idx[n, int(free[0]) if len(free) else 0] = L
    lens = inp.kv_lens + 1
    out, lse = run(tts, inp, idx=idx, kv_lens=lens, kv_cache=cache)
    ro, rl, bad = ref(inp, idx=idx, kv_lens=lens, kv_cache=want)
    assert bad == 0
    assert_close_attn(out.cpu().numpy(), ro, "decode after write")
    assert_lse_close(lse.cpu().numpy(), rl, "decode after write lse")


def test_kv_write_skips_bad_tokens_and_takes_request_ids(tts):
    inp = W.sparse_decode_inputs(kv_lens=(100, 200), seed=65)
    ps = inp.kv_cache.shape[1]
    cache = dev(inp.kv_cache).clone()
    rows = torch.randn(5, inp.kv_cache.shape[2], generator=torch.Generator().manual_seed(66))
    rows = rows.to(torch.bfloat16)
    req = torch.tensor([1, 0, 7, 0, 1], dtype=torch.int32)       # request 7 does not exist
    pos = torch.tensor([5, 3, 0, -1, 10 ** 6], dtype=torch.int32)  # -1, far past the table
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.paged_kv_write(cache, dev(inp.page_tables), dev(rows), dev(pos), req_ids=dev(req),
                       status=st)
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    want = inp.kv_cache.clone()
    want[inp.page_tables[1, 5 // ps], 5 % ps] = rows[0]
    want[inp.page_tables[0, 3 // ps], 3 % ps] = rows[1]
    assert torch.equal(cache.cpu(), want)
