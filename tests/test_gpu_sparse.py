"""GPU parity for tts_sparse_attn_paged against the float64 oracle, plus bitwise
invariance under permutations of every query's index list."""
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


def to_dev(inp: W.SparseInputs):
    dev = torch.device("cuda")
    return (inp.q.to(dev), inp.kv_cache.to(dev), inp.page_table.to(dev), inp.idx.to(dev))


def run(tts, inp, idx=None, status=None):
    q, kv, pt, ix = to_dev(inp)
    if idx is not None:
        ix = idx.to("cuda")
    return tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, dv=inp.dv, status=status)


def ref(inp, idx=None, rows=None):
    q = inp.q.float().numpy()
    ix = (inp.idx if idx is None else idx)
    if rows is not None:
        q = q[rows]
        ix = ix[rows]
    return oracle.sparse_paged(q, inp.kv_cache.float().numpy(), inp.page_table.numpy(),
                               ix.numpy(), inp.kv_len, inp.dv, inp.scale)


@pytest.mark.parametrize("nq,kv_len,topk", [(4, 300, 200), (3, 5000, 2048), (5, 64, 64),
                                            (2, 100, 17), (6, 2590, 1000)])
def test_parity_small(tts, nq, kv_len, topk):
    inp = W.sparse_inputs(nq=nq, kv_len=kv_len, topk=topk, seed=nq * 1000 + topk)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, status=st)
    tts.check_status(st)
    ro, rl, bad = ref(inp)
    assert bad == 0
    assert_close_attn(out.cpu().numpy(), ro, f"sparse nq={nq} topk={topk}")
    assert_lse_close(lse.cpu().numpy(), rl, "sparse lse")


@pytest.mark.parametrize("nq,kv_len,page_size,topk", [
    (2, 20000, 64, 2048),   # kv_len above the counting-sort range: bitonic sort
    (2, 16000, 1, 2048),    # counting sort, page table too large to copy into the scratch
    (2, 20000, 1, 1500),    # bitonic sort, page table read from global memory
    (3, 3000, 1, 2048),     # one-row pages, page table copied into the scratch
])
def test_parity_sort_and_page_table_paths(tts, nq, kv_len, page_size, topk):
    inp = W.sparse_inputs(nq=nq, kv_len=kv_len, page_size=page_size, topk=topk,
                          seed=kv_len + page_size + topk)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, status=st)
    tts.check_status(st)
    ro, rl, bad = ref(inp)
    assert bad == 0
    assert_close_attn(out.cpu().numpy(), ro, f"sparse kv_len={kv_len} page={page_size}")
    assert_lse_close(lse.cpu().numpy(), rl, "sparse lse")
    perm = W.permute_rows(inp.idx, seed=kv_len)
    out_p, lse_p = run(tts, inp, idx=perm)
    assert torch.equal(out_p, out) and torch.equal(lse_p, lse)


@pytest.mark.parametrize("nq", [5, 30, 76, 160])
def test_split_last_wave_matches_unsplit_and_oracle(tts, nq):
    # nq = 5 / 30: every unit split (4 / 2 parts); 76: whole waves only (no split on a
    # 152-SM part); 160: a partial wave of split units after whole ones.
    inp = W.sparse_inputs(nq=nq, kv_len=2590, topk=2048, seed=70 + nq)
    q, kv, pt, ix = to_dev(inp)
    ws = torch.empty(max(16, tts.sparse_workspace_bytes(nq)), dtype=torch.uint8, device="cuda")
    a_out, a_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, workspace=ws)
    b_out, b_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, workspace=ws)
    assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)  # run to run
    perm = W.permute_rows(inp.idx, seed=nq).to("cuda")
    p_out, p_lse = tts.sparse_attn_paged(q, kv, pt, perm, inp.kv_len, inp.scale, workspace=ws)
    assert torch.equal(a_out, p_out) and torch.equal(a_lse, p_lse)  # order invariant
    u_out, u_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, split=False)
    rows = sorted({0, nq // 2, nq - 1})
    ro, rl, _ = ref(inp, rows=rows)
    for o, l, what in ((a_out, a_lse, "split"), (u_out, u_lse, "unsplit")):
        assert_close_attn(o[rows].cpu().numpy(), ro, f"sparse {what} nq={nq}")
        assert_lse_close(l[rows].cpu().numpy(), rl, f"sparse {what} lse")
    # The two schedules agree to rounding: each part rounds its P to bf16 relative to its
    # own reference maximum (relative step 2^-9), so outputs may differ by a few 2^-9 of
    # their scale; lse differs only by fp32 rounding of the merged sums.
    scale = u_out.abs().max().item()
    assert (a_out - u_out).abs().max().item() <= 2.0 ** -7 * scale
    assert (a_lse - u_lse).abs().max().item() < 1e-4


def test_empty_slots_duplicates_and_bad_entries(tts):
    inp = W.sparse_inputs(nq=4, kv_len=700, topk=130, seed=50)
    idx = inp.idx.clone()
    idx[0, 100:] = -1                 # short list
    idx[1, :] = -1                    # nothing valid -> out 0, lse -inf
    idx[2, 5:60] = idx[2, 0]          # duplicates count with multiplicity
    idx[3, 7] = 700                   # out of range -> skipped + flagged
    idx[3, 9] = -5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, idx=idx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    ro, rl, bad = ref(inp, idx=idx)
    assert bad == 2
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    assert_close_attn(out.cpu().numpy(), ro, "slots")
    assert_lse_close(lse.cpu().numpy(), rl, "slots lse")


def test_bad_page_table_entry_flagged(tts):
    inp = W.sparse_inputs(nq=2, kv_len=256, topk=64, seed=51)
    pt = inp.page_table.clone()
    pt[1] = 999  # logical page 1 (positions 64..127) maps outside the cache
    bad_inp = W.SparseInputs(inp.q, inp.kv_cache, pt, inp.idx, inp.kv_len, inp.dv, inp.scale)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, bad_inp, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    ro, rl, _ = ref(bad_inp)
    assert_close_attn(out.cpu().numpy(), ro, "bad page")


def test_full_config_permutation_invariance_and_parity(tts):
    inp = W.sparse_inputs()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run(tts, inp, status=st)
    out_again, lse_again = run(tts, inp, status=st)
    tts.check_status(st)
    assert torch.equal(out, out_again) and torch.equal(lse, lse_again)
    for s in W.PERM_SEEDS:
        o2, l2 = run(tts, inp, idx=W.permute_rows(inp.idx, s), status=st)
        assert torch.equal(o2, out) and torch.equal(l2, lse), f"permutation seed {s}"
    rows = np.array([0, 1, 161, 200, 321, 322] + list(range(7, 323, 29)))
    ro, rl, bad = ref(inp, rows=rows)
    assert bad == 0
    assert_close_attn(out[rows].cpu().numpy(), ro, "sparse full sampled")
    assert_lse_close(lse[rows].cpu().numpy(), rl, "sparse full lse")


def test_chained_topk_then_sparse(tts):
    # top-k over indexer logits feeds the sparse kernel (the attn1 chain of the V32 write-up)
    ti = W.topk_inputs(rows=16, cols=2590, k=2048, seed=52)
    si = W.sparse_inputs(nq=16, kv_len=2590, topk=2048, seed=53)
    dev = torch.device("cuda")
    gidx = tts.topk_select(ti.logits.to(dev), ti.row_starts.to(dev), ti.row_lens.to(dev), 2048)
    oidx, _ = oracle.topk(ti.logits.numpy(), ti.row_starts.numpy(), ti.row_lens.numpy(), 2048)
    assert np.array_equal(gidx.cpu().numpy(), oidx)
    out, lse = tts.sparse_attn_paged(si.q.to(dev), si.kv_cache.to(dev), si.page_table.to(dev),
                                     gidx, si.kv_len, si.scale)
    ro, rl, _ = oracle.sparse_paged(si.q.float().numpy(), si.kv_cache.float().numpy(),
                                    si.page_table.numpy(), oidx, si.kv_len, si.dv, si.scale)
    assert_close_attn(out.cpu().numpy(), ro, "chained")


@pytest.mark.parametrize("nq,kv_len,page_size,topk", [
    (76, 2590, 64, 2048),   # whole waves only on a 152-SM part: no split either way
    (3, 20000, 64, 2048),   # bitonic sort path
    (5, 300, 1, 200),       # one-row pages
])
def test_presorted_lists_match_in_kernel_sort(tts, nq, kv_len, page_size, topk):
    # With a workspace, a first launch writes every query's canonical list and the
    # attention CTAs read it; without one they sort in the kernel. Same lists, so the
    # outputs are bitwise equal whenever neither call splits its last wave.
    inp = W.sparse_inputs(nq=nq, kv_len=kv_len, page_size=page_size, topk=topk,
                          seed=nq + kv_len + topk)
    idx = inp.idx.clone()
    idx[0, :7] = -1            # empty slots and a duplicate survive canonicalisation
    idx[-1, 5] = idx[-1, 6]
    q, kv, pt, _ = to_dev(inp)
    ix = idx.to("cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if torch.cuda.get_device_properties(0).multi_processor_count == 152 and nq == 76:
        ws = torch.empty(tts.sparse_workspace_bytes(nq), dtype=torch.uint8, device="cuda")
        a_out, a_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, workspace=ws,
                                             status=st)
        b_out, b_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, split=False,
                                             status=st)
        assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)
    a_out, a_lse = tts.sparse_attn_paged(q, kv, pt, ix, inp.kv_len, inp.scale, status=st)
    tts.check_status(st)
    ro, rl, bad = ref(inp, idx=idx)
    assert bad == 0
    assert_close_attn(a_out.cpu().numpy(), ro, f"presorted nq={nq} kv_len={kv_len}")
    assert_lse_close(a_lse.cpu().numpy(), rl, "presorted lse")
    perm = W.permute_rows(idx, seed=7).to("cuda")
    p_out, p_lse = tts.sparse_attn_paged(q, kv, pt, perm, inp.kv_len, inp.scale)
    assert torch.equal(p_out, a_out) and torch.equal(p_lse, a_lse)
