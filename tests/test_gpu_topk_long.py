"""GPU parity for tts_topk_select_long (rows split over many CTAs): indices bit-exact
against the float64 oracle's stable descending selection, on rows from just above one
chunk to 2^18 values, with ties across chunk borders, signed zeros, infinities, short
and invalid windows."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts():
    import tiled_top_sparse_gb300 as m
    m.lib()
    return m


def run(tts, inp: W.TopkInputs, status=None):
    dev = torch.device("cuda")
    return tts.topk_select_long(inp.logits.to(dev), inp.row_starts.to(dev),
                                inp.row_lens.to(dev), inp.k, status=status)


def oracle_idx(inp):
    return oracle.topk(inp.logits.numpy(), inp.row_starts.numpy(), inp.row_lens.numpy(), inp.k)


@pytest.mark.parametrize("rows,cols,k", [(4, 16385, 2048), (3, 50000, 4096), (2, 262144, 2048),
                                         (5, 40000, 1), (3, 70001, 7)])
def test_random_rows_bit_exact(tts, rows, cols, k):
    # bf16-grid normal values: plenty of equal values around the k-th
    inp = W.topk_inputs(rows=rows, cols=cols, k=k, seed=cols + k, causal=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = run(tts, inp, st)
    tts.check_status(st)
    ref, bad = oracle_idx(inp)
    assert bad == 0
    assert np.array_equal(a.cpu().numpy(), ref)
    assert torch.equal(a, run(tts, inp))


def test_ties_across_chunks_signed_zero_and_infinities(tts):
    g = torch.Generator().manual_seed(11)
    rows, cols = 6, 100000
    x = torch.randint(-2, 3, (rows, cols), generator=g).float()
    zero = x == 0
    x[zero] = torch.where(torch.rand(int(zero.sum()), generator=g) < 0.5, torch.tensor(0.0),
                          torch.tensor(-0.0))
    x[1] = 1.0                                   # one value everywhere
    x[2, ::3] = float("inf")                     # more +inf than k
    x[3] = float("-inf")
    x[3, 99990:] = 0.5                           # the only finite values at the very end
    x[4, :50000] = -1.0                          # ties of the k-th value in the last chunks
    x[4, 50000:] = -1.0
    x[4, 77777] = 3.0
    inp = W.TopkInputs(x, torch.zeros(rows, dtype=torch.int32),
                       torch.full((rows,), cols, dtype=torch.int32), 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)


def test_windows_short_empty_offset_and_invalid(tts):
    g = torch.Generator().manual_seed(12)
    rows, cols = 7, 70000
    x = torch.randn(rows, cols, generator=g).to(torch.bfloat16).float()
    starts = torch.tensor([0, 100, 33000, 0, 5, 60000, 69999], dtype=torch.int32)
    lens = torch.tensor([70000, 2000, 16384, 0, 40000, 10000, 1], dtype=torch.int32)
    inp = W.TopkInputs(x, starts, lens, 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)
    # a window past the row's end: that row is all -1 and the status reports it
    bad = W.TopkInputs(x[:2].contiguous(), torch.tensor([0, 69000], dtype=torch.int32),
                       torch.tensor([100, 2000], dtype=torch.int32), 16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(tts, bad, st).cpu().numpy()
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    assert (out[1] == -1).all()
    ref_bad, nbad = oracle_idx(bad)
    assert nbad == 1 and np.array_equal(out, ref_bad)


def test_matches_the_one_cta_kernel(tts):
    # below the short kernel's limit both paths must give the same bits
    inp = W.topk_inputs(rows=9, cols=16384, k=2048, seed=5, causal=True)
    dev = torch.device("cuda")
    a = tts.topk_select(inp.logits.to(dev), inp.row_starts.to(dev), inp.row_lens.to(dev), inp.k)
    assert torch.equal(a, run(tts, inp))


def test_picks_clustered_along_the_row(tts):
    # The threshold comes from a sample spread evenly over the window; rows whose large
    # values sit together (in the first 8192 values, in the first 16384, in the later
    # half) or rise steadily along the row make the sample's view of the row uneven:
    # the selection must still be exact.
    g = torch.Generator().manual_seed(23)
    rows, cols = 4, 262144
    x = torch.randn(rows, cols, generator=g).to(torch.bfloat16).float()
    x[0, :8192] += 10.0                                  # every pick in the first round
    x[1, :16384] += 10.0                                 # first chunk, beyond its first round
    x[2, cols // 2:] += 5.0                              # the later half dominates
    x[3] = torch.linspace(-3.0, 3.0, cols).to(torch.bfloat16).float() + 0.01 * x[3]
    inp = W.TopkInputs(x, torch.zeros(rows, dtype=torch.int32),
                       torch.full((rows,), cols, dtype=torch.int32), 2048)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run(tts, inp, st)
    tts.check_status(st)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_finish_radix_fallback_for_crowded_buckets(tts):
    # 600 copies of one large value among the picks: a bucket of more than 512 members
    # sends the finish to its radix select and sort. Row 0 lies on the bf16 grid (the
    # finish splits a value's ties by position: the copies sit in one sixteenth of the
    # row); row 1 holds plain fp32 values (no split: the copies are spread over the row).
    g = torch.Generator().manual_seed(29)
    cols = 262144
    x = torch.randn(2, cols, generator=g)
    x[0] = x[0].to(torch.bfloat16).float()
    x[0, 100:700] = 4.0
    x[1, torch.randperm(cols, generator=g)[:600]] = 4.0
    inp = W.TopkInputs(x, torch.zeros(2, dtype=torch.int32),
                       torch.full((2,), cols, dtype=torch.int32), 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)
