"""GPU parity for tts_topk_select: indices bit-exact against the float64 oracle."""
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
    return tts.topk_select(inp.logits.to(dev), inp.row_starts.to(dev), inp.row_lens.to(dev),
                           inp.k, status=status)


def oracle_idx(inp):
    idx, bad = oracle.topk(inp.logits.numpy(), inp.row_starts.numpy(), inp.row_lens.numpy(),
                           inp.k)
    return idx, bad


def test_full_config_bit_exact_and_repeatable(tts):
    inp = W.topk_inputs()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = run(tts, inp, st)
    b = run(tts, inp, st)
    ref, bad = oracle_idx(inp)
    assert bad == 0
    tts.check_status(st)
    assert np.array_equal(a.cpu().numpy(), ref)
    assert torch.equal(a, b)


@pytest.mark.parametrize("rows,cols,k", [(7, 100, 16), (33, 5000, 4096), (5, 16384, 3000),
                                         (40, 700, 1), (3, 2049, 2048)])
def test_shapes_with_ties(tts, rows, cols, k):
    inp = W.topk_inputs(rows=rows, cols=cols, k=k, seed=rows * 7 + k, causal=True)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)


def test_heavy_ties_and_signed_zero(tts):
    g = torch.Generator().manual_seed(9)
    x = torch.randint(-2, 3, (16, 3000), generator=g).float()
    x[x == 0] = torch.where(torch.rand(int((x == 0).sum()), generator=g) < 0.5,
                            torch.tensor(0.0), torch.tensor(-0.0))
    inp = W.TopkInputs(x, torch.zeros(16, dtype=torch.int32),
                       torch.full((16,), 3000, dtype=torch.int32), 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)


@pytest.mark.parametrize("pattern", ["constant", "signed_zeros", "low_byte", "full_fp32"])
def test_digit_patterns(tts, pattern):
    # The radix passes skip digits that are equal across a window; these rows make 4, 4,
    # 3 and no passes skippable.
    g = torch.Generator().manual_seed(31)
    rows, cols = 12, 2590
    if pattern == "constant":
        x = torch.full((rows, cols), 0.375)
    elif pattern == "signed_zeros":
        x = torch.where(torch.rand(rows, cols, generator=g) < 0.5, torch.tensor(0.0),
                        torch.tensor(-0.0))
    elif pattern == "low_byte":  # 1.0 plus 0..255 units in the last place
        bits = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32) + 0x3F800000
        x = bits.view(torch.float32)
    else:
        x = torch.randn(rows, cols, generator=g)
    inp = W.TopkInputs(x, torch.zeros(rows, dtype=torch.int32),
                       torch.full((rows,), cols, dtype=torch.int32), 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)


def test_short_rows_offsets_and_bad_windows(tts):
    g = torch.Generator().manual_seed(10)
    x = torch.randn(6, 3000, generator=g).to(torch.bfloat16).float()
    starts = torch.tensor([0, 100, 2999, 5, -1, 10], dtype=torch.int32)
    lens = torch.tensor([0, 50, 1, 2990, 10, 2995], dtype=torch.int32)  # rows 4, 5 invalid
    inp = W.TopkInputs(x, starts, lens, 2048)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run(tts, inp, st).cpu().numpy()
    ref, bad = oracle_idx(inp)
    assert bad == 2
    assert np.array_equal(got, ref)
    assert int(st.item()) & tts.TTS_DEV_INDEX_RANGE
    with pytest.raises(tts.TTSError):
        tts.check_status(st)


def test_output_canaries_untouched(tts):
    inp = W.topk_inputs(rows=20, cols=2590, k=2048, seed=11)
    dev = torch.device("cuda")
    buf = torch.full((20 * 2048 + 2 * 4096,), -12345, dtype=torch.int32, device=dev)
    idx = buf[4096:4096 + 20 * 2048].view(20, 2048)
    tts.topk_select(inp.logits.to(dev), inp.row_starts.to(dev), inp.row_lens.to(dev), 2048, idx=idx)
    torch.cuda.synchronize()
    assert bool((buf[:4096] == -12345).all()) and bool((buf[-4096:] == -12345).all())
    ref, _ = oracle_idx(inp)
    assert np.array_equal(idx.cpu().numpy(), ref)


def test_bucket_limit_and_mixed_values(tts):
    # Windows of up to 4096 values are ranked inside value buckets unless one bucket holds
    # more than 128 values, when the whole window is radix-sorted instead; both must give
    # the oracle's indices. Rows: 128 and 129 copies of one value among distinct ones
    # (just inside / just past the limit), infinities and signed zeros among normals,
    # one outlier that stretches the bucket range, all values negative, plain fp32
    # values (not on the bf16 grid), and a 4096-value window.
    g = torch.Generator().manual_seed(11)
    rows = []
    for copies in (128, 129):
        x = torch.randn(3000, generator=g)
        x[torch.randperm(3000, generator=g)[:copies]] = 4.5  # a value no normal draw shares a bucket with
        rows.append(x)
    x = torch.randn(3000, generator=g)
    x[[3, 50, 900]] = float("inf")
    x[[4, 51]] = float("-inf")
    x[[5, 6, 7]] = 0.0
    x[[8, 9]] = -0.0
    rows.append(x)
    x = torch.randn(3000, generator=g)
    x[17] = 3e38
    rows.append(x)
    rows.append(-torch.randn(3000, generator=g).abs())
    rows.append(torch.randn(3000, generator=g) * 1e-3 + 7.0)
    logits = torch.stack(rows)
    n = logits.shape[0]
    inp = W.TopkInputs(logits, torch.zeros(n, dtype=torch.int32),
                       torch.full((n,), 3000, dtype=torch.int32), 2048)
    ref, _ = oracle_idx(inp)
    assert np.array_equal(run(tts, inp).cpu().numpy(), ref)
    full = W.TopkInputs(torch.randn(2, 4096, generator=g), torch.zeros(2, dtype=torch.int32),
                        torch.full((2,), 4096, dtype=torch.int32), 4000)
    ref, _ = oracle_idx(full)
    assert np.array_equal(run(tts, full).cpu().numpy(), ref)


@pytest.mark.parametrize("cols", [3071, 3072, 3073])
def test_per_thread_shape_boundary(tts, cols):
    # Rows of at most 3072 values run with six values per thread (four CTAs per SM),
    # longer ones with eight; either side of the boundary, whole and partial windows of
    # bf16-grid values (buckets of ties), a row of two values only (the radix fallback)
    # and a row that ends exactly at the last thread's last value.
    g = torch.Generator().manual_seed(cols)
    x = torch.randn(6, cols, generator=g).to(torch.bfloat16).float()
    x[1] = torch.where(torch.rand(cols, generator=g) < 0.5, torch.tensor(1.0), torch.tensor(-2.5))
    starts = torch.tensor([0, 0, 1, cols - 1, 0, 7], dtype=torch.int32)
    lens = torch.tensor([cols, cols, cols - 1, 1, 2048, cols - 7], dtype=torch.int32)
    for k in (1, 2048, 3072):
        inp = W.TopkInputs(x, starts, lens, k)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = run(tts, inp, st).cpu().numpy()
        ref, bad = oracle_idx(inp)
        assert bad == 0
        tts.check_status(st)
        assert np.array_equal(got, ref), f"cols {cols} k {k}"
