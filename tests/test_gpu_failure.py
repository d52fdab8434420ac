"""Failure detection without a GPU fault: a bounded device wait that runs out must set
the timeout bit and return, and the context must stay usable afterwards."""
import time

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import tiled_top_sparse_gb300 as tts
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    tts.debug_wait_timeout(st)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(st.item()) & tts.TTS_DEV_TIMEOUT
    assert 0.5 < dt < 30.0
    with pytest.raises(tts.TTSError) as ei:
        tts.check_status(st)
    assert ei.value.code == tts.TTS_ERR_DEVICE_TIMEOUT
    # the context still works: a real call succeeds right after
    ti = W.topk_inputs(rows=4, cols=300, k=64, seed=70)
    idx = tts.topk_select(ti.logits.cuda(), ti.row_starts.cuda(), ti.row_lens.cuda(), 64)
    assert idx.shape == (4, 64) and bool((idx[:, 0] >= 0).all())


def test_status_argument_required():
    import tiled_top_sparse_gb300 as tts
    assert tts.lib().tts_debug_wait_timeout(None, None) == tts.TTS_ERR_INVALID_ARG
