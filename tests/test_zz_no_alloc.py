"""The allocation-free LM-head argmax (dflash_lm_head_argmax_noalloc).

Some callers cannot give the library device memory when they call it — a
serving loop whose memory is entirely reserved up front by its own pool, or
a latency-critical path that must not call cudaMalloc.  The allocation-free
entry point serves them from a fixed internal scratch array.  This file is
collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def model(dfl):
    from synth.gpu import draft_model
    w = synth.with_(synth.WORKLOADS["tiny_f32"], dtype="bf16")
    weights = synth.draft_weights(w.draft, w.dtype, w.seed, device="cuda")
    m = draft_model(w.draft, w.dtype, weights, max_pos=64)
    yield w, m, weights
    m.close()


def test_noalloc_matches_workspace_entry_point_twice(dfl, model):
    w, m, weights = model
    s = w.draft
    rows = 15
    x = torch.randn(rows, s.D, generator=torch.Generator().manual_seed(5)).cuda()
    ids_ref = torch.empty(rows, dtype=torch.int32, device="cuda")
    gap_ref = torch.empty(rows, device="cuda")
    dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids_ref, gap_ref,
                              m.workspace(rows))
    assert dfl.dflash_get_status(m.handle) == 0
    for _ in range(2):                         # the shared scratch keeps the last call's data
        ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        gap = torch.full((rows,), -1.0, device="cuda")
        dfl.dflash_lm_head_argmax_noalloc(m.handle, x, rows, weights["g_f"], ids, gap)
        assert dfl.dflash_get_status(m.handle) == 0
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
        np.testing.assert_allclose(gap.cpu().numpy(), gap_ref.cpu().numpy(), atol=2e-2, rtol=0)


def test_noalloc_rejects_sizes_beyond_its_limit(dfl, model):
    w, m, weights = model
    x = torch.zeros(17, w.draft.D, device="cuda")
    ids = torch.empty(17, dtype=torch.int32, device="cuda")
    with pytest.raises(dfl.DFlashError) as e:
        dfl.dflash_lm_head_argmax_noalloc(m.handle, x, 17, weights["g_f"], ids, None)
    assert e.value.code == 10
