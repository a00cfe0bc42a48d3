"""Error paths: host-detected argument errors and device-detected range
errors.  Every case is rejected before launch or caught by the kernels' own
range checks (the offending writes are skipped); none faults the GPU."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(dfl):
    from synth.gpu import draft_model
    w = synth.WORKLOADS["tiny_f32"]
    weights = synth.draft_weights(w.draft, w.dtype, w.seed, device="cuda")
    m = draft_model(w.draft, w.dtype, weights, max_pos=40)
    yield w, m
    m.close()


def test_capacity_overflow_is_reported(dfl, tiny):
    from synth.gpu import kv_cache
    w, m = tiny
    s = w.draft
    kv = kv_cache(s, 1, 16, w.dtype)
    kv.len.fill_(10)
    H_t = torch.randn(8, s.D, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = torch.tensor([8], dtype=torch.int32, device="cuda")
    dfl.dflash_inject_kv(m.handle, H_t, 8, z, n, 1, kv.struct, m.workspace(8))
    assert dfl.dflash_get_status(m.handle) == dfl.DFlashError(4, "").code
    assert int(kv.len[0]) == 10                   # not advanced
    assert dfl.dflash_get_status(m.handle) == 0   # status was cleared


def test_anchor_out_of_range_is_reported(dfl, tiny):
    from synth.gpu import kv_cache
    w, m = tiny
    kv = kv_cache(w.draft, 1, 16, w.dtype)
    a = torch.tensor([w.draft.V + 5], dtype=torch.int32, device="cuda")
    ids = torch.empty(1, w.B, dtype=torch.int32, device="cuda")
    dfl.dflash_draft_block(m.handle, a, 1, w.B, kv.struct, ids, None, None, m.workspace(w.B))
    assert dfl.dflash_get_status(m.handle) == 8


def test_position_beyond_rope_table_is_reported(dfl, tiny):
    from synth.gpu import kv_cache
    w, m = tiny                                   # max_pos = 40
    kv = kv_cache(w.draft, 1, 64, w.dtype)
    kv.len.fill_(36)                              # block positions 36 .. 43
    a = torch.tensor([5], dtype=torch.int32, device="cuda")
    ids = torch.empty(1, w.B, dtype=torch.int32, device="cuda")
    dfl.dflash_draft_block(m.handle, a, 1, w.B, kv.struct, ids, None, None, m.workspace(w.B))
    assert dfl.dflash_get_status(m.handle) == 8


def test_workspace_and_alignment_errors(dfl, tiny):
    w, m = tiny
    s = w.draft
    hs = [torch.randn(4, s.D, device="cuda") for _ in range(s.n_pick)]
    out = torch.empty(4, s.D, device="cuda")
    with pytest.raises(dfl.DFlashError) as e:
        dfl.dflash_fuse_context(m.handle, hs, 4, out, torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 9
    ws = m.workspace(4)
    bad = [hs[0].data_ptr() + 4] + [h.data_ptr() for h in hs[1:]]
    with pytest.raises(dfl.DFlashError) as e:
        dfl.dflash_fuse_context(m.handle, bad, 4, out, ws)
    assert e.value.code == 3
    from synth.gpu import kv_cache
    kv = kv_cache(s, 1, 16, w.dtype)
    a = torch.zeros(2, dtype=torch.int32, device="cuda")
    ids = torch.empty(2, w.B, dtype=torch.int32, device="cuda")
    with pytest.raises(dfl.DFlashError) as e:       # batch larger than the cache holds
        dfl.dflash_draft_block(m.handle, a, 2, w.B, kv.struct, ids, None, None, ws)
    assert e.value.code == 1


def test_empty_inputs(dfl, tiny):
    from synth.gpu import kv_cache
    w, m = tiny
    s = w.draft
    kv = kv_cache(s, 2, 16, w.dtype)
    ws = m.workspace(8)
    dfl.dflash_fuse_context(m.handle, [torch.empty(0, s.D, device="cuda")] * s.n_pick, 0,
                            torch.empty(0, s.D, device="cuda"), ws)
    z = torch.zeros(2, dtype=torch.int32, device="cuda")
    dfl.dflash_inject_kv(m.handle, torch.empty(1, s.D, device="cuda"), 0, z, z, 2, kv.struct, ws)
    assert dfl.dflash_get_status(m.handle) == 0
    np.testing.assert_array_equal(kv.len.cpu().numpy(), [0, 0])
