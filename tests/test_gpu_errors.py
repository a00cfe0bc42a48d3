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


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_runs_out_and_the_handle_recovers(dfl, tiny, which):
    """A wait that nothing completes (0: an mbarrier no thread arrives at,
    1: a device counter nothing raises) gives up after its limit and records
    DFLASH_ERR_DEVICE_TIMEOUT; the next normal call on the same handle
    succeeds and matches the oracle."""
    import time

    import oracle as O
    from helpers import id_parity, to_np
    from synth.gpu import kv_cache
    w, m = tiny
    s = w.draft
    t0 = time.perf_counter()
    dfl.dflash_selftest_wait(m.handle, which, 200_000)       # 200 us
    assert dfl.dflash_get_status(m.handle) == 7             # DFLASH_ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert dfl.dflash_get_status(m.handle) == 0             # cleared
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    K, V = synth.random_kv_cache(1, s.G, 30, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype, w.seed,
                                 device="cuda")
    kv = kv_cache(s, 1, 30, w.dtype, k=K, v=V)
    kv.len.fill_(30)
    anchors = synth.anchors(1, s.V, s.mask_id, w.seed)
    ids = torch.empty(1, w.B, dtype=torch.int32, device="cuda")
    gap = torch.empty(1, w.B - 1, device="cuda")
    dfl.dflash_draft_block(m.handle, torch.from_numpy(anchors).cuda(), 1, w.B, kv.struct, ids, gap,
                           None, m.workspace(w.B, max_batch=1, max_block=w.B))
    assert dfl.dflash_get_status(m.handle) == 0
    W = to_np(weights)
    cK = [[K[l][0, :, :30].float().cpu().numpy().transpose(1, 0, 2)] for l in range(s.n_layers)]
    cV = [[V[l][0, :, :30].float().cpu().numpy().transpose(1, 0, 2)] for l in range(s.n_layers)]
    oids, ogap = O.draft_block(s, W, cK, cV, anchors, w.B, O.f32)
    assert id_parity(ids.cpu().numpy(), oids, ogap)[0] == 0


def test_selftest_wait_rejects_bad_arguments(dfl, tiny):
    _, m = tiny
    for which, limit in [(2, 10_000), (0, 10), (1, 2_000_000_000)]:
        with pytest.raises(dfl.DFlashError) as e:
            dfl.dflash_selftest_wait(m.handle, which, limit)
        assert e.value.code == 1


@pytest.mark.parametrize("case", ["f32", "bf16_streaming", "bf16_tensor_core"])
def test_argmax_row_without_maximum(dfl, case):
    """A residual row of NaN makes every logit of its row NaN: its id is 0
    (not an index past the vocabulary) with gap 0 and the status reports
    DFLASH_ERR_DEVICE_BOUNDS; the other rows keep the ids they get without
    it (f32 SIMT path, bf16 streaming LM head at 15 rows, bf16 tensor-core
    LM head at 130 rows)."""
    from synth.gpu import draft_model
    from test_gpu_draft import SMALL_BF16
    w = synth.WORKLOADS["tiny_f32"] if case == "f32" else SMALL_BF16
    s = w.draft
    rows = 130 if case == "bf16_tensor_core" else 15
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    m = draft_model(s, w.dtype, weights, max_pos=64)
    x = torch.randn(rows, s.D, generator=torch.Generator().manual_seed(17)).cuda()
    ws = m.workspace(rows)

    def run(xx):
        ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        gap = torch.full((rows,), -1.0, device="cuda")
        dfl.dflash_lm_head_argmax(m.handle, xx, rows, weights["g_f"], ids, gap, ws)
        return ids.cpu().numpy(), gap.cpu().numpy(), dfl.dflash_get_status(m.handle)

    ref_ids, ref_gap, st = run(x)
    assert st == 0
    x[3] = float("nan")
    ids, gap, st = run(x)
    assert st == 8                                          # DFLASH_ERR_DEVICE_BOUNDS
    assert ids[3] == 0 and gap[3] == 0.0
    keep = np.arange(rows) != 3
    np.testing.assert_array_equal(ids[keep], ref_ids[keep])
    np.testing.assert_array_equal(gap[keep], ref_gap[keep])
    m.close()


def test_argmax_row_without_maximum_in_the_persistent_block(dfl):
    """The persistent draft-block kernel: a NaN anchor embedding makes its
    sequence's rows NaN; their ids are 0 and the status reports
    DFLASH_ERR_DEVICE_BOUNDS, while the other sequence's ids are unchanged."""
    from synth.gpu import draft_model, kv_cache
    from test_gpu_draft import SMALL_BF16
    w, s = SMALL_BF16, SMALL_BF16.draft
    B = 8
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    K, V = synth.random_kv_cache(2, s.G, 40, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype, w.seed,
                                 device="cuda")
    kv = kv_cache(s, 2, 40, w.dtype, k=K, v=V)
    anchors = torch.tensor([5, 9], dtype=torch.int32, device="cuda")

    def run(model):
        kv.len.fill_(40)
        ids = torch.full((2, B), -1, dtype=torch.int32, device="cuda")
        model_ws = model.workspace(2 * B, max_batch=2, max_block=B)
        dfl.dflash_draft_block(model.handle, anchors, 2, B, kv.struct, ids, None, None, model_ws)
        return ids.cpu().numpy(), dfl.dflash_get_status(model.handle)

    m = draft_model(s, w.dtype, weights, max_pos=64)
    ref, st = run(m)
    assert st == 0
    m.close()
    weights["embed"][5] = float("nan")
    m = draft_model(s, w.dtype, weights, max_pos=64)
    ids, st = run(m)
    m.close()
    assert st == 8
    np.testing.assert_array_equal(ids[0], [5] + [0] * (B - 1))
    np.testing.assert_array_equal(ids[1], ref[1])
