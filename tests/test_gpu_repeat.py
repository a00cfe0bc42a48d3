"""Repeated identical launches give bit-identical results.

Every kernel here is deterministic by construction: work splits depend only
on shapes, and partial sums are added in a fixed order.  So any difference
between identical launches is a race.  With two co-resident CTAs per SM, the
streaming kernel once returned one consumer warp's 32 output columns wrong
in a few of 300 such launches.  It runs one CTA per SM since then. These
tests keep watching it, the persistent draft-block kernel (two CTAs per SM)
and the tensor-core projection, at the Qwen3-8B shape, and the tcgen05 split
attention at the 35B-A3B shape."""
import dataclasses

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

QWEN3 = synth.WORKLOADS["qwen3_8b_b1"]


@pytest.fixture(scope="module")
def one_layer_model(dfl):
    from synth.gpu import draft_model
    w = synth.with_(QWEN3, draft=dataclasses.replace(QWEN3.draft, n_layers=1))
    weights = synth.draft_weights(w.draft, w.dtype, w.seed, device="cuda")
    m = draft_model(w.draft, w.dtype, weights, max_pos=4096)
    yield w, m, weights
    m.close()


def _repeat(fn, n):
    """Run fn n times; return how many results differ from the first (fn
    returns a tuple of device tensors, compared on the device)."""
    first = [t.clone() for t in fn()]
    bad = 0
    for _ in range(n - 1):
        out = fn()
        if not all(torch.equal(a, b) for a, b in zip(first, out)):
            bad += 1
    return bad


@pytest.mark.parametrize("rows", [30, 480])
def test_lm_head_logits_repeat(dfl, one_layer_model, rows):
    """30 rows: the streaming kernel (the configuration that showed the
    race); 480 rows: the tensor-core kernel."""
    w, m, weights = one_layer_model
    s = w.draft
    x = torch.randn(rows, s.D, generator=torch.Generator().manual_seed(40)).cuda()
    logits = torch.empty(rows, s.V, device="cuda")
    ws = m.workspace(rows)

    def call():
        dfl.dflash_lm_head_logits(m.handle, x, rows, weights["g_f"], logits, ws)
        return (logits,)

    n = 300 if rows == 30 else 100
    bad = _repeat(call, n)
    assert dfl.dflash_get_status(m.handle) == 0
    print(f"LM-head logits, {rows} rows: {bad} of {n - 1} repeats differ")
    assert bad == 0


def test_lm_head_argmax_repeat(dfl, one_layer_model):
    """The streaming LM head with its argmax epilogue and grid barrier."""
    w, m, weights = one_layer_model
    rows = 15
    x = torch.randn(rows, w.draft.D, generator=torch.Generator().manual_seed(41)).cuda()
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    gap = torch.empty(rows, device="cuda")
    ws = m.workspace(rows)

    def call():
        dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids, gap, ws)
        return ids, gap

    bad = _repeat(call, 300)
    assert dfl.dflash_get_status(m.handle) == 0
    assert bad == 0


def test_persistent_draft_block_repeat(dfl):
    """The whole Qwen3-8B-shaped draft block (five layers, L = 2048, B = 16)
    in the persistent kernel, 300 times."""
    from synth.gpu import draft_model, kv_cache
    w, s = QWEN3, QWEN3.draft
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    K, V = synth.random_kv_cache(1, s.G, w.ctx_len, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device="cuda")
    kv = kv_cache(s, 1, w.ctx_len, w.dtype, k=K, v=V)
    kv.len.fill_(w.ctx_len - w.B)
    m = draft_model(s, w.dtype, weights, max_pos=w.ctx_len + 64)
    anchors = torch.from_numpy(synth.anchors(1, s.V, s.mask_id, w.seed)).cuda()
    ids = torch.empty(1, w.B, dtype=torch.int32, device="cuda")
    gap = torch.empty(1, w.B - 1, device="cuda")
    hid = torch.empty(w.B, s.D, device="cuda")
    ws = m.workspace(w.B, max_batch=1, max_block=w.B)

    def call():
        dfl.dflash_draft_block(m.handle, anchors, 1, w.B, kv.struct, ids, gap, hid, ws)
        return ids, gap, hid

    bad = _repeat(call, 300)
    assert dfl.dflash_get_status(m.handle) == 0
    m.close()
    print(f"persistent draft block: {bad} of 299 repeats differ")
    assert bad == 0


@pytest.mark.parametrize("B", [8, 16])
def test_tcgen05_attention_block_repeat(dfl, B):
    """A two-layer 35B-A3B-shaped draft block at batch 4 with ragged contexts
    (32 or 64 rows: the streaming projections and the tcgen05 split
    attention with its TMEM buffers and stage barriers), 200 times."""
    from synth.gpu import draft_model, kv_cache
    w = synth.WORKLOADS["qwen35_a3b_32k"]
    s = dataclasses.replace(w.draft, n_layers=2)
    lens = [5000, 2048, 777, 3333]
    cap = max(lens) + 8
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    K, V = synth.random_kv_cache(4, s.G, cap, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device="cuda")
    kv = kv_cache(s, 4, cap, w.dtype, k=K, v=V)
    kv.len.copy_(torch.tensor(lens, dtype=torch.int32))
    m = draft_model(s, w.dtype, weights, max_pos=cap + B + 8)
    anchors = torch.from_numpy(synth.anchors(4, s.V, s.mask_id, w.seed)).cuda()
    ids = torch.empty(4, B, dtype=torch.int32, device="cuda")
    gap = torch.empty(4, B - 1, device="cuda")
    hid = torch.empty(4 * B, s.D, device="cuda")
    ws = m.workspace(4 * B, max_batch=4, max_block=B)

    def call():
        dfl.dflash_draft_block(m.handle, anchors, 4, B, kv.struct, ids, gap, hid, ws)
        return ids, gap, hid

    bad = _repeat(call, 200)
    assert dfl.dflash_get_status(m.handle) == 0
    m.close()
    print(f"tcgen05 attention block B={B}: {bad} of 199 repeats differ")
    assert bad == 0
