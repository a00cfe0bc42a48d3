"""Losslessness pins of the oracle's greedy speculative loop.

The greedy DFlash loop must emit exactly the target's own greedy
autoregressive output (the verification rule makes the draft's quality
irrelevant to the output)."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import make_all_accept, tiny_e2e, to_np


def _weights(tshape, dshape, seed):
    TW = to_np(synth.target_weights(tshape, "f32", seed))
    DW = to_np(synth.draft_weights(dshape, "f32", seed + 1,
                                   shared={"embed": None, "lm_head": None}))
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    return TW, DW


@pytest.mark.parametrize("B", [4, 6])
def test_speculative_equals_autoregressive(B):
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 50 + B)
    prompt = synth.random_ids(12, tshape.V, seed=3).tolist()
    n_new = 20
    ar = O.ar_generate(tshape, TW, prompt, n_new)
    spec, taus = O.speculative_generate(tshape, TW, dshape, DW, prompt, n_new, B)
    np.testing.assert_array_equal(spec, ar)
    assert all(1 <= t <= B for t in taus)
    assert sum(taus) + 1 >= n_new


def test_speculative_all_accepted_blocks():
    """Every block fully accepted (tau = B): the crop/append bookkeeping of a
    long accepted prefix still reproduces the autoregressive output."""
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 77)
    c = 5
    TW, DW = make_all_accept(TW, DW, tshape, c)
    prompt = synth.random_ids(9, tshape.V, seed=4).tolist() + [c]
    B, n_new = 4, 17
    ar = O.ar_generate(tshape, TW, prompt, n_new)
    assert (ar == c).all()
    spec, taus = O.speculative_generate(tshape, TW, dshape, DW, prompt, n_new, B)
    np.testing.assert_array_equal(spec, ar)
    assert taus == [B] * len(taus)


def test_sampling_loop_low_temperature_is_the_greedy_loop():
    """T -> 0: every softmax is one-hot at the argmax, so the sampling loop
    draws the argmax drafts and verification reduces to the greedy rule:
    the same tokens and taus as the greedy loop, whatever the uniforms."""
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 60)
    prompt = synth.random_ids(11, tshape.V, seed=6).tolist()
    B, n_new = 4, 16
    greedy, gt = O.speculative_generate(tshape, TW, dshape, DW, prompt, n_new, B)
    samp, st = O.speculative_sample_generate(tshape, TW, dshape, DW, prompt, n_new, B, 1e-6,
                                             synth.round_uniforms(1, B))
    np.testing.assert_array_equal(samp, greedy)
    assert st == gt


def test_sampling_loop_taus_in_range():
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 61)
    prompt = synth.random_ids(11, tshape.V, seed=7).tolist()
    B, n_new = 5, 16
    out, taus = O.speculative_sample_generate(tshape, TW, dshape, DW, prompt, n_new, B, 1.0,
                                              synth.round_uniforms(2, B))
    assert len(out) == n_new and all(0 <= t < tshape.V for t in out)
    assert all(1 <= t <= B for t in taus) and sum(taus) + 1 >= n_new


def test_speculative_equals_autoregressive_bf16_storage():
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 91)
    prompt = synth.random_ids(10, tshape.V, seed=5).tolist()
    ar = O.ar_generate(tshape, TW, prompt, 14, store=O.bf16)
    spec, _ = O.speculative_generate(tshape, TW, dshape, DW, prompt, 14, 5, store=O.bf16)
    np.testing.assert_array_equal(spec, ar)


def test_draft_block_anchor_column_and_shapes():
    w = synth.WORKLOADS["tiny_f32"]
    s = w.draft
    DW = to_np(synth.draft_weights(s, "f32", w.seed))
    L = 5
    rng = np.random.default_rng(0)
    cK = [[rng.standard_normal((L, s.G, s.d)) for _ in range(2)] for _ in range(s.n_layers)]
    cV = [[rng.standard_normal((L, s.G, s.d)) for _ in range(2)] for _ in range(s.n_layers)]
    ids, gaps = O.draft_block(s, DW, cK, cV, [3, 900], w.B)
    assert ids.shape == (2, w.B) and gaps.shape == (2, w.B - 1)
    assert list(ids[:, 0]) == [3, 900]
    assert (gaps >= 0).all() and ids.max() < s.V


def test_selected_loop_equals_autoregressive():
    """DFlash 2 candidate selection changes the drafts, not the output: the
    greedy loop with the selector still emits the target's own greedy
    autoregressive tokens (txtmix §13-§14 with the verification of §8)."""
    tshape, dshape = tiny_e2e()
    TW, DW = _weights(tshape, dshape, 91)
    sel = to_np(synth.selector_weights(dshape.D, dshape.V, "f32", 5, rank=32))
    sel["top_k"] = 8
    prompt = synth.random_ids(12, tshape.V, seed=4).tolist()
    n_new = 20
    ar = O.ar_generate(tshape, TW, prompt, n_new)
    spec, taus = O.speculative_generate(tshape, TW, dshape, DW, prompt, n_new, 6, selector=sel)
    np.testing.assert_array_equal(spec, ar)
    assert all(1 <= t <= 6 for t in taus)
