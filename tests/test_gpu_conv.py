"""DFlash 2's grouped dynamic causal conv in the draft layers on the GPU vs
the oracle (txtmix source reading §13-§14), fp32 and bf16, alone and
together with causal / sliding-window layers, through the block call and
the round call."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import to_np
from test_gpu_draft import SMALL_BF16, _random_cache_case

pytestmark = pytest.mark.gpu


def _conv(w, group=16, **masks):
    s = dataclasses.replace(w.draft, conv_group=group, **masks)
    w = synth.with_(w, draft=s)
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    return w, synth.add_conv_weights(weights, s, w.dtype, w.seed + 7, device="cuda")


@pytest.mark.parametrize("group", [16, 64])
def test_conv_f32(dfl, group):
    w, weights = _conv(synth.WORKLOADS["tiny_f32"], group)
    _random_cache_case(dfl, w, w.B, [0, 20, 64], np.arange(3), weights)


@pytest.mark.parametrize("B,lens", [(8, [37, 0]), (16, [300]), (16, [0, 300, 17, 700])])
def test_conv_bf16(dfl, B, lens):
    w, weights = _conv(SMALL_BF16)
    _random_cache_case(dfl, w, B, lens, np.arange(len(lens)), weights)


def test_conv_with_causal_window_layers(dfl):
    w, weights = _conv(synth.WORKLOADS["tiny_f32"], 16, causal_layers=0b11, window_layers=0b10,
                       sliding_window=6)
    _random_cache_case(dfl, w, w.B, [0, 20, 64], np.arange(3), weights)


def test_conv_changes_the_block(dfl):
    """The conv modules are live: the same weights without them give
    another residual stream (so the parity above tests the conv itself)."""
    w, weights = _conv(synth.WORKLOADS["tiny_f32"])
    s = w.draft
    W = to_np(weights)
    rng = np.random.default_rng(3)
    cK = [[rng.standard_normal((9, s.G, s.d))] for _ in range(s.n_layers)]
    cV = [[rng.standard_normal((9, s.G, s.d))] for _ in range(s.n_layers)]
    _, _, h_conv = O.draft_block(s, W, cK, cV, [5], w.B, lm_head=False, return_hidden=True)
    plain = dataclasses.replace(s, conv_group=0)
    _, _, h_plain = O.draft_block(plain, W, cK, cV, [5], w.B, lm_head=False, return_hidden=True)
    assert np.abs(h_conv - h_plain).max() > 1e-2
