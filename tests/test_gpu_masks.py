"""Causal and sliding-window draft layers on the GPU vs the oracle (txtmix
source reading §6), through each attention path: the reference kernel
(fp32), the persistent block kernel (at most 16 bf16 rows) and the planned
split attention (more rows), with the tolerances of the block draft's
tests."""
import dataclasses

import numpy as np
import pytest

import synth
from test_gpu_draft import SMALL_BF16, _random_cache_case

pytestmark = pytest.mark.gpu


def _masked(w, causal, window_layers, window):
    s = dataclasses.replace(w.draft, causal_layers=causal, window_layers=window_layers,
                            sliding_window=window)
    return synth.with_(w, draft=s)


@pytest.mark.parametrize("causal,wl,W", [(0b11, 0, 0), (0b01, 0b10, 5), (0b11, 0b11, 1),
                                         (0, 0b01, 12)])
def test_masks_reference_kernel_f32(dfl, causal, wl, W):
    """fp32: ragged contexts (one empty: a causal anchor sees only itself)."""
    w = _masked(synth.WORKLOADS["tiny_f32"], causal, wl, W)
    _random_cache_case(dfl, w, w.B, [0, 20, 64], np.arange(3))


@pytest.mark.parametrize("B,lens", [(8, [37, 0]), (16, [300]), (5, [64])])
def test_masks_block_kernel_bf16(dfl, B, lens):
    n = SMALL_BF16.draft.n_layers
    w = _masked(SMALL_BF16, (1 << n) - 1, 1, 6)   # every layer causal, layer 0 windowed
    _random_cache_case(dfl, w, B, lens, np.arange(len(lens)))


@pytest.mark.parametrize("B,lens", [(16, [0, 300, 17, 700]), (48, [1000])])
def test_masks_split_attention_bf16(dfl, B, lens):
    n = SMALL_BF16.draft.n_layers
    w = _masked(SMALL_BF16, 1, (1 << n) - 1, 40)   # layer 0 causal, every layer windowed
    _random_cache_case(dfl, w, B, lens, np.arange(len(lens)))


def test_masks_qwen3_8b_batch1(dfl):
    """The Qwen3-8B shape at a 2048 context: every layer causal, alternate
    layers with a 128-key window (most of the context out of reach)."""
    w = synth.WORKLOADS["qwen3_8b_b1"]
    n = w.draft.n_layers
    w = _masked(w, (1 << n) - 1, int("01" * 8, 2) & ((1 << n) - 1), 128)
    _random_cache_case(dfl, w, w.B, [w.ctx_len], np.array([0]))
