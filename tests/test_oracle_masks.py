"""Pins of the oracle's causal / sliding-window draft layers (txtmix source
reading §6: sliding_attention layers are causal by default and keep a
window of sliding_window keys; full_attention layers are bidirectional)."""
import dataclasses

import numpy as np
import pytest

import oracle as O
import synth
from helpers import to_np64
from test_oracle_pins import _tiny_layer

D, H, G, d, F = 32, 4, 2, 8, 48


def _inputs(rng, L, B):
    return (O.f32(rng.standard_normal((B, D))), rng.standard_normal((L, G, d)),
            rng.standard_normal((L, G, d)))


def _layer(rng, x, lay, cK, cV, mask):
    L, B = cK.shape[0], x.shape[0]
    return O.draft_layer(x, lay, cK, cV, np.arange(L, L + B), H, G, d, 1e6, 1e-6, O.f32, mask)


def test_window_of_one_returns_the_rows_own_value():
    """Causal with a window of one key: each row sees only itself, so each
    head's attention output is its own value row (softmax of one score)."""
    rng = np.random.default_rng(1)
    L, B = 5, 4
    q = rng.standard_normal((B, H, d))
    K = rng.standard_normal((L + B, G, d))
    V = rng.standard_normal((L + B, G, d))
    out = O.attention(q, K, V, O.draft_key_visible(L, B, True, 1))
    for hh in range(H):
        np.testing.assert_allclose(out[:, hh], V[L:, hh // (H // G)], atol=1e-12)


def test_causal_rows_ignore_later_rows():
    rng = np.random.default_rng(2)
    L, B = 6, 5
    lay = _tiny_layer(rng, D, H, G, d, F)
    x, cK, cV = _inputs(rng, L, B)
    mask = O.draft_key_visible(L, B, True, 0)
    a = _layer(rng, x, lay, cK, cV, mask)
    for i in range(B - 1):
        y = x.copy()
        y[i + 1:] = O.f32(rng.standard_normal((B - i - 1, D)))
        b = _layer(rng, y, lay, cK, cV, mask)
        np.testing.assert_array_equal(a[:i + 1], b[:i + 1])
        assert not np.allclose(a[i + 1:], b[i + 1:])
    # bidirectional: row 0 does see the later rows
    full = _layer(rng, x, lay, cK, cV, None)
    y = x.copy()
    y[1:] += 1.0
    assert not np.allclose(full[0], _layer(rng, y, lay, cK, cV, None)[0])


@pytest.mark.parametrize("causal", [True, False])
def test_window_ignores_older_context(causal):
    """Block row i at position L + i keeps keys after L + i - W: context
    entries before L - W + 1 are out of every row's window."""
    rng = np.random.default_rng(3)
    L, B, W = 12, 4, 5
    lay = _tiny_layer(rng, D, H, G, d, F)
    x, cK, cV = _inputs(rng, L, B)
    mask = O.draft_key_visible(L, B, causal, W)
    a = _layer(rng, x, lay, cK, cV, mask)
    cut = L - W + 1
    cK2, cV2 = cK.copy(), cV.copy()
    cK2[:cut] = rng.standard_normal((cut, G, d))
    cV2[:cut] = rng.standard_normal((cut, G, d))
    np.testing.assert_array_equal(a, _layer(rng, x, lay, cK2, cV2, mask))
    cK2[cut] += 1.0   # the oldest entry still in row 0's window
    assert not np.allclose(a[0], _layer(rng, x, lay, cK2, cV2, mask)[0])


def test_causal_anchor_is_full_attention_over_sliced_keys():
    """The anchor row of a causal layer equals plain attention over the
    context and the anchor's own key, sliced out explicitly."""
    rng = np.random.default_rng(4)
    L, B = 7, 4
    q = rng.standard_normal((B, H, d))
    K = rng.standard_normal((L + B, G, d))
    V = rng.standard_normal((L + B, G, d))
    masked = O.attention(q, K, V, O.draft_key_visible(L, B, True, 0))
    for i in range(B):
        sliced = O.attention(q[i:i + 1], K[:L + i + 1], V[:L + i + 1])
        np.testing.assert_allclose(masked[i:i + 1], sliced, atol=1e-12)


def test_window_covering_every_key_changes_nothing():
    rng = np.random.default_rng(5)
    L, B = 6, 4
    lay = _tiny_layer(rng, D, H, G, d, F)
    x, cK, cV = _inputs(rng, L, B)
    np.testing.assert_array_equal(_layer(rng, x, lay, cK, cV, O.draft_key_visible(L, B, False, L + B)),
                                  _layer(rng, x, lay, cK, cV, None))


def test_draft_block_reads_the_layer_types():
    """draft_block applies layer l's mask from the shape's bit masks: both
    layers causal, layer 1 also windowed to 3 keys, equals running the
    layers by hand with those masks."""
    rng = np.random.default_rng(6)
    w = synth.WORKLOADS["tiny_f32"]
    s = dataclasses.replace(w.draft, causal_layers=0b11, window_layers=0b10, sliding_window=3)
    Wt = to_np64(synth.draft_weights(s, "f32", 3))
    L = 9
    ctxK = [[rng.standard_normal((L, s.G, s.d))] for _ in range(s.n_layers)]
    ctxV = [[rng.standard_normal((L, s.G, s.d))] for _ in range(s.n_layers)]
    _, _, hid = O.draft_block(s, Wt, ctxK, ctxV, [5], w.B, lm_head=False, return_hidden=True)
    x = O.embed_block(Wt["embed"], 5, s.mask_id, w.B, s.embed_scale)
    pos = np.arange(L, L + w.B)
    for l, lay in enumerate(Wt["layers"]):
        mask = O.draft_key_visible(L, w.B, True, 3 if l == 1 else 0)
        x = O.draft_layer(x, lay, ctxK[l][0], ctxV[l][0], pos, s.H, s.G, s.d, s.rope_theta,
                          s.eps, O.f32, mask)
    np.testing.assert_array_equal(hid[0], x)
