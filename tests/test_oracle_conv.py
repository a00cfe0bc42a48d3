"""Pins of the oracle's DFlash 2 grouped dynamic causal conv (txtmix source
reading §13, §14): closed forms of the two-tap conv, its group sharing and
causality, the reading order of the kernel projection, and its place in a
draft layer."""
import numpy as np

import oracle as O
from oracle.dflash_oracle import _conv_pair
from test_oracle_pins import _tiny_layer

D, H, G, d, F = 32, 4, 2, 8, 48


def test_identity_and_shift_taps():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 12))
    zero = np.zeros((5, 2, 3))
    ident = np.stack([np.ones(12), np.zeros(12)])
    shift = np.stack([np.zeros(12), np.ones(12)])
    np.testing.assert_array_equal(O.dynamic_conv(x, zero, ident, 4), x)
    np.testing.assert_array_equal(O.dynamic_conv(x, zero, shift, 4),
                                  np.concatenate([np.zeros((1, 12)), x[:-1]]))


def test_one_correction_per_channel_group():
    """Unit rows and a zero base kernel: every output is the sum of the
    corrections of its channel's group (the first row has no predecessor)."""
    rng = np.random.default_rng(2)
    corr = rng.standard_normal((4, 2, 3))
    out = O.dynamic_conv(np.ones((4, 12)), corr, np.zeros((2, 12)), 4)
    for t in range(4):
        for ch in range(12):
            want = corr[t, 0, ch // 4] + (corr[t, 1, ch // 4] if t > 0 else 0.0)
            assert out[t, ch] == want


def test_causal():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 8))
    corr, base = rng.standard_normal((6, 2, 2)), rng.standard_normal((2, 8))
    a = O.dynamic_conv(x, corr, base, 4)
    for t in range(5):
        y = x.copy()
        y[t + 1:] += 1.0
        np.testing.assert_array_equal(a[:t + 1], O.dynamic_conv(y, corr, base, 4)[:t + 1])


def test_projection_reading_order():
    """Kernel projection rows are read as [call, tap, group]: a projection
    whose only non-zero row is (call 1, tap 0, group 0) changes only the
    finish call's tap-0 coefficient of channels 0..group-1, by x . row."""
    rng = np.random.default_rng(4)
    B, Dm, g = 4, 8, 4
    ng = Dm // g
    x = rng.standard_normal((B, Dm))
    kp = np.zeros((2 * 2 * ng, Dm))
    kp[1 * 2 * ng + 0 * ng + 0] = rng.standard_normal(Dm)
    base = np.zeros((2, 2, Dm))
    prep, fin = _conv_pair(x, kp, base, g)
    y = rng.standard_normal((B, Dm))
    np.testing.assert_array_equal(prep(y), np.zeros((B, Dm)))
    c = x @ kp[2 * ng]
    out = fin(y)
    np.testing.assert_allclose(out[:, :g], c[:, None] * O.f32(y)[:, :g], atol=1e-12)
    np.testing.assert_array_equal(out[:, g:], 0.0)


def _conv_layer(rng, att_base, mlp_base, kp_zero=True):
    lay = _tiny_layer(rng, D, H, G, d, F)
    ng = D // 4
    for k, base in (("att", att_base), ("mlp", mlp_base)):
        lay[f"conv_{k}_kp"] = np.zeros((4 * ng, D)) if kp_zero else rng.standard_normal((4 * ng, D))
        lay[f"conv_{k}_base"] = base
    return lay


def _run(lay, x, cK, cV, group):
    L, B = cK.shape[0], x.shape[0]
    return O.draft_layer(x, lay, cK, cV, np.arange(L, L + B), H, G, d, 1e6, 1e-6, O.f32, None,
                         group)


def test_identity_convs_leave_the_layer_unchanged():
    rng = np.random.default_rng(5)
    ident = np.stack([np.stack([np.ones(D), np.zeros(D)])] * 2)   # [call, tap, D]
    lay = _conv_layer(rng, ident, ident)
    x = O.f32(rng.standard_normal((5, D)))
    cK, cV = rng.standard_normal((7, G, d)), rng.standard_normal((7, G, d))
    np.testing.assert_allclose(_run(lay, x, cK, cV, 4), _run(lay, x, cK, cV, 0), atol=1e-6)


def test_shifting_finish_conv_shifts_the_attention_increment():
    """With the FFN's output weights zero, a layer's output minus its input
    is the attention sublayer's increment; a finish conv with taps (0, 1)
    moves that increment down one row (the first row gets none)."""
    rng = np.random.default_rng(6)
    ident = np.stack([np.ones(D), np.zeros(D)])
    shift = np.stack([np.zeros(D), np.ones(D)])
    lay = _conv_layer(rng, np.stack([ident, shift]), np.stack([ident, ident]))
    lay["wd"][:] = 0
    x = O.f32(rng.standard_normal((5, D)))
    cK, cV = rng.standard_normal((7, G, d)), rng.standard_normal((7, G, d))
    inc = _run(lay, x, cK, cV, 0) - x
    got = _run(lay, x, cK, cV, 4) - x
    np.testing.assert_allclose(got, np.concatenate([np.zeros((1, D)), inc[:-1]]), atol=1e-6)
