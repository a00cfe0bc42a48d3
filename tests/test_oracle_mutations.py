"""Plant plausible mistakes in the oracle (CPU only) and check that a pin
catches each one: a pin that cannot fail pins nothing."""
import numpy as np
import pytest

import oracle as O
import oracle.dflash_oracle as OM
import test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(OM, name, fn)
    monkeypatch.setattr(O, name, fn)


def _rope_wrong_sign(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    phi = OM.rope_angles(pos, d, theta)[:, None, :]
    c, s = np.cos(phi), np.sin(phi)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)


def _rope_interleaved(x, pos, theta):
    # pairs (2i, 2i+1) instead of (i, i + d/2)
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    phi = OM.rope_angles(pos, d, theta)[:, None, :]
    c, s = np.cos(phi), np.sin(phi)
    x1, x2 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x1 * c - x2 * s
    out[..., 1::2] = x2 * c + x1 * s
    return out


def _attention_modulo_groups(q, K, V, key_visible=None):
    n, H, d = q.shape
    G = K.shape[1]
    out = np.empty((n, H, d))
    for h in range(H):
        g = h % G
        s = (q[:, h] @ K[:, g].T) / np.sqrt(d)
        if key_visible is not None:
            s = np.where(key_visible, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        out[:, h] = (p / p.sum(1, keepdims=True)) @ V[:, g]
    return out


_ATTENTION = OM.attention
_VERIFY = OM.verify_greedy


def _attention_no_scale(q, K, V, key_visible=None):
    return _ATTENTION(q * np.sqrt(q.shape[-1]), K, V, key_visible)


def _fuse_reversed(hiddens, Wc, g_c, eps, store=OM.f32):
    X = np.concatenate([np.asarray(h, dtype=np.float64) for h in hiddens[::-1]], axis=-1)
    return store(OM.rmsnorm(OM.linear(X, Wc), g_c, eps))


def _fuse_no_norm(hiddens, Wc, g_c, eps, store=OM.f32):
    X = np.concatenate([np.asarray(h, dtype=np.float64) for h in hiddens], axis=-1)
    return store(OM.linear(X, Wc))


def _verify_off_by_one(draft, post, start):
    batch, B = draft.shape
    acc = np.zeros(batch, dtype=np.int32)
    bon = np.zeros(batch, dtype=np.int32)
    out = np.full((batch, B), -1, dtype=np.int32)
    nl = np.zeros(batch, dtype=np.int32)
    for b in range(batch):
        a = 0
        while a < B - 1 and draft[b, a + 1] == post[b, a + 1]:
            a += 1
        acc[b], bon[b] = a, post[b, a]
        out[b, :a] = draft[b, 1:a + 1]
        out[b, a] = bon[b]
        nl[b] = start[b] + a + 1
    return acc, bon, out, nl


def _verify_bonus_after(draft, post, start):
    acc, bon, out, nl = _VERIFY(draft, post, start)
    B = draft.shape[1]
    bon = post[np.arange(len(acc)), np.minimum(acc + 1, B - 1)]
    return acc, bon, out, nl


def _argmax_highest(z):
    z = np.asarray(z)
    return (z.shape[-1] - 1 - np.argmax(z[..., ::-1], axis=-1)).astype(np.int32)


def _ids_wrong_end(n_t, n):
    if n == 1:
        return [n_t // 2]
    return [1 + round(i * (n_t - 3) / (n - 1)) for i in range(n)]


def _bf16_truncate(x):
    a = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (a.view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)


def _layer_drop_attn_residual(x, layer, ctx_K, ctx_V, pos, H, G, d, theta, eps, store=OM.f32):
    B = x.shape[0]
    h = store(OM.rmsnorm(x, layer["g_in"], eps))
    q = store(OM.rope(OM.rmsnorm(OM.linear(h, layer["wq"]).reshape(B, H, d), layer["q_norm"], eps), pos, theta))
    k = store(OM.rope(OM.rmsnorm(OM.linear(h, layer["wk"]).reshape(B, G, d), layer["k_norm"], eps), pos, theta))
    v = store(OM.linear(h, layer["wv"]).reshape(B, G, d))
    o = store(OM.attention(q, np.concatenate([ctx_K, k]), np.concatenate([ctx_V, v])).reshape(B, H * d))
    x = OM.f32(OM.linear(o, layer["wo"]))
    h2 = store(OM.rmsnorm(x, layer["g_post"], eps))
    a = store(OM.silu(OM.linear(h2, layer["wg"])) * OM.linear(h2, layer["wu"]))
    return OM.f32(x + OM.linear(a, layer["wd"]))


MUTATIONS = [
    ("rope", _rope_wrong_sign, lambda: P.test_rope_complex_form()),
    ("rope", _rope_interleaved, lambda: P.test_rope_complex_form()),
    ("attention", _attention_modulo_groups, lambda: P.test_attention_vs_sdpa(4, 2)),
    ("attention", _attention_no_scale, lambda: P.test_attention_vs_sdpa(4, 4)),
    ("fuse_context", _fuse_reversed, lambda: P.test_fuse_worked_example()),
    ("fuse_context", _fuse_no_norm, lambda: P.test_fuse_worked_example()),
    ("verify_greedy", _verify_off_by_one, lambda: P.test_verify_exhaustive(3)),
    ("verify_greedy", _verify_bonus_after, lambda: P.test_verify_exhaustive(3)),
    ("argmax_lowest", _argmax_highest, lambda: P.test_argmax_ties_lowest_and_gap()),
    ("build_target_layer_ids", _ids_wrong_end, lambda: P.test_layer_ids_configs(36, [1, 9, 17, 25, 33])),
    ("bf16", _bf16_truncate, lambda: P.test_bf16_rounding_matches_torch()),
    ("draft_layer", _layer_drop_attn_residual, lambda: P.test_draft_layer_identity_without_outputs()),
]


@pytest.mark.parametrize("i", range(len(MUTATIONS)))
def test_pin_catches_planted_mistake(monkeypatch, i):
    name, bad, pin = MUTATIONS[i]
    pin()                                   # passes on the real oracle
    _patch(monkeypatch, name, bad)
    with pytest.raises(AssertionError):
        pin()
