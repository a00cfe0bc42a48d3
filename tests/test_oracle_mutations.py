"""Plant plausible mistakes in the oracle (CPU only) and check that a pin
catches each one: a pin that cannot fail pins nothing."""
import numpy as np
import pytest

import oracle as O
import oracle.dflash_oracle as OM
import test_oracle_conv as C
import test_oracle_masks as M
import test_oracle_pins as P
import test_oracle_pins_layer as PL
import test_oracle_sampling as S
import test_oracle_selector as SEL


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


def _attention_modulo_groups(q, K, V, key_visible=None, arith="f64"):
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


def _attention_no_scale(q, K, V, key_visible=None, arith="f64"):
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


def _layer_drop_attn_residual(x, layer, ctx_K, ctx_V, pos, H, G, d, theta, eps, store=OM.f32,
                              mask=None, conv_group=0, arith="f64"):
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


# ---- mutants of the sampling, selection, conv and mask functions ----------
def _visible_causal_excludes_self(L, B, causal, window):
    p = np.arange(L, L + B)[:, None]
    j = np.arange(L + B)[None, :]
    vis = np.ones((B, L + B), dtype=bool)
    if causal:
        vis &= j < p                     # a row loses its own key
    if window > 0:
        vis &= j > p - window
    return vis


def _visible_window_one_wider(L, B, causal, window):
    p = np.arange(L, L + B)[:, None]
    j = np.arange(L + B)[None, :]
    vis = np.ones((B, L + B), dtype=bool)
    if causal:
        vis &= j <= p
    if window > 0:
        vis &= j >= p - window           # W + 1 keys
    return vis


def _conv_taps_swapped(x, corr, base, group):
    x = np.asarray(x, np.float64)
    k = np.asarray(base, np.float64)[None] + np.repeat(np.asarray(corr, np.float64), group, axis=-1)
    prev = np.concatenate([np.zeros((1, x.shape[1])), x[:-1]], axis=0)
    return k[:, 1] * x + k[:, 0] * prev


def _conv_wraps_first_row(x, corr, base, group):
    x = np.asarray(x, np.float64)
    k = np.asarray(base, np.float64)[None] + np.repeat(np.asarray(corr, np.float64), group, axis=-1)
    return k[:, 0] * x + k[:, 1] * np.roll(x, 1, axis=0)


def _conv_groups_interleaved(x, corr, base, group):
    x = np.asarray(x, np.float64)
    corr = np.asarray(corr, np.float64)
    k = np.asarray(base, np.float64)[None] + np.tile(corr, (1, 1, group))   # channel c -> group c % n
    prev = np.concatenate([np.zeros((1, x.shape[1])), x[:-1]], axis=0)
    return k[:, 0] * x + k[:, 1] * prev


def _sample_left(weights, u):
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    return min(int(np.searchsorted(c, u * c[-1], side="left")), len(c) - 1)


def _verify_rejection_with(accept_rule, residual_rule):
    """verify_rejection with its acceptance test and residual replaced."""
    def verify(draft, q, p, u_accept, u_sample, start):
        draft = np.asarray(draft)
        batch, B = draft.shape
        accept = np.zeros(batch, dtype=np.int32)
        token = np.zeros(batch, dtype=np.int32)
        out = np.full((batch, B), -1, dtype=np.int32)
        new_len = np.zeros(batch, dtype=np.int32)
        for b in range(batch):
            a = 0
            while a < B - 1:
                d = int(draft[b, a + 1])
                if not accept_rule(u_accept[b, a], q[b, a][d], p[b, a][d]):
                    break
                a += 1
            if a < B - 1:
                res = residual_rule(np.asarray(p[b, a], np.float64), np.asarray(q[b, a], np.float64))
                tok = OM.sample_from(res if res.sum() > 0 else p[b, a], float(u_sample[b]))
            else:
                tok = OM.sample_from(p[b, B - 1], float(u_sample[b]))
            accept[b], token[b] = a, tok
            out[b, :a] = draft[b, 1:a + 1]
            out[b, a] = tok
            new_len[b] = int(start[b]) + a + 1
        return accept, token, out, new_len
    return verify


# u * q > p instead of u * q < p
_verify_accept_flipped = _verify_rejection_with(lambda u, qd, pd: u * qd > pd,
                                                lambda p, q: np.maximum(p - q, 0.0))
# residual max(q - p, 0) instead of max(p - q, 0)
_verify_residual_reversed = _verify_rejection_with(lambda u, qd, pd: u * qd < pd,
                                                   lambda p, q: np.maximum(q - p, 0.0))


def _topk_highest_on_ties(z, k):
    z = np.asarray(z)
    out = np.empty(z.shape[:-1] + (k,), dtype=np.int32)
    for idx in np.ndindex(*z.shape[:-1]):
        row = z[idx]
        out[idx] = np.lexsort((-np.arange(row.shape[0]), -row))[:k]
    return out


_real_select = OM.select_candidates


def _select_codebooks_swapped(logits, hidden, anchor, W_h, code_pred, code_succ, top_k):
    return _real_select(logits, hidden, anchor, W_h, code_succ, code_pred, top_k)


_INJECT = OM.inject_kv


def _inject_swapped(H_t, layer, pos, G, d, theta, eps, store=OM.f32, qk_norm=True):
    return _INJECT(H_t, dict(layer, wk=layer["wv"], wv=layer["wk"]), pos, G, d, theta, eps, store,
                   qk_norm)


def _inject_no_knorm(H_t, layer, pos, G, d, theta, eps, store=OM.f32, qk_norm=True):
    return _INJECT(H_t, layer, pos, G, d, theta, eps, store, False)


def _inject_rope_at_row_index(H_t, layer, pos, G, d, theta, eps, store=OM.f32, qk_norm=True):
    return _INJECT(H_t, layer, np.arange(H_t.shape[0]), G, d, theta, eps, store, qk_norm)


def _inject_norm_after_rope(H_t, layer, pos, G, d, theta, eps, store=OM.f32, qk_norm=True):
    T = H_t.shape[0]
    k = OM.linear(H_t, layer["wk"]).reshape(T, G, d)
    k = OM.rmsnorm(OM.rope(k, pos, theta), layer["k_norm"], eps)
    v = OM.linear(H_t, layer["wv"]).reshape(T, G, d)
    return store(k), store(v)


def _layer_variant(swiglu_reversed=False, q_norm=True):
    """draft_layer (no conv) with one planted mistake."""
    def layer_fn(x, layer, ctx_K, ctx_V, pos, H, G, d, theta, eps, store=OM.f32, mask=None,
                 conv_group=0, arith="f64"):
        B = x.shape[0]
        h = store(OM.rmsnorm(x, layer["g_in"], eps))
        q = OM.linear(h, layer["wq"]).reshape(B, H, d)
        k = OM.linear(h, layer["wk"]).reshape(B, G, d)
        v = OM.linear(h, layer["wv"]).reshape(B, G, d)
        q = store(OM.rope(OM.rmsnorm(q, layer["q_norm"], eps) if q_norm else q, pos, theta))
        k = store(OM.rope(OM.rmsnorm(k, layer["k_norm"], eps), pos, theta))
        o = store(OM.attention(q, np.concatenate([ctx_K, k]), np.concatenate([ctx_V, store(v)]),
                               mask).reshape(B, H * d))
        x = OM.f32(x + OM.linear(o, layer["wo"]))
        h2 = store(OM.rmsnorm(x, layer["g_post"], eps))
        g, u = OM.linear(h2, layer["wg"]), OM.linear(h2, layer["wu"])
        a = store(OM.silu(u) * g if swiglu_reversed else OM.silu(g) * u)
        return OM.f32(x + OM.linear(a, layer["wd"]))
    return layer_fn


def _block_variant(pos_from_zero=False, logit_rows_from_anchor=False, final_norm=True):
    """draft_block (bidirectional layers, one planted mistake)."""
    def block_fn(shape, W, ctx_K, ctx_V, anchors, B, store=OM.f32, return_logits=False,
                 lm_head=True, return_hidden=False, arith="f64"):
        ids = np.zeros((len(anchors), B), np.int32)
        gaps = np.zeros((len(anchors), B - 1))
        hidden = []
        for b, a in enumerate(anchors):
            L = ctx_K[0][b].shape[0]
            pos = np.arange(B) if pos_from_zero else np.arange(L, L + B)
            x = OM.embed_block(W["embed"], a, shape.mask_id, B, shape.embed_scale)
            for l, layer in enumerate(W["layers"]):
                x = OM.draft_layer(x, layer, ctx_K[l][b], ctx_V[l][b], pos, shape.H, shape.G,
                                   shape.d, shape.rope_theta, shape.eps, store)
            hidden.append(x)
            ids[b, 0] = a
            if lm_head:
                rows = x[:-1] if logit_rows_from_anchor else x[1:]
                hf = store(OM.rmsnorm(rows, W["g_f"], shape.eps)) if final_norm else rows
                z = OM.lm_head_logits(hf, W["lm_head"])
                ids[b, 1:] = OM.argmax_lowest(z)
                gaps[b] = OM.top2_gap(z)
        return (ids, gaps, np.stack(hidden)) if return_hidden else (ids, gaps)
    return block_fn


def _embed_no_scale(embed, anchor, mask_id, B, scale):
    return OM.f32(np.asarray(embed[[int(anchor)] + [int(mask_id)] * (B - 1)], np.float64))


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
    ("draft_key_visible", _visible_causal_excludes_self, lambda: M.test_causal_anchor_is_full_attention_over_sliced_keys()),
    ("draft_key_visible", _visible_window_one_wider, lambda: M.test_window_ignores_older_context(True)),
    ("dynamic_conv", _conv_taps_swapped, lambda: C.test_identity_and_shift_taps()),
    ("dynamic_conv", _conv_wraps_first_row, lambda: C.test_identity_and_shift_taps()),
    ("dynamic_conv", _conv_groups_interleaved, lambda: C.test_one_correction_per_channel_group()),
    ("sample_from", _sample_left, lambda: S.test_sample_from_buckets()),
    ("verify_rejection", _verify_accept_flipped, lambda: S.test_equal_distributions_accept_everything()),
    ("verify_rejection", _verify_residual_reversed, lambda: S.test_emitted_token_follows_target(0)),
    ("topk_lowest", _topk_highest_on_ties, lambda: SEL.test_topk_matches_brute_force_with_ties(0)),
    ("select_candidates", _select_codebooks_swapped, lambda: SEL.test_planted_bigram_chain_is_followed()),
    ("inject_kv", _inject_swapped, lambda: PL.test_inject_kv_identity_projections_and_positions()),
    ("inject_kv", _inject_no_knorm, lambda: PL.test_inject_kv_identity_projections_and_positions()),
    ("inject_kv", _inject_rope_at_row_index, lambda: PL.test_inject_kv_identity_projections_and_positions()),
    ("inject_kv", _inject_norm_after_rope, lambda: PL.test_inject_kv_identity_projections_and_positions()),
    ("draft_layer", _layer_variant(swiglu_reversed=True), lambda: PL.test_draft_layer_swiglu_orientation()),
    ("draft_layer", _layer_variant(q_norm=False), lambda: PL.test_draft_layer_query_norm()),
    ("draft_block", _block_variant(pos_from_zero=True), lambda: PL.test_draft_block_anchor_at_position_after_context()),
    ("draft_block", _block_variant(logit_rows_from_anchor=True), lambda: PL.test_draft_block_final_norm_and_logit_rows()),
    ("draft_block", _block_variant(final_norm=False), lambda: PL.test_draft_block_final_norm_and_logit_rows()),
    ("embed_block", _embed_no_scale, lambda: PL.test_embed_block_scale()),
]


@pytest.mark.parametrize("i", range(len(MUTATIONS)))
def test_pin_catches_planted_mistake(monkeypatch, i):
    name, bad, pin = MUTATIONS[i]
    pin()                                   # passes on the real oracle
    _patch(monkeypatch, name, bad)
    with pytest.raises(AssertionError):
        pin()
