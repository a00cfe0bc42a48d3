"""Pins of the oracle's K/V injection, draft layer and draft block wiring.

Each pin reduces one function to a closed form, or to library routines on a
special case, that a plausible mistake cannot pass:
  inject_kv    which projection feeds K and which V, k_norm applied, and
               applied before RoPE at the cache positions;
  draft_layer  the SwiGLU orientation silu(gate) * up, and the query norm;
  draft_block  the anchor at position L (right after the L cached entries),
               the final RMSNorm, and logits from rows 1..B-1 only;
  embed_block  the input embedding scale.
tests/test_oracle_mutations.py plants a mistake of each kind and checks that
the pin named for it fails."""
import math

import numpy as np
import torch
import torch.nn.functional as Fn

import oracle as O
import synth


def _rot_complex(x, pos, theta):
    """Rotation of the pairs (i, i + d/2) as complex multiplication by
    exp(i pos theta^(-2i/d)), the form the RoPE pin checks the oracle against."""
    d = x.shape[-1]
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    inv = 1.0 / theta ** (np.arange(0, d, 2) / d)
    z = z * np.exp(1j * np.asarray(pos, np.float64)[:, None, None] * inv)
    return np.concatenate([z.real, z.imag], -1)


def _rmsnorm_t(x, gain, eps=1e-6):
    x = torch.as_tensor(np.asarray(x, np.float64))
    return Fn.rms_norm(x, (x.shape[-1],), torch.as_tensor(np.asarray(gain, np.float64)),
                       eps=eps).numpy()


# --- K/V injection -----------------------------------------------------------------
def test_inject_kv_identity_projections_and_positions():
    """([tutorial] §2.1.2; [reading] §5.)  With k_proj = 3 I and v_proj = 2 I
    (G d = D), K at position 0 is each head's slice of H_t through the
    per-head RMSNorm with the k_norm gains (torch's rms_norm) and V is twice
    the slice.  The same row appended at positions 5 and 1000 gives K equal
    to the position-0 K rotated by those positions: k_norm comes before
    RoPE (the gains differ across the pairs RoPE mixes), at the positions
    given, not at the rows' indices."""
    rng = np.random.default_rng(20)
    G, d, theta, eps = 2, 8, 1e6, 1e-6
    D = G * d
    layer = {"wk": 3.0 * np.eye(D), "wv": 2.0 * np.eye(D), "k_norm": rng.uniform(0.5, 2.0, d)}
    Ht = rng.standard_normal((3, D))
    K, V = O.inject_kv(Ht, layer, np.zeros(3, np.int64), G, d, theta, eps, O.f32)
    sl = Ht.reshape(3, G, d)
    np.testing.assert_allclose(K, _rmsnorm_t(3.0 * sl, layer["k_norm"], eps), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(V, 2.0 * sl, rtol=1e-6, atol=1e-7)
    same = np.repeat(Ht[:1], 3, axis=0)
    pos = np.array([0, 5, 1000])
    K2, _ = O.inject_kv(same, layer, pos, G, d, theta, eps, O.f32)
    np.testing.assert_allclose(K2, _rot_complex(np.repeat(K2[:1], 3, axis=0), pos, theta),
                               rtol=1e-6, atol=1e-6)


# --- draft layer -------------------------------------------------------------------
def _layer(rng, D, H, G, d, F):
    w = lambda *s: rng.standard_normal(s) * 0.3
    return {"wq": w(H * d, D), "wk": w(G * d, D), "wv": w(G * d, D), "wo": w(D, H * d),
            "wg": w(F, D), "wu": w(F, D), "wd": w(D, F), "g_in": np.ones(D),
            "g_post": rng.uniform(0.5, 2.0, D), "q_norm": rng.uniform(0.5, 2.0, d),
            "k_norm": rng.uniform(0.5, 2.0, d)}


def test_draft_layer_swiglu_orientation():
    """([reading] §6: the draft layers are Qwen3 layers, FFN = down(silu(gate)
    * up).)  With o_proj zero the attention adds nothing; with gate = 1.5 I,
    up = -0.7 I and down = I the layer adds silu(1.5 h2) * (-0.7 h2), h2 the
    post-attention RMSNorm of x (torch's silu and rms_norm)."""
    rng = np.random.default_rng(21)
    D = H = 8
    lay = _layer(rng, D, 1, 1, 8, D)
    lay["wo"][:] = 0
    lay["wg"], lay["wu"], lay["wd"] = 1.5 * np.eye(D), -0.7 * np.eye(D), np.eye(D)
    x = O.f32(rng.standard_normal((3, D)))
    out = O.draft_layer(x, lay, rng.standard_normal((4, 1, 8)), rng.standard_normal((4, 1, 8)),
                        np.arange(4, 7), 1, 1, 8, 1e6, 1e-6, O.f32)
    h2 = torch.from_numpy(_rmsnorm_t(x, lay["g_post"]))
    expect = x + (Fn.silu(1.5 * h2) * (-0.7 * h2)).numpy()
    np.testing.assert_allclose(out, expect, rtol=1e-6, atol=1e-6)


def test_draft_layer_query_norm():
    """The per-head query RMSNorm: (1) with q_norm gains zero every query is
    zero, so each row attends uniformly and (o_proj = I, FFN off) adds the
    mean of all values [context ; block] (the block's own values are
    h W_v^T, h the input RMSNorm of x by torch); (2) with nonzero gains the
    layer does not change when W_q is scaled by 7."""
    rng = np.random.default_rng(22)
    D, H, G, d = 8, 1, 1, 8
    lay = _layer(rng, D, H, G, d, D)
    lay["wo"], lay["wg"] = np.eye(D), np.zeros((D, D))
    x = O.f32(rng.standard_normal((3, D)))
    cK, cV = rng.standard_normal((5, G, d)), rng.standard_normal((5, G, d))
    pos = np.arange(5, 8)
    zq = dict(lay, q_norm=np.zeros(d))
    out = O.draft_layer(x, zq, cK, cV, pos, H, G, d, 1e6, 1e-6, O.f32)
    vb = _rmsnorm_t(x, lay["g_in"]) @ lay["wv"].T
    mean_v = np.concatenate([cV[:, 0], vb]).mean(0)
    np.testing.assert_allclose(out, x + mean_v, rtol=1e-6, atol=1e-6)
    a = O.draft_layer(x, lay, cK, cV, pos, H, G, d, 1e6, 1e-6, O.f32)
    b = O.draft_layer(x, dict(lay, wq=7.0 * lay["wq"]), cK, cV, pos, H, G, d, 1e6, 1e-6, O.f32)
    np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-6)
    assert np.abs(a - out).max() > 1e-3       # the gains do matter


# --- draft block -------------------------------------------------------------------
def _shape(D, H, d, V, mask_id, embed_scale=1.0):
    return synth.DraftShape(n_layers=1, D=D, H=H, G=H, d=d, F=D, V=V, mask_id=mask_id,
                            n_target_layers=12, embed_scale=embed_scale)


def test_draft_block_anchor_at_position_after_context():
    """([reading] §9: the block's positions continue from the cached context;
    the anchor sits right after the L entries.)  d = 2, so RoPE turns the one
    pair by p radians at position p.  One cached entry (L = 1) whose key is
    the anchor's own unit-RMS row h turned by 1 radian: an anchor at position
    1 scores that key exactly like its own, attends to both equally, and
    (all projections I, FFN off) the layer adds (v_ctx + h) / 2."""
    s = _shape(D=2, H=1, d=2, V=4, mask_id=3)
    I2, Z2 = np.eye(2), np.zeros((2, 2))
    lay = {"wq": I2, "wk": I2, "wv": I2, "wo": I2, "wg": Z2, "wu": Z2, "wd": Z2,
           "g_in": np.ones(2), "g_post": np.ones(2), "q_norm": np.ones(2), "k_norm": np.ones(2)}
    E = np.array([[0.3, 0.4], [1.0, 0.0], [0.0, 1.0], [0.5, 0.5]])
    W = {"embed": E, "lm_head": np.eye(4, 2), "g_f": np.ones(2), "layers": [lay]}
    h = E[0] / math.sqrt(np.mean(E[0] ** 2))
    kappa = _rot_complex(h[None, None, :], [1], s.rope_theta)[0]
    v_ctx = np.array([[[1.0, -2.0]]])
    _, _, hid = O.draft_block(s, W, [[kappa[None]]], [[v_ctx]], [0], 1, O.f32, lm_head=False,
                              return_hidden=True)
    np.testing.assert_allclose(hid[0, 0], E[0] + (v_ctx[0, 0] + h) / 2, atol=1e-5)


def test_draft_block_final_norm_and_logit_rows():
    """([reading] §6, §14: drafts come from block rows 1..B-1 through the
    final norm and the shared LM head.)  Identity layers (o_proj and down
    zero) keep the embedded block; LM-head row 7 is planted along the final
    norm of the mask embedding and row 5 along that of the anchor, so rows
    1..B-1 draft 7 (the anchor row would draft 5), and each gap is the top-2
    gap of the mask row's normed logits (torch's rms_norm with the g_f
    gains)."""
    rng = np.random.default_rng(23)
    D, V, B, anchor, mask = 8, 16, 4, 4, 15
    s = _shape(D=D, H=1, d=8, V=V, mask_id=mask)
    lay = _layer(rng, D, 1, 1, 8, D)
    lay["wo"][:] = 0
    lay["wd"][:] = 0
    E = rng.standard_normal((V, D)) * 0.02
    g_f = rng.uniform(0.5, 2.0, D)
    lm = rng.standard_normal((V, D)) * 0.1
    hm, ha = _rmsnorm_t(E[mask], g_f), _rmsnorm_t(E[anchor], g_f)
    lm[7] = 5.0 * hm / np.linalg.norm(hm)
    lm[5] = 5.0 * ha / np.linalg.norm(ha)
    W = {"embed": E, "lm_head": lm, "g_f": g_f, "layers": [lay]}
    ctx = [[rng.standard_normal((3, 1, 8))]]
    ids, gap = O.draft_block(s, W, ctx, [[rng.standard_normal((3, 1, 8))]], [anchor], B, O.f32)
    np.testing.assert_array_equal(ids, [[anchor, 7, 7, 7]])
    z = np.sort(torch.from_numpy(hm) @ torch.from_numpy(lm).T)
    np.testing.assert_allclose(gap[0], np.full(B - 1, z[-1] - z[-2]), rtol=1e-5)


def test_embed_block_scale():
    """([reading] §9, §11: input_embedding_scale multiplies the block's
    embedding rows [anchor, mask x (B-1)].)  Identity layers return the
    embedded block as the residual."""
    rng = np.random.default_rng(24)
    D, V = 8, 16
    s = _shape(D=D, H=1, d=8, V=V, mask_id=9, embed_scale=2.5)
    lay = _layer(rng, D, 1, 1, 8, D)
    lay["wo"][:] = 0
    lay["wd"][:] = 0
    E = rng.standard_normal((V, D))
    W = {"embed": E, "lm_head": E, "g_f": np.ones(D), "layers": [lay]}
    ctx = [[rng.standard_normal((2, 1, 8))]]
    _, _, hid = O.draft_block(s, W, ctx, ctx, [3], 4, O.f32, lm_head=False, return_hidden=True)
    np.testing.assert_allclose(hid[0], 2.5 * E[[3, 9, 9, 9]], rtol=1e-7)
