"""Pins of the CPU oracle against facts the pages and mathematics fix.

None of these compare the oracle with itself: each checks a printed value,
a closed form, a library routine on a special case, an invariant, or an
exhaustive brute force.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --- target layer selection -------------------------------------------------
@pytest.mark.parametrize("n_t,expect", [(12, [1, 3, 5, 7, 9]),
                                        (36, [1, 9, 17, 25, 33]),
                                        (8, [1, 2, 3, 4, 5])])
def test_layer_ids_configs(n_t, expect):
    assert O.build_target_layer_ids(n_t, 5) == expect


@pytest.mark.parametrize("n_t", range(6, 80))
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_layer_ids_rule(n_t, n):
    # picks span the second layer to the third-from-last, 0-based, uniformly
    if n_t - 4 < n - 1:
        return
    ids = O.build_target_layer_ids(n_t, n)
    assert ids[0] == 1 and ids[-1] == n_t - 3
    assert len(ids) == n and ids == sorted(set(ids))
    step = (n_t - 4) / (n - 1)
    for i, v in enumerate(ids):
        assert abs(v - (1 + i * step)) <= 0.5


def test_layer_ids_single_pick_is_middle():
    assert O.build_target_layer_ids(12, 1) == [6]
    assert O.build_target_layer_ids(36, 1) == [18]


# --- context fusion ------------------------------------------------------------
def test_fuse_worked_example():
    """The tutorial's printed context_feature[:3, :8] (seed 42 snippet)."""
    rows = []
    with open(os.path.join(GOLDEN, "fuse_worked_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([float(v) for v in line.split()])
    expect = np.array(rows)
    torch.manual_seed(42)
    hs = [torch.randn(10, 64) for _ in range(5)]
    lin = torch.nn.Linear(5 * 64, 64, bias=False)
    got = O.fuse_context([h.numpy() for h in hs], lin.weight.detach().numpy(),
                         np.ones(64), 1e-6, O.f32)
    assert got.shape == (10, 64)
    np.testing.assert_allclose(got[:3, :8], expect, atol=6e-5, rtol=0)


def test_fuse_rms_unit_and_concat_order():
    rng = np.random.default_rng(0)
    hs = [rng.standard_normal((7, 16)) for _ in range(5)]
    Wc = rng.standard_normal((16, 80)) * 0.1
    y = O.fuse_context(hs, Wc, np.ones(16), 1e-6, O.f32)
    # RMS of the output is sqrt(ms / (ms + eps)) for pre-norm mean square ms
    ms = np.mean((np.concatenate(hs, 1) @ Wc.T) ** 2, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, axis=1)), np.sqrt(ms / (ms + 1e-6)),
                               atol=1e-7)
    # a W_c that reads only the 3rd picked layer (columns 2D..3D) reproduces
    # RMSNorm of that layer: the concat is along the hidden axis, ascending
    sel = np.zeros((16, 80))
    sel[:, 32:48] = np.eye(16)
    y = O.fuse_context(hs, sel, np.ones(16), 1e-6, O.f32)
    h = hs[2]
    np.testing.assert_allclose(y, O.f32(h / np.sqrt(np.mean(h * h, 1, keepdims=True) + 1e-6)),
                               atol=1e-6)


def test_wc_sizes():
    # 5 x 2048 x 2048 x 2 B ~ 42 MB for the Qwen3.5-35B-A3B-shaped draft
    s = synth.WORKLOADS["qwen35_a3b_32k"].draft
    assert s.D * s.n_pick * s.D * 2 == 5 * 2048 * 2048 * 2 == 41_943_040
    s = synth.WORKLOADS["qwen3_8b_b1"].draft
    assert s.D * s.n_pick * s.D * 2 == 167_772_160
    # projection activations at batch 1, L = 2048, D = 2048: ~40 MB in, ~8 MB out
    assert 2048 * 5 * 2048 * 2 == 41_943_040 and 2048 * 2048 * 2 == 8_388_608


# --- rmsnorm -------------------------------------------------------------------
def test_rmsnorm_vs_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 33)) * 3
    g = rng.standard_normal(33)
    ref = Fn.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-12)


# --- rope ----------------------------------------------------------------------
def test_rope_complex_form():
    rng = np.random.default_rng(2)
    d, theta = 64, 1e6
    x = rng.standard_normal((9, 3, d))
    pos = rng.integers(0, 40000, size=9)
    got = O.rope(x, pos, theta)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    inv = 1.0 / theta ** (np.arange(0, d, 2) / d)
    z = z * np.exp(1j * pos[:, None, None] * inv[None, None, :])
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag], -1), atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(3)
    d = 128
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    np.testing.assert_allclose(O.rope(q, np.array([0]), 1e6), q, atol=0)
    np.testing.assert_allclose(np.linalg.norm(O.rope(q, np.array([777]), 1e6)),
                               np.linalg.norm(q), rtol=1e-13)
    # <R(p) q, R(p') k> depends only on p - p'
    dots = [float(np.sum(O.rope(q, np.array([p + 5]), 1e6) * O.rope(k, np.array([p]), 1e6)))
            for p in (0, 13, 4096)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# --- attention -----------------------------------------------------------------
@pytest.mark.parametrize("H,G", [(4, 2), (4, 4), (8, 2)])
def test_attention_vs_sdpa(H, G):
    rng = np.random.default_rng(4)
    n, m, d = 8, 72, 64
    q = rng.standard_normal((n, H, d))
    K = rng.standard_normal((m, G, d))
    V = rng.standard_normal((m, G, d))
    got = O.attention(q, K, V)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(H // G, 0)[None]
    tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(H // G, 0)[None]
    ref = Fn.scaled_dot_product_attention(tq, tk, tv)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, atol=1e-12)
    # causal (key j visible to query i iff j <= i + (m - n)) matches is_causal
    vis = np.arange(m)[None, :] <= (np.arange(n)[:, None] + m - n)
    got = O.attention(q, K, V, vis)
    mask = torch.from_numpy(vis)
    ref = Fn.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)[0].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_attention_zero_query_is_mean():
    rng = np.random.default_rng(5)
    V = rng.standard_normal((10, 2, 8))
    out = O.attention(np.zeros((3, 4, 8)), rng.standard_normal((10, 2, 8)), V)
    np.testing.assert_allclose(out[:, 0], np.broadcast_to(V[:, 0].mean(0), (3, 8)), atol=1e-14)
    np.testing.assert_allclose(out[:, 3], np.broadcast_to(V[:, 1].mean(0), (3, 8)), atol=1e-14)


# --- storage rounding ----------------------------------------------------------
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-5, 5, 5000),
                        [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(O.bf16(x), ref.astype(np.float64))


# --- draft layer reductions ------------------------------------------------------
def _tiny_layer(rng, D, H, G, d, F):
    w = lambda *s: rng.standard_normal(s) * 0.05
    return {"wq": w(H * d, D), "wk": w(G * d, D), "wv": w(G * d, D), "wo": w(D, H * d),
            "wg": w(F, D), "wu": w(F, D), "wd": w(D, F), "g_in": np.ones(D),
            "g_post": np.ones(D), "q_norm": np.ones(d), "k_norm": np.ones(d)}


def test_draft_layer_identity_without_outputs():
    rng = np.random.default_rng(7)
    D, H, G, d, F = 32, 4, 2, 8, 48
    lay = _tiny_layer(rng, D, H, G, d, F)
    lay["wo"][:] = 0
    lay["wd"][:] = 0
    x = O.f32(rng.standard_normal((5, D)))
    out = O.draft_layer(x, lay, rng.standard_normal((9, G, d)), rng.standard_normal((9, G, d)),
                        np.arange(9, 14), H, G, d, 1e6, 1e-6, O.f32)
    np.testing.assert_array_equal(out, x)


def test_draft_layer_single_key_grouped_heads():
    """Empty context and a 1-row block: the only key is the row itself, so
    each head's attention output is its group's v (softmax of one score)."""
    rng = np.random.default_rng(8)
    H, G, d = 4, 2, 8
    D = H * d
    F = 40
    lay = _tiny_layer(rng, D, H, G, d, F)
    lay["wv"] = np.eye(G * d, D)           # v = h[:G d]
    lay["wo"] = np.eye(D)                   # attention output added as is
    lay["wg"][:] = 0                        # SiLU(0) = 0: FFN contributes 0
    x = O.f32(rng.standard_normal((1, D)))
    out = O.draft_layer(x, lay, np.zeros((0, G, d)), np.zeros((0, G, d)), np.array([3]),
                        H, G, d, 1e6, 1e-6, O.f32)
    h = O.f32(x / np.sqrt(np.mean(x * x) + 1e-6))
    expect = x.copy()
    for hh in range(H):
        g = hh // (H // G)
        expect[0, hh * d:(hh + 1) * d] += h[0, g * d:(g + 1) * d]
    np.testing.assert_allclose(out, O.f32(expect), atol=1e-6)


def test_draft_layer_zero_query_ignores_context_keys():
    rng = np.random.default_rng(9)
    D, H, G, d, F = 32, 4, 2, 8, 48
    lay = _tiny_layer(rng, D, H, G, d, F)
    lay["wq"][:] = 0
    x = O.f32(rng.standard_normal((3, D)))
    cv = rng.standard_normal((6, G, d))
    a = O.draft_layer(x, lay, rng.standard_normal((6, G, d)), cv, np.arange(6, 9), H, G, d, 1e6, 1e-6)
    b = O.draft_layer(x, lay, rng.standard_normal((6, G, d)), cv, np.arange(6, 9), H, G, d, 1e6, 1e-6)
    np.testing.assert_allclose(a, b, atol=1e-12)


# --- LM head argmax --------------------------------------------------------------
def test_argmax_ties_lowest_and_gap():
    z = np.array([[0.5, 2.0, 2.0, -1.0], [3.0, 1.0, 2.5, 3.0], [0.0, 0.0, 0.0, 0.0],
                  [1.0, 4.0, 3.25, 0.0]])
    np.testing.assert_array_equal(O.argmax_lowest(z), [1, 0, 0, 1])
    np.testing.assert_allclose(O.top2_gap(z), [0.0, 0.0, 0.0, 0.75])
    rng = np.random.default_rng(10)
    z = O.f32(rng.standard_normal((50, 300)))
    z[:, 7] = z.max(1) + 1
    assert (O.argmax_lowest(z) == 7).all()


# --- verification ----------------------------------------------------------------
def _brute_accept(draft, post):
    B = len(draft)
    return max(k for k in range(B) if all(draft[j + 1] == post[j] for j in range(k)))


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_verify_exhaustive(B):
    import itertools
    V = 3
    combos = list(itertools.product(range(V), repeat=B))
    drafts = np.array([c for c in combos for _ in combos])
    posts = np.array([c for _ in combos for c in combos])
    start = np.arange(len(drafts)) % 17
    acc, bon, out, nl = O.verify_greedy(drafts, posts, start)
    for i in range(len(drafts)):
        a = _brute_accept(drafts[i], posts[i])
        assert acc[i] == a
        assert 1 <= a + 1 <= B
        assert bon[i] == posts[i, a]
        assert list(out[i, :a]) == list(drafts[i, 1:a + 1]) and out[i, a] == posts[i, a]
        assert (out[i, a + 1:] == -1).all()
        assert nl[i] == start[i] + a + 1


@pytest.mark.parametrize("p,B,closed", [(0.3, 8, 3.14117), (0.2, 16, 4.85926)])
def test_expected_tau_planted(p, B, closed):
    """E[tau] = sum_k P(prefix_k matches) + 1 under planted Geometric drafts."""
    exact = O.expected_tau_from_prefix([(1 - p) ** k for k in range(1, B)])
    assert abs(exact - closed) < 1e-5
    n = 100_000
    rng = np.random.default_rng(11)
    draft = rng.integers(0, 50, size=(n, B)).astype(np.int32)
    post, k = synth.planted_posterior(draft, p, 50, seed=12)
    acc, _, _, _ = O.verify_greedy(draft, post, np.zeros(n, dtype=np.int32))
    assert (acc == k).all()
    tau = acc + 1
    assert tau.min() >= 1 and tau.max() <= B
    assert abs(tau.mean() - exact) < 4 * tau.std() / math.sqrt(n)
