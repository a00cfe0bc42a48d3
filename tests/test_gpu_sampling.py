"""Sampling at T > 0 on the GPU vs the oracle: per-row softmax with
inverse-CDF draws, rejection verification, the LM-head logits, the draft
block without its LM head, and the sampling loop end to end.

Draws are integers decided by floating point: both sides take them on the
same fp32 inputs, with fp64 running sums.  The GPU's exponentials are fp32,
the oracle's fp64, so a draw may differ only where u * total falls within
that rounding of a CDF boundary; such draws are counted and must be rare."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import float_parity, to_np, to_np64

pytestmark = pytest.mark.gpu

BOUNDARY = 1e-6   # relative distance of u * total from a CDF boundary that may flip a draw


def _handle(dfl, wname="tiny_f32"):
    from synth.gpu import draft_model
    w = synth.WORKLOADS[wname]
    weights = synth.draft_weights(w.draft, w.dtype, w.seed, device="cuda")
    return w, weights, draft_model(w.draft, w.dtype, weights, max_pos=64)


def _near_boundary(weights, u, a, b):
    """True when u * total lies within BOUNDARY * total of a running sum that
    separates indices a and b (the two candidate draws)."""
    c = np.cumsum(np.asarray(weights, np.float64))
    t = u * c[-1]
    lo, hi = min(a, b), max(a, b)
    return bool(np.any(np.abs(c[lo:hi] - t) <= BOUNDARY * c[-1]))


@pytest.mark.parametrize("V,T,skip", [(1024, 1.0, 0), (151936, 1.0, 16), (2048, 0.5, 0),
                                      (4096, 2.0, 5)])
def test_sample_rows_matches_oracle(dfl, V, T, skip):
    """skip > 1: the draws land in the draft slots of [batch, skip] blocks
    (slot 0, the anchor, untouched)."""
    _, _, m = _handle(dfl)
    rng = np.random.default_rng(V + int(10 * T))
    rows = 24 if skip != 16 else 30
    z = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    u = rng.random(rows)
    dev = "cuda"
    n_ids = rows if skip < 2 else rows // (skip - 1) * skip
    ids = torch.full((n_ids,), -1, dtype=torch.int32, device=dev)
    probs = torch.empty(rows, V, device=dev)
    dfl.dflash_sample_rows(m.handle, torch.from_numpy(z).to(dev), rows, V, T,
                           torch.from_numpy(u).to(dev), ids, probs, ids_skip_first_of=skip)
    assert dfl.dflash_get_status(m.handle) == 0
    p = O.softmax_t(z, T)
    np.testing.assert_allclose(probs.cpu().numpy(), p, rtol=2e-5, atol=1e-12)
    # in place (probs is the logits buffer): the same bits and draws
    zin = torch.from_numpy(z).to(dev)
    ids2 = torch.full_like(ids, -1)
    dfl.dflash_sample_rows(m.handle, zin, rows, V, T, torch.from_numpy(u).to(dev), ids2, zin,
                           ids_skip_first_of=skip)
    assert torch.equal(zin, probs) and torch.equal(ids2, ids)
    got = ids.cpu().numpy()
    if skip > 1:
        blk = got.reshape(-1, skip)
        assert (blk[:, 0] == -1).all()
        got = blk[:, 1:].reshape(-1)
    want = np.array([O.sample_from(p[r], u[r]) for r in range(rows)])
    flips = [r for r in range(rows) if got[r] != want[r]]
    assert all(_near_boundary(p[r], u[r], got[r], want[r]) for r in flips), flips
    print(f"V={V} T={T}: {rows} draws, {len(flips)} at a CDF boundary")
    assert len(flips) <= 1
    m.close()


def _pq(rng, batch, B, V, spread):
    zq = rng.standard_normal((batch, B - 1, V)) * 2
    zp = np.concatenate([zq, rng.standard_normal((batch, 1, V)) * 2], axis=1)
    zp = zp + rng.standard_normal(zp.shape) * spread
    # both sides verify the same fp32 distributions
    q = O.softmax_t(zq, 1.0).astype(np.float32)
    p = O.softmax_t(zp, 1.0).astype(np.float32)
    return q, p


@pytest.mark.parametrize("V,B,batch,spread", [(1024, 8, 3, 0.3), (151936, 16, 1, 0.05),
                                              (4096, 16, 4, 0.1), (2048, 4, 5, 0.0)])
def test_verify_rejection_matches_oracle(dfl, V, B, batch, spread):
    """Drafts drawn from q; p a perturbed q (spread 0: p equals q on the
    draft positions, so every draft is accepted)."""
    _, _, m = _handle(dfl)
    dev = "cuda"
    rng = np.random.default_rng(V + B)
    flips, accepted = 0, []
    for trial in range(6):
        q, p = _pq(rng, batch, B, V, spread)
        draft = np.zeros((batch, B), dtype=np.int32)
        draft[:, 0] = rng.integers(0, V, batch)
        for b in range(batch):
            for j in range(1, B):
                draft[b, j] = O.sample_from(q[b, j - 1], rng.random())
        u_acc, u_smp = rng.random((batch, B - 1)), rng.random(batch)
        start = rng.integers(0, 100, batch).astype(np.int32)
        t = lambda a, dt=None: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        acc = torch.empty(batch, dtype=torch.int32, device=dev)
        tau = torch.empty(batch, dtype=torch.int32, device=dev)
        tok = torch.empty(batch, dtype=torch.int32, device=dev)
        out = torch.empty(batch, B, dtype=torch.int32, device=dev)
        nl = torch.empty(batch, dtype=torch.int32, device=dev)
        dfl.dflash_verify_rejection(m.handle, t(draft), t(q), t(p), V, t(u_acc), t(u_smp), batch,
                                    B, t(start), acc, tau, tok, out, nl)
        assert dfl.dflash_get_status(m.handle) == 0
        oa, ot, oo, on = O.verify_rejection(draft, q.astype(np.float64), p.astype(np.float64),
                                            u_acc, u_smp, start)
        # acceptance is decided on identical fp32 values in fp64: exact
        np.testing.assert_array_equal(acc.cpu().numpy(), oa)
        np.testing.assert_array_equal(nl.cpu().numpy(), on)
        np.testing.assert_array_equal(tau.cpu().numpy(), oa + 1)
        g_tok, g_out = tok.cpu().numpy(), out.cpu().numpy()
        for b in range(batch):
            a = oa[b]
            np.testing.assert_array_equal(g_out[b, :a], oo[b, :a])
            assert (g_out[b, a + 1:] == -1).all()
            if g_tok[b] != ot[b]:
                w = (np.maximum(p[b, a].astype(np.float64) - q[b, a], 0.0) if a < B - 1
                     else p[b, B - 1].astype(np.float64))
                assert _near_boundary(w, u_smp[b], g_tok[b], ot[b])
                flips += 1
            assert g_out[b, a] == g_tok[b]
        accepted += list(oa)
    print(f"V={V} B={B}: accepted counts {accepted}, {flips} draws at a CDF boundary")
    assert flips <= 1
    if spread == 0.0:
        assert all(a == B - 1 for a in accepted)
    m.close()


@pytest.mark.parametrize("wname,skip", [("tiny_f32", 0), ("tiny_f32", 8), ("qwen3_8b_b1", 16)])
def test_lm_head_logits(dfl, wname, skip):
    w, weights, m = _handle(dfl, wname)
    s = w.draft
    dev = "cuda"
    rows_in = 32
    x = torch.randn(rows_in, s.D, generator=torch.Generator().manual_seed(5)).to(dev)
    keep = [r for r in range(rows_in) if not skip or r % skip != 0]
    logits = torch.empty(len(keep), s.V, device=dev)
    ws = m.workspace(rows_in)
    dfl.dflash_lm_head_logits(m.handle, x, len(keep), weights["g_f"], logits, ws,
                              skip_first_of=skip)
    assert dfl.dflash_get_status(m.handle) == 0
    st = O.storage(w.dtype)
    hf = st(O.rmsnorm(x.cpu().numpy()[keep].astype(np.float64), to_np64(weights)["g_f"], s.eps))
    ref = O.lm_head_logits(hf, to_np(weights["lm_head"]))
    err, _ = float_parity(logits.cpu().numpy(), ref, w.dtype, f"{wname} logits")
    print(f"{wname} skip={skip}: logits max|err| {err:.3e}")
    m.close()


def test_draft_block_residual_only(dfl):
    """draft_ids = NULL: the LM head is skipped and the residual equals the
    one the full call returns (the persistent launch without its LM-head
    phases, and the multi-launch path)."""
    from synth.gpu import draft_model, kv_cache
    w = synth.WORKLOADS["qwen3_8b_b1"]
    s = w.draft
    dev = "cuda"
    weights = synth.draft_weights(s, w.dtype, w.seed, device=dev)
    m = draft_model(s, w.dtype, weights, max_pos=600)
    for batch, B, L in [(1, 16, 300), (2, 16, 200)]:   # one launch; 32 rows: the launches
        K, V = synth.random_kv_cache(batch, s.G, L + 8, s.d, s.n_layers, 1.3, w.dtype, w.seed,
                                     device=dev)
        kv = kv_cache(s, batch, L + 8, w.dtype, k=K, v=V)
        kv.len.fill_(L)
        a = torch.from_numpy(synth.anchors(batch, s.V, s.mask_id, 3)).to(dev)
        ws = m.workspace(batch * B, max_batch=batch, max_block=B)
        h1 = torch.empty(batch * B, s.D, device=dev)
        h2 = torch.empty(batch * B, s.D, device=dev)
        ids = torch.empty(batch, B, dtype=torch.int32, device=dev)
        dfl.dflash_draft_block(m.handle, a, batch, B, kv.struct, ids, None, h1, ws)
        dfl.dflash_draft_block(m.handle, a, batch, B, kv.struct, None, None, h2, ws)
        assert dfl.dflash_get_status(m.handle) == 0
        assert torch.equal(h1, h2)
    m.close()


def test_e2e_sampling_loop_matches_oracle(dfl):
    """The sampling loop (T = 1) on the GPU and the oracle's, consuming the
    same seeded uniforms: the same tokens and taus."""
    from synth.gpu import draft_model, spec_decoder, target_model
    from test_gpu_e2e import _upload, _weights
    w = synth.WORKLOADS["e2e_f32"]
    TWn, DWn = _weights(w)
    TW, DW = _upload(TWn), _upload(DWn)
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    n_new, T = 24, 1.0
    cap = w.prompt_len + n_new + 2 * w.B
    target = target_model(w.target, w.dtype, TW, max_pos=cap)
    draft = draft_model(w.draft, w.dtype, DW, max_pos=cap)
    dec = spec_decoder(w, target, draft, cap=cap)
    prompt = synth.random_ids(w.prompt_len, w.target.V, seed=w.seed).tolist()
    uni = synth.round_uniforms(11, w.B)
    toks, taus = dec.generate_sampled(prompt, n_new, T, uni)
    assert dfl.dflash_get_status(target.handle) == 0
    assert dfl.dflash_get_status(draft.handle) == 0
    ref, rtaus = O.speculative_sample_generate(w.target, to_np64(TWn), w.draft, to_np64(DWn),
                                               prompt, n_new, w.B, T, uni)
    print(f"sampling loop: rounds {len(taus)}, taus {taus}")
    np.testing.assert_array_equal(np.array(toks), ref)
    assert taus == rtaus
    target.close()
    draft.close()


def _chi2_ok(counts, probs, label, alpha=1e-5):
    """Pearson chi-squared of observed counts against n * probs: bins of zero
    probability must stay empty, and the p-value of the rest exceed alpha."""
    stats = pytest.importorskip("scipy.stats")
    counts, probs = np.asarray(counts, np.float64), np.asarray(probs, np.float64)
    n = counts.sum()
    zero = probs == 0
    assert counts[zero].sum() == 0, f"{label}: drew a token of zero probability"
    e = n * probs[~zero]
    x2 = float(((counts[~zero] - e) ** 2 / e).sum())
    pv = float(stats.chi2.sf(x2, int((~zero).sum()) - 1))
    print(f"{label}: n={int(n)} chi2={x2:.1f} p={pv:.3g}")
    assert pv > alpha, label


def _dist(rng, V, zeros):
    w = rng.gamma(0.7, size=V)
    w[zeros] = 0.0
    return (w / w.sum()).astype(np.float32)


def test_verify_rejection_is_lossless_chi2(dfl):
    """The speculative-sampling guarantee on the GPU verifier: with draft
    tokens drawn from q_j, the token emitted at block position j (whenever
    the round reaches it) is distributed as the target's p_j, whatever q is.
    p and q are fixed per position (so the target's next-token law does not
    depend on the earlier tokens) and each has tokens of zero probability
    the other favours.  Also the acceptance rate of the first draft equals
    sum_x min(p_0, q_0)."""
    _, _, m = _handle(dfl)
    dev = "cuda"
    rng = np.random.default_rng(2024)
    V, B, n = 12, 4, 60000
    p = np.stack([_dist(rng, V, [j % V, 5]) for j in range(B)])
    q = np.stack([_dist(rng, V, [(j + 3) % V]) for j in range(B - 1)])
    cq = np.cumsum(q.astype(np.float64), axis=1)
    draft = np.zeros((n, B), dtype=np.int32)
    draft[:, 0] = rng.integers(0, V, n)
    for j in range(1, B):   # d_j drawn from q_{j-1} by inverse CDF
        t = rng.random(n) * cq[j - 1, -1]
        draft[:, j] = np.minimum(np.searchsorted(cq[j - 1], t, side="right"), V - 1)
    qq = np.ascontiguousarray(np.broadcast_to(q, (n, B - 1, V)))
    pp = np.ascontiguousarray(np.broadcast_to(p, (n, B, V)))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    u_acc, u_smp = rng.random((n, B - 1)), rng.random(n)
    start = np.zeros(n, dtype=np.int32)
    acc = torch.empty(n, dtype=torch.int32, device=dev)
    out = torch.empty(n, B, dtype=torch.int32, device=dev)
    dfl.dflash_verify_rejection(m.handle, t(draft), t(qq), t(pp), V, t(u_acc), t(u_smp), n, B,
                                t(start), acc, None, None, out, None)
    assert dfl.dflash_get_status(m.handle) == 0
    out, acc = out.cpu().numpy(), acc.cpu().numpy()
    for j in range(B):
        col = out[:, j]
        col = col[col >= 0]
        assert len(col) == (acc >= j).sum()
        _chi2_ok(np.bincount(col, minlength=V), p[j], f"position {j}")
    r = float(np.minimum(p[0].astype(np.float64), q[0]).sum())
    z = ((acc >= 1).mean() - r) / np.sqrt(r * (1 - r) / n)
    print(f"first-draft acceptance {(acc >= 1).mean():.4f} vs {r:.4f} (z = {z:.2f})")
    assert abs(z) < 5
    m.close()


def test_sample_rows_chi2(dfl):
    """Draws from one row's softmax(z / T) (T = 0.7) with independent
    uniforms follow that distribution."""
    _, _, m = _handle(dfl)
    dev = "cuda"
    rng = np.random.default_rng(7)
    V, n, T = 24, 60000, 0.7
    z = (rng.standard_normal(V) * 1.5).astype(np.float32)
    zz = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(z, (n, V)))).to(dev)
    ids = torch.empty(n, dtype=torch.int32, device=dev)
    dfl.dflash_sample_rows(m.handle, zz, n, V, T, torch.from_numpy(rng.random(n)).to(dev), ids)
    assert dfl.dflash_get_status(m.handle) == 0
    _chi2_ok(np.bincount(ids.cpu().numpy(), minlength=V), O.softmax_t(z, T), "softmax draws")
    m.close()


def test_verify_rejection_zero_residual(dfl):
    """p_a == q_a and a draft of zero probability under both: the draft is
    rejected (u * 0 < 0 fails), the residual max(p - q, 0) is all zero, and
    the token is drawn from p_a itself; also a draft id out of range fails
    its test and sets the status word."""
    _, _, m = _handle(dfl)
    dev = "cuda"
    rng = np.random.default_rng(99)
    V, B, batch = 5000, 4, 3
    q = O.softmax_t(rng.standard_normal((batch, B - 1, V)) * 2, 1.0).astype(np.float32)
    p = np.concatenate([q, O.softmax_t(rng.standard_normal((batch, 1, V)), 1.0)
                        .astype(np.float32)], axis=1)
    draft = np.zeros((batch, B), dtype=np.int32)
    for b in range(batch):
        for j in range(1, B):
            draft[b, j] = O.sample_from(q[b, j - 1], rng.random())
    for b, j in [(0, 1), (1, 2)]:   # rejection at position j-1, p == q there
        z = int(draft[b, j])
        q[b, j - 1, z] = p[b, j - 1, z] = 0.0
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    u_acc, u_smp = rng.random((batch, B - 1)), rng.random(batch)
    start = np.full(batch, 7, dtype=np.int32)
    acc = torch.empty(batch, dtype=torch.int32, device=dev)
    tok = torch.empty(batch, dtype=torch.int32, device=dev)
    out = torch.empty(batch, B, dtype=torch.int32, device=dev)
    dfl.dflash_verify_rejection(m.handle, t(draft), t(q), t(p), V, t(u_acc), t(u_smp), batch, B,
                                t(start), acc, None, tok, out, None)
    assert dfl.dflash_get_status(m.handle) == 0
    oa, ot, oo, _ = O.verify_rejection(draft, q.astype(np.float64), p.astype(np.float64), u_acc,
                                       u_smp, start)
    assert list(oa[:2]) == [0, 1] and oa[2] == B - 1
    np.testing.assert_array_equal(acc.cpu().numpy(), oa)
    np.testing.assert_array_equal(tok.cpu().numpy(), ot)
    np.testing.assert_array_equal(out.cpu().numpy(), oo)
    # an out-of-range draft id: rejected there, ST_BOUNDS reported
    draft[2, 2] = V + 3
    dfl.dflash_verify_rejection(m.handle, t(draft), t(q), t(p), V, t(u_acc), t(u_smp), batch, B,
                                t(start), acc, None, tok, out, None)
    assert acc.cpu().numpy()[2] == 1
    assert dfl.dflash_get_status(m.handle) == 8   # DFLASH_ERR_DEVICE_BOUNDS
    m.close()
