"""Greedy verification on the GPU vs the oracle: bit-exact integers."""
import itertools

import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu


def run_verify(dfl, draft, post, start, alias_new_len=False):
    dev = "cuda"
    batch, B = draft.shape
    d = torch.from_numpy(np.ascontiguousarray(draft)).to(dev)
    p = torch.from_numpy(np.ascontiguousarray(post)).to(dev)
    st = torch.from_numpy(np.ascontiguousarray(start.astype(np.int32))).to(dev)
    acc = torch.full((batch,), -7, dtype=torch.int32, device=dev)
    tau = torch.full((batch,), -7, dtype=torch.int32, device=dev)
    bon = torch.full((batch,), -7, dtype=torch.int32, device=dev)
    out = torch.full((batch, B), -7, dtype=torch.int32, device=dev)
    nl = st if alias_new_len else torch.full((batch,), -7, dtype=torch.int32, device=dev)
    dfl.dflash_verify_greedy(d, p, batch, B, st, acc, tau, bon, out, nl)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (acc, tau, bon, out, nl)]


def check(dfl, draft, post, start, alias=False):
    acc, tau, bon, out, nl = run_verify(dfl, draft, post, start, alias)
    ra, rb, ro, rn = O.verify_greedy(draft, post, start)
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(bon, rb)
    np.testing.assert_array_equal(out, ro)
    np.testing.assert_array_equal(nl, rn)
    np.testing.assert_array_equal(tau, ra + 1)
    assert tau.min() >= 1 and tau.max() <= draft.shape[1]
    return acc


@pytest.mark.parametrize("wname", ["tiny_f32", "qwen3_8b_b32_ragged", "qwen35_a3b_32k"])
def test_verify_planted_geometric(dfl, wname):
    w = synth.WORKLOADS[wname]
    n = 4096
    draft = synth.random_ids((n, w.B), w.draft.V, seed=w.seed)
    post, k = synth.planted_posterior(draft, w.geom_p, w.draft.V, seed=w.seed + 1)
    start = synth.random_ids((n,), 30000, seed=w.seed + 2)
    acc = check(dfl, draft, post, start)
    np.testing.assert_array_equal(acc, k)          # planted prefix recovered exactly
    # mean tau against E[tau] = 1 + sum_k (1-p)^k, within 4 sigma
    exact = O.expected_tau_from_prefix([(1 - w.geom_p) ** j for j in range(1, w.B)])
    tau = acc + 1
    assert abs(tau.mean() - exact) < 4 * tau.std() / np.sqrt(n) + 1e-9


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_verify_exhaustive(dfl, B):
    combos = list(itertools.product(range(3), repeat=B))
    draft = np.array([c for c in combos for _ in combos], dtype=np.int32)
    post = np.array([c for _ in combos for c in combos], dtype=np.int32)
    start = (np.arange(len(draft)) % 23).astype(np.int32)
    check(dfl, draft, post, start)


def test_verify_trim_in_place(dfl):
    w = synth.WORKLOADS["qwen3_8b_b32_ragged"]
    draft = synth.random_ids((32, 16), w.draft.V, seed=5)
    post, _ = synth.planted_posterior(draft, 0.2, w.draft.V, seed=6)
    start = np.array(synth.ctx_lengths(w), dtype=np.int32)
    check(dfl, draft, post, start, alias=True)


def test_verify_all_accept_and_all_reject(dfl):
    V, B = 1000, 16
    draft = synth.random_ids((64, B), V, seed=9)
    post = np.zeros_like(draft)
    post[:32, :B - 1] = draft[:32, 1:]          # every draft matches: a = B-1
    post[32:, 0] = (draft[32:, 1] + 1) % V       # first draft rejected: a = 0
    acc = check(dfl, draft, post, np.zeros(64, dtype=np.int32))
    assert (acc[:32] == B - 1).all() and (acc[32:] == 0).all()


def test_verify_empty_batch(dfl):
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    dfl.dflash_verify_greedy(z, z, 0, 4, z, z, None, z, z, None)
    torch.cuda.synchronize()
