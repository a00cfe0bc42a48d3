"""The allocation-free LM-head argmax (dflash_lm_head_argmax_noalloc).

Some callers cannot give the library device memory when they call it — a
serving loop whose memory is entirely reserved up front by its own pool, or
a latency-critical path that must not call cudaMalloc.  The allocation-free
entry point serves them from a fixed internal scratch array.  This file is
collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.

Both entry points run the same kernels on the same inputs, so their ids and
gaps must be identical bit for bit; the results must also match the oracle
(ids bit-exact outside top-2 gaps under 1e-3, gaps within 2e-2).  Calls of
two handles of different hidden and vocabulary sizes alternate, so a call
after a larger one finds the shared array holding the larger call's data."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import NEAR_TIE, to_np

pytestmark = pytest.mark.gpu

SMALL = synth.with_(synth.WORKLOADS["tiny_f32"], dtype="bf16")            # D 256, V 1024
LARGE = synth.Workload(                                                    # D 2048, V 40000
    name="noalloc_large", dtype="bf16",
    draft=synth.DraftShape(n_layers=1, D=2048, H=16, G=4, d=128, F=512, V=40000, mask_id=39999,
                           n_target_layers=12),
    batch=1, B=16, ctx_len=0, seed=1011)


def _model(w):
    from synth.gpu import draft_model
    weights = synth.draft_weights(w.draft, w.dtype, w.seed, device="cuda")
    return draft_model(w.draft, w.dtype, weights, max_pos=64), weights


@pytest.fixture(scope="module")
def models(dfl):
    made = {w.name: _model(w) for w in (SMALL, LARGE)}
    yield made
    for m, _ in made.values():
        m.close()


def _rows(w, rows, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, w.draft.D, generator=g) *
            torch.exp(torch.randn(rows, 1, generator=g))).cuda()


def _with_workspace(dfl, m, weights, x, rows):
    ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    gap = torch.full((rows,), -1.0, device="cuda")
    dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids, gap, m.workspace(rows))
    assert dfl.dflash_get_status(m.handle) == 0
    return ids.cpu().numpy(), gap.cpu().numpy()


def _noalloc(dfl, m, weights, x, rows):
    ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    gap = torch.full((rows,), -1.0, device="cuda")
    dfl.dflash_lm_head_argmax_noalloc(m.handle, x, rows, weights["g_f"], ids, gap)
    assert dfl.dflash_get_status(m.handle) == 0
    return ids.cpu().numpy(), gap.cpu().numpy()


def _oracle_check(w, weights, x, ids, gap, label):
    hf = O.bf16(O.rmsnorm(x.double().cpu().numpy(), to_np(weights["g_f"]), w.draft.eps))
    z = O.lm_head_logits(hf, to_np(weights["lm_head"]))
    oids, ogap = O.argmax_lowest(z), O.top2_gap(z)
    near = ogap < NEAR_TIE
    bad = int(((ids != oids) & ~near).sum())
    err = float(np.abs(gap - ogap).max())
    print(f"{label}: ids {len(ids)}, mismatches outside near-ties {bad}, near-ties "
          f"{int(near.sum())}; gap max|err| {err:.3e}")
    assert bad == 0 and err <= 2e-2


def test_noalloc_matches_workspace_entry_point_and_oracle(dfl, models):
    """Two calls in a row on one handle, then calls of a second handle with a
    larger hidden size and vocabulary between calls of the first."""
    cases = [(SMALL, 15, 5), (SMALL, 16, 6), (LARGE, 16, 7), (SMALL, 9, 8), (LARGE, 3, 9),
             (SMALL, 15, 5)]
    for w, rows, seed in cases:
        m, weights = models[w.name]
        x = _rows(w, rows, seed)
        ref_ids, ref_gap = _with_workspace(dfl, m, weights, x, rows)
        ids, gap = _noalloc(dfl, m, weights, x, rows)
        np.testing.assert_array_equal(ids, ref_ids)
        np.testing.assert_array_equal(gap, ref_gap)
        _oracle_check(w, weights, x, ids, gap, f"{w.name} {rows} rows")


def test_noalloc_rejects_sizes_beyond_its_limit(dfl, models):
    m, weights = models[SMALL.name]
    x = torch.zeros(17, SMALL.draft.D, device="cuda")
    ids = torch.empty(17, dtype=torch.int32, device="cuda")
    with pytest.raises(dfl.DFlashError) as e:
        dfl.dflash_lm_head_argmax_noalloc(m.handle, x, 17, weights["g_f"], ids, None)
    assert e.value.code == 10
