"""End-to-end greedy speculative loop on the GPU (fp32): losslessness.

The loop's output must equal the oracle target's own greedy autoregressive
output, token for token; the GPU's own autoregressive decode (one row per
forward) must agree too, which checks that the kernels are row-invariant."""
import collections
import time

import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import make_all_accept, make_partial_accept, to_np, to_np64

pytestmark = pytest.mark.gpu


def _upload(obj, dev="cuda"):
    if isinstance(obj, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(obj)).to(dev)
    if isinstance(obj, dict):
        return {k: _upload(v, dev) for k, v in obj.items()}
    if isinstance(obj, list):
        return [_upload(v, dev) for v in obj]
    return obj


def _run(dfl, w, TWn, DWn, prompt, n_new):
    from synth.gpu import draft_model, spec_decoder, target_model
    TW, DW = _upload(TWn), _upload(DWn)
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    cap = w.prompt_len + n_new + 2 * w.B
    target = target_model(w.target, w.dtype, TW, max_pos=cap)
    draft = draft_model(w.draft, w.dtype, DW, max_pos=cap)
    dec = spec_decoder(w, target, draft, cap=cap)
    spec, taus = dec.generate(prompt, n_new)
    ar = dec.ar_decode(prompt, n_new)
    assert dfl.dflash_get_status(target.handle) == 0
    assert dfl.dflash_get_status(draft.handle) == 0
    target.close()
    draft.close()
    return np.array(spec), np.array(ar), taus


def _weights(w):
    TW = to_np(synth.target_weights(w.target, w.dtype, w.seed))
    DW = to_np(synth.draft_weights(w.draft, w.dtype, w.seed + 1,
                                   shared={"embed": None, "lm_head": None}))
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    return TW, DW


def test_e2e_lossless_256_tokens(dfl):
    w = synth.WORKLOADS["e2e_f32"]
    TW, DW = _weights(w)
    prompt = synth.random_ids(w.prompt_len, w.target.V, seed=w.seed).tolist()
    spec, ar_gpu, taus = _run(dfl, w, TW, DW, prompt, w.new_tokens)
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    ref, ref_taus = O.speculative_generate(w.target, to_np64(TW), w.draft, to_np64(DW), prompt,
                                           w.new_tokens, w.B)
    hist = collections.Counter(taus)
    print(f"e2e: rounds {len(taus)}, mean tau {np.mean(taus):.3f}, "
          f"tau histogram {dict(sorted(hist.items()))}")
    np.testing.assert_array_equal(ar_gpu, ar_ref)
    np.testing.assert_array_equal(spec, ar_ref)
    np.testing.assert_array_equal(ref, ar_ref)
    assert list(taus) == list(ref_taus)
    assert all(1 <= t <= w.B for t in taus)


def test_e2e_partial_acceptance(dfl):
    """A planted greedy cycle that the draft matches one step at a time:
    rounds accept one draft (tau = 2 of B = 16: the target cache is trimmed
    inside the verified block and two rows carry over) or none.  Tokens equal
    the oracle target's greedy decode, and the tau sequence equals the
    oracle loop's, on the host-synchronised and the device-resident loops."""
    from synth.gpu import draft_model, spec_decoder, target_model
    w = synth.with_(synth.WORKLOADS["e2e_f32"], new_tokens=120)
    TW, DW = _weights(w)
    cycle = [11, 222, 3333, 444, 55, 666, 7]
    TW, DW = make_partial_accept(TW, DW, w.target, cycle, m_index=2)
    prompt = synth.random_ids(w.prompt_len - 1, w.target.V, seed=3).tolist() + [cycle[0]]
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    ref, ref_taus = O.speculative_generate(w.target, to_np64(TW), w.draft, to_np64(DW), prompt,
                                           w.new_tokens, w.B)
    np.testing.assert_array_equal(ref, ar_ref)
    assert 2 in ref_taus and 1 in ref_taus and max(ref_taus) == 2
    Tg, Dg = _upload(TW), _upload(DW)
    Dg["embed"], Dg["lm_head"] = Tg["embed"], Tg["lm_head"]
    cap = w.prompt_len + w.new_tokens + 12 * w.B
    target = target_model(w.target, w.dtype, Tg, max_pos=cap)
    draft = draft_model(w.draft, w.dtype, Dg, max_pos=cap)
    dec = spec_decoder(w, target, draft, cap=cap)
    spec, taus = dec.generate(prompt, w.new_tokens)
    res, res_taus = dec.generate_resident(prompt, w.new_tokens)
    assert dfl.dflash_get_status(target.handle) == 0
    assert dfl.dflash_get_status(draft.handle) == 0
    target.close()
    draft.close()
    print(f"partial acceptance: {len(taus)} rounds, tau histogram "
          f"{dict(sorted(collections.Counter(taus).items()))}")
    np.testing.assert_array_equal(np.array(spec), ar_ref)
    np.testing.assert_array_equal(np.array(res)[:w.new_tokens], ar_ref)
    assert list(taus) == list(ref_taus)
    assert list(res_taus)[:len(ref_taus)] == list(ref_taus)


def test_e2e_lossless_all_blocks_accepted(dfl):
    """Every draft accepted (tau = B each round): exercises long accepted
    prefixes, the cache trim and multi-row context injection per round."""
    w = synth.with_(synth.WORKLOADS["e2e_f32"], new_tokens=96)
    TW, DW = _weights(w)
    c = 77
    TW, DW = make_all_accept(TW, DW, w.target, c)
    prompt = synth.random_ids(w.prompt_len - 1, w.target.V, seed=2).tolist() + [c]
    spec, ar_gpu, taus = _run(dfl, w, TW, DW, prompt, w.new_tokens)
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    np.testing.assert_array_equal(spec, ar_ref)
    np.testing.assert_array_equal(ar_gpu, ar_ref)
    assert taus == [w.B] * len(taus)


def _run_both(dfl, w, TWn, DWn, prompt, n_new, **kw):
    """The host-synchronised loop and the device-resident loop on the same
    models, each timed (after a warm-up of both)."""
    from synth.gpu import draft_model, spec_decoder, target_model
    TW, DW = _upload(TWn), _upload(DWn)
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    cap = w.prompt_len + n_new + 12 * w.B
    target = target_model(w.target, w.dtype, TW, max_pos=cap)
    draft = draft_model(w.draft, w.dtype, DW, max_pos=cap)
    dec = spec_decoder(w, target, draft, cap=cap)
    dec.generate(prompt, 8)
    dec.generate_resident(prompt, 8, **kw)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    host, host_taus = dec.generate(prompt, n_new)
    t1 = time.perf_counter()
    res, res_taus = dec.generate_resident(prompt, n_new, **kw)
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    assert dfl.dflash_get_status(target.handle) == 0
    assert dfl.dflash_get_status(draft.handle) == 0
    print(f"host-synchronised loop {n_new / (t1 - t0):.0f} tokens/s ({len(host_taus)} rounds), "
          f"device-resident loop {n_new / (t2 - t1):.0f} tokens/s ({len(res_taus)} rounds, {kw})")
    target.close()
    draft.close()
    return np.array(host), host_taus, np.array(res), res_taus


def test_e2e_resident_loop_matches_host_loop(dfl):
    """Device-resident rounds (dflash_draft_round, state on the device, a
    host read every 4 rounds): the same tokens and the same tau per round as
    the host-synchronised loop, and lossless."""
    w = synth.WORKLOADS["e2e_f32"]
    TW, DW = _weights(w)
    prompt = synth.random_ids(w.prompt_len, w.target.V, seed=w.seed).tolist()
    host, host_taus, res, res_taus = _run_both(dfl, w, TW, DW, prompt, w.new_tokens,
                                               check_every=4)
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    np.testing.assert_array_equal(host, ar_ref)
    np.testing.assert_array_equal(res, ar_ref)
    # the resident loop may run a few rounds past the end before its check
    assert res_taus[:len(host_taus)] == host_taus
    assert all(1 <= t <= w.B for t in res_taus)


def test_e2e_resident_loop_block_schedule(dfl):
    """Block sizes scheduled between 8 and 16 from the last window's taus:
    still the target's own greedy output (any B is lossless)."""
    w = synth.WORKLOADS["e2e_f32"]
    TW, DW = _weights(w)
    prompt = synth.random_ids(w.prompt_len, w.target.V, seed=w.seed + 5).tolist()
    _, _, res, res_taus = _run_both(dfl, w, TW, DW, prompt, w.new_tokens, check_every=4,
                                    block_sizes=(8, 16))
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    np.testing.assert_array_equal(res, ar_ref)
    hist = collections.Counter(res_taus)
    print(f"scheduled blocks: rounds {len(res_taus)}, tau histogram {dict(sorted(hist.items()))}")
    # short accepted prefixes move the schedule to 8-row blocks after the first window
    if max(res_taus[:4]) < 8:
        assert max(res_taus[4:8]) <= 8


def test_e2e_resident_loop_all_accepted(dfl):
    """Every draft accepted: tau = B every round, and the schedule stays at
    the largest block."""
    w = synth.with_(synth.WORKLOADS["e2e_f32"], new_tokens=96)
    TW, DW = _weights(w)
    c = 77
    TW, DW = make_all_accept(TW, DW, w.target, c)
    prompt = synth.random_ids(w.prompt_len - 1, w.target.V, seed=2).tolist() + [c]
    _, _, res, res_taus = _run_both(dfl, w, TW, DW, prompt, w.new_tokens, check_every=2,
                                    block_sizes=(8, 16))
    ar_ref = O.ar_generate(w.target, to_np64(TW), prompt, w.new_tokens)
    np.testing.assert_array_equal(res, ar_ref)
    assert res_taus == [w.B] * len(res_taus)


def test_e2e_selected_loop(dfl):
    """The greedy loop with DFlash 2 candidate selection: the GPU's tokens
    and taus equal the oracle's selected loop, and the tokens are the
    target's own greedy output (lossless whatever the drafts)."""
    from synth.gpu import draft_model, spec_decoder, target_model
    w = synth.WORKLOADS["e2e_f32"]
    TWn, DWn = _weights(w)
    TW, DW = _upload(TWn), _upload(DWn)
    DW["embed"], DW["lm_head"] = TW["embed"], TW["lm_head"]
    n_new = 40
    cap = w.prompt_len + n_new + 2 * w.B
    target = target_model(w.target, w.dtype, TW, max_pos=cap)
    draft = draft_model(w.draft, w.dtype, DW, max_pos=cap)
    dec = spec_decoder(w, target, draft, cap=cap)
    sel = synth.selector_weights(w.draft.D, w.draft.V, "f32", 13, rank=64, device="cuda")
    sel["top_k"] = 16
    prompt = synth.random_ids(w.prompt_len, w.target.V, seed=w.seed).tolist()
    toks, taus = dec.generate(prompt, n_new, selector=sel)
    assert dfl.dflash_get_status(draft.handle) == 0
    sel_np = to_np64({k: v for k, v in sel.items() if k != "top_k"})
    sel_np["top_k"] = 16
    ref, rtaus = O.speculative_generate(w.target, to_np64(TWn), w.draft, to_np64(DWn), prompt,
                                        n_new, w.B, selector=sel_np)
    ar = O.ar_generate(w.target, to_np64(TWn), prompt, n_new)
    print(f"selected loop: rounds {len(taus)}, taus {taus}")
    np.testing.assert_array_equal(np.array(toks), ref)
    np.testing.assert_array_equal(np.array(toks), ar)
    assert taus == rtaus
    target.close()
    draft.close()
