"""One speculative round through dflash_draft_round vs the oracle: fusion of
the pending target features, their K/V injection after each sequence's cached
context, and the block draft over the grown caches.  Blocks of at most 16
rows run it as one persistent launch; larger ones run the three calls."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import F32_DRAWS, float_parity, oracle_block, to_np, to_np64
from test_gpu_draft import SMALL_BF16, _compare

pytestmark = pytest.mark.gpu


def _round_case(dfl, w, B, lens, nrows, compare=None):
    """compare: test_gpu_draft._compare unless given (same arguments)."""
    from synth.gpu import draft_model, kv_cache
    s = w.draft
    dev = "cuda"
    batch = len(lens)
    lens, nrows = np.asarray(lens, np.int32), np.asarray(nrows, np.int32)
    n_in = int(nrows.sum())
    row0 = np.concatenate([[0], np.cumsum(nrows)[:-1]]).astype(np.int32)
    cap = int((lens + nrows).max()) + 8
    weights = synth.draft_weights(s, w.dtype, w.seed, device=dev)
    K, V = synth.random_kv_cache(batch, s.G, cap, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device=dev)
    # the cache beyond each length is cleared, so the test also sees that the
    # round writes exactly the appended rows
    for l in range(s.n_layers):
        for b in range(batch):
            K[l][b, :, lens[b]:] = 0
            V[l][b, :, lens[b]:] = 0
    K0 = [k.float().cpu().numpy() for k in K]
    V0 = [v.float().cpu().numpy() for v in V]
    kv = kv_cache(s, batch, cap, w.dtype, k=K, v=V)
    kv.len.copy_(torch.from_numpy(lens))
    m = draft_model(s, w.dtype, weights, max_pos=cap + B + 8)
    hidden = synth.target_hidden_states(max(n_in, 1), s.D, s.n_pick, w.dtype, w.seed + 3, device=dev)
    anchors = synth.anchors(batch, s.V, s.mask_id, w.seed)
    td = synth.torch_dtype(w.dtype)
    ht = torch.zeros(max(n_in, 1), s.D, dtype=td, device=dev)
    ids = torch.full((batch, B), -5, dtype=torch.int32, device=dev)
    gap = torch.empty(batch, max(B - 1, 1), device=dev)
    hid = torch.empty(batch * B, s.D, device=dev)
    ws = m.workspace(max(batch * B, n_in), max_batch=batch, max_block=B)
    dfl.dflash_draft_round(m.handle, hidden, n_in, torch.from_numpy(row0).to(dev),
                           torch.from_numpy(nrows).to(dev), ht,
                           torch.from_numpy(anchors).to(dev), batch, B, kv.struct, ids, gap, hid, ws)
    assert dfl.dflash_get_status(m.handle) == 0
    np.testing.assert_array_equal(kv.len.cpu().numpy(), lens + nrows)
    label = f"round {w.name} B={B} lens={lens.tolist()} pending={nrows.tolist()}"

    # oracle: fusion, injection, draft, from the same inputs only
    W = to_np(weights)
    W64 = to_np64(weights)
    store = O.storage(w.dtype)
    Ht = O.fuse_context([to_np(h)[:n_in] for h in hidden], W64["wc"], W64["g_c"], s.eps, store)
    if n_in:
        err, exact = float_parity(ht.float().cpu().numpy()[:n_in], Ht, w.dtype, f"{label} H_t")
        print(f"{label}: H_t max|err| {err:.3e}, bit-equal {exact:.5f}")
        assert exact > 0.99
    cK, cV = [], []
    for l in range(s.n_layers):
        Kg, Vg = kv.k[l].float().cpu().numpy(), kv.v[l].float().cpu().numpy()
        Kl, Vl = [], []
        for b in range(batch):
            L, n, r0 = lens[b], nrows[b], row0[b]
            k, v = O.inject_kv(Ht[r0:r0 + n], W64["layers"][l], np.arange(L, L + n), s.G, s.d,
                               s.rope_theta, s.eps, store)
            if n:
                # within tolerance element by element; bit-equal for nearly all: the GPU
                # injects its own H_t, which differs from the oracle's in ~0.1% of its bf16
                # values (a one-ulp flip where the fp32 sum lands at a rounding midpoint),
                # and each K/V value sums D such products, so a few percent of them round
                # the other way (with the oracle's H_t as input both sides agree, see
                # test_inject_parity_ragged)
                _, ek = float_parity(Kg[b, :, L:L + n].transpose(1, 0, 2), k, w.dtype, f"K l{l} b{b}")
                _, ev = float_parity(Vg[b, :, L:L + n].transpose(1, 0, 2), v, w.dtype, f"V l{l} b{b}")
                print(f"{label}: layer {l} seq {b}: K bit-equal {ek:.4f}, V {ev:.4f}")
                assert ek > 0.9 and ev > 0.9
            # the old context is untouched and nothing past the new length is written
            np.testing.assert_array_equal(Kg[b, :, :L], K0[l][b, :, :L])
            np.testing.assert_array_equal(Vg[b, :, :L], V0[l][b, :, :L])
            assert not Kg[b, :, L + n:].any() and not Vg[b, :, L + n:].any()
            Kl.append(np.concatenate([K0[l][b, :, :L].transpose(1, 0, 2), k]))
            Vl.append(np.concatenate([V0[l][b, :, :L].transpose(1, 0, 2), v]))
        cK.append(Kl)
        cV.append(Vl)
    ids, gap, hid = ids.cpu().numpy(), gap.cpu().numpy(), hid.cpu().numpy().reshape(batch, B, s.D)
    assert (ids[:, 0] == anchors).all()
    if B == 1:
        m.close()
        return
    m.close()
    o64 = oracle_block(s, W, cK, cV, anchors, B, store, with_logits=True)
    o32 = ([oracle_block(s, W, cK, cV, anchors, B, store, arith=a) for a in F32_DRAWS]
           if w.dtype == "bf16" else None)
    (compare or _compare)(w, ids, gap, hid, o64, label, o32)


@pytest.mark.parametrize("B,lens,nrows", [
    (16, [64], [16]),                    # one sequence, 16 pending rows
    (8, [0, 37], [5, 3]),                # an empty old context
    (4, [5, 100, 0, 64], [2, 0, 4, 1]),  # a sequence with nothing pending
    (5, [30], [16]),                     # more pending rows than block rows
    (16, [40, 20], [10, 12]),            # 32 block rows: the three calls
])
def test_round_small_bf16(dfl, B, lens, nrows):
    _round_case(dfl, SMALL_BF16, B, lens, nrows)


def test_round_block_size_one(dfl):
    """B = 1: the block is the anchors; the round still fuses and injects."""
    _round_case(dfl, SMALL_BF16, 1, [3, 9, 0], [1, 2, 1])


def test_round_qwen3_8b(dfl):
    """Qwen3-8B-shaped draft: 16 pending rows after 2032 cached positions,
    then the B = 16 block (the per-round shape of the bench step)."""
    _round_case(dfl, synth.WORKLOADS["qwen3_8b_b1"], 16, [2032], [16])
