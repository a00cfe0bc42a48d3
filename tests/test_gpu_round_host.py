"""One greedy round through dflash_round_host: inputs copied in from pinned
host memory, the round drafted and verified, results copied back out.

The results must equal, bit for bit, those of the same round run through
the device-buffer calls (dflash_draft_round + dflash_verify_greedy), which
proves the copies and the result layout.  They are also held to the oracle:
the draft ids equal the oracle's outside its near-ties, and for every
sequence whose ids equal the oracle's, the accepted prefix, bonus, emitted
tokens and trimmed length equal oracle.verify_greedy's.  The target's
posterior is built from the oracle's own ids, so the accepted prefixes span
0 .. B-1 (txtmix §9: accept the longest prefix the target agrees with, then
add its token at the first disagreement)."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import NEAR_TIE, oracle_block, to_np, to_np64
from test_gpu_draft import SMALL_BF16

pytestmark = pytest.mark.gpu


def _oracle_ids(s, w, weights, K0, V0, hidden, lens, nrows, row0, anchors, B):
    """Fusion, injection and the block draft from the test's inputs only."""
    W, W64 = to_np(weights), to_np64(weights)
    store = O.storage(w.dtype)
    n_in = int(nrows.sum())
    Ht = (O.fuse_context([to_np(h)[:n_in] for h in hidden], W64["wc"], W64["g_c"], s.eps, store)
          if n_in else np.zeros((0, s.D)))
    cK, cV = [], []
    for l in range(s.n_layers):
        Kl, Vl = [], []
        for b in range(len(lens)):
            L, n, r0 = lens[b], nrows[b], row0[b]
            k, v = O.inject_kv(Ht[r0:r0 + n], W64["layers"][l], np.arange(L, L + n), s.G, s.d,
                               s.rope_theta, s.eps, store)
            Kl.append(np.concatenate([K0[l][b, :, :L].transpose(1, 0, 2), k]))
            Vl.append(np.concatenate([V0[l][b, :, :L].transpose(1, 0, 2), v]))
        cK.append(Kl)
        cV.append(Vl)
    ids, gap, _ = oracle_block(s, W, cK, cV, anchors, B, store)
    return ids, gap


def _posterior(oids, V, seed):
    """A target argmax that agrees with the oracle's drafts for a chosen
    prefix of each sequence (0, all B-1, and values between), then not."""
    batch, B = oids.shape
    rng = np.random.default_rng(seed)
    post = rng.integers(0, V, size=(batch, B)).astype(np.int32)
    for b in range(batch):
        a = [0, B - 1, (B - 1) // 2, 1][b % 4] if B > 1 else 0
        post[b, :a] = oids[b, 1:a + 1]
        if a < B - 1:
            post[b, a] = (oids[b, a + 1] + 1 + b) % V
    return post


@pytest.mark.parametrize("B,lens,nrows", [
    (4, [64, 37, 0, 100], [3, 3, 5, 1]),   # 16 block rows, 12 pending: the persistent launch
    (16, [40, 20], [10, 12]),              # 32 block rows: the three calls
    (8, [30, 50], [0, 0]),                 # nothing pending: the block alone
])
def test_round_host_matches_device_calls_and_oracle(dfl, B, lens, nrows):
    from synth.gpu import draft_model, kv_cache
    w = SMALL_BF16
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
    K0 = [k.float().cpu().numpy() for k in K]
    V0 = [v.float().cpu().numpy() for v in V]
    kv = kv_cache(s, batch, cap, w.dtype, k=K, v=V)
    m = draft_model(s, w.dtype, weights, max_pos=cap + B + 8)
    hidden = synth.target_hidden_states(max(n_in, 1), s.D, s.n_pick, w.dtype, w.seed + 3,
                                        device=dev)
    anchors = synth.anchors(batch, s.V, s.mask_id, w.seed)
    oids, ogap = _oracle_ids(s, w, weights, K0, V0, hidden, lens, nrows, row0, anchors, B)
    post = _posterior(oids, s.V, w.seed + 7)
    start = (lens + 3).astype(np.int32)
    o_acc, o_bonus, o_tok, o_len = O.verify_greedy(oids, post, start)

    td = synth.torch_dtype(w.dtype)
    ws = m.workspace(max(batch * B, n_in, 1), max_batch=batch, max_block=B)
    r0_d, nr_d = torch.from_numpy(row0).to(dev), torch.from_numpy(nrows).to(dev)
    ht = torch.zeros(max(n_in, 1), s.D, dtype=td, device=dev)
    feats = torch.stack([h[:max(n_in, 1)] for h in hidden])          # [n_pick, rows, D]
    ints_in = np.concatenate([anchors.astype(np.int32), post.reshape(-1)])
    n_out = dfl.dflash_round_out_len(batch, B)
    P = (batch + 3) // 4 * 4
    assert n_out == 2 * batch * B + 3 * P

    # the device-buffer calls
    kv.len.copy_(torch.from_numpy(lens))
    start_d = torch.from_numpy(start).to(dev)
    new_len_d = torch.empty(batch, dtype=torch.int32, device=dev)
    ids = torch.full((batch, B), -5, dtype=torch.int32, device=dev)
    acc = torch.empty(batch, dtype=torch.int32, device=dev)
    tau = torch.empty_like(acc)
    bonus = torch.empty_like(acc)
    tok = torch.empty(batch, B, dtype=torch.int32, device=dev)
    post_d = torch.from_numpy(post).to(dev)
    dfl.dflash_draft_round(m.handle, [feats[i] for i in range(s.n_pick)], n_in, r0_d, nr_d, ht,
                           torch.from_numpy(anchors).to(dev), batch, B, kv.struct, ids, None,
                           None, ws)
    dfl.dflash_verify_greedy(ids, post_d, batch, B, start_d, acc, tau, bonus, tok, new_len_d)
    assert dfl.dflash_get_status(m.handle) == 0
    ref = np.full(n_out, -7, np.int32)
    ref[:batch * B] = ids.cpu().numpy().reshape(-1)
    ref[batch * B:2 * batch * B] = tok.cpu().numpy().reshape(-1)
    for i, t in enumerate((acc, tau, bonus)):
        ref[2 * batch * B + i * P:2 * batch * B + i * P + batch] = t.cpu().numpy()
    ref_len = new_len_d.cpu().numpy()

    # the host-buffer call, on the restored cache lengths
    kv.len.copy_(torch.from_numpy(lens))
    h_feat = feats.cpu().pin_memory() if n_in else None
    h_in = torch.from_numpy(ints_in).pin_memory()
    h_out = torch.full((n_out,), -7, dtype=torch.int32).pin_memory()
    d_in = torch.empty(len(ints_in), dtype=torch.int32, device=dev)
    d_out = torch.full((n_out,), -7, dtype=torch.int32, device=dev)
    d_feat = torch.empty_like(feats) if n_in else None
    new_len2 = torch.empty(batch, dtype=torch.int32, device=dev)
    dfl.dflash_round_host(m.handle, h_feat, d_feat, n_in, h_in, d_in, h_out, d_out, r0_d, nr_d,
                          ht, batch, B, kv.struct, start_d, new_len2, ws)
    torch.cuda.current_stream().synchronize()
    assert dfl.dflash_get_status(m.handle) == 0
    np.testing.assert_array_equal(kv.len.cpu().numpy(), lens + nrows)
    m.close()
    got = h_out.numpy().copy()
    pad = np.ones(n_out, bool)
    pad[:2 * batch * B] = False
    for i in range(3):
        pad[2 * batch * B + i * P:2 * batch * B + i * P + batch] = False
    np.testing.assert_array_equal(got[~pad], ref[~pad])
    np.testing.assert_array_equal(new_len2.cpu().numpy(), ref_len)

    # against the oracle
    g_ids = got[:batch * B].reshape(batch, B)
    g_tok = got[batch * B:2 * batch * B].reshape(batch, B)
    g_acc, g_tau, g_bonus = (got[2 * batch * B + i * P:2 * batch * B + i * P + batch]
                             for i in range(3))
    near = np.zeros((batch, B), bool)
    near[:, 1:] = ogap < NEAR_TIE
    assert ((g_ids == oids) | near).all()
    same = (g_ids == oids).all(axis=1)
    print(f"B={B} lens={lens.tolist()} pending={nrows.tolist()}: accept {g_acc.tolist()} "
          f"(oracle {o_acc.tolist()}), sequences compared {int(same.sum())}/{batch}")
    assert same.sum() >= (batch + 1) // 2
    np.testing.assert_array_equal(g_acc[same], o_acc[same])
    np.testing.assert_array_equal(g_tau[same], o_acc[same] + 1)
    np.testing.assert_array_equal(g_bonus[same], o_bonus[same])
    np.testing.assert_array_equal(g_tok[same], o_tok[same])
    np.testing.assert_array_equal(new_len2.cpu().numpy()[same], o_len[same])
    if B > 1 and batch >= 2:
        assert len(set(o_acc.tolist())) >= 2        # the prefixes differ in length
