"""Block draft forward on the GPU vs the oracle.

Ids are bit-exact outside near-ties (oracle top-2 gap < 1e-3, counted and
reported); the residual stream after the last layer and the gaps meet the
float tolerance against the oracle run with the same storage points."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import (F32_DRAWS, NEAR_TIE, bf16_draft_parity, float_parity, id_parity, oracle_block,
                     to_np, to_np64)

pytestmark = pytest.mark.gpu


def _gpu_draft(dfl, m, anchors, batch, B, kv, D):
    dev = "cuda"
    a = torch.from_numpy(np.asarray(anchors, dtype=np.int32)).to(dev)
    ids = torch.full((batch, B), -5, dtype=torch.int32, device=dev)
    gap = torch.empty(batch, max(B - 1, 1), device=dev)
    hid = torch.empty(batch * B, D, device=dev)
    dfl.dflash_draft_block(m.handle, a, batch, B, kv.struct, ids, gap, hid,
                           m.workspace(batch * B, max_batch=batch, max_block=B))
    assert dfl.dflash_get_status(m.handle) == 0
    return ids.cpu().numpy(), gap.cpu().numpy(), hid.cpu().numpy().reshape(batch, B, D)


def _oracle_ctx(kv, lens, seqs, n_layers):
    K = [[kv.k[l][b, :, :lens[b]].float().cpu().numpy().transpose(1, 0, 2) for b in seqs]
         for l in range(n_layers)]
    V = [[kv.v[l][b, :, :lens[b]].float().cpu().numpy().transpose(1, 0, 2) for b in seqs]
         for l in range(n_layers)]
    return K, V


def _compare(w, ids, gap, hid, o64, label, o32=None):
    """fp32 path: ids bit-exact outside near-ties (oracle gap < 1e-3), floats
    within 1e-4 of the oracle.  bf16 path: helpers.bf16_draft_parity against
    the oracle with bf16 storage points (o32: the same oracle in fp32
    arithmetic, which sets the case's floor)."""
    oids, ogap, ohid = o64[:3]
    if w.dtype == "f32":
        bad, near, n = id_parity(ids, oids, ogap)
        print(f"{label}: ids compared {n}, mismatches {bad}, near-ties (<{NEAR_TIE}) {near}")
        assert bad == 0
        far = (ogap >= NEAR_TIE) & (np.asarray(ids)[:, 1:] == np.asarray(oids)[:, 1:])
        e_h, _ = float_parity(hid, ohid, "f32", f"{label} residual")
        e_g, _ = float_parity(gap[far], ogap[far], "f32", "gap")
        print(f"{label}: residual max err {e_h:.3e}, gap max err {e_g:.3e}")
        return
    bf16_draft_parity(label, ids, gap, hid, o64, o32)


def test_draft_chain_tiny(dfl):
    """fuse -> inject -> draft on the tiny fp32 instance, against the same
    chain in the oracle."""
    from synth.gpu import draft_model, kv_cache
    w = synth.WORKLOADS["tiny_f32"]
    s, L, B = w.draft, w.ctx_len, w.B
    dev = "cuda"
    weights = synth.draft_weights(s, w.dtype, w.seed, device=dev)
    hs = synth.target_hidden_states(L, s.D, s.n_pick, w.dtype, w.seed, device=dev)
    m = draft_model(s, w.dtype, weights, max_pos=256)
    kv = kv_cache(s, 1, 128, w.dtype)
    ws = m.workspace(L)
    H_t = torch.empty(L, s.D, device=dev)
    dfl.dflash_fuse_context(m.handle, hs, L, H_t, ws)
    z = torch.zeros(1, dtype=torch.int32, device=dev)
    dfl.dflash_inject_kv(m.handle, H_t, L, z, torch.tensor([L], dtype=torch.int32, device=dev), 1,
                         kv.struct, ws)
    anchors = synth.anchors(1, s.V, s.mask_id, w.seed)
    ids, gap, hid = _gpu_draft(dfl, m, anchors, 1, B, kv, s.D)
    assert int(kv.len[0]) == L
    W = to_np64(weights)
    Ht = O.fuse_context([to_np(h) for h in hs], W["wc"], W["g_c"], s.eps, O.f32)
    cK, cV = [], []
    for lay in W["layers"]:
        k, v = O.inject_kv(Ht, lay, np.arange(L), s.G, s.d, s.rope_theta, s.eps, O.f32)
        cK.append([k])
        cV.append([v])
    o64 = O.draft_block(s, W, cK, cV, anchors, B, O.f32, return_hidden=True)
    _compare(w, ids, gap, hid, o64, "tiny chain")
    m.close()


def _random_cache_case(dfl, w, B, lens, sample, weights=None):
    from synth.gpu import draft_model, kv_cache
    s = w.draft
    batch = len(lens)
    cap = max(max(lens), 1)
    dev = "cuda"
    if weights is None:
        weights = synth.draft_weights(s, w.dtype, w.seed, device=dev)
    K, V = synth.random_kv_cache(batch, s.G, cap, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device=dev)
    kv = kv_cache(s, batch, cap, w.dtype, k=K, v=V)
    kv.len.copy_(torch.tensor(lens, dtype=torch.int32))
    m = draft_model(s, w.dtype, weights, max_pos=cap + B + 8)
    anchors = synth.anchors(batch, s.V, s.mask_id, w.seed)
    ids, gap, hid = _gpu_draft(dfl, m, anchors, batch, B, kv, s.D)
    assert (ids[:, 0] == anchors).all()
    assert (ids >= 0).all() and (ids < s.V).all()
    W = to_np(weights)
    cK, cV = _oracle_ctx(kv, lens, sample, s.n_layers)
    o64 = oracle_block(s, W, cK, cV, anchors[sample], B, O.storage(w.dtype), with_logits=True)
    o32 = None
    if w.dtype == "bf16":
        o32 = [oracle_block(s, W, cK, cV, anchors[sample], B, O.storage(w.dtype), arith=a)
               for a in F32_DRAWS]
    _compare(w, ids[sample], gap[sample], hid[sample], o64, f"{w.name} B={B} seqs={list(sample)}",
             o32)
    m.close()
    return weights


def test_draft_tiny_batch32_ragged(dfl):
    w = synth.with_(synth.WORKLOADS["tiny_f32"], batch=32)
    lens = [int(x) for x in np.random.default_rng(1).integers(0, 65, 32)]
    lens[3] = 0                                   # empty context: block attends to itself only
    _random_cache_case(dfl, w, w.B, lens, np.arange(32))


def test_draft_qwen3_8b_batch1(dfl):
    w = synth.WORKLOADS["qwen3_8b_b1"]
    _random_cache_case(dfl, w, w.B, [w.ctx_len], np.array([0]))


def test_draft_qwen3_8b_batch32_ragged(dfl):
    """Batch 32, contexts U{512..8192}, five layers: a seeded quarter of the
    sequences with the shortest and the longest context among them (the
    oracle re-reads every weight per sequence and per run; the one-layer
    case in test_gpu_bf16_parity compares a seeded half)."""
    w = synth.WORKLOADS["qwen3_8b_b32_ragged"]
    lens = synth.ctx_lengths(w)
    order = np.argsort(lens)
    part = np.random.default_rng(w.seed + 31).choice(w.batch, w.batch // 4 - 2, replace=False)
    sample = np.array(sorted(set(part.tolist()) | {int(order[0]), int(order[-1])}))
    _random_cache_case(dfl, w, w.B, lens, sample)


def test_draft_35b_batch8_narrow_tiles(dfl):
    """35B-A3B-shaped draft, 8 sequences x 16 rows = 128 rows: every layer
    projection runs on the tensor-core kernel with 128-column tiles (the
    head-norm + RoPE, SwiGLU and residual epilogues at that width)."""
    w = synth.with_(synth.WORKLOADS["qwen35_a3b_32k"], batch=8)
    lens = [int(x) for x in np.random.default_rng(8).integers(1, 1500, 8)]
    lens[5] = 0
    _random_cache_case(dfl, w, w.B, lens, np.array([2, 5]))


@pytest.mark.parametrize("B", [8, 16])
def test_draft_long_context_32k(dfl, B):
    """Batch 4 at L = 32768: all four sequences."""
    w = synth.WORKLOADS["qwen35_a3b_32k"]
    _random_cache_case(dfl, w, B, [w.ctx_len] * w.batch, np.arange(w.batch))


def test_draft_block_size_one(dfl):
    """B = 1: the block is the anchor alone; no logits, ids = anchors."""
    from synth.gpu import draft_model, kv_cache
    w = synth.WORKLOADS["tiny_f32"]
    s = w.draft
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    m = draft_model(s, w.dtype, weights, max_pos=64)
    kv = kv_cache(s, 2, 16, w.dtype)
    ids, _, _ = _gpu_draft(dfl, m, [11, 22], 2, 1, kv, s.D)
    np.testing.assert_array_equal(ids[:, 0], [11, 22])
    m.close()


@pytest.mark.parametrize("wname", ["tiny_f32", "qwen3_8b_b1"])
def test_lm_head_argmax_ties_and_gap(dfl, wname):
    """Duplicate LM-head rows make exact logit ties: the lowest index wins
    (33 and 700 sit in different 128-row vocabulary tiles, 900 and 901 in
    the same one) and the gap is zero; elsewhere ids and gaps match."""
    from synth.gpu import draft_model
    w = synth.WORKLOADS[wname]
    s = w.draft
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    rows = 6
    x = torch.randn(rows, s.D, generator=torch.Generator().manual_seed(3)).cuda()
    hf = x / torch.sqrt((x * x).mean(1, keepdim=True) + s.eps)
    lm = weights["lm_head"]
    lm[700] = (hf[0] * 0.5).to(lm.dtype)
    lm[33] = (hf[0] * 0.5).to(lm.dtype)    # same row twice: exact tie, 33 < 700
    lm[900] = (hf[1] * 0.5).to(lm.dtype)
    lm[901] = (hf[1] * 0.5).to(lm.dtype)
    m = draft_model(s, w.dtype, weights, max_pos=64)
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    gap = torch.empty(rows, device="cuda")
    dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids, gap, m.workspace(rows))
    torch.cuda.synchronize()
    ids, gap = ids.cpu().numpy(), gap.cpu().numpy()
    assert ids[0] == 33 and ids[1] == 900 and gap[0] == 0 and gap[1] == 0
    st = O.storage(w.dtype)
    z = O.lm_head_logits(st(O.rmsnorm(x.cpu().numpy(), np.ones(s.D), s.eps)), to_np(lm))
    og = O.top2_gap(z)
    far = og >= NEAR_TIE
    np.testing.assert_array_equal(ids[2:][far[2:]], O.argmax_lowest(z)[2:][far[2:]])
    np.testing.assert_allclose(gap, og, atol=1e-4 if w.dtype == "f32" else 2e-3)
    m.close()


# ---- short blocks (at most 16 rows): the single persistent launch ----------
# A small bf16 shape that the persistent kernel accepts (head dim 128, D a
# multiple of 128): its projections have fewer (tile, k-chunk) units than the
# kernel has CTAs, so most CTAs own no unit of a phase.
SMALL_BF16 = synth.Workload(
    name="small_bf16", dtype="bf16",
    draft=synth.DraftShape(n_layers=2, D=256, H=4, G=2, d=128, F=768, V=2048, mask_id=2047,
                           n_target_layers=12),
    batch=1, B=16, ctx_len=64, seed=1005)


@pytest.mark.parametrize("B,lens", [
    (16, [64]),                  # one sequence, 16 rows
    (5, [37]),                   # 5 rows: a partial 16-row tile
    (8, [0, 37]),                # two sequences, one with an empty context
    (4, [5, 100, 0, 64]),        # four ragged sequences
])
def test_draft_short_block_small_bf16(dfl, B, lens):
    _random_cache_case(dfl, SMALL_BF16, B, lens, np.arange(len(lens)))


@pytest.mark.parametrize("B,lens", [
    (16, [0, 3000, 17, 700]),    # 64 rows: streaming launches, ragged split-attention items
    (48, [1000]),                # 96 query rows per kv head: two query groups
])
def test_draft_split_attention_small_bf16(dfl, B, lens):
    """Blocks above 16 rows run the per-projection launches and the planned
    split attention (items cut from the device-side lengths)."""
    _random_cache_case(dfl, SMALL_BF16, B, lens, np.arange(len(lens)))


def test_draft_short_block_b1_batch16(dfl):
    """16 sequences of block size 1: the block is the anchors; the final
    residual still matches the oracle and the ids are the anchors."""
    from synth.gpu import draft_model, kv_cache
    w, s = SMALL_BF16, SMALL_BF16.draft
    lens = [int(x) for x in np.random.default_rng(5).integers(0, 70, 16)]
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    K, V = synth.random_kv_cache(16, s.G, 70, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device="cuda")
    kv = kv_cache(s, 16, 70, w.dtype, k=K, v=V)
    kv.len.copy_(torch.tensor(lens, dtype=torch.int32))
    m = draft_model(s, w.dtype, weights, max_pos=128)
    anchors = synth.anchors(16, s.V, s.mask_id, w.seed)
    ids, _, hid = _gpu_draft(dfl, m, anchors, 16, 1, kv, s.D)
    np.testing.assert_array_equal(ids[:, 0], anchors)
    W = to_np(weights)
    cK, cV = _oracle_ctx(kv, lens, range(16), s.n_layers)
    o64 = oracle_block(s, W, cK, cV, anchors, 1, O.storage(w.dtype))
    o32 = [oracle_block(s, W, cK, cV, anchors, 1, O.storage(w.dtype), arith=a) for a in F32_DRAWS]
    bf16_draft_parity("B=1 x 16", ids, np.zeros((16, 0)), hid, o64, o32)
    m.close()


def test_draft_qwen3_8b_two_sequences(dfl):
    """Qwen3-8B-shaped draft, two sequences of 8 rows (16 rows: one launch)
    with contexts of 2048 and 300."""
    w = synth.WORKLOADS["qwen3_8b_b1"]
    _random_cache_case(dfl, w, 8, [2048, 300], np.array([0, 1]))


def test_draft_qwen3_8b_batch2_rows32(dfl):
    """32 rows: above the persistent kernel's limit, the per-projection
    streaming launches run."""
    w = synth.WORKLOADS["qwen3_8b_b1"]
    _random_cache_case(dfl, w, 16, [1500, 2048], np.array([0, 1]))
