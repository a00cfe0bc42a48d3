"""bf16 draft path against the oracle at the stated tolerance.

The tolerance: floats within max-abs-err 2e-2 (plus one bf16 ulp of the
value where that is larger, tests/helpers.float_parity) of the oracle run
with the same bf16 storage points; draft ids bit-exact wherever the
oracle's top-2 logit gap is at least 1e-3 (positions under it counted and
printed).  Where the result depends only on the test's inputs through one
storage point — the LM head and argmax on a given residual, the fused
context H_t and the K/V entries a round appends — it is asserted as stated.
Through a draft layer, a bf16 storage point turns any difference in the
arithmetic before it (fp32 against fp64 sums) into whole-ulp flips of a few
of its values, which the next RMSNorm amplifies, so the oracle itself, run
with fp32 products and sums (arith="f32", in three summation orders),
departs from its fp64 run by a floor no fp32 implementation gets under.
helpers.bf16_draft_parity holds the GPU to the stated tolerance wherever
that floor is below half of it, and to small multiples of the floor
elsewhere; each case prints the GPU's distance, the floor, and the ids that
differ by gap band.

Shapes: the Qwen3-8B-shaped draft (D 4096, 32/8 heads, F 12288, vocabulary
151936) with one layer at batch 1 and L = 2048 (the persistent launch), two
sequences of 8 rows (the same launch), 32 rows (the streaming launches) and
batch 32 with ragged contexts (the tensor-core launches); the
Qwen3.5-35B-A3B-shaped draft (D 2048, 16/4 heads) with one layer at batch 4
and L = 32768, blocks of 8 and 16."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from helpers import F32_DRAWS, NEAR_TIE, bf16_draft_parity, float_parity, oracle_block, to_np

pytestmark = pytest.mark.gpu


def one_layer(w: synth.Workload, **kw) -> synth.Workload:
    return synth.with_(w, draft=dataclasses.replace(w.draft, n_layers=1), **kw)


def compare(w, ids, gap, hid, o64, label, o32):
    bf16_draft_parity(label, ids, gap, hid, o64, o32)


def draft_case(dfl, w, lens, sample):
    from synth.gpu import draft_model, kv_cache
    s, B = w.draft, w.B
    batch = len(lens)
    cap = max(max(lens), 1)
    dev = "cuda"
    weights = synth.draft_weights(s, w.dtype, w.seed, device=dev)
    K, V = synth.random_kv_cache(batch, s.G, cap, s.d, s.n_layers, 0.02 * np.sqrt(s.D), w.dtype,
                                 w.seed, device=dev)
    kv = kv_cache(s, batch, cap, w.dtype, k=K, v=V)
    kv.len.copy_(torch.tensor(lens, dtype=torch.int32))
    m = draft_model(s, w.dtype, weights, max_pos=cap + B + 8)
    anchors = synth.anchors(batch, s.V, s.mask_id, w.seed)
    a = torch.from_numpy(anchors).to(dev)
    ids = torch.full((batch, B), -5, dtype=torch.int32, device=dev)
    gap = torch.empty(batch, B - 1, device=dev)
    hid = torch.empty(batch * B, s.D, device=dev)
    dfl.dflash_draft_block(m.handle, a, batch, B, kv.struct, ids, gap, hid,
                           m.workspace(batch * B, max_batch=batch, max_block=B))
    assert dfl.dflash_get_status(m.handle) == 0
    ids, gap = ids.cpu().numpy(), gap.cpu().numpy()
    hid = hid.cpu().numpy().reshape(batch, B, s.D)
    assert (ids[:, 0] == anchors).all()
    W = to_np(weights)
    cK = [[kv.k[l][b, :, :lens[b]].float().cpu().numpy().transpose(1, 0, 2) for b in sample]
          for l in range(s.n_layers)]
    cV = [[kv.v[l][b, :, :lens[b]].float().cpu().numpy().transpose(1, 0, 2) for b in sample]
          for l in range(s.n_layers)]
    m.close()
    store = O.storage(w.dtype)
    o64 = oracle_block(s, W, cK, cV, anchors[sample], B, store, with_logits=True)
    o32 = [oracle_block(s, W, cK, cV, anchors[sample], B, store, arith=a) for a in F32_DRAWS]
    bf16_draft_parity(f"one-layer {w.name} B={B} batch {batch} seqs {sample.tolist()}",
                      ids[sample], gap[sample], hid[sample], o64, o32)


QWEN3 = synth.WORKLOADS["qwen3_8b_b1"]
A3B = synth.WORKLOADS["qwen35_a3b_32k"]


def test_one_layer_qwen3_8b_batch1(dfl):
    """16 rows: the persistent launch (the bench's block)."""
    draft_case(dfl, one_layer(QWEN3), [QWEN3.ctx_len], np.array([0]))


def test_one_layer_qwen3_8b_two_sequences(dfl):
    """Two sequences of 8 rows, contexts 2048 and 300: the persistent launch."""
    draft_case(dfl, one_layer(QWEN3, B=8, batch=2), [2048, 300], np.array([0, 1]))


def test_one_layer_qwen3_8b_rows32(dfl):
    """32 rows: the streaming projections and the planned split attention."""
    draft_case(dfl, one_layer(QWEN3, batch=2), [1500, 2048], np.array([0, 1]))


def test_one_layer_qwen3_8b_batch32_ragged(dfl):
    """512 rows, contexts U{512..8192}: the tensor-core projections; a seeded
    half of the sequences is compared."""
    w = one_layer(synth.WORKLOADS["qwen3_8b_b32_ragged"])
    lens = synth.ctx_lengths(w)
    sample = np.sort(np.random.default_rng(w.seed + 29).choice(w.batch, w.batch // 2,
                                                               replace=False))
    draft_case(dfl, w, lens, sample)


@pytest.mark.parametrize("B", [8, 16])
def test_one_layer_35b_a3b_batch4_32k(dfl, B):
    """Batch 4 at L = 32768 (32 and 64 rows): all four sequences."""
    draft_case(dfl, one_layer(A3B, B=B), [A3B.ctx_len] * A3B.batch, np.arange(A3B.batch))


def test_one_layer_round_qwen3_8b(dfl):
    """One speculative round of a one-layer Qwen3-8B-shaped draft through
    dflash_draft_round (16 pending rows after 2032 cached positions, then the
    B = 16 block: the bench's launch): H_t and the appended K/V within the
    stated tolerance, then the block as above."""
    from test_gpu_round import _round_case
    _round_case(dfl, one_layer(QWEN3), 16, [2032], [16], compare=compare)


@pytest.mark.parametrize("rows", [15, 64, 480])
def test_lm_head_argmax_qwen3_vocab(dfl, rows):
    """Final RMSNorm + LM head + argmax alone at vocabulary 151936 on seeded
    fp32 residual rows of varied scale (15 and 64 rows: the streaming kernel;
    480: the tensor-core kernel)."""
    from synth.gpu import draft_model
    w = one_layer(QWEN3)
    s = w.draft
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    g = torch.Generator().manual_seed(31 + rows)
    x = torch.randn(rows, s.D, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))
    m = draft_model(s, w.dtype, weights, max_pos=64)
    ids = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    gap = torch.empty(rows, device="cuda")
    dfl.dflash_lm_head_argmax(m.handle, x.cuda(), rows, weights["g_f"], ids, gap,
                              m.workspace(rows))
    assert dfl.dflash_get_status(m.handle) == 0
    m.close()
    W_lm = to_np(weights["lm_head"])
    hf = O.bf16(O.rmsnorm(x.double().numpy(), to_np(weights["g_f"]), s.eps))
    z = O.lm_head_logits(hf, W_lm)
    oids, ogap = O.argmax_lowest(z), O.top2_gap(z)
    ids, gap = ids.cpu().numpy(), gap.cpu().numpy()
    near = ogap < NEAR_TIE
    bad = int(((ids != oids) & ~near).sum())
    e_g, _ = float_parity(gap, ogap, "bf16", "LM-head gap")
    print(f"LM head {rows} rows: ids compared {int((~near).sum())}, mismatches {bad}, "
          f"near-ties {int(near.sum())}, differing in all {int((ids != oids).sum())}; "
          f"gap max|err| {e_g:.3e}, bound 2e-2")
    assert bad == 0
