"""Test plumbing: tensor conversion and small workload builders."""
import numpy as np
import torch

import oracle as O
import synth


def to_np(obj):
    """torch tensors (any float dtype) -> float32 numpy; ints kept; recursive."""
    if isinstance(obj, torch.Tensor):
        t = obj.detach().cpu()
        if t.is_floating_point():
            return t.float().numpy()
        return t.numpy()
    if isinstance(obj, dict):
        return {k: to_np(v) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [to_np(v) for v in obj]
    return obj


def tiny_e2e(D=64, H=4, d=16, F=96, V=128, t_layers=8, d_layers=2):
    """A small target/draft pair with the end-to-end workload's structure."""
    tshape = synth.TargetShape(n_layers=t_layers, D=D, H=H, G=H, d=d, F=F, V=V)
    dshape = synth.DraftShape(n_layers=d_layers, D=D, H=H, G=H, d=d, F=F, V=V,
                              mask_id=V - 1, n_target_layers=t_layers)
    return tshape, dshape


def make_all_accept(TW, DW, tshape, c):
    """Make greedy decoding collapse onto a fixed token c that every draft
    row predicts: the target's blocks become identities (zero W_o and W_d),
    so its next token is a function of the current token only; the LM head
    row c is aligned with the normalised embedding of c, and the mask token
    shares c's embedding, so the draft (also identity layers) proposes c at
    every masked position."""
    for lay in TW["layers"] + DW["layers"]:
        lay["wo"] = lay["wo"] * 0
        lay["wd"] = lay["wd"] * 0
    e = TW["embed"][c].astype(np.float64)
    e = e / np.sqrt(np.mean(e * e) + tshape.eps)
    TW["lm_head"][c] = (10.0 * e / np.linalg.norm(e)).astype(TW["lm_head"].dtype)
    TW["embed"][tshape.V - 1] = TW["embed"][c]
    return TW, DW


def make_partial_accept(TW, DW, tshape, cycle, m_index):
    """Plant greedy decoding with partial agreement.  Identity blocks (zero
    W_o and W_d) in both models make every position's next token a function
    of its own token only; LM-head row cycle[k+1] is aligned with the
    normalised embedding of cycle[k], so the target follows the cycle
    cycle[0] -> cycle[1] -> ... -> cycle[0].  The mask token shares the
    embedding of cycle[m_index], so the draft proposes cycle[m_index + 1] at
    every masked position: a round whose anchor is cycle[m_index] accepts
    one draft and rejects the next (tau = 2, with a cycle of three or more),
    every other round accepts none (tau = 1)."""
    for lay in TW["layers"] + DW["layers"]:
        lay["wo"] = lay["wo"] * 0
        lay["wd"] = lay["wd"] * 0
    n = len(cycle)
    for k in range(n):
        e = TW["embed"][cycle[k]].astype(np.float64)
        e = e / np.sqrt(np.mean(e * e) + tshape.eps)
        TW["lm_head"][cycle[(k + 1) % n]] = (e / np.linalg.norm(e)).astype(TW["lm_head"].dtype)
    TW["embed"][tshape.V - 1] = TW["embed"][cycle[m_index]]
    return TW, DW


def to_np64(obj):
    """Like to_np but float64 (weights upcast once for the oracle)."""
    if isinstance(obj, torch.Tensor):
        t = obj.detach().cpu()
        if t.is_floating_point():
            return t.double().numpy()
        return t.numpy()
    if isinstance(obj, dict):
        return {k: to_np64(v) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [to_np64(v) for v in obj]
    return obj


NEAR_TIE = 1e-3      # top-2 logit gap under which an id is reported, not compared
TOL = {"f32": 1e-4, "bf16": 2e-2}


def id_parity(gpu_ids, ora_ids, ora_gap, thresh=NEAR_TIE):
    """(mismatches outside near-ties, near-tie count, compared count) for the
    draft columns 1..B-1."""
    g = np.asarray(gpu_ids)[:, 1:]
    o = np.asarray(ora_ids)[:, 1:]
    near = np.asarray(ora_gap) < thresh
    bad = (g != o) & ~near
    return int(bad.sum()), int(near.sum()), int((~near).sum())


def float_excess(got, ref, dtype):
    """(max error, elements beyond the float_parity bound, bit-equal share),
    without asserting."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = TOL[dtype]
    bound = np.maximum(tol, np.abs(ref) * 2.0 ** -7) if dtype == "bf16" else tol
    err = np.abs(got - ref)
    return (float(err.max()) if err.size else 0.0, int((err > bound).sum()),
            float(np.mean(got == ref)) if got.size else 1.0)


def float_parity(got, ref, dtype, what=""):
    """Element-wise float parity against the oracle run with the same
    storage points.  Bound: TOL[dtype] absolute; in bf16 also one bf16 ulp
    of the oracle value (2^-7 |v|), since a stored value whose fp32 result
    sits within rounding noise of a bf16 midpoint may round either way and
    one ulp exceeds 2e-2 once |v| >= 4.  Returns (max error, bit-equal share)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    tol = TOL[dtype]
    bound = np.maximum(tol, np.abs(ref) * 2.0 ** -7) if dtype == "bf16" else tol
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond tolerance, "
                           f"max err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0, float(np.mean(got == ref)) if got.size else 1.0


F32_DRAWS = ("f32", "f32.1", "f32.2")


def bf16_draft_parity(label, ids, gap, hid, o64, o32s):
    """A bf16 draft block against the oracle run with the same bf16 storage
    points.  o64 = (ids, gaps, residual) of the oracle in fp64 arithmetic;
    o32s = the same oracle with every product and sum in fp32, once per
    summation order in F32_DRAWS (arith="f32", "f32.1", ...).

    The stated tolerance is max-abs-err 2e-2 (one bf16 ulp where larger, as
    in float_parity) and ids bit-exact outside top-2 gaps under 1e-3.  A
    bf16 storage point turns any arithmetic difference before it (fp32
    against fp64 sums) into whole-ulp flips of a few of its values, and the
    RMSNorms amplify them, so the oracle's own fp32 runs depart from its
    fp64 run by a case-dependent floor that no fp32 implementation gets
    under; each summation order is an independent draw of it.  With f the
    largest departure over the draws (max and rms of the residual, max of
    the gaps) and s the rms of all gap departures pooled over draws and
    positions: every residual element within max(stated bound, 2 f_max) —
    the stated tolerance itself wherever the floor is below half of it — and
    the rms error within 2 f_rms + 5e-4; gaps (where the ids agree) within
    max(2e-2, 2 f_gap, 8 s); ids equal to the fp64 oracle's, except that
    where they differ the GPU's id must be one the oracle's own logits
    (o64[3]) rank within max(1e-3, 2 f_gap, 8 s) of their best — a
    near-maximiser at the noise fp32 arithmetic itself makes.  Prints the
    distances, the floor, the counts beyond the stated tolerance and every
    differing id with its oracle deficit."""
    rms = lambda a: float(np.sqrt(np.mean(np.square(a)))) if np.size(a) else 0.0
    oids, ogap, ohid = (np.asarray(a) for a in o64[:3])
    ologits = o64[3] if len(o64) > 3 else None
    ids, gap, hid = np.asarray(ids), np.asarray(gap, np.float64), np.asarray(hid, np.float64)
    assert hid.shape == ohid.shape and np.isfinite(hid).all(), label
    f_max = max(float(np.abs(np.asarray(o[2]) - ohid).max()) for o in o32s)
    f_rms = max(rms(np.asarray(o[2]) - ohid) for o in o32s)
    dg = np.concatenate([(np.asarray(o[1]) - ogap).ravel() for o in o32s])
    f_gap = float(np.abs(dg).max()) if dg.size else 0.0
    sg = rms(dg)
    flips32 = max(int((np.asarray(o[0])[:, 1:] != oids[:, 1:]).sum()) for o in o32s)
    err = np.abs(hid - ohid)
    stated = np.maximum(TOL["bf16"], np.abs(ohid) * 2.0 ** -7)
    bound = np.maximum(stated, 2.0 * f_max)
    g, o = ids[:, 1:], oids[:, 1:]
    same = g == o
    gerr = np.abs(gap - ogap)[same]
    gbound = max(TOL["bf16"], 2.0 * f_gap, 8.0 * sg)
    dbound = max(NEAR_TIE, 2.0 * f_gap, 8.0 * sg)
    diff = g != o
    worst = 0.0
    for b, i in zip(*np.nonzero(diff)):
        z = np.asarray(ologits[b, i], np.float64)
        deficit = float(z.max() - z[g[b, i]])
        worst = max(worst, deficit)
        print(f"  {label}: differing id seq {b} pos {i + 1}: gpu {g[b, i]}, oracle {o[b, i]} "
              f"(oracle gap {ogap[b, i]:.3e}); oracle logit deficit of the gpu id {deficit:.3e}")
    print(f"{label}: residual |gpu - oracle| max {err.max():.3e} rms {rms(hid - ohid):.3e} "
          f"({int((err > stated).sum())} of {err.size} beyond the stated bound); fp32-arithmetic "
          f"floor over {len(o32s)} orders max {f_max:.3e} rms {f_rms:.3e}; gap max err "
          f"{gerr.max() if gerr.size else 0:.3e} (floor max {f_gap:.3e}, rms {sg:.3e}); ids "
          f"{g.size}: differing {int(diff.sum())} (oracle gap < 1e-3: "
          f"{int((diff & (ogap < NEAR_TIE)).sum())} of {int((ogap < NEAR_TIE).sum())}; worst oracle "
          f"logit deficit {worst:.3e}, bound {dbound:.3e}); the fp32 draws' ids differ at up to "
          f"{flips32}")
    assert not (err > bound).any(), f"{label}: {int((err > bound).sum())} residual elements beyond bound"
    assert rms(hid - ohid) <= 2.0 * f_rms + 5e-4, label
    assert not (gerr > gbound).any(), f"{label}: gap error {gerr.max():.3e} beyond {gbound:.3e}"
    assert worst <= dbound, f"{label}: an id differs with oracle deficit {worst:.3e} > {dbound:.3e}"


def oracle_block(shape, W, cK, cV, anchors, B, store, arith="f64", with_logits=False):
    """oracle.draft_block over the given sequences, with the final norm and
    LM head of all their rows taken in one pass (the same oracle functions
    draft_block calls per sequence; one pass over a vocabulary-sized LM head
    instead of one per sequence).  Returns (ids, gaps, residual), and the
    logits [n, B-1, V] after them when with_logits."""
    _, _, hid = O.draft_block(shape, W, cK, cV, anchors, B, store, lm_head=False,
                              return_hidden=True, arith=arith)
    n = len(anchors)
    if B == 1:
        out = (np.asarray(anchors, np.int32)[:, None], np.zeros((n, 0)), hid)
        return out + (np.zeros((n, 0, shape.V)),) if with_logits else out
    hf = store(O.rmsnorm(hid[:, 1:].reshape(n * (B - 1), shape.D), W["g_f"], shape.eps))
    z = O.lm_head_logits(hf, W["lm_head"], arith=arith)
    ids = np.concatenate([np.asarray(anchors, np.int32)[:, None],
                          O.argmax_lowest(z).reshape(n, B - 1)], axis=1)
    out = (ids, O.top2_gap(z).reshape(n, B - 1), hid)
    return out + (z.reshape(n, B - 1, -1),) if with_logits else out
