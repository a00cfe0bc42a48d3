"""Test plumbing: tensor conversion and small workload builders."""
import numpy as np
import torch

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
