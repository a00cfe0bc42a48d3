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
