"""Device-side setup of the synthetic workloads (needs the built library).

Creates library handles and caches for a workload from the seeded
generators in ``synth``; no arithmetic of the method happens here.
"""
from __future__ import annotations

import torch

import block_diffusion_drafter_layer_gb300 as dfl
from block_diffusion_drafter_layer_gb300.loop import SpecDecoder

from . import DraftShape, TargetShape, Workload


def draft_model(s: DraftShape, dtype: str, weights: dict, max_pos: int) -> dfl.Model:
    ids = dfl.dflash_build_target_layer_ids(s.n_target_layers, s.n_pick)
    return dfl.Model(D=s.D, H=s.H, G=s.G, d=s.d, F=s.F, V=s.V, n_layers=s.n_layers, dtype=dtype,
                     weights=weights, max_pos=max_pos, qk_norm=True, mask_id=s.mask_id,
                     n_target_layers=s.n_target_layers, n_pick=s.n_pick, target_layer_ids=ids,
                     rope_theta=s.rope_theta, eps=s.eps, embed_scale=s.embed_scale,
                     causal_layers=s.causal_layers, window_layers=s.window_layers,
                     sliding_window=s.sliding_window, conv_group=s.conv_group)


def target_model(t: TargetShape, dtype: str, weights: dict, max_pos: int) -> dfl.Model:
    return dfl.Model(D=t.D, H=t.H, G=t.G, d=t.d, F=t.F, V=t.V, n_layers=t.n_layers, dtype=dtype,
                     weights=weights, max_pos=max_pos, qk_norm=False, mask_id=t.V - 1,
                     rope_theta=t.rope_theta, eps=t.eps)


def kv_cache(s: DraftShape, batch: int, cap: int, dtype: str, k=None, v=None,
             device="cuda") -> dfl.KVCache:
    return dfl.KVCache(s.n_layers, batch, s.G, cap, s.d, dtype, device, k=k, v=v)


def spec_decoder(w: Workload, target: dfl.Model, draft: dfl.Model, cap: int,
                 device="cuda") -> SpecDecoder:
    t, s = w.target, w.draft
    return SpecDecoder(target, draft, t_layers=t.n_layers, t_kv_heads=t.G, d_layers=s.n_layers,
                       d_kv_heads=s.G, head_dim=s.d, D=s.D, n_target_layers=s.n_target_layers,
                       n_pick=s.n_pick, B=w.B, max_prompt=w.prompt_len, cap=cap, device=device)
