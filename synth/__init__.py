"""Seeded synthetic workloads for the DFlash draft path.

This module holds the workload shapes and the seeded random generators that
feed both the CUDA path and the CPU oracle.  It holds none of the method's
arithmetic: every function here only draws random numbers of a stated
distribution and shape.  Both sides receive the same bytes, so parity
compares like with like.

Shapes follow the workloads described for DFlash ("Block Diffusion for Flash
Speculative Decoding"): a tiny fp32 instance, a Qwen3-8B-shaped draft at
batch 1, the same draft at batch 32 with ragged contexts, a
Qwen3.5-35B-A3B-shaped draft at 32K context, and an end-to-end fp32 loop
with a small Llama-style target.  Weights are random-init N(0, 0.02), RMSNorm
gains are 1, target hidden states are N(0, 1).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch

WEIGHT_STD = 0.02


@dataclass(frozen=True)
class DraftShape:
    """Shape of a draft model (all Qwen3-style draft layers)."""
    n_layers: int
    D: int            # hidden size (shared with the target)
    H: int            # query heads
    G: int            # key/value heads (GQA groups)
    d: int            # head dim
    F: int            # SwiGLU intermediate size
    V: int            # vocabulary (shared embedding / LM head)
    mask_id: int      # mask_token_id
    n_target_layers: int
    n_pick: int = 5
    rope_theta: float = 1e6
    eps: float = 1e-6
    embed_scale: float = 1.0
    causal_layers: int = 0    # bit l: layer l is causal (a sliding_attention layer)
    window_layers: int = 0    # bit l: layer l keeps sliding_window keys
    sliding_window: int = 0
    conv_group: int = 0       # channels per conv correction (0: no conv modules)


@dataclass(frozen=True)
class TargetShape:
    """Shape of the small random-init Llama-style causal target (E2E only)."""
    n_layers: int
    D: int
    H: int
    G: int
    d: int
    F: int
    V: int
    rope_theta: float = 1e6
    eps: float = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                    # "f32" or "bf16": storage type of weights/activations
    draft: DraftShape
    batch: int
    B: int                        # block size (anchor + B-1 masks)
    ctx_len: int = 0              # fixed context length (when ctx_range is None)
    ctx_range: Optional[tuple] = None   # (lo, hi) inclusive uniform ragged lengths
    geom_p: float = 0.3           # planted acceptance ~ Geometric(p)
    target: Optional[TargetShape] = None
    prompt_len: int = 0
    new_tokens: int = 0
    seed: int = 1000


QWEN3_8B_DRAFT = DraftShape(n_layers=5, D=4096, H=32, G=8, d=128, F=12288,
                            V=151936, mask_id=151935, n_target_layers=36)

WORKLOADS: Dict[str, Workload] = {
    # tiny fp32 instance
    "tiny_f32": Workload(
        name="tiny_f32", dtype="f32",
        draft=DraftShape(n_layers=2, D=256, H=4, G=2, d=64, F=768, V=1024,
                         mask_id=1023, n_target_layers=12),
        batch=1, B=8, ctx_len=64, geom_p=0.3, seed=1000),
    # Qwen3-8B-shaped draft, batch 1, L = 2048
    "qwen3_8b_b1": Workload(
        name="qwen3_8b_b1", dtype="bf16", draft=QWEN3_8B_DRAFT,
        batch=1, B=16, ctx_len=2048, geom_p=0.2, seed=1001),
    # same draft, batch 32, ragged contexts U{512..8192}
    "qwen3_8b_b32_ragged": Workload(
        name="qwen3_8b_b32_ragged", dtype="bf16", draft=QWEN3_8B_DRAFT,
        batch=32, B=16, ctx_range=(512, 8192), geom_p=0.2, seed=1002),
    # Qwen3.5-35B-A3B-shaped draft at 32K context, batch 4
    "qwen35_a3b_32k": Workload(
        name="qwen35_a3b_32k", dtype="bf16",
        draft=DraftShape(n_layers=5, D=2048, H=16, G=4, d=128, F=6144,
                         V=151936, mask_id=151935, n_target_layers=40),
        batch=4, B=16, ctx_len=32768, geom_p=0.2, seed=1003),
    # end-to-end greedy loop, fp32
    "e2e_f32": Workload(
        name="e2e_f32", dtype="f32",
        draft=DraftShape(n_layers=3, D=512, H=8, G=8, d=64, F=1536, V=4096,
                         mask_id=4095, n_target_layers=8),
        target=TargetShape(n_layers=8, D=512, H=8, G=8, d=64, F=1536, V=4096),
        batch=1, B=16, prompt_len=128, new_tokens=256, geom_p=0.2, seed=1004),
}


def with_(w: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller test cases)."""
    return dataclasses.replace(w, **kw)


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, gen, device, dtype) -> torch.Tensor:
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t.to(dtype)


def draft_weights(shape: DraftShape, dtype: str, seed: int, device="cpu",
                  shared: Optional[dict] = None) -> dict:
    """Random-init draft weights.

    Linear weights are stored out x in (the ``nn.Linear.weight`` layout),
    N(0, 0.02), in ``dtype``.  RMSNorm gains are fp32 ones.  ``shared``
    supplies the target's embedding and LM head when the draft shares them.
    """
    td = torch_dtype(dtype)
    g = _gen(seed, device)
    D, H, G, d, F, V = shape.D, shape.H, shape.G, shape.d, shape.F, shape.V
    ones = lambda n: torch.ones(n, dtype=torch.float32, device=device)
    w = {
        "wc": _normal((D, shape.n_pick * D), WEIGHT_STD, g, device, td),
        "g_c": ones(D),
        "g_f": ones(D),
        "layers": [],
    }
    for _ in range(shape.n_layers):
        w["layers"].append({
            "wq": _normal((H * d, D), WEIGHT_STD, g, device, td),
            "wk": _normal((G * d, D), WEIGHT_STD, g, device, td),
            "wv": _normal((G * d, D), WEIGHT_STD, g, device, td),
            "wo": _normal((D, H * d), WEIGHT_STD, g, device, td),
            "wg": _normal((F, D), WEIGHT_STD, g, device, td),
            "wu": _normal((F, D), WEIGHT_STD, g, device, td),
            "wd": _normal((D, F), WEIGHT_STD, g, device, td),
            "g_in": ones(D), "g_post": ones(D),
            "q_norm": ones(d), "k_norm": ones(d),
        })
    if shared is not None:
        w["embed"] = shared["embed"]
        w["lm_head"] = shared["lm_head"]
    else:
        w["embed"] = _normal((V, D), WEIGHT_STD, g, device, td)
        w["lm_head"] = _normal((V, D), WEIGHT_STD, g, device, td)
    return w


def target_weights(shape: TargetShape, dtype: str, seed: int, device="cpu") -> dict:
    """Random-init Llama-style target (no q/k norm), same layout conventions."""
    td = torch_dtype(dtype)
    g = _gen(seed, device)
    D, H, G, d, F, V = shape.D, shape.H, shape.G, shape.d, shape.F, shape.V
    ones = lambda n: torch.ones(n, dtype=torch.float32, device=device)
    w = {
        "embed": _normal((V, D), WEIGHT_STD, g, device, td),
        "lm_head": _normal((V, D), WEIGHT_STD, g, device, td),
        "g_final": ones(D),
        "layers": [],
    }
    for _ in range(shape.n_layers):
        w["layers"].append({
            "wq": _normal((H * d, D), WEIGHT_STD, g, device, td),
            "wk": _normal((G * d, D), WEIGHT_STD, g, device, td),
            "wv": _normal((G * d, D), WEIGHT_STD, g, device, td),
            "wo": _normal((D, H * d), WEIGHT_STD, g, device, td),
            "wg": _normal((F, D), WEIGHT_STD, g, device, td),
            "wu": _normal((F, D), WEIGHT_STD, g, device, td),
            "wd": _normal((D, F), WEIGHT_STD, g, device, td),
            "g_in": ones(D), "g_post": ones(D),
        })
    return w


def target_hidden_states(T: int, D: int, n: int, dtype: str, seed: int,
                         device="cpu") -> List[torch.Tensor]:
    """``n`` synthetic target-layer hidden states, each [T, D], N(0, 1)."""
    g = _gen(seed + 7, device)
    return [_normal((T, D), 1.0, g, device, torch_dtype(dtype)) for _ in range(n)]


def ctx_lengths(w: Workload) -> List[int]:
    """Per-sequence context lengths (fixed, or uniform ragged in ctx_range)."""
    if w.ctx_range is None:
        return [w.ctx_len] * w.batch
    rng = np.random.default_rng(w.seed + 11)
    lo, hi = w.ctx_range
    return [int(x) for x in rng.integers(lo, hi + 1, size=w.batch)]


def anchors(batch: int, V: int, mask_id: int, seed: int) -> np.ndarray:
    """Anchor tokens, uniform over the vocabulary without the mask id."""
    rng = np.random.default_rng(seed + 13)
    a = rng.integers(0, V - 1, size=batch).astype(np.int32)
    return np.where(a >= mask_id, a + 1, a).astype(np.int32)


def random_kv_cache(batch: int, G: int, cap: int, d: int, n_layers: int,
                    v_std: float, dtype: str, seed: int, device="cpu"):
    """Synthetic injected context K/V, [batch, G, cap, d] per layer.

    K entries are N(0, 1) (a k_norm'd, rotated key has unit RMS); V entries
    are N(0, v_std^2) with v_std = 0.02 * sqrt(D) (a unit-RMS feature through
    an N(0, 0.02) projection)."""
    g = _gen(seed + 17, device)
    td = torch_dtype(dtype)
    K = [_normal((batch, G, cap, d), 1.0, g, device, td) for _ in range(n_layers)]
    V = [_normal((batch, G, cap, d), v_std, g, device, td) for _ in range(n_layers)]
    return K, V


def random_ids(shape, V: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, V, size=shape).astype(np.int32)


def planted_posterior(draft: np.ndarray, p: float, V: int, seed: int):
    """Target posterior ids planted to match a draft for a Geometric prefix.

    ``draft`` is [batch, B] (column 0 = anchor).  For each sequence a match
    length k ~ Geometric(p) on {0, 1, ...} (P(k) = (1-p)^k p) is capped at
    B-1.  For j < k, post[j] = draft[j+1]; if k < B-1, post[k] is forced to
    differ from draft[k+1]; every other entry is uniform over the vocabulary.
    Returns (post, k).
    """
    rng = np.random.default_rng(seed)
    batch, B = draft.shape
    post = rng.integers(0, V, size=(batch, B)).astype(np.int64)
    k = np.minimum(rng.geometric(p, size=batch) - 1, B - 1)
    for b in range(batch):
        kb = int(k[b])
        post[b, :kb] = draft[b, 1:kb + 1]
        if kb < B - 1:
            r = int(rng.integers(0, V - 1))
            post[b, kb] = (int(draft[b, kb + 1]) + 1 + r) % V
    return post.astype(np.int32), k.astype(np.int32)


def round_uniforms(seed: int, B: int):
    """Seeded uniform [0, 1) draws of a sampling loop (T > 0), as a function
    of the round r: (u_first, u_draft [B-1], u_accept [B-1], u_sample).
    u_first draws the first token from the prefill's last row (round 0);
    u_draft draws the B-1 drafts, u_accept decides each draft's acceptance
    and u_sample draws the token after the accepted prefix.  Both the GPU
    loop and the oracle's loop consume these same numbers."""
    def draws(r: int):
        g = np.random.default_rng([seed, r])
        return (float(g.random()), g.random(B - 1), g.random(B - 1), float(g.random()))
    return draws


def selector_weights(D: int, V: int, dtype: str, seed: int, rank: int = 256,
                     device="cpu") -> dict:
    """Random-init weights of a DFlash 2 candidate selector: the context-gate
    projection w_h [rank, D] with N(0, 1/D) entries (unit-scale gates from
    unit-RMS rows) and two codebooks [V, rank] with N(0, rank^-1/2) entries,
    so that a pair term summed over the rank has unit scale, comparable to
    the draft logits' gaps."""
    td = torch_dtype(dtype)
    g = _gen(seed, device)
    return {"w_h": _normal((rank, D), D ** -0.5, g, device, td),
            "code_pred": _normal((V, rank), rank ** -0.25, g, device, td),
            "code_succ": _normal((V, rank), rank ** -0.25, g, device, td)}


def add_conv_weights(weights: dict, shape: DraftShape, dtype: str, seed: int,
                     device="cpu") -> dict:
    """Random-init conv modules (one around attention, one around the FFN)
    added to each layer of ``weights``: kernel projections [2 * 2 * (D //
    conv_group), D] with N(0, 0.1^2 / D) entries (corrections of about 0.1
    from unit-RMS rows) and fp32 base kernels [2 (call), 2 (tap), D] near
    the identity (tap 0 about 1, tap 1 about 0.3 in size)."""
    td = torch_dtype(dtype)
    g = _gen(seed, device)
    D, ng = shape.D, shape.D // shape.conv_group
    for lay in weights["layers"]:
        for k in ("att", "mlp"):
            lay[f"conv_{k}_kp"] = _normal((4 * ng, D), 0.1 * D ** -0.5, g, device, td)
            base = _normal((2, 2, D), 0.3, g, device, torch.float32)
            base[:, 0] += 1.0
            lay[f"conv_{k}_base"] = base
    return weights
