"""DFlash oracle: numpy fp64 restatement of the draft path (test infrastructure).

Pages cited (by title and section):
  [tutorial]  "A3-dflash — DFlash: Block Diffusion for Flash Speculative
              Decoding" (llm-paper-tutorials), §2.1.1 feature extraction
              (worked example), §2.1.2 KV injection, §2.1.3 parallel drafting.
  [translation] papercache.org translation of the paper, §3.1 speedup
              analysis, §4.1 inference design, experimental setup.
  [notes]     tom-jerr notes on DFlash, "DFlash Inference Workflow" and the
              acceptance-length identity (proof §1).
  [reading]   txtmix "DFlash：把扩散模型关进草稿阶段…" source reading, §5 target
              feature KV injection, §6 one-step denoising, §8 losslessness
              from the verification rule, §9 one request through the system,
              §11 dflash_config fields, §13-§14 DFlash 2 (the candidate
              selector).

Arithmetic: every dot product and reduction in fp64.  Values are then
rounded at the "storage points" where the GPU path stores a tensor, using
``store`` (fp32 rounding in f32 mode, fp32-then-bf16 round-to-nearest-even
in bf16 mode).  The residual stream, the softmax and the logits are fp32.
Argmax is taken on fp32-rounded logits, lowest index first on ties.

What pins each function (tests/test_oracle_*.py):
  build_target_layer_ids   rule table + end points + 1-pick middle layer
  fuse_context             printed worked example ([tutorial] §2.1.1),
                           RMS = 1 invariant, W_c byte counts
  rmsnorm                  torch.nn.functional.rms_norm, RMS = 1
  rope                     complex-multiplication form, relative-position
                           invariance, identity at position 0, norm kept
  attention                torch scaled_dot_product_attention (fp64) with
                           grouped K/V heads, uniform-score closed form
  draft_key_visible        causal window of one: each row's own value
                           exactly; causal rows ignore later rows; a window
                           ignores older context; the anchor's causal output
                           equals full attention over explicitly sliced keys;
                           a window covering all keys changes nothing
  dynamic_conv             taps (1, 0) are the identity and (0, 1) a shift
                           by one row; one correction per channel group;
                           causal (a row ignores later rows); in a layer,
                           identity convs change nothing and a shifting
                           finish conv shifts the sublayer's increment
  inject_kv                identity k/v projections of distinct scales:
                           K is the per-head RMSNorm (torch) with the k_norm
                           gains, V the scaled slice; a row appended at
                           positions p is the position-0 K rotated by p
                           (complex form): k_norm before RoPE, at the cache
                           positions
  draft_layer/draft_block  reductions: zero W_o and W_d give the identity;
                           zero W_q gives uniform attention (closed form);
                           context enters only through K/V; SwiGLU with
                           diagonal gate/up/down equals torch's
                           silu(gate) * up; zero q_norm gains give the mean of
                           all values, and a scaled W_q changes nothing;
                           a d = 2 head places the anchor at position L (it
                           scores a key turned by L radians like its own);
                           planted LM-head rows: drafts come from rows 1..B-1
                           through the final norm (torch rms_norm gap)
  embed_block              identity layers return scale x the block's rows
  lm_head_argmax           brute force with planted ties / gaps
  verify_greedy            exhaustive enumeration on tiny B and V;
                           tau in [1, B]; E[tau] closed form under planted
                           Geometric acceptance (Monte Carlo)
  target_forward + loops   losslessness: speculative output equals the
                           target's own greedy autoregressive output
  sample_from              hand-computed inverse-CDF buckets (zero weights
                           skipped, scale invariance), Monte Carlo frequencies
  verify_rejection         the speculative-sampling theorem (chi-square: the
                           emitted token follows p whatever q is), acceptance
                           rate sum_x min(p, q), p = q accepts everything,
                           one-hot p and q reduce to verify_greedy
                           (exhaustive on tiny B and V)
  speculative_sample_generate  T -> 0 limit equals the greedy loop
  topk_lowest              brute force by repeated argmax on tiny rows with
                           planted ties
  select_candidates        k = 1 and a zero codebook reduce the walk to the
                           argmax; a planted bigram chain (pair term on the
                           predecessor's and successor's own codebooks) is
                           followed from the anchor; relabelling the
                           vocabulary relabels the path
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "build_target_layer_ids", "f32", "bf16", "storage", "rmsnorm",
    "rope_angles", "rope", "linear", "attention", "fuse_context", "inject_kv",
    "embed_block", "draft_layer", "draft_block", "lm_head_logits",
    "argmax_lowest", "top2_gap", "verify_greedy", "expected_tau_from_prefix",
    "TargetCache", "target_forward", "ar_generate", "speculative_generate",
    "softmax_t", "sample_from", "verify_rejection", "acceptance_probability",
    "speculative_sample_generate", "topk_lowest", "select_candidates", "draft_key_visible",
    "dynamic_conv",
]


# ---------------------------------------------------------------------------
# target layer selection  ([reading] §5; [translation] experimental setup)
# ---------------------------------------------------------------------------
def build_target_layer_ids(num_target_layers: int, n_pick: int) -> List[int]:
    """Uniformly spaced 0-based layer ids in [1, num_target_layers - 3].

    [reading] §5: picks are spread uniformly between the second layer and
    the third-from-last (0-based 1 .. num_target_layers-3); a draft that
    takes a single pick takes the middle layer.  The pages do not say how a
    non-integer spacing rounds; this reads it as round-half-up.  The middle
    layer is read as num_target_layers // 2.
    """
    if n_pick < 1:
        raise ValueError("n_pick must be >= 1")
    if n_pick == 1:
        return [num_target_layers // 2]
    lo, hi = 1, num_target_layers - 3
    if hi < lo:
        raise ValueError("target too shallow")
    span = hi - lo
    ids = []
    for i in range(n_pick):
        # round_half_up(i * span / (n_pick - 1)) in exact integer arithmetic
        num = 2 * i * span + (n_pick - 1)
        ids.append(lo + num // (2 * (n_pick - 1)))
    return ids


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------
def f32(x) -> np.ndarray:
    """Round to fp32 (round-to-nearest-even) and return as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16(x) -> np.ndarray:
    """Round to fp32, then to bfloat16 (round-to-nearest-even), as fp64.

    bfloat16 keeps the upper 16 bits of an IEEE fp32 word; rounding adds
    0x7FFF plus the lowest kept bit before truncating."""
    a = np.asarray(x, dtype=np.float64).astype(np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def storage(dtype: str):
    """The rounding applied where the path stores an activation tensor."""
    return {"f32": f32, "bf16": bf16}[dtype]


# ---------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gain over the last axis.

    [tutorial] §2.1.1 (the fusion snippet's RMSNorm: eps 1e-6, gain applied
    after normalisation)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, dtype=np.float64)


def _f32_order(arith: str):
    """None for fp64 arithmetic; else the seed of the order fp32 sums take
    (0: natural order; k > 0: the reduction axis permuted by a permutation
    seeded with k, the same sum in another order)."""
    if arith == "f64":
        return None
    if arith == "f32":
        return 0
    if arith.startswith("f32."):
        return int(arith[4:])
    raise ValueError(arith)


def linear(x: np.ndarray, W: np.ndarray, chunk: int = 1 << 14, arith: str = "f64") -> np.ndarray:
    """y = x W^T with W stored out x in (``nn.Linear.weight``), fp64.

    Large W are upcast a block of output rows at a time.  arith="f32" (or
    "f32.k", the sum over the input axis in the order of a seeded
    permutation) takes the products and sums in fp32 instead (numpy's fp32
    matmul): the arithmetic-precision reference the bf16 tests measure their
    floor with (the storage points are unchanged)."""
    order = _f32_order(arith)
    if order is not None:
        x32 = np.asarray(x, dtype=np.float32)
        perm = np.random.default_rng(order).permutation(x32.shape[-1]) if order else None
        if perm is not None:
            x32 = x32[..., perm]
        out = np.empty(x32.shape[:-1] + (W.shape[0],), dtype=np.float64)
        for s in range(0, W.shape[0], chunk):
            Wc = np.asarray(W[s:s + chunk], dtype=np.float32)
            out[..., s:s + chunk] = x32 @ (Wc[:, perm] if perm is not None else Wc).T
        return out
    x = np.asarray(x, dtype=np.float64)
    n_out = W.shape[0]
    if W.dtype == np.float64 or n_out <= chunk:
        return x @ np.asarray(W, dtype=np.float64).T
    out = np.empty(x.shape[:-1] + (n_out,), dtype=np.float64)
    for s in range(0, n_out, chunk):
        out[..., s:s + chunk] = x @ W[s:s + chunk].astype(np.float64).T
    return out


def rope_angles(pos: np.ndarray, d: int, theta: float) -> np.ndarray:
    """phi[p, i] = pos_p * theta^(-2i/d), i < d/2 (fp64)."""
    i = np.arange(d // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary embedding with rotate-half pairing (i, i + d/2).

    x: [n, heads, d]; pos: [n].  Pair (x_i, x_{i+d/2}) is rotated by
    phi = pos * theta^(-2i/d):
        x_i'       = x_i cos(phi) - x_{i+d/2} sin(phi)
        x_{i+d/2}' = x_{i+d/2} cos(phi) + x_i sin(phi)
    (Qwen3/Llama convention, which the draft and target layers follow.)"""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    phi = rope_angles(pos, d, theta)[:, None, :]      # [n, 1, d/2]
    c, s = np.cos(phi), np.sin(phi)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray,
              key_visible: Optional[np.ndarray] = None, arith: str = "f64") -> np.ndarray:
    """Softmax attention with grouped K/V heads, fp64.

    q: [n, H, d]; K, V: [m, G, d]; query head h reads K/V head
    h // (H / G).  Scale 1/sqrt(d).  ``key_visible`` [n, m] (bool) masks
    keys; None means every key is visible (the draft's bidirectional block
    over [context ; block], [reading] §6: full-attention layers are
    non-causal).  arith="f32" / "f32.k": scores, softmax and the weighted
    sum in fp32, for "f32.k" over the keys in a seeded permuted order (see
    ``linear``).  Returns [n, H, d]."""
    n, H, d = q.shape
    m, G, _ = K.shape
    rep = H // G
    order = _f32_order(arith)
    if order is not None:
        q, K, V = (np.asarray(a, dtype=np.float32) for a in (q, K, V))
        if order:
            perm = np.random.default_rng(order).permutation(m)
            K, V = K[perm], V[perm]
            if key_visible is not None:
                key_visible = key_visible[:, perm]
    out = np.empty((n, H, d), dtype=np.float64)
    for h in range(H):
        g = h // rep
        s = (q[:, h, :] @ K[:, g, :].T) / q.dtype.type(math.sqrt(d))   # [n, m]
        if key_visible is not None:
            s = np.where(key_visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, g, :]
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------------------
# context fusion ([tutorial] §2.1.1 formula and snippet; [reading] §5)
# ---------------------------------------------------------------------------
def fuse_context(hiddens: Sequence[np.ndarray], Wc: np.ndarray, g_c: np.ndarray,
                 eps: float, store=f32) -> np.ndarray:
    """H_t = RMSNorm(W_c [H^(l1); ...; H^(l5)]).

    The picked layers' hidden states are concatenated along the hidden axis
    in ascending layer order ([T, 5D]), projected by W_c (D x 5D, no bias:
    y = x W_c^T) and RMS-normalised.  H_t is stored (``store``)."""
    X = np.concatenate([np.asarray(h, dtype=np.float64) for h in hiddens], axis=-1)
    Y = linear(X, Wc)
    return store(rmsnorm(Y, g_c, eps))


# ---------------------------------------------------------------------------
# K/V injection ([tutorial] §2.1.2; [reading] §5; [translation] §4.1)
# ---------------------------------------------------------------------------
def inject_kv(H_t: np.ndarray, layer: dict, pos: np.ndarray, G: int, d: int,
              theta: float, eps: float, store=f32, qk_norm: bool = True):
    """Context K/V entries of one draft layer.

    The context feature goes through this layer's k_proj and v_proj only
    (never Q, o_proj or the FFN): K = RoPE(k_norm(H_t W_k^T), pos),
    V = H_t W_v^T.  Returns stored K, V of shape [T, G, d]."""
    T = H_t.shape[0]
    k = linear(H_t, layer["wk"]).reshape(T, G, d)
    if qk_norm:
        k = rmsnorm(k, layer["k_norm"], eps)
    k = rope(k, pos, theta)
    v = linear(H_t, layer["wv"]).reshape(T, G, d)
    return store(k), store(v)


# ---------------------------------------------------------------------------
# block draft forward ([reading] §5, §6, §9; [tutorial] §2.1.2–2.1.3)
# ---------------------------------------------------------------------------
def embed_block(embed: np.ndarray, anchor: int, mask_id: int, B: int,
                scale: float) -> np.ndarray:
    """Block input [anchor, mask x (B-1)] through the shared embedding, times
    input_embedding_scale ([reading] §6 and §9), as the fp32 residual."""
    ids = [int(anchor)] + [int(mask_id)] * (B - 1)
    return f32(np.asarray(embed[ids], dtype=np.float64) * scale)


def draft_key_visible(L: int, B: int, causal: bool, window: int) -> np.ndarray:
    """Which keys each block row sees in a draft layer ([reading] §6: a
    sliding_attention layer is causal unless configured otherwise, and its
    visible range is cut to the sliding window; a full_attention layer is
    bidirectional).  Keys are [context ; block] at positions 0 .. L+B-1,
    block row i at position p = L + i.  A causal row sees keys at or before
    p; a window of W keeps keys after p - W.  Returns [B, L + B] bool."""
    p = np.arange(L, L + B)[:, None]
    j = np.arange(L + B)[None, :]
    vis = np.ones((B, L + B), dtype=bool)
    if causal:
        vis &= j <= p
    if window > 0:
        vis &= j > p - window
    return vis


def dynamic_conv(x: np.ndarray, corr: np.ndarray, base: np.ndarray, group: int) -> np.ndarray:
    """DFlash 2's two-tap grouped dynamic causal conv over one block
    ([reading] §13, §14): out_t = k_t0 * x_t + k_t1 * x_(t-1), depthwise,
    with each coefficient the learned base kernel plus a correction computed
    from the row's hidden state, one correction per group of ``group``
    channels.  The block's first row has no predecessor (zero: the module
    keeps no state across steps; every later row reads the one before it,
    so the first mask position reads the anchor).

    x: [B, D]; corr: [B, 2, D // group] (tap, group); base: [2, D] (tap,
    channel).  Returns [B, D] fp64."""
    x = np.asarray(x, np.float64)
    k = np.asarray(base, np.float64)[None] + np.repeat(np.asarray(corr, np.float64), group, axis=-1)
    prev = np.concatenate([np.zeros((1, x.shape[1])), x[:-1]], axis=0)
    return k[:, 0] * x + k[:, 1] * prev


def _conv_pair(x: np.ndarray, kp: np.ndarray, base: np.ndarray, group: int, arith: str = "f64"):
    """The corrections of a conv module's two calls from the rows x:
    kernel_projection kp [2 * 2 * (D // group), D] (no bias), read as
    [call, tap, group]; base [2 (call), 2 (tap), D].  Returns the prepare
    and finish functions (y -> conv of y with that call's coefficients; the
    prepared rows are stored in fp32, and the sublayer output y is stored in
    fp32 before its finish conv)."""
    B, D = x.shape
    corr = linear(x, kp, arith=arith).reshape(B, 2, 2, D // group)
    return (lambda y: f32(dynamic_conv(y, corr[:, 0], base[0], group)),
            lambda y: dynamic_conv(f32(y), corr[:, 1], base[1], group))


def draft_layer(x: np.ndarray, layer: dict, ctx_K: np.ndarray, ctx_V: np.ndarray,
                pos: np.ndarray, H: int, G: int, d: int, theta: float, eps: float,
                store=f32, mask: Optional[np.ndarray] = None, conv_group: int = 0,
                arith: str = "f64") -> np.ndarray:
    """One Qwen3-style draft decoder layer over one sequence's block.

    x: [B, D] fp32 residual.  ctx_K, ctx_V: [L, G, d] injected context.
    Queries come from the block only; keys/values are [context ; block]
    concatenated along the sequence ([tutorial] §2.1.2; [reading] §5);
    attention is bidirectional unless ``mask`` (draft_key_visible) says
    otherwise.  Then o_proj + residual and a SwiGLU FFN + residual, each
    sublayer pre-normalised.

    conv_group > 0 (DFlash 2, [reading] §13, §14): each sublayer has its own
    conv module (layer["conv_att_kp"] / ["conv_att_base"] and the "mlp"
    pair).  Its corrections come from the residual entering the sublayer;
    the prepare call convolves that residual before the sublayer's norm and
    the finish call convolves the sublayer's output before the residual
    add (x + finish(f(norm(prepare(x)))))."""
    B = x.shape[0]
    prep = fin = lambda y: y
    if conv_group:
        prep, fin = _conv_pair(x, layer["conv_att_kp"], layer["conv_att_base"], conv_group, arith)
    h = store(rmsnorm(prep(x), layer["g_in"], eps))
    q = linear(h, layer["wq"], arith=arith).reshape(B, H, d)
    k = linear(h, layer["wk"], arith=arith).reshape(B, G, d)
    v = linear(h, layer["wv"], arith=arith).reshape(B, G, d)
    q = store(rope(rmsnorm(q, layer["q_norm"], eps), pos, theta))
    k = store(rope(rmsnorm(k, layer["k_norm"], eps), pos, theta))
    v = store(v)
    K = np.concatenate([ctx_K, k], axis=0)
    Vv = np.concatenate([ctx_V, v], axis=0)
    o = store(attention(q, K, Vv, mask, arith=arith).reshape(B, H * d))
    x = f32(x + fin(linear(o, layer["wo"], arith=arith)))
    if conv_group:
        prep, fin = _conv_pair(x, layer["conv_mlp_kp"], layer["conv_mlp_base"], conv_group, arith)
    h2 = store(rmsnorm(prep(x), layer["g_post"], eps))
    a = store(silu(linear(h2, layer["wg"], arith=arith)) * linear(h2, layer["wu"], arith=arith))
    return f32(x + fin(linear(a, layer["wd"], arith=arith)))


def lm_head_logits(hf: np.ndarray, W_lm: np.ndarray, arith: str = "f64") -> np.ndarray:
    """fp32 logits hf W_lm^T (the target's shared LM head)."""
    return f32(linear(hf, W_lm, arith=arith))


def argmax_lowest(z: np.ndarray) -> np.ndarray:
    """Argmax over the last axis; ties go to the lowest index."""
    return np.argmax(z, axis=-1).astype(np.int32)


def top2_gap(z: np.ndarray) -> np.ndarray:
    """Largest minus second-largest value over the last axis (0 on a tie)."""
    part = np.partition(z, -2, axis=-1)
    return part[..., -1] - part[..., -2]


def draft_block(shape, W: dict, ctx_K: List[List[np.ndarray]],
                ctx_V: List[List[np.ndarray]], anchors: Sequence[int], B: int,
                store=f32, return_logits: bool = False, lm_head: bool = True,
                return_hidden: bool = False, arith: str = "f64"):
    """Single-pass draft of one block per sequence.

    ``shape`` has D, H, G, d, eps, rope_theta, mask_id, embed_scale.
    ``ctx_K[l][b]`` / ``ctx_V[l][b]``: [L_b, G, d] injected context of
    layer l, sequence b.  The block [anchor, mask x (B-1)] sits at positions
    L_b .. L_b + B - 1 ([reading] §9: positions run from start - ctx_len).
    Every row goes through every layer (the anchor's K/V feed the others);
    layer l is causal when bit l of shape.causal_layers is set and keeps a
    window of shape.sliding_window keys when bit l of shape.window_layers is
    (draft_key_visible; both default to none: bidirectional layers);
    the final RMSNorm and the shared LM head run on rows 1..B-1 only, and
    each draft id is the argmax of its fp32 logits ([reading] §6, §14).

    Returns ids [batch, B] (column 0 = anchor), gap [batch, B-1] and,
    if asked, logits [batch, B-1, V] and the fp32 residual stream after the
    last layer [batch, B, D].  With lm_head=False only the residual stream is
    computed (ids and gaps are left zero).  arith="f32" runs every product
    and sum in fp32 with the same storage points (``linear``): the distance
    of that run from the fp64 one is the floor any fp32 implementation of
    the block sits at."""
    batch = len(anchors)
    ids = np.zeros((batch, B), dtype=np.int32)
    gaps = np.zeros((batch, B - 1), dtype=np.float64)
    all_logits, hidden = [], []
    for b in range(batch):
        L = ctx_K[0][b].shape[0]
        pos = np.arange(L, L + B)
        x = embed_block(W["embed"], anchors[b], shape.mask_id, B, shape.embed_scale)
        for l, layer in enumerate(W["layers"]):
            causal = bool((getattr(shape, "causal_layers", 0) >> l) & 1)
            window = (getattr(shape, "sliding_window", 0)
                      if (getattr(shape, "window_layers", 0) >> l) & 1 else 0)
            mask = draft_key_visible(L, B, causal, window) if causal or window else None
            x = draft_layer(x, layer, ctx_K[l][b], ctx_V[l][b], pos, shape.H,
                            shape.G, shape.d, shape.rope_theta, shape.eps, store, mask,
                            getattr(shape, "conv_group", 0), arith=arith)
        hidden.append(x)
        ids[b, 0] = anchors[b]
        if not lm_head:
            continue
        hf = store(rmsnorm(x[1:], W["g_f"], shape.eps))
        z = lm_head_logits(hf, W["lm_head"], arith=arith)
        ids[b, 1:] = argmax_lowest(z)
        gaps[b] = top2_gap(z)
        if return_logits:
            all_logits.append(z)
    out = [ids, gaps]
    if return_logits:
        out.append(np.stack(all_logits))
    if return_hidden:
        out.append(np.stack(hidden))
    return tuple(out)


# ---------------------------------------------------------------------------
# greedy verification ([reading] §8, §9; [translation] §3.1)
# ---------------------------------------------------------------------------
def verify_greedy(draft: np.ndarray, post: np.ndarray, start: np.ndarray):
    """Longest matching prefix plus a bonus token, per sequence.

    draft[b] = [anchor, d_1 .. d_{B-1}]; post[b, j] is the target's argmax at
    block position j.  a_b counts the leading j >= 1 with
    draft[b, j] == post[b, j-1] (the first mismatch ends the prefix);
    bonus_b = post[b, a_b]; tau_b = a_b + 1 in [1, B].  The emitted tokens
    are draft[b, 1..a_b] then the bonus; the target cache keeps
    start_b + a_b + 1 entries.

    Returns (accept, bonus, out_tokens [batch, B] padded with -1, new_len)."""
    draft = np.asarray(draft)
    post = np.asarray(post)
    batch, B = draft.shape
    accept = np.zeros(batch, dtype=np.int32)
    bonus = np.zeros(batch, dtype=np.int32)
    out = np.full((batch, B), -1, dtype=np.int32)
    new_len = np.zeros(batch, dtype=np.int32)
    for b in range(batch):
        a = 0
        while a < B - 1 and draft[b, a + 1] == post[b, a]:
            a += 1
        accept[b] = a
        bonus[b] = post[b, a]
        out[b, :a] = draft[b, 1:a + 1]
        out[b, a] = bonus[b]
        new_len[b] = int(start[b]) + a + 1
    return accept, bonus, out, new_len


def expected_tau_from_prefix(prefix_match_prob: Sequence[float]) -> float:
    """E[tau] = 1 + sum_k P(first k drafts all match), k = 1 .. B-1.

    [notes] proof §1: for a non-negative integer match length,
    E = sum_k P(match length >= k) = sum_k P(prefix of length k matches);
    the bonus token adds one ([translation] §3.1: tau in [1, gamma + 1])."""
    return 1.0 + float(np.sum(prefix_match_prob))


# ---------------------------------------------------------------------------
# sampling verification, T > 0 ([reading] §8: the acceptance probability is
# p/q, the prefix ends at the first rejection, and the token after it is
# drawn from max(p - q, 0) normalised; [translation] T = 1 experiments)
# ---------------------------------------------------------------------------
def softmax_t(z: np.ndarray, T: float) -> np.ndarray:
    """softmax(z / T) over the last axis in fp64, T > 0."""
    if not T > 0:
        raise ValueError("temperature must be positive")
    a = np.asarray(z, dtype=np.float64) / T
    a = a - a.max(axis=-1, keepdims=True)
    e = np.exp(a)
    return e / e.sum(axis=-1, keepdims=True)


def sample_from(weights: np.ndarray, u: float) -> int:
    """Inverse-CDF draw from non-negative weights (need not sum to 1): the
    smallest index i whose running sum (fp64, in index order) exceeds
    u * total, u in [0, 1).  An index of zero weight is never drawn."""
    w = np.asarray(weights, dtype=np.float64)
    c = np.cumsum(w)
    i = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(i, len(w) - 1)


def verify_rejection(draft: np.ndarray, q: np.ndarray, p: np.ndarray,
                     u_accept: np.ndarray, u_sample: np.ndarray, start: np.ndarray):
    """Speculative sampling verification per sequence.

    draft[b] = [anchor, d_1 .. d_{B-1}], d_j drawn from q[b, j-1], the
    draft's distribution at block position j.  p[b, j] (j = 0 .. B-1) is the
    target's distribution of the token that follows block position j.  d_j
    is accepted when u_accept[b, j-1] * q[b, j-1][d_j] < p[b, j-1][d_j]
    (probability min(1, p/q)); the first rejection ends the prefix, a_b
    drafts accepted.  The token after the prefix is drawn with u_sample[b]:
    from max(p[b, a] - q[b, a], 0) renormalised when d_{a+1} was rejected,
    from p[b, B-1] when every draft was accepted.  tau_b = a_b + 1.

    Returns (accept, token, out_tokens [batch, B] padded with -1, new_len),
    shaped like verify_greedy's result (token in the bonus's place)."""
    draft = np.asarray(draft)
    batch, B = draft.shape
    accept = np.zeros(batch, dtype=np.int32)
    token = np.zeros(batch, dtype=np.int32)
    out = np.full((batch, B), -1, dtype=np.int32)
    new_len = np.zeros(batch, dtype=np.int32)
    for b in range(batch):
        a = 0
        while a < B - 1:
            d = int(draft[b, a + 1])
            if u_accept[b, a] * q[b, a][d] < p[b, a][d]:
                a += 1
            else:
                break
        if a < B - 1:
            res = np.maximum(np.asarray(p[b, a], np.float64) - np.asarray(q[b, a], np.float64), 0.0)
            tok = sample_from(res if res.sum() > 0 else p[b, a], float(u_sample[b]))
        else:
            tok = sample_from(p[b, B - 1], float(u_sample[b]))
        accept[b] = a
        token[b] = tok
        out[b, :a] = draft[b, 1:a + 1]
        out[b, a] = tok
        new_len[b] = int(start[b]) + a + 1
    return accept, token, out, new_len


def acceptance_probability(p: np.ndarray, q: np.ndarray) -> float:
    """P(a draft drawn from q is accepted against p) = sum_x min(p(x), q(x))."""
    return float(np.minimum(np.asarray(p, np.float64), np.asarray(q, np.float64)).sum())


# ---------------------------------------------------------------------------
# DFlash 2 candidate selection  ([reading] §13, §14)
# ---------------------------------------------------------------------------
def topk_lowest(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values of each row of z, ordered by value
    (descending) and, among equal values, by index (ascending)."""
    z = np.asarray(z)
    out = np.empty(z.shape[:-1] + (k,), dtype=np.int32)
    for idx in np.ndindex(*z.shape[:-1]):
        row = z[idx]
        order = np.lexsort((np.arange(row.shape[0]), -row))
        out[idx] = order[:k]
    return out


def select_candidates(logits: np.ndarray, hidden: np.ndarray, anchor: int,
                      W_h: np.ndarray, code_pred: np.ndarray, code_succ: np.ndarray,
                      top_k: int):
    """The DFlash 2 candidate selector on one block, greedy.

    logits: [n, V], the draft's logits at block positions 1..n (the anchor
    makes none); hidden: [n, D], the final-normed rows that produced them.
    Each position keeps its top_k tokens (topk_lowest) with their logits as
    unary scores U_t.  The context gate is H_t = W_h hidden_t (W_h [r, D],
    no bias).  Starting from the anchor, the walk scores every candidate b
    of position t after the chosen predecessor a as
        S_t(a, b) = U_t(b) + sum_r code_pred[a, r] * H_t[r] * code_succ[b, r]
    and keeps the best (the earlier candidate on a tie); the kept token is
    the next predecessor.  Returns (path [n], candidates [n, top_k],
    chosen scores [n])."""
    logits = np.asarray(logits, np.float64)
    n = logits.shape[0]
    cand = topk_lowest(logits, top_k)
    unary = np.take_along_axis(logits, cand, axis=-1)
    H = np.asarray(hidden, np.float64) @ np.asarray(W_h, np.float64).T
    A = np.asarray(code_pred, np.float64)
    Bc = np.asarray(code_succ, np.float64)
    path = np.zeros(n, dtype=np.int32)
    best = np.zeros(n)
    pred = int(anchor)
    for t in range(n):
        gate = A[pred] * H[t]
        scores = unary[t] + Bc[cand[t]] @ gate
        j = int(np.argmax(scores))
        path[t] = cand[t, j]
        best[t] = scores[j]
        pred = int(path[t])
    return path, cand, best


# ---------------------------------------------------------------------------
# end-to-end check: Llama-style causal target and the two decoders
# ([reading] §9; [tutorial] data-flow section)
# ---------------------------------------------------------------------------
class TargetCache:
    """Per-layer causal K/V history of one sequence ([G, len, d] lists)."""

    def __init__(self, n_layers: int):
        self.K = [[] for _ in range(n_layers)]
        self.V = [[] for _ in range(n_layers)]

    def __len__(self):
        return len(self.K[0])

    def crop(self, n: int):
        """Keep the first n positions (the trim after verification)."""
        for l in range(len(self.K)):
            del self.K[l][n:]
            del self.V[l][n:]


def target_forward(tshape, TW: dict, cache: TargetCache, tokens: Sequence[int],
                   tap_ids: Sequence[int], store=f32, logits_out: list = None):
    """Causal forward of the target over ``tokens`` appended to ``cache``.

    One row at a time (row i at position len(cache) sees keys 0..pos), so a
    row's result does not depend on how many rows are processed together.
    Returns (argmax ids per row, taps [n_pick, n, D] fp32): a tap is the
    residual stream after 0-based decoder layer ``id``.  ``logits_out``
    (a list), when given, receives each row's fp32 logits."""
    D, H, G, d = tshape.D, tshape.H, tshape.G, tshape.d
    ids_out, taps = [], [[] for _ in tap_ids]
    for tok in tokens:
        p = len(cache)
        x = f32(np.asarray(TW["embed"][int(tok)], dtype=np.float64))[None, :]
        for l, layer in enumerate(TW["layers"]):
            h = store(rmsnorm(x, layer["g_in"], tshape.eps))
            q = linear(h, layer["wq"]).reshape(1, H, d)
            k = linear(h, layer["wk"]).reshape(1, G, d)
            v = linear(h, layer["wv"]).reshape(1, G, d)
            q = store(rope(q, np.array([p]), tshape.rope_theta))
            k = store(rope(k, np.array([p]), tshape.rope_theta))
            v = store(v)
            cache.K[l].append(k[0])
            cache.V[l].append(v[0])
            K = np.stack(cache.K[l])          # keys 0..p
            Vv = np.stack(cache.V[l])
            o = store(attention(q, K, Vv).reshape(1, H * d))
            x = f32(x + linear(o, layer["wo"]))
            h2 = store(rmsnorm(x, layer["g_post"], tshape.eps))
            a = store(silu(linear(h2, layer["wg"])) * linear(h2, layer["wu"]))
            x = f32(x + linear(a, layer["wd"]))
            for j, tid in enumerate(tap_ids):
                if tid == l:
                    taps[j].append(x[0].copy())
        hf = store(rmsnorm(x, TW["g_final"], tshape.eps))
        z = lm_head_logits(hf, TW["lm_head"])
        if logits_out is not None:
            logits_out.append(z[0])
        ids_out.append(int(argmax_lowest(z)[0]))
    return np.array(ids_out, dtype=np.int32), np.array(taps, dtype=np.float64)


def ar_generate(tshape, TW: dict, prompt: Sequence[int], n_new: int,
                store=f32) -> np.ndarray:
    """The target's own greedy autoregressive decode: n_new tokens."""
    cache = TargetCache(tshape.n_layers)
    ids, _ = target_forward(tshape, TW, cache, prompt, [], store)
    out = [int(ids[-1])]
    while len(out) < n_new:
        ids, _ = target_forward(tshape, TW, cache, [out[-1]], [], store)
        out.append(int(ids[0]))
    return np.array(out, dtype=np.int32)


def speculative_generate(tshape, TW: dict, dshape, DW: dict,
                         prompt: Sequence[int], n_new: int, B: int,
                         store=f32, selector: Optional[dict] = None):
    """Greedy DFlash loop ([reading] §9 steps 2-6).

    Prefill the target (first token = first anchor; taps of every prompt
    position become the context); then per round: inject the pending
    context rows into every draft layer's cache, draft the block
    [anchor, mask x (B-1)], verify it with one target forward, keep the
    accepted prefix plus the bonus, crop the target cache to the new start,
    and keep only the accepted positions' taps as the next context.
    selector (DFlash 2, [reading] §13-§14): {"w_h", "code_pred",
    "code_succ", "top_k"}; the drafts are then select_candidates over the
    block's logits and final-normed rows instead of the argmax.

    Returns (tokens [n_new], list of tau per round)."""
    tap_ids = build_target_layer_ids(dshape.n_target_layers, dshape.n_pick)
    cache = TargetCache(tshape.n_layers)
    ids, taps = target_forward(tshape, TW, cache, prompt, tap_ids, store)
    out = [int(ids[-1])]
    start = len(prompt)
    ctx_K = [np.zeros((0, dshape.G, dshape.d)) for _ in DW["layers"]]
    ctx_V = [np.zeros((0, dshape.G, dshape.d)) for _ in DW["layers"]]
    pending = taps                         # [n_pick, T, D]
    taus = []
    while len(out) < n_new:
        # K/V injection of the pending context rows at their own positions
        T = pending.shape[1]
        H_t = fuse_context(list(pending), DW["wc"], DW["g_c"], dshape.eps, store)
        pos = np.arange(start - T, start)
        for l, layer in enumerate(DW["layers"]):
            k, v = inject_kv(H_t, layer, pos, dshape.G, dshape.d,
                             dshape.rope_theta, dshape.eps, store)
            ctx_K[l] = np.concatenate([ctx_K[l], k], axis=0)
            ctx_V[l] = np.concatenate([ctx_V[l], v], axis=0)
        if selector is None:
            draft, _ = draft_block(dshape, DW, [[k] for k in ctx_K],
                                   [[v] for v in ctx_V], [out[-1]], B, store)
        else:
            draft, _, z, hid = draft_block(dshape, DW, [[k] for k in ctx_K],
                                           [[v] for v in ctx_V], [out[-1]], B, store,
                                           return_logits=True, return_hidden=True)
            hn = rmsnorm(hid[0, 1:], DW["g_f"], dshape.eps)
            path, _, _ = select_candidates(z[0], hn, out[-1], selector["w_h"],
                                           selector["code_pred"], selector["code_succ"],
                                           selector["top_k"])
            draft = draft.copy()
            draft[0, 1:] = path
        post, vtaps = target_forward(tshape, TW, cache, draft[0], tap_ids, store)
        accept, bonus, toks, new_len = verify_greedy(draft, post[None, :],
                                                     np.array([start]))
        a = int(accept[0])
        out.extend(int(t) for t in toks[0, :a + 1])
        cache.crop(int(new_len[0]))
        pending = vtaps[:, :a + 1, :]
        start = int(new_len[0])
        taus.append(a + 1)
    return np.array(out[:n_new], dtype=np.int32), taus


def speculative_sample_generate(tshape, TW: dict, dshape, DW: dict,
                                prompt: Sequence[int], n_new: int, B: int, T: float,
                                uniforms, store=f32):
    """The DFlash loop at temperature T > 0 ([reading] §8, §9): drafts drawn
    from the draft's softmax(z / T), verification by verify_rejection
    against the target's softmax(z / T).  ``uniforms(round)`` returns that
    round's (u_first, u_draft [B-1], u_accept [B-1], u_sample) draws; u_first
    (round 0 only) draws the first token from the prefill's last row.

    Returns (tokens [n_new], list of tau per round)."""
    tap_ids = build_target_layer_ids(dshape.n_target_layers, dshape.n_pick)
    cache = TargetCache(tshape.n_layers)
    z_pre = []
    _, taps = target_forward(tshape, TW, cache, prompt, tap_ids, store, z_pre)
    u_first, _, _, _ = uniforms(0)
    out = [sample_from(softmax_t(z_pre[-1], T), u_first)]
    start = len(prompt)
    ctx_K = [np.zeros((0, dshape.G, dshape.d)) for _ in DW["layers"]]
    ctx_V = [np.zeros((0, dshape.G, dshape.d)) for _ in DW["layers"]]
    pending = taps
    taus = []
    r = 0
    while len(out) < n_new:
        _, u_draft, u_accept, u_sample = uniforms(r)
        Tn = pending.shape[1]
        H_t = fuse_context(list(pending), DW["wc"], DW["g_c"], dshape.eps, store)
        pos = np.arange(start - Tn, start)
        for l, layer in enumerate(DW["layers"]):
            k, v = inject_kv(H_t, layer, pos, dshape.G, dshape.d,
                             dshape.rope_theta, dshape.eps, store)
            ctx_K[l] = np.concatenate([ctx_K[l], k], axis=0)
            ctx_V[l] = np.concatenate([ctx_V[l], v], axis=0)
        _, _, z = draft_block(dshape, DW, [[k] for k in ctx_K], [[v] for v in ctx_V],
                              [out[-1]], B, store, return_logits=True)
        q = softmax_t(z[0], T)                                       # [B-1, V]
        draft = np.array([[out[-1]] + [sample_from(q[j], u_draft[j]) for j in range(B - 1)]])
        z_ver = []
        _, vtaps = target_forward(tshape, TW, cache, draft[0], tap_ids, store, z_ver)
        pv = softmax_t(np.array(z_ver), T)                           # [B, V]
        accept, _, toks, new_len = verify_rejection(draft, q[None], pv[None],
                                                    np.asarray(u_accept)[None],
                                                    np.array([u_sample]), np.array([start]))
        a = int(accept[0])
        out.extend(int(t) for t in toks[0, :a + 1])
        cache.crop(int(new_len[0]))
        pending = vtaps[:, :a + 1, :]
        start = int(new_len[0])
        taus.append(a + 1)
        r += 1
    return np.array(out[:n_new], dtype=np.int32), taus
