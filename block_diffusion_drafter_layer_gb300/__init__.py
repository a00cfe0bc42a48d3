"""Python binding of libdflash (the DFlash draft path on GB300, sm_103a).

Thin ctypes marshalling over the C ABI in ``include/dflash.h``: every
function here has the C function's name, turns torch tensors into device
pointers and the current CUDA stream into a ``cudaStream_t``, and raises
``DFlashError`` on a non-zero status.  All arithmetic runs in the library's
CUDA kernels; PyTorch only provides device memory and streams.  Importing
this module fails loudly if ``libdflash.so`` has not been built.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash.so")

MAX_LAYERS = 16
MAX_PICK = 8
F32, BF16 = 0, 1
(K_WEIGHT_GEMM, K_ATTENTION, K_LM_HEAD, K_DENSE_GEMM, K_ELEMENTWISE, K_VERIFY,
 K_DRAFT_CHAIN) = range(7)
K_NCLASS = 7


class DFlashError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {dflash_strerror(code)} (code {code})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"libdflash.so is not built ({LIB_PATH}); run "
                      "block_diffusion_drafter_layer_gb300/build.py")
_lib = C.CDLL(LIB_PATH)


class dflash_config(C.Structure):
    _fields_ = [("hidden", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("ffn", C.c_int32), ("vocab", C.c_int32),
                ("n_layers", C.c_int32), ("n_target_layers", C.c_int32), ("n_pick", C.c_int32),
                ("target_layer_ids", C.c_int32 * MAX_PICK), ("mask_token_id", C.c_int32),
                ("max_pos", C.c_int32), ("qk_norm", C.c_int32), ("dtype", C.c_int32),
                ("rope_theta", C.c_float), ("rms_eps", C.c_float), ("embed_scale", C.c_float),
                ("causal_layers", C.c_int32), ("window_layers", C.c_int32),
                ("sliding_window", C.c_int32), ("conv_group", C.c_int32)]


class dflash_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd",
                                          "g_in", "g_post", "q_norm", "k_norm",
                                          "conv_att_kp", "conv_att_base", "conv_mlp_kp",
                                          "conv_mlp_base")]


class dflash_weights(C.Structure):
    _fields_ = [("wc", C.c_void_p), ("g_c", C.c_void_p), ("g_f", C.c_void_p),
                ("embed", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", dflash_layer_weights * MAX_LAYERS)]


class dflash_kv(C.Structure):
    _fields_ = [("k", C.c_void_p * MAX_LAYERS), ("v", C.c_void_p * MAX_LAYERS),
                ("len", C.c_void_p), ("cap", C.c_int32), ("batch_cap", C.c_int32)]


_P = C.c_void_p
_sig = {
    "dflash_create": (C.c_int, [C.POINTER(dflash_config), C.POINTER(dflash_weights), C.POINTER(_P)]),
    "dflash_destroy": (C.c_int, [_P]),
    "dflash_workspace_bytes": (C.c_size_t, [_P, C.c_int32, C.c_int32, C.c_int64]),
    "dflash_build_target_layer_ids": (C.c_int, [C.c_int32, C.c_int32, C.POINTER(C.c_int32)]),
    "dflash_fuse_context": (C.c_int, [_P, C.POINTER(_P), C.c_int64, _P, _P, C.c_size_t, _P]),
    "dflash_inject_kv": (C.c_int, [_P, _P, C.c_int64, _P, _P, C.c_int32, C.POINTER(dflash_kv),
                                   _P, C.c_size_t, _P]),
    "dflash_draft_block": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.POINTER(dflash_kv), _P, _P,
                                     _P, _P, C.c_size_t, _P]),
    "dflash_draft_round": (C.c_int, [_P, C.POINTER(_P), C.c_int32, _P, _P, _P, _P, C.c_int32,
                                     C.c_int32, C.POINTER(dflash_kv), _P, _P, _P, _P, C.c_size_t,
                                     _P]),
    "dflash_verify_greedy": (C.c_int, [_P, _P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_emit_tokens": (C.c_int, [_P, _P, _P, C.c_int32, C.c_int32, _P, C.c_int32, _P, _P,
                                     C.c_int32, _P, _P]),
    "dflash_round_host": (C.c_int, [_P, _P, _P, C.c_int32, _P, _P, _P, _P, _P, _P, _P, C.c_int32,
                                    C.c_int32, C.POINTER(dflash_kv), _P, _P, _P, C.c_size_t, _P]),
    "dflash_round_out_len": (C.c_int64, [C.c_int32, C.c_int32]),
    "dflash_lm_head_argmax": (C.c_int, [_P, _P, C.c_int32, _P, _P, _P, _P, C.c_size_t, _P]),
    "dflash_lm_head_logits": (C.c_int, [_P, _P, C.c_int32, _P, C.c_int32, _P, _P, C.c_size_t,
                                        _P]),
    "dflash_sampling_ws_bytes": (C.c_size_t, [C.c_int32, C.c_int32]),
    "dflash_sample_rows": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.c_float, _P, _P, C.c_int32,
                                     _P, _P, C.c_size_t, _P]),
    "dflash_verify_rejection": (C.c_int, [_P, _P, _P, _P, C.c_int32, _P, _P, C.c_int32,
                                          C.c_int32, _P, _P, _P, _P, _P, _P, _P, C.c_size_t,
                                          _P]),
    "dflash_select_ws_bytes": (C.c_size_t, [_P, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "dflash_select_candidates": (C.c_int, [_P, _P, _P, _P, _P, C.c_int32, C.c_int32, C.c_int32,
                                           _P, C.c_int32, _P, _P, C.c_int32, _P, _P, _P, _P,
                                           C.c_size_t, _P]),
    "dflash_target_forward": (C.c_int, [_P, _P, C.c_int32, C.c_int32, C.POINTER(dflash_kv),
                                        C.POINTER(C.c_int32), C.c_int32, _P, _P, _P, C.c_size_t,
                                        _P]),
    "dflash_lm_head_argmax_noalloc": (C.c_int, [_P, _P, C.c_int32, _P, _P, _P, _P]),
    "dflash_selftest_wait": (C.c_int, [_P, C.c_int32, C.c_int64, _P]),
    "dflash_get_status": (C.c_int, [_P, _P]),
    "dflash_strerror": (C.c_char_p, [C.c_int]),
    "dflash_launch_count": (C.c_int64, []),
    "dflash_timing_enable": (C.c_int, [_P, C.c_int]),
    "dflash_timing_read": (C.c_int, [_P, C.c_int32, C.POINTER(C.c_double), C.POINTER(C.c_int64)]),
    "dflash_chain_trace_enable": (C.c_int, [_P, C.c_int]),
    "dflash_chain_trace_read": (C.c_int, [_P, C.POINTER(C.c_int64), C.c_int32,
                                          C.POINTER(C.c_int32)]),
    "dflash_chain_trace_events": (C.c_int, [_P, C.POINTER(C.c_int64), C.c_int64,
                                            C.POINTER(C.c_int64)]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != 0:
        raise DFlashError(rc, where)


def dflash_strerror(code: int) -> str:
    return _lib.dflash_strerror(code).decode()


def dflash_launch_count() -> int:
    return int(_lib.dflash_launch_count())


def dflash_build_target_layer_ids(n_target_layers: int, n_pick: int) -> list:
    out = (C.c_int32 * max(n_pick, 1))()
    _check(_lib.dflash_build_target_layer_ids(n_target_layers, n_pick, out),
           "dflash_build_target_layer_ids")
    return list(out)[:n_pick]


def dflash_create(cfg: dflash_config, w: dflash_weights) -> int:
    h = _P()
    _check(_lib.dflash_create(C.byref(cfg), C.byref(w), C.byref(h)), "dflash_create")
    return h.value


def dflash_destroy(h: int):
    _check(_lib.dflash_destroy(h), "dflash_destroy")


def dflash_workspace_bytes(h: int, max_batch: int, max_block: int, max_rows: int) -> int:
    return int(_lib.dflash_workspace_bytes(h, max_batch, max_block, max_rows))


def dflash_fuse_context(h: int, hidden: Sequence[torch.Tensor], T: int, h_t_out: torch.Tensor,
                        ws: torch.Tensor, stream=None):
    arr = (_P * len(hidden))(*[_ptr(x) for x in hidden])
    _check(_lib.dflash_fuse_context(h, arr, T, _ptr(h_t_out), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "dflash_fuse_context")


def dflash_inject_kv(h: int, h_t: torch.Tensor, n_rows: int, seq_row0: torch.Tensor,
                     seq_rows: torch.Tensor, batch: int, kv: dflash_kv, ws: torch.Tensor,
                     stream=None):
    _check(_lib.dflash_inject_kv(h, _ptr(h_t), n_rows, _ptr(seq_row0), _ptr(seq_rows), batch,
                                 C.byref(kv), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(stream)), "dflash_inject_kv")


def dflash_draft_block(h: int, anchor: torch.Tensor, batch: int, B: int, kv: dflash_kv,
                       draft_ids: torch.Tensor, top2_gap: Optional[torch.Tensor],
                       hidden_out: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    _check(_lib.dflash_draft_block(h, _ptr(anchor), batch, B, C.byref(kv), _ptr(draft_ids),
                                   _ptr(top2_gap), _ptr(hidden_out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_draft_block")


def dflash_draft_round(h: int, hidden: Sequence[torch.Tensor], n_rows: int,
                       seq_row0: torch.Tensor, seq_rows: torch.Tensor, h_t_out: torch.Tensor,
                       anchor: torch.Tensor, batch: int, B: int, kv: dflash_kv,
                       draft_ids: torch.Tensor, top2_gap: Optional[torch.Tensor],
                       hidden_out: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    """Fusion + injection of the n_rows pending features, then the block draft."""
    arr = (_P * len(hidden))(*[_ptr(x) for x in hidden])
    _check(_lib.dflash_draft_round(h, arr, n_rows, _ptr(seq_row0), _ptr(seq_rows), _ptr(h_t_out),
                                   _ptr(anchor), batch, B, C.byref(kv), _ptr(draft_ids),
                                   _ptr(top2_gap), _ptr(hidden_out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_draft_round")


def dflash_emit_tokens(h: int, out_tokens: torch.Tensor, tau: torch.Tensor, batch: int, B: int,
                       out_buf: torch.Tensor, out_len: torch.Tensor,
                       tau_log: Optional[torch.Tensor] = None,
                       n_rounds: Optional[torch.Tensor] = None, stream=None):
    """Append a round's emitted tokens (and its tau) on the device."""
    log_cap = tau_log.shape[-1] if tau_log is not None else 0
    _check(_lib.dflash_emit_tokens(h, _ptr(out_tokens), _ptr(tau), batch, B, _ptr(out_buf),
                                   out_buf.shape[-1], _ptr(out_len), _ptr(tau_log), log_cap,
                                   _ptr(n_rounds), _stream(stream)), "dflash_emit_tokens")


def dflash_round_out_len(batch: int, B: int) -> int:
    return int(_lib.dflash_round_out_len(batch, B))


def dflash_round_host(h: int, host_features: Optional[torch.Tensor],
                      dev_features: Optional[torch.Tensor], n_rows: int, host_in: torch.Tensor,
                      dev_in: torch.Tensor, host_out: torch.Tensor, dev_out: torch.Tensor,
                      seq_row0: torch.Tensor, seq_rows: torch.Tensor, h_t_out: torch.Tensor,
                      batch: int, B: int, kv: dflash_kv, start: torch.Tensor,
                      new_len: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    """One greedy round from host buffers to host buffers (copies queued on
    the stream; host_out is valid once the stream is synchronised)."""
    _check(_lib.dflash_round_host(h, _ptr(host_features), _ptr(dev_features), n_rows,
                                  _ptr(host_in), _ptr(dev_in), _ptr(host_out), _ptr(dev_out),
                                  _ptr(seq_row0), _ptr(seq_rows), _ptr(h_t_out), batch, B,
                                  C.byref(kv), _ptr(start), _ptr(new_len), _ptr(ws),
                                  ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_round_host")


def dflash_lm_head_logits(h: int, x: torch.Tensor, rows: int, norm_gain: torch.Tensor,
                          logits: torch.Tensor, ws: torch.Tensor, skip_first_of: int = 0,
                          stream=None):
    _check(_lib.dflash_lm_head_logits(h, _ptr(x), rows, _ptr(norm_gain), skip_first_of,
                                      _ptr(logits), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "dflash_lm_head_logits")


def dflash_sampling_ws_bytes(rows: int, vocab: int) -> int:
    return int(_lib.dflash_sampling_ws_bytes(rows, vocab))


def _sampling_ws(ws, rows, vocab, like):
    if ws is None:   # scratch from torch's caching allocator
        ws = torch.empty(dflash_sampling_ws_bytes(rows, vocab), dtype=torch.uint8,
                         device=like.device)
    return ws


def dflash_sample_rows(h: int, logits: torch.Tensor, rows: int, vocab: int, temperature: float,
                       u: Optional[torch.Tensor], ids: Optional[torch.Tensor],
                       probs: Optional[torch.Tensor] = None, ids_skip_first_of: int = 0,
                       ws: Optional[torch.Tensor] = None, stream=None):
    ws = _sampling_ws(ws, rows, vocab, logits)
    _check(_lib.dflash_sample_rows(h, _ptr(logits), rows, vocab, temperature, _ptr(u), _ptr(ids),
                                   ids_skip_first_of, _ptr(probs), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_sample_rows")


def dflash_verify_rejection(h: int, draft: torch.Tensor, q_probs: torch.Tensor,
                            p_probs: torch.Tensor, vocab: int, u_accept: torch.Tensor,
                            u_sample: torch.Tensor, batch: int, B: int, start: torch.Tensor,
                            accept: torch.Tensor, tau: Optional[torch.Tensor],
                            token: Optional[torch.Tensor], out_tokens: torch.Tensor,
                            new_len: Optional[torch.Tensor], ws: Optional[torch.Tensor] = None,
                            stream=None):
    ws = _sampling_ws(ws, batch, vocab, p_probs)
    _check(_lib.dflash_verify_rejection(h, _ptr(draft), _ptr(q_probs), _ptr(p_probs), vocab,
                                        _ptr(u_accept), _ptr(u_sample), batch, B, _ptr(start),
                                        _ptr(accept), _ptr(tau), _ptr(token), _ptr(out_tokens),
                                        _ptr(new_len), _ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)), "dflash_verify_rejection")


def dflash_select_ws_bytes(h: int, batch: int, B: int, top_k: int, rank: int) -> int:
    return int(_lib.dflash_select_ws_bytes(h, batch, B, top_k, rank))


def dflash_select_candidates(h: int, logits: torch.Tensor, hidden: torch.Tensor,
                             norm_gain: torch.Tensor, anchor: torch.Tensor, batch: int, B: int,
                             top_k: int, w_h: torch.Tensor, code_pred: torch.Tensor,
                             code_succ: torch.Tensor, draft_ids: torch.Tensor,
                             candidates: Optional[torch.Tensor] = None,
                             scores: Optional[torch.Tensor] = None,
                             ws: Optional[torch.Tensor] = None, stream=None):
    rank, n_codes = int(w_h.shape[0]), int(code_pred.shape[0])
    if ws is None:   # scratch from torch's caching allocator
        ws = torch.empty(dflash_select_ws_bytes(h, batch, B, top_k, rank), dtype=torch.uint8,
                         device=logits.device)
    _check(_lib.dflash_select_candidates(h, _ptr(logits), _ptr(hidden), _ptr(norm_gain),
                                         _ptr(anchor), batch, B, top_k, _ptr(w_h), rank,
                                         _ptr(code_pred), _ptr(code_succ), n_codes,
                                         _ptr(draft_ids), _ptr(candidates), _ptr(scores),
                                         _ptr(ws), ws.numel() * ws.element_size(),
                                         _stream(stream)), "dflash_select_candidates")


def dflash_verify_greedy(draft: torch.Tensor, post: torch.Tensor, batch: int, B: int,
                         start: torch.Tensor, accept: torch.Tensor, tau: Optional[torch.Tensor],
                         bonus: torch.Tensor, out_tokens: torch.Tensor,
                         new_len: Optional[torch.Tensor], stream=None):
    _check(_lib.dflash_verify_greedy(_ptr(draft), _ptr(post), batch, B, _ptr(start), _ptr(accept),
                                     _ptr(tau), _ptr(bonus), _ptr(out_tokens), _ptr(new_len),
                                     _stream(stream)), "dflash_verify_greedy")


def dflash_lm_head_argmax(h: int, x: torch.Tensor, rows: int, norm_gain: torch.Tensor,
                          ids: torch.Tensor, top2_gap: Optional[torch.Tensor], ws: torch.Tensor,
                          stream=None):
    _check(_lib.dflash_lm_head_argmax(h, _ptr(x), rows, _ptr(norm_gain), _ptr(ids), _ptr(top2_gap),
                                      _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_lm_head_argmax")


def dflash_target_forward(h: int, tokens: torch.Tensor, batch: int, T: int, kv: dflash_kv,
                          tap_ids: Sequence[int], taps_out: Optional[torch.Tensor],
                          argmax_out: torch.Tensor, ws: torch.Tensor, stream=None):
    ids = (C.c_int32 * max(len(tap_ids), 1))(*tap_ids)
    _check(_lib.dflash_target_forward(h, _ptr(tokens), batch, T, C.byref(kv), ids, len(tap_ids),
                                      _ptr(taps_out), _ptr(argmax_out), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)),
           "dflash_target_forward")


def dflash_lm_head_argmax_noalloc(h: int, x: torch.Tensor, rows: int, norm_gain: torch.Tensor,
                                  ids: torch.Tensor, top2_gap: Optional[torch.Tensor], stream=None):
    """LM-head argmax with the library's fixed internal scratch (no workspace),
    for callers that cannot provide device memory at call time."""
    _check(_lib.dflash_lm_head_argmax_noalloc(h, _ptr(x), rows, _ptr(norm_gain), _ptr(ids),
                                              _ptr(top2_gap), _stream(stream)),
           "dflash_lm_head_argmax_noalloc")


def dflash_selftest_wait(h: int, which: int, limit_ns: int, stream=None):
    """One bounded wait that nothing completes (0: an mbarrier, 1: a device
    counter); the next dflash_get_status reports the timeout."""
    _check(_lib.dflash_selftest_wait(h, which, limit_ns, _stream(stream)), "dflash_selftest_wait")


def dflash_get_status(h: int, stream=None) -> int:
    return int(_lib.dflash_get_status(h, _stream(stream)))


def dflash_timing_enable(h: int, on: bool):
    _check(_lib.dflash_timing_enable(h, 1 if on else 0), "dflash_timing_enable")


def dflash_timing_read(h: int, kclass: int):
    ms, n = C.c_double(), C.c_int64()
    _check(_lib.dflash_timing_read(h, kclass, C.byref(ms), C.byref(n)), "dflash_timing_read")
    return ms.value, n.value


def dflash_chain_trace_enable(h: int, on: bool):
    _check(_lib.dflash_chain_trace_enable(h, 1 if on else 0), "dflash_chain_trace_enable")


TRACE_COLS = ("first_start", "last_start", "first_end", "last_end", "mma_done",
              "mark_a", "mark_b", "mark_c")


def dflash_chain_trace_read(h: int, n: int = 128):
    """Per phase of the latest traced persistent launch: a tuple of ns times
    named by TRACE_COLS (0 where a phase has no such event)."""
    k = len(TRACE_COLS)
    buf = (C.c_int64 * (k * n))()
    np_ = C.c_int32()
    _check(_lib.dflash_chain_trace_read(h, buf, n, C.byref(np_)), "dflash_chain_trace_read")
    return [tuple(buf[k * i: k * i + k]) for i in range(min(np_.value, n))]


EV_CTAS, EV_PHASES, EV_UNITS = 4, 169, 12
EV_SLOTS = 2 + 4 * EV_UNITS


def dflash_chain_trace_events(h: int):
    """Raw event log [EV_CTAS][EV_PHASES][EV_SLOTS] (SM cycles, comparable
    within one CTA) of the latest traced launch (zeros unless the library was
    built with -DDFLASH_CH_EVLOG=1)."""
    n = EV_CTAS * EV_PHASES * EV_SLOTS
    buf = (C.c_int64 * n)()
    cnt = C.c_int64()
    _check(_lib.dflash_chain_trace_events(h, buf, n, C.byref(cnt)), "dflash_chain_trace_events")
    return [[list(buf[(c * EV_PHASES + p) * EV_SLOTS:(c * EV_PHASES + p + 1) * EV_SLOTS])
             for p in range(EV_PHASES)] for c in range(EV_CTAS)]


# ---------------------------------------------------------------------------
# marshalling helpers: build the C structs from tensors and keep them alive
# ---------------------------------------------------------------------------
class Model:
    """A created handle plus the tensors its weight struct points at."""

    def __init__(self, *, D, H, G, d, F, V, n_layers, dtype: str, weights: dict, max_pos: int,
                 qk_norm: bool, mask_id: int = 0, n_target_layers: int = 0, n_pick: int = 5,
                 target_layer_ids: Sequence[int] = (), rope_theta=1e6, eps=1e-6,
                 embed_scale=1.0, causal_layers=0, window_layers=0, sliding_window=0,
                 conv_group=0):
        cfg = dflash_config()
        cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim = D, H, G, d
        cfg.ffn, cfg.vocab, cfg.n_layers = F, V, n_layers
        cfg.n_target_layers, cfg.n_pick = n_target_layers, n_pick
        for i, v in enumerate(target_layer_ids):
            cfg.target_layer_ids[i] = v
        cfg.mask_token_id, cfg.max_pos, cfg.qk_norm = mask_id, max_pos, 1 if qk_norm else 0
        cfg.dtype = BF16 if dtype == "bf16" else F32
        cfg.rope_theta, cfg.rms_eps, cfg.embed_scale = rope_theta, eps, embed_scale
        cfg.causal_layers, cfg.window_layers = causal_layers, window_layers
        cfg.sliding_window, cfg.conv_group = sliding_window, conv_group
        w = dflash_weights()
        w.wc, w.g_c = _ptr(weights.get("wc")), _ptr(weights.get("g_c"))
        w.g_f = _ptr(weights.get("g_f", weights.get("g_final")))
        w.embed, w.lm_head = _ptr(weights["embed"]), _ptr(weights["lm_head"])
        for l, lay in enumerate(weights["layers"]):
            for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_in", "g_post",
                         "q_norm", "k_norm", "conv_att_kp", "conv_att_base", "conv_mlp_kp",
                         "conv_mlp_base"):
                setattr(w.layers[l], name, _ptr(lay.get(name)))
        self.cfg, self.w, self.weights = cfg, w, weights
        self.dtype = dtype
        self.vocab, self.n_layers = V, n_layers
        self.final_gain = weights.get("g_f", weights.get("g_final"))   # the final RMSNorm's gain
        self.handle = dflash_create(cfg, w)

    def workspace(self, max_rows: int, device="cuda", max_batch: int = 0,
                  max_block: int = 0) -> torch.Tensor:
        """Workspace for calls of up to max_rows rows and draft blocks of up to
        max_batch x max_block rows (default: one sequence of max_rows rows)."""
        if max_batch == 0:
            max_batch, max_block = 1, max_rows
        n = dflash_workspace_bytes(self.handle, max_batch, max_block, max_rows)
        return torch.empty(n, dtype=torch.uint8, device=device)

    def close(self):
        if self.handle:
            dflash_destroy(self.handle)
            self.handle = None


class KVCache:
    """Per-layer [batch_cap, G, cap, d] K/V tensors and the int32 length vector."""

    def __init__(self, n_layers: int, batch_cap: int, G: int, cap: int, d: int, dtype: str,
                 device="cuda", k=None, v=None):
        td = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.k = k if k is not None else [torch.zeros(batch_cap, G, cap, d, dtype=td, device=device)
                                          for _ in range(n_layers)]
        self.v = v if v is not None else [torch.zeros(batch_cap, G, cap, d, dtype=td, device=device)
                                          for _ in range(n_layers)]
        self.len = torch.zeros(batch_cap, dtype=torch.int32, device=device)
        s = dflash_kv()
        for l in range(n_layers):
            s.k[l], s.v[l] = _ptr(self.k[l]), _ptr(self.v[l])
        s.len, s.cap, s.batch_cap = _ptr(self.len), cap, batch_cap
        self.struct = s
