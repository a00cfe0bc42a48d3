"""Greedy DFlash speculative loop on one GPU, driven through the C ABI.

Host-side orchestration only (txtmix source reading §9, steps 2-6): prefill
the target, then per round fuse and inject the pending context rows, draft
one block, verify it with one target forward, keep the accepted prefix plus
the bonus token, trim the target cache, and carry the accepted positions'
taps into the next round.  Every step runs in libdflash kernels; the host
reads back the accepted length once per round (as the reference loop does).
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import torch

from . import (KVCache, Model, dflash_build_target_layer_ids, dflash_draft_block,
               dflash_draft_round, dflash_emit_tokens, dflash_fuse_context, dflash_inject_kv,
               dflash_lm_head_logits, dflash_sample_rows, dflash_sampling_ws_bytes,
               dflash_select_candidates, dflash_select_ws_bytes,
               dflash_target_forward,
               dflash_verify_greedy, dflash_verify_rejection)


def next_block_size(sizes: Sequence[int], B: int, longest_tau: int) -> int:
    """Block size for the next rounds of the resident loop, from the longest
    tau of the last window: the largest listed size once tau reached the
    current size (every draft accepted: a longer block may pay), else the
    smallest listed size that still covers longest_tau + 1 (a block that is
    never filled costs target and draft rows for nothing).  sizes ascending."""
    if longest_tau >= B:
        return sizes[-1]
    fit = [b for b in sizes if b >= longest_tau + 1]
    return fit[0] if fit else sizes[-1]

class SpecDecoder:
    def __init__(self, target: Model, draft: Model, *, t_layers: int, t_kv_heads: int,
                 d_layers: int, d_kv_heads: int, head_dim: int, D: int, n_target_layers: int,
                 n_pick: int, B: int, max_prompt: int, cap: int, device="cuda"):
        self.target, self.draft, self.B, self.D = target, draft, B, D
        self.device = device
        self.dtype = target.dtype
        td = torch.bfloat16 if self.dtype == "bf16" else torch.float32
        self.tap_ids = dflash_build_target_layer_ids(n_target_layers, n_pick)
        self.n_pick = n_pick
        rows = max(max_prompt, B)
        self.tkv = KVCache(t_layers, 1, t_kv_heads, cap, head_dim, self.dtype, device)
        self.dkv = KVCache(d_layers, 1, d_kv_heads, cap, head_dim, self.dtype, device)
        self.ws_t = target.workspace(rows, device)
        self.ws_d = draft.workspace(rows, device)
        self.h_t = torch.empty(rows, D, dtype=td, device=device)
        self.draft_ids = torch.empty(1, B, dtype=torch.int32, device=device)
        self.post = torch.empty(B, dtype=torch.int32, device=device)
        self.start = torch.zeros(1, dtype=torch.int32, device=device)
        self.accept = torch.zeros(1, dtype=torch.int32, device=device)
        self.tau = torch.zeros(1, dtype=torch.int32, device=device)
        self.bonus = torch.zeros(1, dtype=torch.int32, device=device)
        self.out_tokens = torch.zeros(1, B, dtype=torch.int32, device=device)
        self.row0 = torch.zeros(1, dtype=torch.int32, device=device)
        self.taps_block = torch.empty(n_pick, B, D, dtype=td, device=device)

    def reset(self):
        self.tkv.len.zero_()
        self.dkv.len.zero_()

    def generate(self, prompt: Sequence[int], n_new: int,
                 selector: Optional[dict] = None) -> Tuple[List[int], List[int]]:
        """The greedy loop, reading the accepted length every round.
        selector (DFlash 2's candidate selection, txtmix §13-§14): {"w_h",
        "code_pred", "code_succ", "top_k"}; the block is then drafted without
        its argmax head, and the drafts are dflash_select_candidates over its
        LM-head logits (greedy verification keeps the output the target's
        own).  Returns (tokens, tau per round)."""
        self.reset()
        dev, B = self.device, self.B
        if selector is not None:
            V = self.draft.vocab
            hid = torch.empty(B, self.D, dtype=torch.float32, device=dev)
            z_d = torch.empty(B - 1, V, dtype=torch.float32, device=dev)
            rank = int(selector["w_h"].shape[0])
            ws_sel = torch.empty(dflash_select_ws_bytes(self.draft.handle, 1, B,
                                                        selector["top_k"], rank),
                                 dtype=torch.uint8, device=dev)
        P = len(prompt)
        td = self.taps_block.dtype
        taps_pre = torch.empty(self.n_pick, P, self.D, dtype=td, device=dev)
        argmax_pre = torch.empty(P, dtype=torch.int32, device=dev)
        tokens = torch.tensor(prompt, dtype=torch.int32, device=dev)[None]
        dflash_target_forward(self.target.handle, tokens, 1, P, self.tkv.struct, self.tap_ids,
                              taps_pre, argmax_pre, self.ws_t)
        out = [int(argmax_pre[-1].item())]
        pending, T = taps_pre, P
        taus = []
        while len(out) < n_new:
            # inject the pending context rows at positions start - T .. start - 1
            dflash_fuse_context(self.draft.handle, [pending[j] for j in range(self.n_pick)], T,
                                self.h_t, self.ws_d)
            nrows = torch.tensor([T], dtype=torch.int32, device=dev)
            dflash_inject_kv(self.draft.handle, self.h_t, T, self.row0, nrows, 1,
                             self.dkv.struct, self.ws_d)
            anchor = torch.tensor([out[-1]], dtype=torch.int32, device=dev)
            if selector is None:
                dflash_draft_block(self.draft.handle, anchor, 1, B, self.dkv.struct,
                                   self.draft_ids, None, None, self.ws_d)
            else:
                g_d = self.draft.final_gain
                dflash_draft_block(self.draft.handle, anchor, 1, B, self.dkv.struct, None, None,
                                   hid, self.ws_d)
                dflash_lm_head_logits(self.draft.handle, hid, B - 1, g_d, z_d, self.ws_d,
                                      skip_first_of=B)
                dflash_select_candidates(self.draft.handle, z_d, hid, g_d, anchor, 1, B,
                                         selector["top_k"], selector["w_h"],
                                         selector["code_pred"], selector["code_succ"],
                                         self.draft_ids, ws=ws_sel)
            # verify: one target forward over [anchor, d_1 .. d_{B-1}]
            self.start.copy_(self.tkv.len[:1])
            dflash_target_forward(self.target.handle, self.draft_ids, 1, B, self.tkv.struct,
                                  self.tap_ids, self.taps_block, self.post, self.ws_t)
            dflash_verify_greedy(self.draft_ids, self.post, 1, B, self.start, self.accept,
                                 self.tau, self.bonus, self.out_tokens, self.tkv.len)
            a = int(self.accept.item())
            out.extend(int(t) for t in self.out_tokens[0, :a + 1].tolist())
            pending, T = self.taps_block, a + 1
            taus.append(a + 1)
        return out[:n_new], taus

    def generate_resident(self, prompt: Sequence[int], n_new: int, check_every: int = 8,
                          block_sizes: Sequence[int] = ()) -> Tuple[List[int], List[int]]:
        """The same loop with every round's state on the device: the round's
        fusion + injection + draft is one dflash_draft_round call whose
        pending rows are the previous round's tau (device) and whose anchor
        is its bonus (device); dflash_emit_tokens appends the emitted tokens
        and tau on the device.  The host reads the output length only every
        `check_every` rounds (it may then run a few rounds past n_new, whose
        tokens are dropped).

        block_sizes: block sizes to schedule between (e.g. (16, 8)); at each
        check the next rounds use the smallest listed size that still covers
        the longest tau of the last window plus one (a block that is never
        filled costs target rows and draft rows for nothing), and the largest
        once a window's longest tau reaches the current size.  Empty: the
        decoder's own B throughout.  Returns (tokens, tau per round)."""
        self.reset()
        dev = self.device
        sizes = sorted(set(block_sizes)) or [self.B]
        if sizes[-1] > self.B:
            raise ValueError("block sizes above the decoder's B")
        P = len(prompt)
        td = self.taps_block.dtype
        taps_pre = torch.empty(self.n_pick, P, self.D, dtype=td, device=dev)
        argmax_pre = torch.empty(P, dtype=torch.int32, device=dev)
        tokens = torch.tensor(prompt, dtype=torch.int32, device=dev)[None]
        dflash_target_forward(self.target.handle, tokens, 1, P, self.tkv.struct, self.tap_ids,
                              taps_pre, argmax_pre, self.ws_t)
        cap = n_new + (check_every + 1) * self.B
        out_buf = torch.zeros(1, cap, dtype=torch.int32, device=dev)
        out_buf[0, 0] = argmax_pre[-1]
        out_len = torch.ones(1, dtype=torch.int32, device=dev)
        max_rounds = n_new + check_every
        tau_log = torch.zeros(1, max_rounds, dtype=torch.int32, device=dev)
        n_rounds = torch.zeros(1, dtype=torch.int32, device=dev)
        anchor = argmax_pre[-1:]
        pending, n_rows = taps_pre, P
        seq_rows = torch.tensor([P], dtype=torch.int32, device=dev)
        B = sizes[-1]
        rounds = 0
        while True:
            dflash_draft_round(self.draft.handle, [pending[j] for j in range(self.n_pick)],
                               n_rows, self.row0, seq_rows, self.h_t, anchor, 1, B,
                               self.dkv.struct, self.draft_ids, None, None, self.ws_d)
            self.start.copy_(self.tkv.len[:1])
            dflash_target_forward(self.target.handle, self.draft_ids, 1, B, self.tkv.struct,
                                  self.tap_ids, self.taps_block, self.post, self.ws_t)
            dflash_verify_greedy(self.draft_ids, self.post, 1, B, self.start, self.accept,
                                 self.tau, self.bonus, self.out_tokens, self.tkv.len)
            dflash_emit_tokens(self.draft.handle, self.out_tokens, self.tau, 1, B, out_buf,
                               out_len, tau_log, n_rounds)
            anchor, pending, n_rows, seq_rows = self.bonus, self.taps_block, B, self.tau
            rounds += 1
            if rounds % check_every == 0 or rounds >= max_rounds:
                if int(out_len.item()) >= n_new or rounds >= max_rounds:
                    break
                if len(sizes) > 1:
                    recent = tau_log[0, rounds - check_every:rounds]
                    B = next_block_size(sizes, B, int(recent.max().item()))
        taus = tau_log[0, :int(n_rounds.item())].tolist()
        n = min(int(out_len.item()), cap)
        return out_buf[0, :n].tolist()[:n_new], taus

    def generate_sampled(self, prompt: Sequence[int], n_new: int, temperature: float,
                         uniforms) -> Tuple[List[int], List[int]]:
        """The loop at temperature T > 0 (txtmix §8): each draft is drawn
        from the draft's softmax(z / T) (dflash_draft_block without its LM
        head, dflash_lm_head_logits, dflash_sample_rows), verified against
        the target's softmax(z / T) by dflash_verify_rejection.  The target's
        final hidden rows come from a tap at its last layer.  ``uniforms(r)``
        gives round r's (u_first, u_draft [B-1], u_accept [B-1], u_sample).
        Returns (tokens, tau per round)."""
        self.reset()
        dev, B, D = self.device, self.B, self.D
        T = float(temperature)
        V = self.target.vocab
        L = self.target.n_layers
        taps_ids = list(self.tap_ids) + [L - 1]
        n_t = len(taps_ids)
        P = len(prompt)
        td = self.taps_block.dtype
        taps_pre = torch.empty(n_t, P, D, dtype=td, device=dev)
        argmax_pre = torch.empty(P, dtype=torch.int32, device=dev)
        tokens = torch.tensor(prompt, dtype=torch.int32, device=dev)[None]
        dflash_target_forward(self.target.handle, tokens, 1, P, self.tkv.struct, taps_ids,
                              taps_pre, argmax_pre, self.ws_t)
        f64 = lambda a: torch.as_tensor(a, dtype=torch.float64).reshape(-1).to(dev)
        g_t, g_d = self.target.final_gain, self.draft.final_gain
        z_t = torch.empty(B, V, dtype=torch.float32, device=dev)
        p_t = torch.empty(1, B, V, dtype=torch.float32, device=dev)
        z_d = torch.empty(B - 1, V, dtype=torch.float32, device=dev)
        q_d = torch.empty(1, B - 1, V, dtype=torch.float32, device=dev)
        hid = torch.empty(B, D, dtype=torch.float32, device=dev)
        first = torch.empty(1, dtype=torch.int32, device=dev)
        ws_s = torch.empty(dflash_sampling_ws_bytes(B, V), dtype=torch.uint8, device=dev)
        u_first, _, _, _ = uniforms(0)
        last = taps_pre[n_t - 1, P - 1:P].float()
        dflash_lm_head_logits(self.target.handle, last, 1, g_t, z_t, self.ws_t)
        dflash_sample_rows(self.target.handle, z_t, 1, V, T, f64([u_first]), first, ws=ws_s)
        out = [int(first.item())]
        taps_blk = torch.empty(n_t, B, D, dtype=td, device=dev)
        pending, Tn = taps_pre, P
        taus = []
        r = 0
        while len(out) < n_new:
            _, u_draft, u_accept, u_sample = uniforms(r)
            dflash_fuse_context(self.draft.handle, [pending[j] for j in range(self.n_pick)], Tn,
                                self.h_t, self.ws_d)
            nrows = torch.tensor([Tn], dtype=torch.int32, device=dev)
            dflash_inject_kv(self.draft.handle, self.h_t, Tn, self.row0, nrows, 1,
                             self.dkv.struct, self.ws_d)
            self.draft_ids[0, 0] = out[-1]
            anchor = self.draft_ids[0, :1].clone()
            dflash_draft_block(self.draft.handle, anchor, 1, B, self.dkv.struct, None, None,
                               hid, self.ws_d)
            dflash_lm_head_logits(self.draft.handle, hid, B - 1, g_d, z_d, self.ws_d,
                                  skip_first_of=B)
            dflash_sample_rows(self.draft.handle, z_d, B - 1, V, T, f64(u_draft),
                               self.draft_ids[0, 1:], q_d[0], ws=ws_s)
            self.start.copy_(self.tkv.len[:1])
            dflash_target_forward(self.target.handle, self.draft_ids, 1, B, self.tkv.struct,
                                  taps_ids, taps_blk, self.post, self.ws_t)
            dflash_lm_head_logits(self.target.handle, taps_blk[n_t - 1].float().contiguous(), B,
                                  g_t, z_t, self.ws_t)
            dflash_sample_rows(self.target.handle, z_t, B, V, T, None, None, p_t[0], ws=ws_s)
            dflash_verify_rejection(self.target.handle, self.draft_ids, q_d, p_t, V,
                                    f64(u_accept), f64([u_sample]), 1, B, self.start,
                                    self.accept, self.tau, self.bonus, self.out_tokens,
                                    self.tkv.len, ws=ws_s)
            a = int(self.accept.item())
            out.extend(int(t) for t in self.out_tokens[0, :a + 1].tolist())
            pending, Tn = taps_blk, a + 1
            taus.append(a + 1)
            r += 1
        return out[:n_new], taus

    def ar_decode(self, prompt: Sequence[int], n_new: int) -> List[int]:
        """The target's own greedy decode, one token per forward (M = 1)."""
        self.reset()
        dev = self.device
        P = len(prompt)
        argmax = torch.empty(P, dtype=torch.int32, device=dev)
        tokens = torch.tensor(prompt, dtype=torch.int32, device=dev)[None]
        dflash_target_forward(self.target.handle, tokens, 1, P, self.tkv.struct, [], None, argmax,
                              self.ws_t)
        out = [int(argmax[-1].item())]
        one = torch.empty(1, dtype=torch.int32, device=dev)
        while len(out) < n_new:
            tok = torch.tensor([[out[-1]]], dtype=torch.int32, device=dev)
            dflash_target_forward(self.target.handle, tok, 1, 1, self.tkv.struct, [], None, one,
                                  self.ws_t)
            out.append(int(one.item()))
        return out
