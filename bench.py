"""Throughput of the DFlash draft path on GB300: draft blocks per second.

One step = one speculative round of the hot path on one batch: fuse the
pending target features (B rows per sequence) and inject them into every
draft layer's cache, draft one block [anchor, mask x (B-1)] per sequence,
and verify it greedily against a synthetic target posterior.  The context
length is reset to L at the start of each step so every step sees the same
context.  Weights and caches are random-init, seeded; inputs live in HBM
before the timed region (the value) or in pinned host memory (e2e).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "draft blocks/sec & µs per B=16 block (batch 1/32); % of HBM roofline"
DEFAULT_WORKLOAD = "qwen3_8b_b1"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes / flops per unit of work
# ---------------------------------------------------------------------------
def layer_weight_bytes(s, esz):
    per = (s.H * s.d * s.D + 2 * s.G * s.d * s.D + s.D * s.H * s.d + 3 * s.F * s.D)
    return per * s.n_layers * esz


def step_flops(w, lens):
    """Multiply-add flops of one round (x2): every projection over the rows
    it multiplies, the LM head over rows 1..B-1, and attention (scores and
    weighted sum) of every block row over [context ; block]."""
    s = w.draft
    batch, B = w.batch, w.B
    rows = batch * B
    per_layer = s.H * s.d * s.D + 2 * s.G * s.d * s.D + s.D * s.H * s.d + 3 * s.F * s.D
    f = 2.0 * rows * per_layer * s.n_layers
    f += 2.0 * batch * (B - 1) * s.V * s.D
    f += 2.0 * rows * (s.n_pick * s.D * s.D + 2 * s.G * s.d * s.D * s.n_layers)
    f += sum(4.0 * (int(l) + B) * B * s.H * s.d for l in lens) * s.n_layers
    return f


def step_bytes(w, lens, esz):
    """Bytes a step must move at least once: every weight it reads, the
    cached context K/V, and the small activations in and out."""
    s = w.draft
    batch, B = w.batch, w.B
    rows = batch * B
    out = {}
    out["weight_gemm"] = layer_weight_bytes(s, esz) + s.n_layers * rows * (s.D + s.H * s.d + s.F) * esz
    out["lm_head"] = s.V * s.D * esz + batch * (B - 1) * s.D * esz
    ctx = sum(int(l) + B for l in lens)     # context after this step's injection
    out["attention"] = ctx * s.G * s.d * 2 * esz * s.n_layers
    out["dense_gemm"] = (s.D * s.n_pick * s.D + 2 * s.G * s.d * s.D * s.n_layers) * esz + \
        rows * s.n_pick * s.D * esz
    # the persistent kernel runs the whole round: the fusion and injection
    # weights, the layer weights, the LM head and the context K/V
    out["draft_chain"] = out["weight_gemm"] + out["lm_head"] + out["attention"] + out["dense_gemm"]
    return out


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampling during the timed region.

    The sampler is started first and waited on until it writes its first
    line, then `mark()` brackets the timed region; only samples whose
    timestamp falls inside that bracket count (if the region is shorter than
    the sampling period, the first sample after its start stands in)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, index):
        try:
            u = str(torch.cuda.get_device_properties(index).uuid)
            self.index = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            self.index = str(index)
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        self.t = [None, None]

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
            return
        t_end = time.time() + 10.0
        while time.time() < t_end and self.p.poll() is None:
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.01)

    def mark(self, i):
        self.t[i] = time.time()

    @staticmethod
    def _when(stamp):
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2.0 * self.PERIOD_MS / 1e3)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append((self._when(parts[0]), parts[1:]))
        os.unlink(self.f.name)
        t0, t1 = self.t
        inside = [r for w, r in rows if w is not None and t0 is not None and t0 <= w <= t1]
        if not inside:
            after = [r for w, r in rows if w is not None and t0 is not None and w >= t0]
            inside = after[:1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "period_ms": self.PERIOD_MS}


# ---------------------------------------------------------------------------
class Draft:
    """Device state of one replica: weights, cache, workspace, step buffers."""

    def __init__(self, w, rank, n_steps_total, with_model=True, weights=None):
        self.w = w
        s = w.draft
        dev = "cuda"
        self.lens = synth.ctx_lengths(w)
        self.L_max = max(self.lens)
        self.batch, self.B = w.batch, w.B
        rows = self.batch * self.B
        self.rows = rows
        td = synth.torch_dtype(w.dtype)
        seed = w.seed + 100 * rank
        self.weights = weights if weights is not None else synth.draft_weights(s, w.dtype, seed,
                                                                                device=dev)
        self.len0 = torch.tensor(self.lens, dtype=torch.int32, device=dev)
        # a step's inputs (the 5 target feature slices, anchors, posterior) and
        # results (ids, accepted, tau, bonus, tokens) each live in one buffer,
        # so the end-to-end run moves them with one copy per direction
        hid = synth.target_hidden_states(rows, s.D, s.n_pick, w.dtype, seed + 1, device=dev)
        self.hidden_all = torch.stack(hid)
        del hid
        self.hidden = [self.hidden_all[i] for i in range(s.n_pick)]
        nb, bb = self.batch, self.batch * self.B
        self.ints_in = torch.empty(nb + bb, dtype=torch.int32, device=dev)
        self.anchor = self.ints_in[:nb]
        self.post = self.ints_in[nb:].view(nb, self.B)
        self.anchor.copy_(torch.from_numpy(synth.anchors(nb, s.V, s.mask_id, seed)))
        self.post.copy_(torch.from_numpy(synth.random_ids((nb, self.B), s.V, seed + 2)))
        self.start = torch.tensor(self.lens, dtype=torch.int32, device=dev)
        if not with_model:
            return
        import block_diffusion_drafter_layer_gb300 as dfl
        from synth.gpu import draft_model, kv_cache
        self.dfl = dfl
        cap = self.L_max + 2 * self.B + 8
        self.model = draft_model(s, w.dtype, self.weights, max_pos=cap + 8)
        self.kv = kv_cache(s, self.batch, cap, w.dtype)
        self.ws = self.model.workspace(rows, max_batch=self.batch, max_block=self.B)
        # prefill context: fuse + inject every sequence's L_b rows
        self.T_pre = sum(self.lens)
        self.pre_hidden = synth.target_hidden_states(self.T_pre, s.D, s.n_pick, w.dtype, seed,
                                                     device=dev)
        self.pre_Ht = torch.empty(self.T_pre, s.D, dtype=td, device=dev)
        cu = np.concatenate([[0], np.cumsum(self.lens)[:-1]]).astype(np.int32)
        self.pre_row0 = torch.from_numpy(cu).to(dev)
        self.pre_rows = torch.tensor(self.lens, dtype=torch.int32, device=dev)
        # per-step buffers: B pending feature rows per sequence in, ids out
        self.Ht = torch.empty(rows, s.D, dtype=td, device=dev)
        self.row0 = torch.arange(0, rows, self.B, dtype=torch.int32, device=dev)
        self.nrow = torch.full((self.batch,), self.B, dtype=torch.int32, device=dev)
        # results: ids and tokens [batch, B], then accepted, tau, bonus [batch],
        # each view starting on a 16-byte boundary
        pad = lambda n: (n + 3) // 4 * 4
        offs = np.cumsum([0, bb, bb, pad(nb), pad(nb), pad(nb)])
        self.ints_out = torch.empty(int(offs[-1]), dtype=torch.int32, device=dev)
        view = lambda i, *sh: self.ints_out[int(offs[i]):int(offs[i]) + int(np.prod(sh))].view(*sh)
        self.ids, self.out_tokens = view(0, nb, self.B), view(1, nb, self.B)
        self.acc, self.tau, self.bonus = view(2, nb), view(3, nb), view(4, nb)

    def prefill(self):
        d, m = self.dfl, self.model
        self.kv.len.zero_()
        d.dflash_fuse_context(m.handle, self.pre_hidden, self.T_pre, self.pre_Ht, self.ws)
        d.dflash_inject_kv(m.handle, self.pre_Ht, self.T_pre, self.pre_row0, self.pre_rows,
                           self.batch, self.kv.struct, self.ws)

    def step(self):
        """One round: fusion + injection of the B pending rows per sequence and
        the block draft (dflash_draft_round: one persistent launch for blocks
        of at most 16 rows), then greedy verification."""
        d, m = self.dfl, self.model
        self.kv.len.copy_(self.len0)
        d.dflash_draft_round(m.handle, self.hidden, self.rows, self.row0, self.nrow, self.Ht,
                             self.anchor, self.batch, self.B, self.kv.struct, self.ids, None,
                             None, self.ws)
        d.dflash_verify_greedy(self.ids, self.post, self.batch, self.B, self.start, self.acc,
                               self.tau, self.bonus, self.out_tokens, None)


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, world):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def time_steps(fn, K, world):
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(K):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    _barrier(world)
    return e0.elapsed_time(e1) / 1e3


# ---------------------------------------------------------------------------
def oracle_inputs(st):
    """Host inputs of one replica for the CPU oracle: the same seeded weights
    (fp64), step rows, anchors and posterior; the cached context is a seeded
    synthetic K/V of the same lengths (the oracle never reads anything the
    CUDA path computed)."""
    s = st.w.draft
    to64 = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    W = {"wc": to64(st.weights["wc"]), "g_c": to64(st.weights["g_c"]),
         "g_f": to64(st.weights["g_f"]), "embed": st.weights["embed"].float().cpu().numpy(),
         "lm_head": to64(st.weights["lm_head"]),
         "layers": [{k: to64(v) for k, v in lay.items()} for lay in st.weights["layers"]]}
    K, V = synth.random_kv_cache(st.batch, s.G, st.L_max, s.d, s.n_layers, 0.02 * np.sqrt(s.D),
                                 st.w.dtype, st.w.seed, device="cuda")
    cK = [[K[l][b, :, :st.lens[b]].float().cpu().numpy().astype(np.float64).transpose(1, 0, 2)
           for b in range(st.batch)] for l in range(s.n_layers)]
    cV = [[V[l][b, :, :st.lens[b]].float().cpu().numpy().astype(np.float64).transpose(1, 0, 2)
           for b in range(st.batch)] for l in range(s.n_layers)]
    del K, V
    hid = [h.float().cpu().numpy().astype(np.float64) for h in st.hidden]
    return W, cK, cV, hid, st.anchor.cpu().numpy(), st.post.cpu().numpy(), st.start.cpu().numpy()


def oracle_step(w, W, cK, cV, hid, anchors, post, start, seqs):
    """One oracle round for the sequences in ``seqs``: fuse + inject of the
    B pending rows, draft block, verify."""
    import oracle as O
    s, B = w.draft, w.B
    store = O.storage(w.dtype)
    rows = np.concatenate([np.arange(b * B, (b + 1) * B) for b in seqs])
    Ht = O.fuse_context([h[rows] for h in hid], W["wc"], W["g_c"], s.eps, store)
    K2, V2 = [], []
    for l, lay in enumerate(W["layers"]):
        Kl, Vl = [], []
        for j, b in enumerate(seqs):
            L = cK[l][b].shape[0]
            k, v = O.inject_kv(Ht[j * B:(j + 1) * B], lay, np.arange(L, L + B), s.G, s.d,
                               s.rope_theta, s.eps, store)
            Kl.append(np.concatenate([cK[l][b], k]))
            Vl.append(np.concatenate([cV[l][b], v]))
        K2.append(Kl)
        V2.append(Vl)
    ids, _ = O.draft_block(s, W, K2, V2, anchors[list(seqs)], B, store)
    O.verify_greedy(ids, post[list(seqs)], start[list(seqs)])


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(st, budget_s=12.0):
    """The oracle as it stands, on this host's cores, one sequence per round,
    repeated until ``budget_s`` of CPU work; scaled to blocks/s."""
    W, cK, cV, hid, anchors, post, start = oracle_inputs(st)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(st.w, W, cK, cV, hid, anchors, post, start, [n % st.batch])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 64:
            break
    return {"value": n / el, "unit": "blocks/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} oracle rounds (fuse+inject of {st.B} rows, one B={st.B} draft block, "
                      f"verify) of one sequence each, {el:.1f} s, numpy fp64"}


# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The CPU oracle on the same workload: each step is one sequence's round
    (the whole batch's rows are independent), scaled to blocks/s."""
    if rank != 0:
        return
    w = _workload(args)
    st = Draft(w, 0, 1, with_model=False)
    W, cK, cV, hid, anchors, post, start = oracle_inputs(st)
    del st
    torch.cuda.empty_cache()
    for i in range(args.warmup):
        oracle_step(w, W, cK, cV, hid, anchors, post, start, [i % w.batch])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(w, W, cK, cV, hid, anchors, post, start, [i % w.batch])
    el = time.perf_counter() - t0
    value = args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "blocks/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(w, st_lens=synth.ctx_lengths(w)),
            "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": cpu_cores(),
                             "kind": "oracle",
                             "sample": f"each step is one sequence's round (fuse+inject of {w.B} "
                                       f"rows, one B={w.B} draft block, verify), numpy fp64"},
            "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config(w, st_lens):
    s = w.draft
    return {"workload": w.name, "draft": f"{s.n_layers} layers, D={s.D}, H={s.H}, G={s.G}, "
                                         f"d={s.d}, F={s.F}, V={s.V}",
            "batch": w.batch, "B": w.B, "ctx_len": (w.ctx_len if w.ctx_range is None
                                                    else f"U{list(w.ctx_range)} mean {np.mean(st_lens):.0f}"),
            "step": f"fuse+inject {w.B} rows/seq, draft block, verify",
            "l2": "inputs larger than L2 (weights streamed every step)",
            "parallelism": "replicas"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustain-s", type=float, default=1.0, metavar="S",
                    help="seconds of the sustained region after the timed steps (0: K steps)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batch-32 and long-context blocks of the default line")
    ap.add_argument("--trace", action="store_true",
                    help="print the persistent kernel's per-phase timeline of one step "
                         "(a table, not the JSON line) and exit")
    ap.add_argument("--ctx-len", type=int, default=0, metavar="L",
                    help="replace the workload's context length (fixed-length workloads)")
    ap.add_argument("--lm-head", type=int, default=0, metavar="ROWS",
                    help="time the LM head + argmax alone on ROWS rows of the workload's "
                         "shape (a one-layer draft, so a profiler capture stays small), "
                         "print one line and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        if args.trace:
            if rank == 0:
                run_trace(args)
            return
        if args.lm_head > 0:
            if rank == 0:
                run_lm_head(args)
            return
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


def run_lm_head(args):
    """CUDA-event time of one LM head + argmax call (final RMSNorm, the
    vocabulary projection and the per-row top-2) on args.lm_head rows."""
    import dataclasses
    import block_diffusion_drafter_layer_gb300 as dfl
    from synth.gpu import draft_model
    w = _workload(args)
    s = dataclasses.replace(w.draft, n_layers=1)
    weights = synth.draft_weights(s, w.dtype, w.seed, device="cuda")
    m = draft_model(s, w.dtype, weights, max_pos=64)
    rows = args.lm_head
    x = torch.randn(rows, s.D, device="cuda", generator=torch.Generator("cuda").manual_seed(w.seed))
    ids = torch.empty(rows, dtype=torch.int32, device="cuda")
    gap = torch.empty(rows, device="cuda")
    ws = m.workspace(rows)
    for _ in range(args.warmup):
        dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids, gap, ws)
    torch.cuda.synchronize()
    if dfl.dflash_get_status(m.handle) != 0:
        raise RuntimeError("device status %d" % dfl.dflash_get_status(m.handle))
    st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st.record()
    for _ in range(args.steps):
        dfl.dflash_lm_head_argmax(m.handle, x, rows, weights["g_f"], ids, gap, ws)
    en.record()
    torch.cuda.synchronize()
    us = st.elapsed_time(en) / args.steps * 1000
    flops = 2.0 * rows * s.V * s.D
    print(json.dumps({"lm_head_rows": rows, "workload": w.name, "us_per_call": round(us, 2),
                      "tflops": round(flops / us / 1e6, 1)}))
    m.close()


PHASE_NAMES = ("q/k/v", "q/k/v reduce", "attention", "combine", "o_proj", "o_proj reduce",
               "gate/up", "gate/up reduce", "down", "down reduce")


def run_trace(args):
    """Per-phase device timeline of the draft block in one bench step."""
    import block_diffusion_drafter_layer_gb300 as dfl
    w = _workload(args)
    st = Draft(w, 0, 8)
    st.prefill()
    for _ in range(max(args.warmup, 3)):
        st.step()
    dfl.dflash_chain_trace_enable(st.model.handle, True)
    st.step()
    tr = dfl.dflash_chain_trace_read(st.model.handle)
    dfl.dflash_chain_trace_enable(st.model.handle, False)
    torch.cuda.synchronize()
    if not tr:
        print(f"{w.name}: the draft block did not run as one persistent launch (no timeline)")
        return
    names = ["fuse", "fuse reduce", "fuse norm", "inject", "inject reduce", "embed"]
    if len(tr) < len(names) + PHASE_NAMES.__len__() * w.draft.n_layers:
        names = ["embed"]   # a draft block without the round's phases
    for l in range(w.draft.n_layers):
        names += [f"layer {l} {n}" for n in PHASE_NAMES]
    names += ["LM head", "LM head reduce", "LM head merge"][:len(tr) - len(names)]
    t0 = tr[0][0]
    print(f"# {w.name}: persistent draft-block launch, {len(tr)} phases; times in us from the "
          f"first CTA's start (device %globaltimer, ~1 us resolution)")
    print("| phase | start | first CTA in -> last CTA done | gap after previous | last CTA in | "
          "marks (latest over the grid, from the phase start) |")
    print("|---|---|---|---|---|---|")
    prev = t0
    tot = {}
    for nm, row in zip(names, tr):
        s0, e1 = row[0], row[3]
        marks = " ".join(f"{c}={(v - s0) / 1e3:.2f}" for c, v in
                         zip(("mma_done", "a", "b", "c"), row[4:8]) if v)
        print(f"| {nm} | {(s0 - t0) / 1e3:.1f} | {(e1 - s0) / 1e3:.2f} | {(s0 - prev) / 1e3:.2f} | "
              f"{(row[1] - s0) / 1e3:.2f} | {marks} |")
        key = nm.split(" ", 2)[-1] if nm.startswith("layer") else nm
        tot[key] = tot.get(key, 0.0) + (e1 - prev) / 1e3
        prev = e1
    print(f"\ntotal {(prev - t0) / 1e3:.1f} us; per phase kind (incl. the barrier before it): " +
          ", ".join(f"{k} {v:.1f}" for k, v in tot.items()))


def _traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu record, if that
    record was taken on the current source of the kernel (else None)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    r = rec.get(kernel)
    if not r or r.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for rel in r.get("sources", []):
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                h.update(f.read())
        except OSError:
            return None
    return r.get("dram_bytes_per_launch") if h.hexdigest() == r.get("sha256") else None


def _workload(args):
    """The named workload, with its context length replaced by --ctx-len
    (fixed-length workloads only; a smaller case for profiler captures)."""
    w = synth.WORKLOADS[args.workload]
    if args.ctx_len > 0:
        if w.ctx_range is not None:
            raise SystemExit("--ctx-len applies to fixed-length workloads")
        w = synth.with_(w, ctx_len=args.ctx_len)
    return w


def extra_block(args, w, hbm, tf_sust, weights=None, min_s=0.3):
    """Time the round of another workload (its own weights unless given,
    its own caches, prefilled): at least args.steps steps and at least
    min_s seconds, after args.warmup untimed steps.  Returns the JSON object
    and the replica (so a second block size can share its weights)."""
    st = Draft(w, 0, 1, weights=weights)
    st.prefill()
    for _ in range(max(args.warmup, 3)):
        st.step()
    t1 = time_steps(st.step, 3, 1) / 3
    k = max(args.steps, int(np.ceil(min_s / max(t1, 1e-6))))
    t = time_steps(st.step, k, 1)
    ms = t / k * 1e3
    nbytes = step_bytes(w, st.lens, 2)
    by = sum(nbytes[c] for c in ("weight_gemm", "lm_head", "attention", "dense_gemm"))
    fl = step_flops(w, st.lens)
    hb = by / (ms / 1e3) / 1e9
    tf = fl / (ms / 1e3) / 1e12
    roof_h, roof_t = by / hbm / 1e9 * 1e3, fl / tf_sust / 1e12 * 1e3
    out = {"workload": w.name, "batch": w.batch, "B": w.B,
           "ctx_len": w.ctx_len if w.ctx_range is None else
           {"range": list(w.ctx_range), "mean": float(np.mean(st.lens))},
           "steps": k, "ms_per_step": ms, "blocks_per_s": w.batch / (ms / 1e3),
           "us_per_sequence_block": ms * 1e3 / w.batch,
           "algorithmic_bytes_per_step": by, "flops_per_step": fl,
           "hbm": {"achieved_gbs": hb, "frac_measured": hb / hbm, "frac_8tbs": hb / 8000.0,
                   "roof_ms": roof_h},
           "tensor": {"achieved_tflops": tf, "frac_sustained": tf / tf_sust, "roof_ms": roof_t},
           "binding": "hbm" if roof_h >= roof_t else "tensor",
           "frac_of_binding_roof": max(roof_h, roof_t) / ms}
    return out, st


def run_ours(args, rank, world, local):
    import block_diffusion_drafter_layer_gb300 as dfl
    w = _workload(args)
    if w.dtype != "bf16" or w.target is not None:
        raise SystemExit("bench.py times the bf16 draft workloads")
    hbm, tf_burst, tf_sust, peak_kind = _peaks()
    st = Draft(w, rank, args.steps * 3 + args.warmup * 3)
    esz = 2

    # prefill: the context projection at L (timed on its own)
    st.prefill()
    torch.cuda.synchronize()
    t_fuse = []
    s = torch.cuda.current_stream()
    for i in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        dfl.dflash_fuse_context(st.model.handle, st.pre_hidden, st.T_pre, st.pre_Ht, st.ws)
        e1.record(s)
        torch.cuda.synchronize()
        if i:
            t_fuse.append(e0.elapsed_time(e1) / 1e3)
    st.prefill()
    torch.cuda.synchronize()
    fuse_flops = 2.0 * st.T_pre * w.draft.D * w.draft.n_pick * w.draft.D
    fuse_tf = fuse_flops / np.median(t_fuse) / 1e12

    # device-resident timed region
    for _ in range(args.warmup):
        st.step()
    n0 = dfl.dflash_launch_count()
    clocks = Clocks(local)
    clocks.start()
    clocks.mark(0)
    t = time_steps(st.step, args.steps, world)
    launches = dfl.dflash_launch_count() - n0
    # the same step again for at least a second, so the clock record of the
    # measurement holds many samples (the value above stays the K-step time)
    n_sus = max(args.steps, int(np.ceil(args.sustain_s / max(t / args.steps, 1e-6))))
    t_sus = _max_over_ranks(time_steps(st.step, n_sus, world), world)
    clocks.mark(1)
    clk = clocks.stop()
    clk["region"] = f"the {args.steps} timed steps and the {n_sus} sustained steps after them"
    t = _max_over_ranks(t, world)
    blocks = w.batch * args.steps * world
    value = blocks / t
    ms_step = t / args.steps * 1e3
    sustained = {"steps": n_sus, "seconds": t_sus, "ms_per_step": t_sus / n_sus * 1e3}

    # per-kernel-class device time over an identical region (events per launch)
    dfl.dflash_timing_enable(st.model.handle, True)
    for k in range(dfl.K_NCLASS):
        dfl.dflash_timing_read(st.model.handle, k)
    time_steps(st.step, args.steps, world)
    cls = {}
    names = {dfl.K_WEIGHT_GEMM: "weight_gemm", dfl.K_ATTENTION: "attention",
             dfl.K_LM_HEAD: "lm_head", dfl.K_DENSE_GEMM: "dense_gemm",
             dfl.K_ELEMENTWISE: "elementwise", dfl.K_DRAFT_CHAIN: "draft_chain"}
    for k, name in names.items():
        ms, n = dfl.dflash_timing_read(st.model.handle, k)
        cls[name] = (ms / args.steps, n / args.steps)
    dfl.dflash_timing_enable(st.model.handle, False)
    nbytes = step_bytes(w, st.lens, esz)
    dom = max(["weight_gemm", "lm_head", "attention", "dense_gemm", "draft_chain"],
              key=lambda k: cls[k][0])
    ach = nbytes[dom] / (cls[dom][0] / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
            "frac": ach / hbm, "peak_kind": peak_kind, "frac_of_8tbs": ach / 8000.0,
            "traffic": _traffic(dom, w.name), "launches_per_step": cls[dom][1],
            "algorithmic_bytes_per_step": nbytes[dom],
            "class_ms_per_step": {k: round(v[0], 4) for k, v in cls.items()}}
    total_bytes = sum(nbytes[k] for k in ("weight_gemm", "lm_head", "attention", "dense_gemm"))
    step_frac = total_bytes / (ms_step / 1e3) / 1e9 / hbm

    # end to end through the C ABI from pinned host memory: every step is one
    # dflash_round_host call, which copies the inputs in (features, anchors
    # and posterior: two buffers), drafts and verifies, and copies the results
    # out (one buffer); the host then waits for them
    h_hidden = torch.empty_like(st.hidden_all, device="cpu").pin_memory()
    h_hidden.copy_(st.hidden_all)
    h_ints_in = st.ints_in.cpu().pin_memory()
    h_ints_out = torch.empty_like(st.ints_out, device="cpu").pin_memory()
    h2d = h_hidden.numel() * h_hidden.element_size() + h_ints_in.numel() * 4
    d2h = h_ints_out.numel() * 4

    assert h_ints_out.numel() == dfl.dflash_round_out_len(st.batch, st.B)

    def e2e_step():
        st.kv.len.copy_(st.len0)
        dfl.dflash_round_host(st.model.handle, h_hidden, st.hidden_all, st.rows, h_ints_in,
                              st.ints_in, h_ints_out, st.ints_out, st.row0, st.nrow, st.Ht,
                              st.batch, st.B, st.kv.struct, st.start, None, st.ws)
        torch.cuda.current_stream().synchronize()

    for _ in range(args.warmup):
        e2e_step()
    t0 = time.perf_counter()
    _barrier(world)
    for _ in range(args.steps):
        e2e_step()
    _barrier(world)
    te = _max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": w.batch * args.steps * world / te, "unit": "blocks/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(st)

    # the metric's batch-32 block and the long-context block (one GPU only)
    batch32 = long_ctx = None
    if world == 1 and not args.no_extra and w.name == DEFAULT_WORKLOAD:
        kept = argparse.Namespace(lens=st.lens, T_pre=st.T_pre)
        del st, h_hidden, h_ints_in, h_ints_out, e2e_step
        torch.cuda.empty_cache()
        st = kept
        batch32, st32 = extra_block(args, synth.WORKLOADS["qwen3_8b_b32_ragged"], hbm, tf_sust)
        del st32
        torch.cuda.empty_cache()
        w4 = synth.WORKLOADS["qwen35_a3b_32k"]
        b16, st4 = extra_block(args, w4, hbm, tf_sust)
        b8, st8 = extra_block(args, synth.with_(w4, B=8), hbm, tf_sust, weights=st4.weights)
        del st4, st8
        torch.cuda.empty_cache()
        long_ctx = {"B16": b16, "B8": b8}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "us_per_block": ms_step * 1e3 / w.batch,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic", "config": _config(w, st.lens),
                "roofline": roof,
                "step_hbm_frac": step_frac,
                "step_algorithmic_bytes": total_bytes,
                "context_projection": {"T": st.T_pre, "tflops": fuse_tf, "peak": tf_burst,
                                       "frac": fuse_tf / tf_burst, "unit": "TFLOP/s",
                                       "peak_kind": f"bf16 burst, {peak_kind}"},
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
                "clocks": clk, "sustained": sustained, "batch32": batch32,
                "long_context": long_ctx}
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
