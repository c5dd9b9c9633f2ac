#!/usr/bin/env python3
"""Benchmark of the drafter hot path on GB300.

One step = one pass of the whole hot path for one batch of requests:
  S1+S2  catch-up materialisation of the W pending target-feature rows of every request
         (the rows the previous round committed) into the context rings -- inside the
         round call: the feature projection first, then each layer's context K/V in the
         same product as the block's Q/K/V,
  S3..S9 one masked-block draft round (all layers, DSpine injection),
  S10    tied LM head + per-row argmax.
The same step with the catch-up as a separate materialisation call is timed beside it.
Default workload: the 27B-geometry DSpine-b16 round at B=1 (window 2048 over a
4096-token context, W=16); the B=8 round (contexts uniform in [512, 16384]) is timed in
the same run and reported under "b8".  Inputs are seeded synthetic tensors, resident in
HBM when the timed region starts; the 4.8 GB of weights streamed per step exceed the
129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun (N > 1) every rank runs an independent replica (the round has no
cross-GPU exchange); rank 0 prints one JSON line with the whole-job rate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bdsynth  # noqa: E402

TOPK = 16  # candidates per proposal row of the top-k head (timed beside the step)
METRIC = "draft rounds/s (B=1, W=16, 27B DSpine-b16 geometry)"
UNIT = "rounds/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-b8", action="store_true")
    ap.add_argument("--workload", default="b1", choices=["b1", "b8"],
                    help="the main line's workload (b1: the metric's configuration)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--profile-full", action="store_true",
                    help="with --profile-case: all draft layers instead of one")
    ap.add_argument("--profile-case", action="store_true",
                    help="run two steps of a one-layer 27B-geometry round (batch from "
                         "--workload) and exit: the small case the ncu captures use")
    return ap.parse_args()


# ----------------------------------------------------------------------------- dist
def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)], stdout=open(self.path, "w"),
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- state
class State:
    """Weights, rings and step inputs of one workload, all resident on the GPU."""

    def __init__(self, geo, seed, weights=None):
        from block_drafter_gb300.session import DraftSession
        self.geo = geo
        dev = "cuda"
        self.w = weights if weights is not None else bdsynth.make_weights(geo, seed, device=dev)
        self.mask = bdsynth.mask_token_id(geo, seed)
        self.F = bdsynth.frontiers(geo, seed)
        self.anchors_l = bdsynth.anchor_ids(geo, seed)
        B, W = geo.batch, geo.W
        self.sess = DraftSession(geo, self.w, self.mask, b_max=B, max_masks=geo.n_masks,
                                 max_ctx_rows=2048)
        front = torch.tensor(self.F, dtype=torch.int64, device=dev)
        # committed context: every request's live window, materialised chunk by chunk
        pend_feats, pend_pos, pend_req = [], [], []
        for b in range(B):
            lo, hi = bdsynth.live_window(geo, self.F[b])
            ci = 0
            for c0 in range(lo, hi, 2048):
                n = min(2048, hi - c0)
                f = bdsynth.target_features(geo, n, seed, stream=b * 4096 + ci, device=dev)
                self.sess.materialize(f, torch.full((n,), b, dtype=torch.int32, device=dev),
                                      torch.arange(c0, c0 + n, dtype=torch.int64, device=dev), front)
                ci += 1
                last = f
                last_c0 = c0
            # the W newest rows are this step's pending catch-up work
            take = min(W, hi - lo)
            pend_feats.append(last[-take:].clone())
            pend_pos.append(torch.arange(hi - take, hi, dtype=torch.int64, device=dev))
            pend_req.append(torch.full((take,), b, dtype=torch.int32, device=dev))
        self.feats = torch.cat(pend_feats).contiguous()
        self.row_pos = torch.cat(pend_pos)
        self.row_req = torch.cat(pend_req)
        self.front = front
        self.anchors = torch.tensor(self.anchors_l, dtype=torch.int32, device=dev)
        self.head_in, self.tokens, self.maxl, _ = self.sess.alloc_outputs(B, geo.n_masks)
        rows = self.head_in.shape[0]
        self.cand = torch.empty(rows, TOPK, dtype=torch.int32, device=dev)
        self.cand_score = torch.empty(rows, TOPK, dtype=torch.float32, device=dev)
        self.tail = self.sess.alloc_tail_state(B, geo.n_masks)
        self.refined = torch.empty(rows, dtype=torch.int32, device=dev)
        torch.cuda.synchronize()

    def materialize(self):
        self.sess.materialize(self.feats, self.row_req, self.row_pos, self.front)

    def round(self):
        """The round with this step's pending rows caught up inside the call."""
        self.sess.round(self.anchors, self.front, self.geo.n_masks, self.head_in,
                        pending=(self.feats, self.row_req, self.row_pos))

    def round_plain(self):
        """The round alone (its context already complete)."""
        self.sess.round(self.anchors, self.front, self.geo.n_masks, self.head_in)

    def head(self):
        self.sess.head(self.head_in, self.tokens, self.maxl)

    def head_topk(self):
        self.sess.head_topk(self.head_in, TOPK, self.cand, self.cand_score)

    def head_topk_fp8(self):
        """FP8 retrieval of 128 candidates per row, BF16 rescoring, the 16 best."""
        self.sess.head_topk_fp8(self.head_in, 128, TOPK, self.cand, self.cand_score)

    def round_with_tail(self):
        self.sess.round(self.anchors, self.front, self.geo.n_masks, self.head_in,
                        tail_state=self.tail, pending=(self.feats, self.row_req, self.row_pos))

    def refine(self):
        self.sess.refine_tail(self.tail, self.cand, self.cand_score, self.geo.batch,
                              self.geo.n_masks, self.refined)

    def step(self):
        self.round()
        self.head()

    def step_separate(self):
        """The same step with the catch-up as its own materialisation call."""
        self.materialize()
        self.round_plain()
        self.head()

    # algorithmic bytes of one step: every weight byte once, the windowed context K/V
    # each request reads once, the pending feature rows read and their K/V written
    def bytes_per_step(self) -> dict:
        geo = self.geo
        el = 2 if geo.dtype == "bf16" else 4

        def nb(t):
            return 0 if t is None else t.numel() * t.element_size()
        w = self.w
        shared = sum(nb(w.get(k)) for k in ("w_feature", "context_norm", "final_norm",
                                             "codebook", "g_recv", "g_pred", "a_val", "gate_bias"))
        layers = sum(nb(t) for lw in w["layers"] for t in lw.values())
        head = nb(w["embed_head"])
        kv = 0
        for b in range(geo.batch):
            for l in range(geo.n_layers):
                S = geo.windows[l]
                ctx = min(self.F[b], S - 1) if S > 0 else self.F[b]
                kv += ctx * geo.n_kv_heads * geo.head_dim * el * 2
        rows = self.feats.shape[0]
        pend = rows * geo.n_target_layers * geo.hidden * el \
            + rows * geo.n_layers * geo.n_kv_heads * geo.head_dim * el * 2
        # the codebook is read one row per request, not streamed
        shared -= nb(w.get("codebook"))
        shared += geo.batch * geo.code_width * el
        return {"weights": shared + layers + head, "head": head, "kv": kv, "pending": pend,
                "total": shared + layers + head + kv + pend}

    def flops_per_step(self) -> float:
        geo = self.geo
        T = geo.batch * geo.W
        w = self.w
        lin = sum(t.numel() for lw in w["layers"] for t in lw.values() if t.dim() == 2)
        f = 2.0 * T * lin + 2.0 * geo.batch * geo.n_masks * w["embed_head"].numel()
        if geo.code_width:
            f += 2.0 * T * 3 * geo.msg_width * geo.code_width
        rows = self.feats.shape[0]
        f += 2.0 * rows * w["w_feature"].numel()
        f += 2.0 * rows * sum(lw["wk"].numel() + lw["wv"].numel() for lw in w["layers"])
        for b in range(geo.batch):
            for l in range(geo.n_layers):
                S = geo.windows[l]
                ctx = (min(self.F[b], S - 1) if S > 0 else self.F[b]) + geo.W
                f += 4.0 * geo.head_dim * geo.n_q_heads * geo.W * ctx
        return f


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graphs(st: State, steps: int, warmup: int, world: int):
    """Replays [round with catch-up | head] graphs back to back; events between them give
    the per-call times, the outer pair the step time."""
    g_round, g_head = capture(st.round), capture(st.head)
    for _ in range(warmup):
        g_round.replay()
        g_head.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for k in range(steps):
        ev[k][0].record()
        g_round.replay()
        ev[k][1].record()
        g_head.replay()
        ev[k][2].record()
    torch.cuda.synchronize()
    barrier(world)
    tot = ev[0][0].elapsed_time(ev[-1][2])
    per = {"round_with_catch_up": sum(e[0].elapsed_time(e[1]) for e in ev) / steps,
           "head": sum(e[1].elapsed_time(e[2]) for e in ev) / steps}
    return tot / steps, per


def time_call(fn, steps: int, warmup: int):
    """Mean device time (ms) of one call replayed from a captured graph."""
    g = capture(fn)
    for _ in range(warmup):
        g.replay()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(steps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def round_only(st: State, args) -> dict:
    """The round without pending rows (its context already complete)."""
    us = 1000.0 * time_call(st.round_plain, args.steps, args.warmup)
    return {"us": us, "rounds_per_s": 1e6 / us}


def separate_catch_up(st: State, args) -> dict:
    """The catch-up as its own materialisation call, and the whole step done that way."""
    mat = 1000.0 * time_call(st.materialize, args.steps, args.warmup)
    step = 1000.0 * time_call(st.step_separate, args.steps, args.warmup)
    return {"materialize_us": mat, "step_us": step}


def dflash2_lines(args, world, hbm) -> dict:
    """The DFlash2 variant at the same 27B geometry (dynamic grouped convolution around
    both branches, no DSpine bridge): the same step (round with the fused catch-up + LM
    head) at B=1 and B=8."""
    out = {}
    w = None
    for geo in (bdsynth.DFLASH2_27B_B1, bdsynth.DFLASH2_27B_B8):
        st = State(geo, args.seed, weights=w)
        w = st.w
        ms, per = time_graphs(st, args.steps, args.warmup, world)
        ms = max_over_ranks(ms, world)
        by = st.bytes_per_step()
        gbs = by["total"] / (ms * 1e-3) / 1e9
        out["b%d" % geo.batch] = {
            "workload": geo.name, "us_per_step": 1000.0 * ms, "rounds_per_s": world * 1000.0 / ms,
            "breakdown_us": {k: 1000.0 * v for k, v in per.items()},
            "round_only": round_only(st, args), "achieved_step_gbs": gbs,
            "frac_of_measured_hbm": gbs / hbm, "algorithmic_bytes_per_step": by}
        del st
    return out


def refine_us(st: State, args) -> float:
    """Device time of the last-write refinement (tables + walk) after a round that exported
    its tail state and a top-16 head that produced the candidates."""
    st.round_with_tail()
    st.head_topk()
    torch.cuda.synchronize()
    return 1000.0 * time_call(st.refine, args.steps, args.warmup)


def time_e2e(st: State, steps: int, warmup: int):
    """Public API per step with host buffers: H2D of the step's pending feature rows,
    anchors and frontiers from pinned memory, the three C-ABI calls, D2H of the tokens."""
    h_feats = st.feats.cpu().pin_memory()
    h_anch = st.anchors.cpu().pin_memory()
    h_front = st.front.cpu().pin_memory()
    h_tok = torch.empty_like(st.tokens, device="cpu").pin_memory()
    bi = h_feats.numel() * h_feats.element_size() + h_anch.numel() * 4 + h_front.numel() * 8
    bo = h_tok.numel() * 4

    def one():
        st.feats.copy_(h_feats, non_blocking=True)
        st.anchors.copy_(h_anch, non_blocking=True)
        st.front.copy_(h_front, non_blocking=True)
        st.step()
        h_tok.copy_(st.tokens, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    for _ in range(warmup):
        one()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, bi, bo


def recorded_traffic():
    """DRAM bytes per launch of the roofline kernel from the committed ncu record, if the
    kernel's sources are unchanged since the counters were taken (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    h = hashlib.sha256()
    for f in rec["source_files"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    return rec["traffic_bytes_per_launch"] if h.hexdigest() == rec["source_sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d.get("bf16_tflops_sustained", 1715.0), "measured"
    return 6800.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- oracle
def oracle_step_sample(geo, w_host, F, anchors, mask, feats_np, pos_np, n_layers=None):
    """The oracle's step for request 0: catch-up materialisation of its pending rows,
    the round (optionally limited to the first n_layers layers) and the head."""
    import numpy as np

    from oracle import dspine_oracle as O
    g = geo if n_layers is None else geo.with_(n_layers=n_layers)
    t0 = time.perf_counter()
    rings = {"k": [np.zeros((1, g.n_kv_heads, g.capacity(l), g.head_dim), np.float32)
                   for l in range(g.n_layers)],
             "v": [np.zeros((1, g.n_kv_heads, g.capacity(l), g.head_dim), np.float32)
                   for l in range(g.n_layers)]}
    O.materialize(g, w_host, feats_np, pos_np, F[0], rings=rings)
    O.draft_round(g, w_host, rings, [anchors[0]], [F[0]], mask, g.n_masks)
    return time.perf_counter() - t0


def host_weights(w):
    import numpy as np
    out = {}
    for k, v in w.items():
        if k == "layers":
            out[k] = [{kk: vv.float().cpu().numpy() for kk, vv in lw.items()} for lw in v]
        else:
            out[k] = None if v is None else v.float().cpu().numpy()
    return out


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main
def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, on the host cores.  Each step
    is one full oracle step of request 0 of the B=1 workload (catch-up materialisation of
    its 16 pending rows, the 5-layer round over the 2047-position window, the LM head),
    i.e. exactly the per-request work of one GPU step at B=1."""
    if rank != 0:
        return
    import numpy as np
    geo = bdsynth.DSPINE27B_B1
    w = bdsynth.make_weights(geo, args.seed, device="cpu")
    wh = {k: (None if v is None else v.float().numpy()) for k, v in w.items() if k != "layers"}
    wh["layers"] = [{kk: vv.float().numpy() for kk, vv in lw.items()} for lw in w["layers"]]
    del w
    F = bdsynth.frontiers(geo, args.seed)
    anchors = bdsynth.anchor_ids(geo, args.seed)
    mask = bdsynth.mask_token_id(geo, args.seed)
    feats = bdsynth.target_features(geo, geo.W, args.seed).float().numpy()
    pos = np.arange(F[0] - geo.W, F[0])
    ts = []
    for k in range(args.warmup + args.steps):
        t = oracle_step_sample(geo, wh, F, anchors, mask, feats, pos)
        if k >= args.warmup:
            ts.append(t)
    t_step = statistics.mean(ts)
    val = 1.0 / t_step
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": geo.name, "B": 1, "W": geo.W, "context": F[0],
                       "window": geo.windows[0]},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": "one full oracle step of request 0 per step: catch-up of "
                                       "16 rows, 5-layer round, full LM head"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    from block_drafter_gb300 import binding, builder
    builder.build()
    binding.lib()
    if args.profile_case:
        # One warm step, then the profiled step inside the NVTX range "profiled_step"
        # (ncu --nvtx --nvtx-include "profiled_step/").  GEMM launch order of the B=1 step:
        # [0] W_feature (catch-up), [1] QKV (+ the pending rows' K/V), [2] W_o, [3] gate/up,
        # [4] down, [5] LM head (the bridge runs as one bridge_kernel launch).  At B=8 the
        # pending rows' K/V is its own product after QKV, and the bridge's code read,
        # gate/value maps and write are GEMMs after the down projection.
        base = bdsynth.DSPINE27B_B1 if args.workload == "b1" else bdsynth.DSPINE27B_B8
        geo = base if args.profile_full else base.with_(n_layers=1, windows=(2048,))
        st = State(geo, args.seed)
        st.step()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("profiled_step")
        st.step()
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        binding.sync_status()
        print(json.dumps({"profile_case": geo.name, "layers": geo.n_layers, "ok": True}))
        return

    geo = bdsynth.DSPINE27B_B1 if args.workload == "b1" else bdsynth.DSPINE27B_B8
    st = State(geo, args.seed)
    n0 = binding.kernel_launches()
    st.step()
    torch.cuda.synchronize()
    launches_per_step = binding.kernel_launches() - n0
    binding.sync_status()

    clocks = Clocks(local)
    clocks.start()
    ms, per = time_graphs(st, args.steps, args.warmup, world)
    ck = clocks.stop()
    ms = max_over_ranks(ms, world)
    hbm, tf, peak_kind = peaks()
    by = st.bytes_per_step()
    head_bytes = by["head"] + st.head_in.numel() * st.head_in.element_size()  # weights + fp32 rows
    head_gbs = head_bytes / (per["head"] * 1e-3) / 1e9
    step_gbs = by["total"] / (ms * 1e-3) / 1e9
    e2e_ms, bi, bo = time_e2e(st, max(10, args.steps // 2), 3)
    e2e_ms = max_over_ranks(e2e_ms, world)

    line = {
        "metric": METRIC, "value": world * 1000.0 / ms, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the 27B DSpine-b16 drafter geometry)",
        "config": {"workload": geo.name, "B": geo.batch, "W": geo.W, "context": st.F[0],
                   "window": geo.windows[0], "hidden": geo.hidden, "layers": geo.n_layers,
                   "vocab": geo.vocab,
                   "step": "draft round with the catch-up of 16 pending rows per request fused in "
                           "+ LM head argmax",
                   "l2": "inputs larger than L2 (weights streamed per step >> 129 MB)",
                   "operands": "bf16 weights (packed image: MLP and head converted exactly to fp16); "
                               "fp16 activations in the MLP, head and attention products, bf16 "
                               "hi+lo pairs in the others; fp32 accumulation and residual stream",
                   "parallelism": f"replicas x{world}"},
        "us_per_step": 1000.0 * ms,
        "breakdown_us": {k: 1000.0 * v for k, v in per.items()},
        "round_only": round_only(st, args),
        "separate_catch_up": separate_catch_up(st, args),
        "achieved_step_gbs": step_gbs,
        "step_roofline_frac": {"of_measured_hbm": step_gbs / hbm, "of_8tbs": step_gbs / 8000.0},
        "algorithmic_bytes_per_step": by,
        "roofline": {"bound": "hbm", "kernel": "LM head call (tcgen05 GEMM + split-vocab argmax reduce)",
                     "achieved": head_gbs, "peak": hbm, "unit": "GB/s", "frac": head_gbs / hbm,
                     "traffic": recorded_traffic(), "algorithmic_bytes": head_bytes,
                     "peak_kind": peak_kind},
        "clocks": ck,
        "e2e": {"value": world * 1000.0 / e2e_ms, "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_per_step": launches_per_step,
        "head_topk16_us": 1000.0 * time_call(st.head_topk, args.steps, args.warmup),
        "head_topk16_fp8_us": 1000.0 * time_call(st.head_topk_fp8, args.steps, args.warmup),
        "refine_tail_us": refine_us(st, args),
    }
    if not args.no_b8 and args.workload == "b1":
        geo8 = bdsynth.DSPINE27B_B8
        st8 = State(geo8, args.seed, weights=st.w)
        ms8, per8 = time_graphs(st8, args.steps, args.warmup, world)
        ms8 = max_over_ranks(ms8, world)
        by8 = st8.bytes_per_step()
        gbs8 = by8["total"] / (ms8 * 1e-3) / 1e9
        line["b8"] = {"workload": geo8.name, "contexts": st8.F, "us_per_step": 1000.0 * ms8,
                      "rounds_per_s": world * 1000.0 / ms8,
                      "breakdown_us": {k: 1000.0 * v for k, v in per8.items()},
                      "round_only": round_only(st8, args),
                      "separate_catch_up": separate_catch_up(st8, args),
                      "achieved_step_gbs": gbs8, "frac_of_measured_hbm": gbs8 / hbm,
                      "algorithmic_bytes_per_step": by8,
                      "head_topk16_us": 1000.0 * time_call(st8.head_topk, args.steps, args.warmup),
                      "head_topk16_fp8_us": 1000.0 * time_call(st8.head_topk_fp8, args.steps,
                                                               args.warmup),
                      "refine_tail_us": refine_us(st8, args)}
        del st8
    if not args.no_b8 and args.workload == "b1":
        line["dflash2"] = dflash2_lines(args, world, hbm)
    if rank == 0 and not args.no_cpu_baseline:
        import numpy as np
        wh = host_weights(st.w)
        feats = st.feats[:geo.W].float().cpu().numpy()
        pos = st.row_pos[:geo.W].cpu().numpy()
        t = oracle_step_sample(geo, wh, st.F, st.anchors_l, st.mask, feats, pos)
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": UNIT, "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": "one full step of request 0 (catch-up of 16 rows, "
                                          "5-layer round, full LM head) at B=1, timed once"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
