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
CPU_SAMPLES = 4  # oracle steps timed for the cpu_baseline (about 3 s each on 16 cores)
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


def dflash35b_line(args, world, hbm, peak_kind) -> dict:
    """Plain DFlash at the 35B-A3B draft geometry, B=8 (5 local layers with window 4096 and
    one full-context layer, contexts uniform in [4096, 32768], no injection): the same step
    (round with the fused catch-up + LM head) and the round alone."""
    geo = bdsynth.DFLASH35B_B8
    st = State(geo, args.seed)
    ms, per = time_graphs(st, args.steps, args.warmup, world)
    ms = max_over_ranks(ms, world)
    by = st.bytes_per_step()
    gbs = by["total"] / (ms * 1e-3) / 1e9
    ro = round_only(st, args)
    kt = kernel_times(st, min(args.steps, 10), args.warmup, hbm)
    dom = dominant(kt)
    out = {"workload": geo.name, "contexts": st.F, "us_per_step": 1000.0 * ms,
           "rounds_per_s": world * 1000.0 / ms,
           "breakdown_us": {k: 1000.0 * v for k, v in per.items()}, "round_only": ro,
           "achieved_step_gbs": gbs, "frac_of_measured_hbm": gbs / hbm,
           "algorithmic_bytes_per_step": by,
           "roofline": roofline_entry(dom, kt, hbm, peak_kind, KIND_NAMES[dom]), "kernels": kt}
    del st
    torch.cuda.empty_cache()
    return out


def refine_us(st: State, args) -> float:
    """Device time of the last-write refinement (tables + walk) after a round that exported
    its tail state and a top-16 head that produced the candidates."""
    st.round_with_tail()
    st.head_topk()
    torch.cuda.synchronize()
    return 1000.0 * time_call(st.refine, args.steps, args.warmup)


KERNEL_KINDS = ("qkv", "attention", "wo", "gate_up", "down", "bridge", "head")


def kernel_bytes(st: State) -> dict:
    """Algorithmic bytes of each kernel kind's launches in one step (weights as stored,
    2 bytes per element; the attention's windowed context K/V of every request; the head
    adds its fp32 input rows)."""
    geo = st.geo
    H, D = geo.hidden, geo.head_dim
    QD, KD = geo.n_q_heads * D, geo.n_kv_heads * D
    el = 2 if geo.dtype == "bf16" else 4
    att = []
    for l in range(geo.n_layers):
        S = geo.windows[l]
        ctx = sum((min(F, S - 1) if S > 0 else F) for F in st.F)
        att.append(ctx * KD * el * 2)
    out = {"qkv": [(QD + 2 * KD) * H * el] * geo.n_layers, "attention": att,
           "wo": [H * QD * el] * geo.n_layers, "gate_up": [2 * geo.ffn * H * el] * geo.n_layers,
           "down": [H * geo.ffn * el] * geo.n_layers,
           "head": [geo.vocab * H * el + st.head_in.numel() * 4]}
    if geo.code_width and geo.batch * geo.W <= 32:  # the one-launch bridge (small blocks)
        Rc, Mc = geo.code_width, geo.msg_width
        out["bridge"] = [(Rc * H + H * Mc + 3 * Mc * Rc) * el] * geo.n_layers
    return out


def kernel_times(st: State, steps: int, warmup: int, hbm: float) -> dict:
    """Per-launch device time of each kernel kind of the step, from CUDA events the library
    records around those launches (bd_set_timing_events) in a captured step, averaged over
    the layers and ``steps`` replays.  An event between two launches removes their
    programmatic overlap, so this runs apart from the timed step; the bracketed launch
    itself is measured from the moment its predecessor has finished."""
    from block_drafter_gb300 import binding
    nbytes = kernel_bytes(st)
    out = {}
    for kind in KERNEL_KINDS:
        if kind not in nbytes:
            continue
        n = len(nbytes[kind])
        b = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        binding.set_timing_events(kind, b, e)
        try:
            g = capture(st.step)
        finally:
            binding.set_timing_events(None)
        for _ in range(warmup):
            g.replay()
        tot = [0.0] * n
        try:
            for _ in range(steps):
                g.replay()
                torch.cuda.synchronize()
                for i in range(n):
                    tot[i] += b[i].elapsed_time(e[i])
        except RuntimeError as ex:  # an event was never recorded
            torch.cuda.synchronize()
            out[kind] = {"error": str(ex)[:200]}
            continue
        us = [1000.0 * t / steps for t in tot]
        by = sum(nbytes[kind])
        gbs = by / (sum(us) * 1e-6) / 1e9
        out[kind] = {"launches": n, "us_per_launch": sum(us) / n, "us_per_step": sum(us),
                     "bytes_per_launch": by / n, "achieved_gbs": gbs, "frac_of_measured_hbm": gbs / hbm}
        del g
    return out


def dominant(kt: dict) -> str:
    """The kernel kind with the largest device time per step."""
    ok = {k: v for k, v in kt.items() if "us_per_step" in v}
    if not ok:
        raise RuntimeError(f"no kernel kind was timed: {kt}")
    return max(ok, key=lambda k: ok[k]["us_per_step"])


def roofline_entry(kind: str, kt: dict, hbm: float, peak_kind: str, what: str) -> dict:
    k = kt[kind]
    return {"bound": "hbm", "kernel": what, "achieved": k["achieved_gbs"], "peak": hbm, "unit": "GB/s",
            "frac": k["achieved_gbs"] / hbm, "traffic": recorded_traffic(kind),
            "algorithmic_bytes": k["bytes_per_launch"], "us_per_launch": k["us_per_launch"],
            "peak_kind": peak_kind}


KIND_NAMES = {"qkv": "Q/K/V product (tcgen05 GEMM, head RMSNorm + RoPE epilogue)", "attention": "block attention",
              "wo": "output projection (tcgen05 GEMM, residual epilogue)",
              "gate_up": "SwiGLU gate/up product (tcgen05 GEMM, SwiGLU epilogue)",
              "down": "down projection (tcgen05 GEMM, residual epilogue)",
              "bridge": "fused DSpine bridge (code read + gate/message + write)",
              "head": "LM head product (tcgen05 GEMM, per-tile argmax epilogue)"}


def materialize_line(st: State, steps: int, warmup: int, tf_sust: float, tf_burst: float,
                     hbm: float) -> dict:
    """Context K/V materialisation of a 2048-row prefill chunk at positions 0..2047 (27B
    geometry: W_feature 25600 -> 5120 with the context norm, then every layer's W_k|W_v,
    head norm, RoPE and ring store).  Uses the B=1 state's weights and request-0 rings."""
    geo = st.geo
    n = 2048
    dev = "cuda"
    feats = bdsynth.target_features(bdsynth.CTX27B, n, 0, stream=77, device=dev)
    req = torch.zeros(n, dtype=torch.int32, device=dev)
    pos = torch.arange(n, dtype=torch.int64, device=dev)
    front = torch.tensor([n], dtype=torch.int64, device=dev)

    def call():
        st.sess.materialize(feats, req, pos, front)
    ms = time_call(call, steps, warmup)
    H = geo.hidden
    KD = geo.n_kv_heads * geo.head_dim
    flops = 2.0 * n * geo.n_target_layers * H * H + 2.0 * n * geo.n_layers * 2 * KD * H
    by = (H * geo.n_target_layers * H + geo.n_layers * 2 * KD * H) * 2 + n * geo.n_target_layers * H * 2 \
        + geo.n_layers * n * 2 * KD * 2
    tfs = flops / (ms * 1e-3) / 1e12
    return {"workload": bdsynth.CTX27B.name, "rows": n, "us": 1000.0 * ms, "tflops": tfs,
            "flops": flops, "frac_of_sustained_bf16": tfs / tf_sust, "frac_of_burst_bf16": tfs / tf_burst,
            "bound": "tensor", "algorithmic_bytes": by,
            "frac_of_measured_hbm": by / (ms * 1e-3) / 1e9 / hbm}


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


def recorded_traffic(kind: str):
    """DRAM bytes per launch of one kernel kind from the committed ncu record, if the
    kernel's sources are unchanged since the counters were taken (else None)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get("kernels", {}).get(kind)
    if rec is None:
        return None
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
        return (d["hbm_gbs"], d.get("bf16_tflops_sustained", 1715.0), d.get("bf16_tflops", 1875.0),
                "measured")
    return 6800.0, 1700.0, 1900.0, "fallback"


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
def reference_line(geo, args) -> dict:
    """The reference arm's JSON line for workload ``geo``: the fp64 CPU oracle as it stands,
    on the host cores.  Each step is one full oracle step of request 0 (catch-up
    materialisation of its W pending rows, the round over its context window, the LM head),
    i.e. exactly the per-request work of one GPU step at B=1."""
    import numpy as np
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
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": geo.name, "B": 1, "W": geo.W, "context": int(F[0]),
                       "window": geo.windows[0]},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"one full oracle step of request 0 per step: catch-up of "
                                       f"{geo.W} rows, {geo.n_layers}-layer round, full LM head"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args, rank, world):
    """The reference arm on the metric's workload (the 27B B=1 round); rank 0 only."""
    if rank != 0:
        return
    print(json.dumps(reference_line(bdsynth.DSPINE27B_B1, args)), flush=True)


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
    hbm, tf, tf_burst, peak_kind = peaks()
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
                   "operands": "bf16 weights (packed image: Q/K/V, W_o, MLP and head converted "
                               "to fp16); fp16 activations in those products, bf16 hi+lo pairs "
                               "in the feature projection, the bridge products and the "
                               "attention's scores and probabilities; fp32 accumulation and "
                               "residual stream",
                   "parallelism": f"replicas x{world}"},
        "us_per_step": 1000.0 * ms,
        "breakdown_us": {k: 1000.0 * v for k, v in per.items()},
        "round_only": round_only(st, args),
        "separate_catch_up": separate_catch_up(st, args),
        "achieved_step_gbs": step_gbs,
        "step_roofline_frac": {"of_measured_hbm": step_gbs / hbm, "of_8tbs": step_gbs / 8000.0},
        "algorithmic_bytes_per_step": by,
        "roofline_lm_head_call": {"bound": "hbm",
                                  "kernel": "LM head call (tcgen05 GEMM + split-vocab argmax reduce)",
                                  "achieved": head_gbs, "peak": hbm, "unit": "GB/s",
                                  "frac": head_gbs / hbm, "algorithmic_bytes": head_bytes,
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
    # per-kernel device times inside the step; the roofline entry is the kernel kind with
    # the largest share of the step
    kt = kernel_times(st, min(args.steps, 10), args.warmup, hbm)
    dom = dominant(kt)
    line["roofline"] = roofline_entry(dom, kt, hbm, peak_kind, KIND_NAMES[dom])
    line["kernels"] = kt
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
        kt8 = kernel_times(st8, min(args.steps, 10), args.warmup, hbm)
        dom8 = dominant(kt8)
        line["b8"]["roofline"] = roofline_entry(dom8, kt8, hbm, peak_kind, KIND_NAMES[dom8])
        line["b8"]["kernels"] = kt8
        del st8
    if not args.no_b8 and args.workload == "b1":
        line["dflash2"] = dflash2_lines(args, world, hbm)
        line["dflash_35b_b8"] = dflash35b_line(args, world, hbm, peak_kind)
    if rank == 0 and not args.no_cpu_baseline:
        wh = host_weights(st.w)
        feats = st.feats[:geo.W].float().cpu().numpy()
        pos = st.row_pos[:geo.W].cpu().numpy()
        ts = [oracle_step_sample(geo, wh, st.F, st.anchors_l, st.mask, feats, pos)
              for _ in range(CPU_SAMPLES)]
        t = statistics.mean(ts)
        line["cpu_baseline"] = {"value": 1.0 / t, "unit": UNIT, "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"one full step of request 0 (catch-up of 16 rows, "
                                          f"5-layer round, full LM head) at B=1, mean of "
                                          f"{CPU_SAMPLES} runs",
                                "seconds_per_sample": ts}
    if args.workload == "b1":
        # last: it overwrites request 0's rings of the B=1 state
        line["ctx_materialize_2048"] = materialize_line(st, args.steps, args.warmup, tf, tf_burst, hbm)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
