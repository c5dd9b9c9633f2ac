"""Glue for the parity tests: seeded inputs (bdsynth) -> CUDA path (C ABI) and oracle.

Nothing here computes any step of the method; it only moves tensors between the
seeded generator, the library and the oracle, and measures errors.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

import bdsynth
from oracle import dspine_oracle as O


def np32(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16/fp32 tensor to a float32 NumPy array."""
    return t.detach().to(torch.float32).cpu().numpy()


def weights_to_np(w: dict) -> dict:
    out = {}
    for k, v in w.items():
        if k == "layers":
            out[k] = [None if lw is None else {kk: np32(vv) for kk, vv in lw.items()} for lw in v]
        elif v is None:
            out[k] = None
        else:
            out[k] = np32(v)
    return out


def weights_to(w: dict, device) -> dict:
    out = {}
    for k, v in w.items():
        if k == "layers":
            out[k] = [None if lw is None else {kk: vv.to(device).contiguous() for kk, vv in lw.items()}
                      for lw in v]
        elif v is None:
            out[k] = None
        else:
            out[k] = v.to(device).contiguous()
    return out


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| over the whole tensor."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


class Case:
    """One seeded workload instance on the GPU plus what the oracle needs."""

    def __init__(self, geo: bdsynth.Workload, seed: int = 0, *, zero_write=False, gate_bias=False,
                 frontiers: Optional[List[int]] = None, anchors: Optional[List[int]] = None,
                 gen_device="cpu", max_ctx_rows: int = 2048, weights=None, packed: bool = True):
        from block_drafter_gb300.session import DraftSession
        self.geo, self.seed = geo, seed
        self.mask_id = bdsynth.mask_token_id(geo, seed)
        self.anchors = anchors if anchors is not None else bdsynth.anchor_ids(geo, seed)
        self.frontiers = frontiers if frontiers is not None else bdsynth.frontiers(geo, seed)
        w = weights if weights is not None else bdsynth.make_weights(
            geo, seed, gen_device, zero_write=zero_write, gate_bias=gate_bias)
        self.w_dev = weights_to(w, "cuda")
        self.w_host = w
        self.gen_device = gen_device
        self.sess = DraftSession(geo, self.w_dev, self.mask_id, b_max=geo.batch,
                                 max_masks=geo.n_masks, max_ctx_rows=max_ctx_rows, packed=packed)
        self.max_ctx_rows = max_ctx_rows

    # ---- context
    def request_rows(self, b: int):
        lo, hi = bdsynth.live_window(self.geo, self.frontiers[b])
        return lo, hi

    def features(self, b: int, lo: int, n: int, chunk_index: int = 0) -> torch.Tensor:
        """Captured target rows of request b for positions [lo, lo+n) (one draw per
        (request, chunk))."""
        return bdsynth.target_features(self.geo, n, self.seed, stream=b * 4096 + chunk_index,
                                       device=self.gen_device)

    def fill_rings(self) -> Dict[int, list]:
        """Materialise every request's live window through the C ABI, in chunks of at
        most max_ctx_rows rows.  Returns {b: [(lo, feats_cpu), ...]} for the oracle."""
        dev = "cuda"
        front = torch.tensor(self.frontiers, dtype=torch.int64, device=dev)
        used = {}
        for b in range(self.geo.batch):
            lo, hi = self.request_rows(b)
            used[b] = []
            ci = 0
            for c0 in range(lo, hi, self.max_ctx_rows):
                n = min(self.max_ctx_rows, hi - c0)
                f = self.features(b, c0, n, ci).to(dev)
                req = torch.full((n,), b, dtype=torch.int32, device=dev)
                pos = torch.arange(c0, c0 + n, dtype=torch.int64, device=dev)
                self.sess.materialize(f, req, pos, front)
                used[b].append((c0, f))
                ci += 1
        torch.cuda.synchronize()
        return used

    def rings_np(self, requests: Optional[List[int]] = None) -> dict:
        reqs = list(range(self.geo.batch)) if requests is None else requests
        return {"k": [np32(k[reqs]) for k in self.sess.k], "v": [np32(v[reqs]) for v in self.sess.v]}

    # ---- round + head on the GPU
    def run_gpu(self, layers_out=True):
        g = self.geo
        Bn, K = g.batch, g.n_masks
        dev = "cuda"
        anchors = torch.tensor(self.anchors, dtype=torch.int32, device=dev)
        front = torch.tensor(self.frontiers, dtype=torch.int64, device=dev)
        head_in, tokens, maxl, hidden = self.sess.alloc_outputs(Bn, K)
        lo = (torch.empty(g.n_layers, Bn * (K + 1), g.hidden, dtype=torch.float32, device=dev)
              if layers_out else None)
        self.sess.round(anchors, front, K, head_in, hidden_out=hidden, layers_out=lo)
        self.sess.head(head_in, tokens, maxl)
        from block_drafter_gb300 import binding
        binding.sync_status()
        return {"head_in": head_in, "tokens": tokens, "max_logit": maxl, "hidden": hidden,
                "layers": lo}

    # ---- oracle (reads the GPU's context rings: round parity independent of S1/S2)
    def run_oracle(self, requests: Optional[List[int]] = None, with_head=True):
        reqs = list(range(self.geo.batch)) if requests is None else requests
        rings = self.rings_np(reqs)
        wnp = weights_to_np(self.w_host)
        return O.draft_round(self.geo, wnp, rings, [self.anchors[b] for b in reqs],
                             [self.frontiers[b] for b in reqs], self.mask_id, self.geo.n_masks,
                             with_head=with_head)


def compare_round(case: Case, gpu: dict, ref: dict, requests: Optional[List[int]] = None,
                  tol: float = 2e-2, gap_min: float = 1e-2) -> dict:
    """Per-layer residual and final-norm relative errors; token agreement where the
    oracle's top-2 gap exceeds gap_min."""
    g = case.geo
    reqs = list(range(g.batch)) if requests is None else requests
    W, H, K = g.W, g.hidden, g.n_masks
    rep = {"layer_err": [], "h_err": None, "token_mismatch": 0, "tokens_compared": 0}
    if gpu["layers"] is not None:
        lay = np32(gpu["layers"]).reshape(g.n_layers, g.batch, W, H)[:, reqs]
        for l in range(g.n_layers):
            rep["layer_err"].append(rel_err(lay[l], ref["x_layers"][l]))
    hid = np32(gpu["hidden"]).reshape(g.batch, W, H)[reqs]
    rep["h_err"] = rel_err(hid, ref["h"])
    if "tokens" in ref:
        tok = gpu["tokens"].cpu().numpy().reshape(g.batch, K)[reqs]
        sel = ref["gap"] > gap_min
        rep["tokens_compared"] = int(sel.sum())
        rep["token_mismatch"] = int((tok[sel] != ref["tokens"][sel]).sum())
        rep["min_gap"] = float(ref["gap"].min())
    rep["ok"] = (all(e <= tol for e in rep["layer_err"]) and rep["h_err"] <= tol
                 and rep["token_mismatch"] == 0)
    return rep
