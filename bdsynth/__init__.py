"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the fp64 oracle.

This module holds workload SHAPES and random DRAWS only.  It contains none of the
drafter's arithmetic (no norm, projection, attention or injection): both sides take
the tensors it returns and compute on their own.  Nothing here imports the oracle or
the CUDA package.

Draw recipe (the same for every workload):
  * every tensor has its own index ``i`` in a fixed table and is drawn with
    ``torch.Generator(device).manual_seed(seed * 1_000_000 + i)``;
  * projection matrices ~ N(0, 0.02), drawn in fp32 and rounded to the workload dtype;
  * RMSNorm / head-norm gains ~ 1 + N(0, 0.02) (a gain drawn N(0, 0.02) would collapse
    every activation towards zero and make the argmax comparison vacuous);
  * token-code table rows are N(0, 1) rows scaled to unit L2 norm before rounding
    (the DSpine pages build the table from normalised vectors);
  * DFlash2 convolution: base coefficients of the current tap 1 + N(0, 0.1), of the
    previous tap N(0, 0.1); delta projections N(0, 0.002) (the pages give no
    initialisation; these keep every coefficient near its base at H = 5120);
  * captured target residuals ~ N(0, 1) times a per-captured-layer scale ~ U[0.5, 4];
  * anchor ids ~ U[0, V) with the MASK id excluded; frontiers as each workload states.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

BF16 = "bf16"
F32 = "f32"


@dataclasses.dataclass(frozen=True)
class Workload:
    """Geometry of one drafter workload (the fields mirror a DFlash draft config)."""

    name: str
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    n_target_layers: int
    windows: tuple            # per layer: sliding window S, or 0 for a full-context layer
    code_width: int           # Rc; 0 disables the DSpine bridge (plain DFlash)
    msg_width: int            # Mc
    batch: int                # B requests
    n_masks: int              # K; the block is W = K + 1 rows
    dtype: str
    eps: float = 1e-6
    rope_theta: float = 1e7
    mask_token_id: int = -1   # -1: drawn per seed (small vocabularies)
    ctx_min: int = 0          # committed context length range (inclusive)
    ctx_max: int = 0
    full_capacity: int = 0    # ring capacity of full-context layers (>= ctx_max)
    block_causal: bool = False
    conv_group: int = 0       # DFlash2 grouped convolution group width (0: none)

    @property
    def W(self) -> int:
        return self.n_masks + 1

    @property
    def tokens(self) -> int:
        return self.batch * self.W

    def capacity(self, layer: int) -> int:
        s = self.windows[layer]
        return s if s > 0 else self.full_capacity

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the drafter is measured and checked on.
TINY = Workload(
    name="tiny_fp32", hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=64,
    ffn=768, vocab=1024, n_target_layers=2, windows=(0, 0), code_width=64, msg_width=32,
    batch=1, n_masks=7, dtype=F32, ctx_min=128, ctx_max=128, full_capacity=128)

CTX27B = Workload(
    name="ctx_materialize_27b", hidden=5120, n_layers=5, n_q_heads=32, n_kv_heads=8,
    head_dim=128, ffn=17408, vocab=151936, n_target_layers=5, windows=(2048,) * 5,
    code_width=1024, msg_width=512, batch=1, n_masks=15, dtype=BF16,
    mask_token_id=151669, ctx_min=2048, ctx_max=2048)

DSPINE27B_B1 = Workload(
    name="dspine_b16_27b_b1", hidden=5120, n_layers=5, n_q_heads=32, n_kv_heads=8,
    head_dim=128, ffn=17408, vocab=151936, n_target_layers=5, windows=(2048,) * 5,
    code_width=1024, msg_width=512, batch=1, n_masks=15, dtype=BF16,
    mask_token_id=151669, ctx_min=4096, ctx_max=4096)

DSPINE27B_B8 = DSPINE27B_B1.with_(name="dspine_b16_27b_b8", batch=8, ctx_min=512, ctx_max=16384)

# DFlash2 at the same 27B geometry: the dynamic grouped convolution (two taps, group
# width 16) around both branches, no DSpine bridge.
DFLASH2_27B_B1 = DSPINE27B_B1.with_(name="dflash2_27b_b1", code_width=0, msg_width=0,
                                    conv_group=16)
DFLASH2_27B_B8 = DFLASH2_27B_B1.with_(name="dflash2_27b_b8", batch=8, ctx_min=512,
                                      ctx_max=16384)

DFLASH35B_B8 = Workload(
    name="dflash_35b_a3b_b8", hidden=2048, n_layers=6, n_q_heads=32, n_kv_heads=8,
    head_dim=128, ffn=6144, vocab=151936, n_target_layers=8,
    windows=(4096, 4096, 4096, 4096, 4096, 0), code_width=0, msg_width=0, batch=8,
    n_masks=15, dtype=BF16, mask_token_id=151669, ctx_min=4096, ctx_max=32768,
    full_capacity=32768)

WORKLOADS: Dict[str, Workload] = {w.name: w for w in
                                  (TINY, CTX27B, DSPINE27B_B1, DSPINE27B_B8, DFLASH2_27B_B1,
                                   DFLASH2_27B_B8, DFLASH35B_B8)}


def torch_dtype(dt: str) -> torch.dtype:
    return torch.bfloat16 if dt == BF16 else torch.float32


# --------------------------------------------------------------------------- draws
def _gen(seed: int, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_000 + index)
    return g


def normal(shape, seed: int, index: int, *, std: float = 1.0, mean: float = 0.0,
           device="cpu", dtype=torch.float32) -> torch.Tensor:
    """fp32 N(mean, std) draw from its own seeded generator, rounded to ``dtype``."""
    g = _gen(seed, index, device)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def uniform(shape, lo: float, hi: float, seed: int, index: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, index, device)
    return torch.rand(tuple(shape), generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def randint(lo: int, hi_inclusive: int, n: int, seed: int, index: int) -> List[int]:
    g = _gen(seed, index, "cpu")
    return torch.randint(lo, hi_inclusive + 1, (n,), generator=g).tolist()


# Tensor index table.  Per-layer tensors use LAYER_BASE + 20 * layer + slot.
IDX_W_FEATURE, IDX_CONTEXT_NORM, IDX_FINAL_NORM, IDX_EMBED, IDX_CODEBOOK = 0, 1, 2, 3, 4
IDX_G_RECV, IDX_G_PRED, IDX_A_VAL, IDX_GATE_BIAS = 5, 6, 7, 8
IDX_ANCHORS, IDX_MASK_ID, IDX_FRONTIER, IDX_FEAT_SCALE = 9, 10, 11, 12
IDX_FEATURES = 10_000          # + stream (one independent draw per request)
LAYER_BASE = 100
LAYER_SLOTS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm",
               "w_gate", "w_up", "w_down", "r_read", "w_write", "conv_delta_a", "conv_base_a",
               "conv_delta_m", "conv_base_m")
CONV_BASE_SLOTS = ("conv_base_a", "conv_base_m")
CONV_DELTA_STD = 0.002  # delta ~ N(0, 0.14) per group at H = 5120
NORM_SLOTS = ("in_norm", "q_norm", "k_norm", "post_norm")


def layer_shapes(w: Workload) -> Dict[str, tuple]:
    H, D = w.hidden, w.head_dim
    s = {
        "in_norm": (H,), "wq": (w.n_q_heads * D, H), "wk": (w.n_kv_heads * D, H),
        "wv": (w.n_kv_heads * D, H), "q_norm": (D,), "k_norm": (D,),
        "wo": (H, w.n_q_heads * D), "post_norm": (H,), "w_gate": (w.ffn, H),
        "w_up": (w.ffn, H), "w_down": (H, w.ffn),
    }
    if w.code_width > 0:
        s["r_read"] = (w.code_width, H)
        s["w_write"] = (H, w.msg_width)
    if w.conv_group > 0:
        for br in ("a", "m"):
            s["conv_delta_" + br] = (4 * H // w.conv_group, H)
            s["conv_base_" + br] = (2, 2, H)
    return s


def make_weights(w: Workload, seed: int = 0, device="cpu", *, gate_bias: bool = False,
                 zero_write: bool = False, layers: Optional[List[int]] = None) -> dict:
    """All drafter weights of ``w`` in its dtype.  Returns a nested dict of tensors.

    ``zero_write`` draws every per-layer write matrix as zeros (the identity start of
    the injection).  ``layers`` restricts the per-layer draws (others are omitted).
    """
    dt = torch_dtype(w.dtype)
    H = w.hidden
    out = {
        "w_feature": normal((H, w.n_target_layers * H), seed, IDX_W_FEATURE, std=0.02,
                            device=device, dtype=dt),
        "context_norm": normal((H,), seed, IDX_CONTEXT_NORM, std=0.02, mean=1.0,
                               device=device, dtype=dt),
        "final_norm": normal((H,), seed, IDX_FINAL_NORM, std=0.02, mean=1.0, device=device,
                             dtype=dt),
        "embed_head": normal((w.vocab, H), seed, IDX_EMBED, std=0.02, device=device, dtype=dt),
        "layers": [],
    }
    if w.code_width > 0:
        Rc, Mc = w.code_width, w.msg_width
        cb = normal((w.vocab, Rc), seed, IDX_CODEBOOK, device=device, dtype=torch.float32)
        cb = cb / cb.norm(dim=1, keepdim=True)
        out["codebook"] = cb.to(dt)
        out["g_recv"] = normal((Mc, Rc), seed, IDX_G_RECV, std=0.02, device=device, dtype=dt)
        out["g_pred"] = normal((Mc, Rc), seed, IDX_G_PRED, std=0.02, device=device, dtype=dt)
        out["a_val"] = normal((Mc, Rc), seed, IDX_A_VAL, std=0.02, device=device, dtype=dt)
        out["gate_bias"] = (normal((Mc,), seed, IDX_GATE_BIAS, std=0.02, device=device, dtype=dt)
                            if gate_bias else None)
    shapes = layer_shapes(w)
    for l in range(w.n_layers):
        if layers is not None and l not in layers:
            out["layers"].append(None)
            continue
        d = {}
        for slot_i, name in enumerate(LAYER_SLOTS):
            if name not in shapes:
                continue
            idx = LAYER_BASE + 20 * l + slot_i
            if name in NORM_SLOTS:
                d[name] = normal(shapes[name], seed, idx, std=0.02, mean=1.0, device=device,
                                 dtype=dt)
            elif name == "w_write" and zero_write:
                d[name] = torch.zeros(shapes[name], device=device, dtype=dt)
            elif name in CONV_BASE_SLOTS:
                b = normal(shapes[name], seed, idx, std=0.1, device=device)
                b[:, 0] += 1.0
                d[name] = b.to(dt)
            elif name.startswith("conv_delta"):
                d[name] = normal(shapes[name], seed, idx, std=CONV_DELTA_STD, device=device,
                                 dtype=dt)
            else:
                d[name] = normal(shapes[name], seed, idx, std=0.02, device=device, dtype=dt)
        out["layers"].append(d)
    return out


def mask_token_id(w: Workload, seed: int = 0) -> int:
    if w.mask_token_id >= 0:
        return w.mask_token_id
    return randint(0, w.vocab - 1, 1, seed, IDX_MASK_ID)[0]


def anchor_ids(w: Workload, seed: int = 0) -> List[int]:
    """Uniform anchors in [0, V) that are never the MASK id."""
    mask = mask_token_id(w, seed)
    ids = randint(0, w.vocab - 2, w.batch, seed, IDX_ANCHORS)
    return [i + 1 if i >= mask else i for i in ids]


def frontiers(w: Workload, seed: int = 0) -> List[int]:
    """Committed context length F_b per request (uniform in the workload's range)."""
    if w.ctx_min == w.ctx_max:
        return [w.ctx_min] * w.batch
    return randint(w.ctx_min, w.ctx_max, w.batch, seed, IDX_FRONTIER)


def feature_scales(w: Workload, seed: int = 0) -> torch.Tensor:
    """Per captured target layer scale ~ U[0.5, 4]."""
    return uniform((w.n_target_layers,), 0.5, 4.0, seed, IDX_FEAT_SCALE)


def target_features(w: Workload, n_rows: int, seed: int = 0, stream: int = 0,
                    device="cpu") -> torch.Tensor:
    """``n_rows`` captured target residual rows [n_rows, n_target_layers * H] in the
    workload dtype: N(0,1) per element times the captured layer's scale.

    ``stream`` selects an independent draw (e.g. one per request)."""
    H = w.hidden
    scales = feature_scales(w, seed).to(device)
    t = normal((n_rows, w.n_target_layers, H), seed, IDX_FEATURES + stream, device=device)
    t.mul_(scales.view(1, -1, 1))
    return t.reshape(n_rows, w.n_target_layers * H).to(torch_dtype(w.dtype))


def live_window(w: Workload, frontier: int) -> tuple:
    """[lo, hi) context positions any layer of ``w`` can read at this frontier:
    the largest ring capacity bounds it (full layers: everything)."""
    caps = [w.capacity(l) for l in range(w.n_layers)]
    lo = max(0, frontier - max(caps))
    return lo, frontier


__all__ = [n for n in dir() if not n.startswith("_")]
