"""Thin ctypes binding of ``libblockdrafter.so`` (argument marshalling only).

The functions carry the C ABI's names without the ``bd_`` prefix and take torch tensors
(device memory) or plain ints; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if the library is missing the import of this
module's functions raises.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

from .builder import LIBPATH

MAX_LAYERS = 16
BF16, F32 = 0, 1
BIDIRECTIONAL, CAUSAL = 0, 1

STATUS = {0: "BD_OK", -1: "BD_ERR_INVALID_ARG", -2: "BD_ERR_UNSUPPORTED", -3: "BD_ERR_CUDA",
          -4: "BD_ERR_DEVICE_TIMEOUT", -5: "BD_ERR_WORKSPACE", -6: "BD_ERR_RANGE"}

EXPORTS = ("bd_abi_version", "bd_workspace_bytes", "bd_ctx_kv_materialize", "bd_draft_round",
           "bd_lm_head_argmax", "bd_last_error", "bd_sync_status", "bd_kernel_launches",
           "bd_packed_bytes", "bd_pack_weights", "bd_lm_head_argmax_noalloc", "bd_lm_head_topk",
           "bd_refine_tail", "bd_head_fp8_bytes", "bd_pack_head_fp8", "bd_lm_head_topk_fp8",
           "bd_selftest_wait", "bd_set_timing_events")

TOPK_MAX = 16


class BdError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("n_layers", C.c_int), ("n_q_heads", C.c_int),
                ("n_kv_heads", C.c_int), ("head_dim", C.c_int), ("ffn", C.c_int),
                ("vocab", C.c_int), ("n_target_layers", C.c_int),
                ("window", C.c_int * MAX_LAYERS), ("ring_capacity", C.c_int * MAX_LAYERS),
                ("eps", C.c_float), ("rope_theta", C.c_float), ("mask_token_id", C.c_int),
                ("code_width", C.c_int), ("msg_width", C.c_int), ("block_mask", C.c_int),
                ("dtype", C.c_int), ("conv_group", C.c_int)]


LAYER_FIELDS = ("in_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "post_norm", "w_gate",
                "w_up", "w_down", "r_read", "w_write", "conv_delta_a", "conv_base_a",
                "conv_delta_m", "conv_base_m")


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in LAYER_FIELDS]


class Weights(C.Structure):
    _fields_ = [("w_feature", C.c_void_p), ("context_norm", C.c_void_p),
                ("final_norm", C.c_void_p), ("embed_head", C.c_void_p), ("codebook", C.c_void_p),
                ("g_recv", C.c_void_p), ("g_pred", C.c_void_p), ("a_val", C.c_void_p),
                ("gate_bias", C.c_void_p), ("layer", LayerWeights * MAX_LAYERS),
                ("packed", C.c_void_p)]


class KvCache(C.Structure):
    _fields_ = [("k", C.c_void_p * MAX_LAYERS), ("v", C.c_void_p * MAX_LAYERS),
                ("b_max", C.c_int)]


class Pending(C.Structure):
    _fields_ = [("feats", C.c_void_p), ("request", C.c_void_p), ("pos", C.c_void_p),
                ("n_rows", C.c_int)]


_lib = None


def lib() -> C.CDLL:
    """Load the library (built by ``block_drafter_gb300.builder.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBPATH):
            raise RuntimeError(f"libblockdrafter.so is not built ({LIBPATH}); run "
                               "block_drafter_gb300.builder.build() first")
        L = C.CDLL(LIBPATH)
        vp, i, sz = C.c_void_p, C.c_int, C.c_size_t
        L.bd_abi_version.restype = i
        L.bd_workspace_bytes.restype = sz
        L.bd_workspace_bytes.argtypes = [C.POINTER(Config), i, i, i]
        L.bd_ctx_kv_materialize.restype = i
        L.bd_ctx_kv_materialize.argtypes = [C.POINTER(Config), C.POINTER(Weights),
                                            C.POINTER(KvCache), vp, vp, vp, vp, i, vp, sz, vp]
        L.bd_draft_round.restype = i
        L.bd_draft_round.argtypes = [C.POINTER(Config), C.POINTER(Weights), C.POINTER(KvCache),
                                     vp, vp, i, i, vp, vp, vp, vp, C.POINTER(Pending), vp, sz, vp]
        L.bd_refine_tail.restype = i
        L.bd_refine_tail.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, vp, vp, i, i, i,
                                     vp, vp, vp, vp, sz, vp]
        L.bd_lm_head_argmax.restype = i
        L.bd_lm_head_argmax.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, i, vp, vp,
                                        vp, sz, vp]
        L.bd_last_error.restype = C.c_char_p
        L.bd_sync_status.restype = i
        L.bd_sync_status.argtypes = [vp]
        L.bd_kernel_launches.restype = C.c_uint64
        L.bd_packed_bytes.restype = sz
        L.bd_packed_bytes.argtypes = [C.POINTER(Config)]
        L.bd_pack_weights.restype = i
        L.bd_pack_weights.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, sz, vp]
        L.bd_lm_head_argmax_noalloc.restype = i
        L.bd_lm_head_argmax_noalloc.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, i, vp,
                                                vp, vp]
        L.bd_lm_head_topk.restype = i
        L.bd_lm_head_topk.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, i, i, vp, vp, vp,
                                      sz, vp]
        L.bd_selftest_wait.restype = i
        L.bd_selftest_wait.argtypes = [vp, i, vp]
        L.bd_head_fp8_bytes.restype = sz
        L.bd_head_fp8_bytes.argtypes = [C.POINTER(Config)]
        L.bd_pack_head_fp8.restype = i
        L.bd_pack_head_fp8.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, sz, vp]
        L.bd_lm_head_topk_fp8.restype = i
        L.bd_lm_head_topk_fp8.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, vp, i, i, i,
                                          vp, vp, vp, sz, vp]
        L.bd_set_timing_events.restype = i
        L.bd_set_timing_events.argtypes = [i, C.POINTER(vp), C.POINTER(vp), i]
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise BdError(status, lib().bd_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


# ------------------------------------------------------------------ marshalling
def make_config(*, hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab,
                n_target_layers, windows: Sequence[int], ring_capacity: Sequence[int], eps,
                rope_theta, mask_token_id, code_width=0, msg_width=0, block_causal=False,
                dtype=BF16, conv_group=0) -> Config:
    c = Config()
    c.hidden, c.n_layers, c.n_q_heads, c.n_kv_heads = hidden, n_layers, n_q_heads, n_kv_heads
    c.head_dim, c.ffn, c.vocab, c.n_target_layers = head_dim, ffn, vocab, n_target_layers
    for l in range(n_layers):
        c.window[l] = int(windows[l])
        c.ring_capacity[l] = int(ring_capacity[l])
    c.eps, c.rope_theta, c.mask_token_id = eps, rope_theta, mask_token_id
    c.code_width, c.msg_width = code_width, msg_width
    c.block_mask = CAUSAL if block_causal else BIDIRECTIONAL
    c.dtype = dtype
    c.conv_group = conv_group
    return c


def make_weights(cfg: Config, w: dict) -> Weights:
    """``w``: dict of device tensors with the keys of ``bd_weights`` (and a ``layers``
    list of per-layer dicts with the keys of ``bd_layer_weights``)."""
    s = Weights()
    for k in ("w_feature", "context_norm", "final_norm", "embed_head", "codebook", "g_recv",
              "g_pred", "a_val", "gate_bias"):
        t = w.get(k)
        setattr(s, k, _ptr(t) if t is not None else None)
    for l, lw in enumerate(w["layers"][:cfg.n_layers]):
        for k in LAYER_FIELDS:
            t = lw.get(k) if lw is not None else None
            setattr(s.layer[l], k, _ptr(t) if t is not None else None)
    return s


def make_kv(k: Sequence[torch.Tensor], v: Sequence[torch.Tensor], b_max: int) -> KvCache:
    s = KvCache()
    for l, (kk, vv) in enumerate(zip(k, v)):
        s.k[l] = kk.data_ptr()
        s.v[l] = vv.data_ptr()
    s.b_max = b_max
    return s


# ------------------------------------------------------------------ entry points
def abi_version() -> int:
    return lib().bd_abi_version()


def packed_bytes(cfg: Config) -> int:
    n = lib().bd_packed_bytes(C.byref(cfg))
    if n == 0:
        raise BdError(-1, "invalid config for bd_packed_bytes")
    return n


def pack_weights(cfg: Config, weights: Weights, packed: torch.Tensor, stream=None) -> int:
    """Writes the packed image into ``packed`` (uint8 device tensor) at its first
    1024-byte aligned address and returns that address (to store in weights.packed)."""
    base = packed.data_ptr()
    aligned = (base + 1023) // 1024 * 1024
    nbytes = packed.numel() - (aligned - base)
    _check(lib().bd_pack_weights(C.byref(cfg), C.byref(weights), aligned, nbytes, _stream(stream)))
    return aligned


def head_fp8_bytes(cfg: Config) -> int:
    return lib().bd_head_fp8_bytes(C.byref(cfg))


def pack_head_fp8(cfg: Config, weights: Weights, image: torch.Tensor, stream=None) -> int:
    """Writes the FP8 head copy into ``image`` (uint8 device tensor) at its first 1024-byte
    aligned address and returns that address."""
    base = image.data_ptr()
    aligned = (base + 1023) // 1024 * 1024
    nbytes = image.numel() - (aligned - base)
    _check(lib().bd_pack_head_fp8(C.byref(cfg), C.byref(weights), aligned, nbytes, _stream(stream)))
    return aligned


def lm_head_topk_fp8(cfg: Config, weights: Weights, head_fp8: int, hidden: torch.Tensor,
                     n_cand: int, k: int, token_out: torch.Tensor, workspace: torch.Tensor,
                     score_out: Optional[torch.Tensor] = None, stream=None):
    """FP8 retrieval of n_cand candidates per hidden row, BF16 rescoring, the k best."""
    _check(lib().bd_lm_head_topk_fp8(
        C.byref(cfg), C.byref(weights), head_fp8, _ptr(hidden), int(hidden.shape[0]), int(n_cand),
        int(k), _ptr(token_out), _ptr(score_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def workspace_bytes(cfg: Config, b_max: int, max_masks: int, max_ctx_rows: int) -> int:
    n = lib().bd_workspace_bytes(C.byref(cfg), b_max, max_masks, max_ctx_rows)
    if n == 0:
        raise BdError(-1, "invalid config or sizes for bd_workspace_bytes")
    return n


def ctx_kv_materialize(cfg: Config, weights: Weights, kv: KvCache, target_feats: torch.Tensor,
                       row_request: torch.Tensor, row_pos: torch.Tensor,
                       ctx_frontier: torch.Tensor, workspace: torch.Tensor, stream=None):
    _check(lib().bd_ctx_kv_materialize(
        C.byref(cfg), C.byref(weights), C.byref(kv), _ptr(target_feats), _ptr(row_request),
        _ptr(row_pos), _ptr(ctx_frontier), int(target_feats.shape[0]), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def draft_round(cfg: Config, weights: Weights, kv: KvCache, anchor_ids: torch.Tensor,
                frontier: torch.Tensor, n_masks: int, head_in: torch.Tensor,
                workspace: torch.Tensor, hidden_out: Optional[torch.Tensor] = None,
                layers_out: Optional[torch.Tensor] = None, stream=None,
                tail_state: Optional[torch.Tensor] = None, pending: Optional[tuple] = None):
    """pending = (feats [n, n_tgt*H], request int32 [n], pos int64 [n]) or None: context
    rows the round materialises before it drafts (frontier is the frontier they complete)."""
    pd = None
    if pending is not None:
        feats, req, pos = pending
        pd = Pending(_ptr(feats), _ptr(req), _ptr(pos), int(feats.shape[0]))
    _check(lib().bd_draft_round(
        C.byref(cfg), C.byref(weights), C.byref(kv), _ptr(anchor_ids), _ptr(frontier),
        int(anchor_ids.shape[0]), int(n_masks), _ptr(head_in), _ptr(hidden_out),
        _ptr(layers_out), _ptr(tail_state), None if pd is None else C.byref(pd), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def tail_state_floats(cfg: Config, B: int, n_masks: int) -> int:
    """Size of bd_draft_round's tail_state: T*H + T + T*Mc floats, T = B*(n_masks+1)."""
    T = B * (n_masks + 1)
    return T * (cfg.hidden + 1 + cfg.msg_width)


def refine_tail(cfg: Config, weights: Weights, tail_state: torch.Tensor, cand_ids: torch.Tensor,
                cand_scores: torch.Tensor, B: int, n_masks: int, token_out: torch.Tensor,
                workspace: torch.Tensor, pick_out: Optional[torch.Tensor] = None,
                table_out: Optional[torch.Tensor] = None, stream=None):
    """Last-write refinement + transition tables + greedy walk (bd_refine_tail)."""
    _check(lib().bd_refine_tail(
        C.byref(cfg), C.byref(weights), _ptr(tail_state), _ptr(cand_ids), _ptr(cand_scores),
        int(B), int(n_masks), int(cand_ids.shape[1]), _ptr(token_out), _ptr(pick_out),
        _ptr(table_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def lm_head_argmax(cfg: Config, weights: Weights, hidden: torch.Tensor, token_out: torch.Tensor,
                   workspace: torch.Tensor, max_logit_out: Optional[torch.Tensor] = None,
                   stream=None):
    _check(lib().bd_lm_head_argmax(
        C.byref(cfg), C.byref(weights), _ptr(hidden), int(hidden.shape[0]), _ptr(token_out),
        _ptr(max_logit_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def lm_head_topk(cfg: Config, weights: Weights, hidden: torch.Tensor, k: int,
                 token_out: torch.Tensor, workspace: torch.Tensor,
                 score_out: Optional[torch.Tensor] = None, stream=None):
    """The k best candidates per hidden row: token_out / score_out [rows, k]."""
    _check(lib().bd_lm_head_topk(
        C.byref(cfg), C.byref(weights), _ptr(hidden), int(hidden.shape[0]), int(k), _ptr(token_out),
        _ptr(score_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def lm_head_argmax_noalloc(cfg: Config, weights: Weights, hidden: torch.Tensor,
                           token_out: torch.Tensor, max_logit_out: Optional[torch.Tensor] = None,
                           stream=None):
    """bd_lm_head_argmax without a workspace (scratch in the library's static device array)."""
    _check(lib().bd_lm_head_argmax_noalloc(
        C.byref(cfg), C.byref(weights), _ptr(hidden), int(hidden.shape[0]), _ptr(token_out),
        _ptr(max_logit_out), _stream(stream)))


TIME_KINDS = {"qkv": 1, "attention": 2, "wo": 3, "gate_up": 4, "down": 5, "bridge": 6, "head": 7}


def set_timing_events(kind: Optional[str], begin=(), end=()):
    """Bracket the launches of one kernel kind with CUDA events (bd_set_timing_events);
    ``begin``/``end`` are torch.cuda.Event objects with timing enabled.  kind None clears."""
    if kind is None:
        _check(lib().bd_set_timing_events(0, None, None, 0))
        return
    n = len(begin)
    assert n == len(end) and n > 0
    for ev in list(begin) + list(end):  # torch creates the CUDA event on first record
        if ev.cuda_event == 0:
            ev.record()
    arr_b = (C.c_void_p * n)(*[ev.cuda_event for ev in begin])
    arr_e = (C.c_void_p * n)(*[ev.cuda_event for ev in end])
    _check(lib().bd_set_timing_events(TIME_KINDS[kind], arr_b, arr_e, n))


def kernel_launches() -> int:
    return int(lib().bd_kernel_launches())


def selftest_wait(flag: torch.Tensor, limit_us: int, stream=None):
    """One bounded wait for flag[0] >= 1 (int32 device tensor); see bd_selftest_wait."""
    _check(lib().bd_selftest_wait(_ptr(flag), int(limit_us), _stream(stream)))


def sync_status(stream=None):
    _check(lib().bd_sync_status(_stream(stream)))
