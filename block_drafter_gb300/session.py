"""Convenience wrapper: owns the device buffers (rings, workspace, outputs) a user of the
C ABI would allocate, and calls the three entry points.  Allocation uses torch; all
computation happens in the library's kernels.

``geo`` is any object with the draft-geometry fields (hidden, n_layers, n_q_heads,
n_kv_heads, head_dim, ffn, vocab, n_target_layers, windows, code_width, msg_width, eps,
rope_theta, block_causal, dtype ("bf16"/"f32")) and a ``capacity(layer)`` method.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


def config_of(geo, mask_id: int) -> B.Config:
    return B.make_config(
        hidden=geo.hidden, n_layers=geo.n_layers, n_q_heads=geo.n_q_heads,
        n_kv_heads=geo.n_kv_heads, head_dim=geo.head_dim, ffn=geo.ffn, vocab=geo.vocab,
        n_target_layers=geo.n_target_layers, windows=geo.windows,
        ring_capacity=[geo.capacity(l) for l in range(geo.n_layers)], eps=geo.eps,
        rope_theta=geo.rope_theta, mask_token_id=mask_id, code_width=geo.code_width,
        msg_width=geo.msg_width, block_causal=geo.block_causal,
        dtype=B.BF16 if geo.dtype == "bf16" else B.F32, conv_group=geo.conv_group)


class DraftSession:
    def __init__(self, geo, weights: dict, mask_id: int, b_max: int, max_masks: int = 15,
                 max_ctx_rows: int = 2048, device="cuda", packed: bool = True):
        self.geo = geo
        self.device = torch.device(device)
        self.dtype = torch.bfloat16 if geo.dtype == "bf16" else torch.float32
        self.cfg = config_of(geo, mask_id)
        self.weights = weights
        self.wstruct = B.make_weights(self.cfg, weights)
        self.packed = None
        if packed:  # one-time packed image: GEMMs stream contiguous weight tiles from it
            self.packed = torch.empty(B.packed_bytes(self.cfg) + 1024, dtype=torch.uint8,
                                      device=self.device)
            self.wstruct.packed = B.pack_weights(self.cfg, self.wstruct, self.packed)
        self.b_max = b_max
        self.k = [torch.zeros(b_max, geo.n_kv_heads, geo.capacity(l), geo.head_dim,
                              dtype=self.dtype, device=self.device) for l in range(geo.n_layers)]
        self.v = [torch.zeros_like(t) for t in self.k]
        self.kv = B.make_kv(self.k, self.v, b_max)
        nbytes = B.workspace_bytes(self.cfg, b_max, max_masks, max_ctx_rows)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)

    # S1 + S2
    def materialize(self, feats: torch.Tensor, row_request: torch.Tensor, row_pos: torch.Tensor,
                    ctx_frontier: torch.Tensor, stream=None):
        B.ctx_kv_materialize(self.cfg, self.wstruct, self.kv, feats, row_request, row_pos,
                             ctx_frontier, self.workspace, stream)

    # S3 .. S9 + final norm
    def round(self, anchor_ids: torch.Tensor, frontier: torch.Tensor, n_masks: int,
              head_in: torch.Tensor, hidden_out: Optional[torch.Tensor] = None,
              layers_out: Optional[torch.Tensor] = None, stream=None,
              tail_state: Optional[torch.Tensor] = None, pending: Optional[tuple] = None):
        """pending = (feats, row_request, row_pos): context rows (at most 16 per request)
        materialised inside the round before it drafts; frontier is the frontier they
        complete."""
        B.draft_round(self.cfg, self.wstruct, self.kv, anchor_ids, frontier, n_masks, head_in,
                      self.workspace, hidden_out, layers_out, stream, tail_state, pending)

    def alloc_tail_state(self, Bn: int, n_masks: int) -> torch.Tensor:
        return torch.empty(B.tail_state_floats(self.cfg, Bn, n_masks), dtype=torch.float32,
                           device=self.device)

    def refine_tail(self, tail_state: torch.Tensor, cand_ids: torch.Tensor,
                    cand_scores: torch.Tensor, Bn: int, n_masks: int, token_out: torch.Tensor,
                    pick_out: Optional[torch.Tensor] = None,
                    table_out: Optional[torch.Tensor] = None, stream=None):
        B.refine_tail(self.cfg, self.wstruct, tail_state, cand_ids, cand_scores, Bn, n_masks,
                      token_out, self.workspace, pick_out, table_out, stream)

    # S10
    def head(self, hidden: torch.Tensor, token_out: torch.Tensor,
             max_logit_out: Optional[torch.Tensor] = None, stream=None):
        B.lm_head_argmax(self.cfg, self.wstruct, hidden, token_out, self.workspace,
                         max_logit_out, stream)

    def head_topk(self, hidden: torch.Tensor, k: int, token_out: torch.Tensor,
                  score_out: Optional[torch.Tensor] = None, stream=None):
        B.lm_head_topk(self.cfg, self.wstruct, hidden, k, token_out, self.workspace, score_out,
                       stream)

    def head_topk_fp8(self, hidden: torch.Tensor, n_cand: int, k: int, token_out: torch.Tensor,
                      score_out: Optional[torch.Tensor] = None, stream=None):
        """FP8 retrieval head; the FP8 head copy is built on first use."""
        if getattr(self, "head_fp8", None) is None:
            self.head_fp8_buf = torch.empty(B.head_fp8_bytes(self.cfg) + 1024, dtype=torch.uint8,
                                            device=self.device)
            self.head_fp8 = B.pack_head_fp8(self.cfg, self.wstruct, self.head_fp8_buf, stream)
        B.lm_head_topk_fp8(self.cfg, self.wstruct, self.head_fp8, hidden, n_cand, k, token_out,
                           self.workspace, score_out, stream)

    def alloc_outputs(self, Bn: int, n_masks: int):
        W = n_masks + 1
        H = self.geo.hidden
        head_in = torch.empty(Bn * n_masks, H, dtype=torch.float32, device=self.device)
        tokens = torch.empty(Bn * n_masks, dtype=torch.int32, device=self.device)
        maxl = torch.empty(Bn * n_masks, dtype=torch.float32, device=self.device)
        hidden = torch.empty(Bn * W, H, dtype=torch.float32, device=self.device)
        return head_in, tokens, maxl, hidden
