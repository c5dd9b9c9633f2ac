"""GPU-vs-oracle parity of the top-k candidate head (bd_lm_head_topk) through the C ABI.

The oracle ranks exact fp64 logits.  The GPU ranks fp32 accumulations (bf16 weights,
hidden rows as bf16 hi+lo pairs; tf32 products in the fp32 configuration), so a rank is
compared id for id only where the oracle's neighbouring scores differ by more than EPS,
and the candidate set only where the k-th and (k+1)-th scores do.  Every returned score
is checked against the exact logit of the returned id, the order must be descending
with ties to the lower id, and the first candidate must be the argmax head's token.
"""
import numpy as np
import pytest
import torch

import bdsynth
import harness as Hn
from oracle import dspine_oracle as O

pytestmark = pytest.mark.gpu

EPS = {"bf16": 2e-3, "f32": 4e-3}   # absolute logit tolerance (|logit| <~ 8 here)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_drafter_gb300 import builder
    builder.build()


def _setup(dtype, H, V, rows, seed, tie_rows=None):
    from block_drafter_gb300 import binding as B
    from block_drafter_gb300.session import config_of
    geo = bdsynth.TINY.with_(hidden=H, vocab=V, dtype=dtype)
    dt = bdsynth.torch_dtype(dtype)
    g = torch.Generator().manual_seed(seed)
    E = torch.randn(V, H, generator=g) * 0.02
    h = torch.randn(rows, H, generator=g)
    if tie_rows is not None:  # identical rows inside one 128-row tile, made the best ones
        base = E[tie_rows[0]] * 0 + h[0] / h[0].norm() * 0.5
        for r in tie_rows:
            E[r] = base
    E = E.to(dt)
    cfg = config_of(geo, 0)
    wd = {"w_feature": E, "context_norm": E, "final_norm": E, "embed_head": E, "layers": []}
    wd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in wd.items()}
    ws_struct = B.make_weights(cfg, wd)
    ws = torch.empty(B.workspace_bytes(cfg, 8, 15, 16), dtype=torch.uint8, device="cuda")
    ws_struct.keep = wd  # the struct holds raw pointers: keep the device tensors alive with it
    return B, cfg, ws_struct, ws, E, h


def _run(B, cfg, ws_struct, ws, h, k):
    rows = h.shape[0]
    hd = h.cuda()
    tok = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    am = torch.empty(rows, dtype=torch.int32, device="cuda")
    for _ in range(2):  # twice: the tile counters must reset themselves
        B.lm_head_topk(cfg, ws_struct, hd, k, tok, ws, sc)
        B.sync_status()
    B.lm_head_argmax(cfg, ws_struct, hd, am, ws)
    B.sync_status()
    return tok.cpu().numpy(), sc.cpu().numpy(), am.cpu().numpy()


def _check(dtype, logits, k, tok, sc, am):
    eps = EPS[dtype]
    V = logits.shape[1]
    ids_r, sc_r = O.lm_head_topk(logits, min(k + 1, V))
    stats = {"ranks_compared": 0, "sets_compared": 0}
    for i in range(logits.shape[0]):
        assert len(set(tok[i])) == k and (tok[i] >= 0).all() and (tok[i] < V).all()
        # every returned score is the logit of the returned id
        np.testing.assert_allclose(sc[i], logits[i, tok[i]], atol=eps, rtol=0)
        # descending, ties to the lower id
        for j in range(1, k):
            assert sc[i, j] < sc[i, j - 1] or (sc[i, j] == sc[i, j - 1] and tok[i, j] > tok[i, j - 1])
        assert tok[i, 0] == am[i]
        for j in range(k):
            sep_prev = j == 0 or sc_r[i, j - 1] - sc_r[i, j] > 2 * eps
            sep_next = j + 1 >= sc_r.shape[1] or sc_r[i, j] - sc_r[i, j + 1] > 2 * eps
            if sep_prev and sep_next:
                assert tok[i, j] == ids_r[i, j], (i, j, tok[i], ids_r[i])
                stats["ranks_compared"] += 1
        if k < V and sc_r[i, k - 1] - sc_r[i, k] > 2 * eps:
            assert set(tok[i]) == set(ids_r[i, :k])
            stats["sets_compared"] += 1
    return stats


@pytest.mark.parametrize("dtype,H,V,rows,k", [
    ("bf16", 256, 1000, 1, 16), ("bf16", 512, 4000, 15, 16), ("bf16", 384, 1280, 120, 8),
    ("f32", 256, 1024, 7, 16), ("bf16", 256, 1000, 3, 1), ("bf16", 5120, 151936, 15, 16),
    ("bf16", 5120, 151936, 120, 16)])
def test_lm_head_topk_matches_oracle(dtype, H, V, rows, k):
    B, cfg, ws_struct, ws, E, h = _setup(dtype, H, V, rows, H + V + rows + k)
    tok, sc, am = _run(B, cfg, ws_struct, ws, h, k)
    logits = O.lm_head_logits(Hn.np32(h), Hn.np32(E))
    stats = _check(dtype, logits, k, tok, sc, am)
    print(dtype, H, V, rows, k, stats)
    assert stats["ranks_compared"] >= rows  # the comparison is not vacuous


def test_lm_head_topk_exact_ties_keep_lower_ids_first():
    tie = [300, 301, 302, 340]  # inside vocabulary tile 2 (rows 256..383)
    B, cfg, ws_struct, ws, E, h = _setup("bf16", 256, 1000, 2, 7, tie_rows=tie)
    tok, sc, am = _run(B, cfg, ws_struct, ws, h, 16)
    assert list(tok[0, :4]) == tie, tok[0]
    assert sc[0, 0] == sc[0, 1] == sc[0, 2] == sc[0, 3]
    logits = O.lm_head_logits(Hn.np32(h), Hn.np32(E))
    _check("bf16", logits, 16, tok, sc, am)
