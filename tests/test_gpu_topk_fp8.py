"""GPU parity of the FP8 retrieval head (bd_pack_head_fp8 + bd_lm_head_topk_fp8) through
the C ABI.

Against the oracle's FP8 pipeline (R-fp8) on small heads: the returned ids rank by rank
where the oracle's neighbouring exact scores differ by more than EPS, and every returned
score is the exact logit of its id.  The GPU's approximate scores are fp32 sums of the
same e4m3 products the oracle adds in fp64, so the candidate sets can differ only at
near-ties at the n_cand boundary, far below the returned ranks.  At the 27B head size the
result is checked against the exact head: the FP8 retrieval of 128 candidates recovers
the exact top 16 of every row.  Degenerate rows (all scores equal) exercise the
threshold ties: the k lowest ids of the candidate set, in id order.
"""
import numpy as np
import pytest
import torch

import bdsynth
from oracle import dspine_oracle as O

pytestmark = pytest.mark.gpu

EPS = 2e-3   # absolute logit tolerance (|logit| <~ 8 here)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_drafter_gb300 import builder
    builder.build()


def _setup(H, V, rows, seed, gen_device="cpu"):
    from block_drafter_gb300 import binding as B
    from block_drafter_gb300.session import config_of
    geo = bdsynth.TINY.with_(hidden=H, vocab=V, dtype="bf16")
    g = torch.Generator(device=gen_device).manual_seed(seed)
    E = (torch.randn(V, H, generator=g, device=gen_device) * 0.02).to(torch.bfloat16)
    h = torch.randn(rows, H, generator=g, device=gen_device)
    cfg = config_of(geo, 0)
    Ed = E.cuda()
    wd = {"w_feature": Ed, "context_norm": Ed, "final_norm": Ed, "embed_head": Ed, "layers": []}
    ws_struct = B.make_weights(cfg, wd)
    ws = torch.empty(B.workspace_bytes(cfg, 8, 15, 16), dtype=torch.uint8, device="cuda")
    img = torch.empty(B.head_fp8_bytes(cfg) + 1024, dtype=torch.uint8, device="cuda")
    head8 = B.pack_head_fp8(cfg, ws_struct, img)
    # the weights struct holds raw pointers: keep the device tensors alive with it
    return B, cfg, ws_struct, ws, (img, head8, wd), E, h


def _run(B, cfg, ws_struct, ws, head8, h, n_cand, k):
    rows = h.shape[0]
    hd = h.cuda()
    tok = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(rows, k, dtype=torch.float32, device="cuda")
    for _ in range(2):  # twice: the tile counters must reset themselves
        B.lm_head_topk_fp8(cfg, ws_struct, head8[1], hd, n_cand, k, tok, ws, sc)
        B.sync_status()
    return tok.cpu().numpy(), sc.cpu().numpy()


def _check_ranks(ref_ids, ref_sc, logits, tok, sc, k):
    compared = 0
    for i in range(tok.shape[0]):
        assert len(set(tok[i])) == k
        np.testing.assert_allclose(sc[i], logits[i, tok[i]], atol=EPS, rtol=0)
        for j in range(1, k):
            assert sc[i, j] < sc[i, j - 1] or (sc[i, j] == sc[i, j - 1] and tok[i, j] > tok[i, j - 1])
        for j in range(k):
            sep_prev = j == 0 or ref_sc[i, j - 1] - ref_sc[i, j] > 2 * EPS
            sep_next = j + 1 >= ref_sc.shape[1] or ref_sc[i, j] - ref_sc[i, j + 1] > 2 * EPS
            if sep_prev and sep_next:
                assert tok[i, j] == ref_ids[i, j], (i, j, tok[i], ref_ids[i])
                compared += 1
    return compared


@pytest.mark.parametrize("H,V,rows,n_cand,k", [(512, 4000, 15, 128, 16), (256, 1000, 1, 128, 16),
                                               (256, 1000, 7, 16, 16), (384, 3000, 120, 256, 8),
                                               (512, 4096, 4, 128, 1)])
def test_fp8_retrieval_matches_oracle(H, V, rows, n_cand, k):
    B, cfg, ws_struct, ws, head8, E, h = _setup(H, V, rows, seed=H + V + rows)
    tok, sc = _run(B, cfg, ws_struct, ws, head8, h, n_cand, k)
    Enp, hnp = E.float().numpy(), h.numpy()
    ref_ids, ref_sc, _ = O.lm_head_topk_fp8(hnp, Enp, n_cand, min(k + 1, n_cand))
    logits = O.lm_head_logits(hnp, Enp)
    compared = _check_ranks(ref_ids, ref_sc, logits, tok, sc, k)
    assert compared >= rows * k // 2, compared


def test_fp8_retrieval_equal_scores_take_the_lowest_ids():
    """Zero hidden rows: every approximate and exact score is 0.  Each tile's 16 lowest ids
    enter, the n_cand lowest of those are the candidates, and the k lowest are returned."""
    B, cfg, ws_struct, ws, head8, E, h = _setup(256, 1000, 3, seed=5)
    h = torch.zeros_like(h)
    tok, sc = _run(B, cfg, ws_struct, ws, head8, h, 128, 16)
    assert (tok == np.arange(16)[None, :]).all() and (sc == 0).all()
    ref_ids, _, cand = O.lm_head_topk_fp8(h.numpy(), E.float().numpy(), 128, 16)
    np.testing.assert_array_equal(ref_ids, tok)
    assert sorted(cand[0]) == sorted([t * 128 + j for t in range(8) for j in range(16)])


@pytest.mark.slow
@pytest.mark.parametrize("rows", [15, 120])
def test_fp8_retrieval_recovers_exact_top16_at_27b_size(rows):
    B, cfg, ws_struct, ws, head8, E, h = _setup(5120, 151936, rows, seed=rows, gen_device="cuda")
    tok, sc = _run(B, cfg, ws_struct, ws, head8, h, 128, 16)
    logits = (h.double() @ E.double().T).cpu().numpy()
    ref_ids, ref_sc = O.lm_head_topk(logits, 17)
    compared = _check_ranks(ref_ids, ref_sc, logits, tok, sc, 16)
    assert compared >= rows * 12, compared
