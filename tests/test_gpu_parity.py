"""GPU-vs-oracle parity through the C ABI on small seeded cases.

Tolerances (hidden states): max|gpu - ref| / max|ref| <= 2e-2 (bf16 storage, fp32
accumulation).  The fp32 configuration runs its products on tf32 tensor cores (10-bit
mantissa, relative product error below 2^-11), so the same bound applies; the measured
values are printed.  Argmax tokens are compared bit-exactly wherever the oracle's top-2
logit gap exceeds 1e-2.
"""
import numpy as np
import pytest
import torch

import bdsynth
import harness as Hn
from oracle import dspine_oracle as O

pytestmark = pytest.mark.gpu

TOL = 2e-2

SMALL_BF16 = bdsynth.Workload(
    name="small_bf16", hidden=512, n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128,
    ffn=1024, vocab=4000, n_target_layers=3, windows=(64, 0), code_width=128, msg_width=64,
    batch=3, n_masks=15, dtype="bf16", ctx_min=40, ctx_max=300, full_capacity=320)

SMALL_D64 = bdsynth.Workload(
    name="small_d64_bf16", hidden=256, n_layers=2, n_q_heads=4, n_kv_heads=1, head_dim=64,
    ffn=768, vocab=1000, n_target_layers=2, windows=(24, 24), code_width=64, msg_width=32,
    batch=2, n_masks=7, dtype="bf16", ctx_min=5, ctx_max=90, full_capacity=0)


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_drafter_gb300 import builder
    builder.build()


# ---------------------------------------------------------------- LM head (GEMM core)
@pytest.mark.parametrize("dtype,H,V,rows", [("bf16", 256, 1000, 1), ("bf16", 512, 4000, 15),
                                            ("bf16", 384, 1280, 120), ("f32", 256, 1024, 7),
                                            ("bf16", 5120, 151936, 15)])
def test_lm_head_argmax_matches_oracle(dtype, H, V, rows):
    from block_drafter_gb300 import binding as B
    geo = bdsynth.TINY.with_(hidden=H, vocab=V, dtype=dtype)
    dt = bdsynth.torch_dtype(dtype)
    g = torch.Generator().manual_seed(H + V + rows)
    E = (torch.randn(V, H, generator=g) * 0.02).to(dt)
    h = torch.randn(rows, H, generator=g)  # fp32 hidden rows (the head's input type)
    from block_drafter_gb300.session import config_of
    cfg = config_of(geo, 0)
    wd = {"w_feature": E, "context_norm": E, "final_norm": E, "embed_head": E, "layers": []}
    wd = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in wd.items()}
    ws_struct = B.make_weights(cfg, wd)
    ws = torch.empty(B.workspace_bytes(cfg, 8, 15, 16), dtype=torch.uint8, device="cuda")
    tok = torch.empty(rows, dtype=torch.int32, device="cuda")
    mx = torch.empty(rows, dtype=torch.float32, device="cuda")
    hd = h.cuda()
    for _ in range(2):  # twice: the stream-K counters must reset themselves
        B.lm_head_argmax(cfg, ws_struct, hd, tok, ws, mx)
        B.sync_status()
    logits = O.lm_head_logits(Hn.np32(h), Hn.np32(E))
    ref_tok = O.argmax_lowest(logits)
    gap = O.top2_gap(logits)
    got = tok.cpu().numpy()
    sel = gap > 1e-3
    assert (got[sel] == ref_tok[sel]).all(), (got, ref_tok, gap)
    np.testing.assert_allclose(mx.cpu().numpy(), logits.max(axis=1), rtol=2e-3, atol=2e-3)


# ---------------------------------------------------------------- materialisation
@pytest.mark.parametrize("geo", [SMALL_BF16, SMALL_D64, bdsynth.TINY])
def test_materialize_matches_oracle(geo):
    case = Hn.Case(geo, seed=1, max_ctx_rows=128)
    used = case.fill_rings()
    wnp = Hn.weights_to_np(case.w_host)
    for b in range(geo.batch):
        rings = None
        for (c0, f) in used[b]:
            n = f.shape[0]
            rings = O.materialize(geo, wnp, Hn.np32(f), np.arange(c0, c0 + n),
                                  case.frontiers[b], rings=rings)
        for l in range(geo.n_layers):
            cap = geo.capacity(l)
            lo, hi = O.ring_live_interval(case.frontiers[b], cap)
            slots = np.arange(lo, hi) % cap
            for key, ring in (("k", case.sess.k[l]), ("v", case.sess.v[l])):
                got = Hn.np32(ring[b])[:, slots]
                ref = rings[key][l][0][:, slots]
                err = Hn.rel_err(got, ref)
                assert err <= TOL, (geo.name, b, l, key, err)


# ---------------------------------------------------------------- round
# DFlash2 dynamic grouped convolution (group width 16 / 8), alone and with the bridge
SMALL_DFLASH2 = SMALL_BF16.with_(name="small_dflash2_bf16", code_width=0, msg_width=0,
                                 conv_group=16)
SMALL_DFLASH2_BRIDGE = SMALL_BF16.with_(name="small_dflash2_bridge_bf16", conv_group=8)
TINY_DFLASH2 = bdsynth.TINY.with_(name="tiny_dflash2_fp32", conv_group=16)


@pytest.mark.parametrize("geo,seed", [(bdsynth.TINY, 0), (bdsynth.TINY, 1), (SMALL_BF16, 0),
                                      (SMALL_BF16, 2), (SMALL_D64, 0), (SMALL_DFLASH2, 0),
                                      (SMALL_DFLASH2, 1), (SMALL_DFLASH2_BRIDGE, 2),
                                      (TINY_DFLASH2, 0),
                                      (SMALL_DFLASH2.with_(n_masks=6, batch=5), 3),
                                      # blocks of at most 32 rows: the one-launch bridge
                                      (SMALL_BF16.with_(batch=2), 4), (SMALL_BF16.with_(batch=1), 5),
                                      (SMALL_BF16.with_(batch=4, n_masks=7), 6),
                                      # 8 rows in a 16-row tile; a code of 192 (a partial
                                      # 128-row tile) with a 128-wide message
                                      (SMALL_BF16.with_(batch=1, n_masks=7), 7),
                                      (SMALL_BF16.with_(batch=2, code_width=192, msg_width=128), 8),
                                      # 96 rows: small-weight products take 64-token tiles (a
                                      # full one and a ragged one of 32)
                                      (SMALL_BF16.with_(batch=6), 9)])
def test_round_matches_oracle(geo, seed):
    case = Hn.Case(geo, seed=seed, max_ctx_rows=128)
    case.fill_rings()
    gpu = case.run_gpu()
    ref = case.run_oracle()
    rep = Hn.compare_round(case, gpu, ref, tol=TOL)
    print(geo.name, seed, rep)
    assert rep["ok"], rep


def test_round_block_causal_matches_oracle():
    geo = SMALL_BF16.with_(block_causal=True)
    case = Hn.Case(geo, seed=3, max_ctx_rows=128)
    case.fill_rings()
    rep = Hn.compare_round(case, case.run_gpu(), case.run_oracle(), tol=TOL)
    assert rep["ok"], rep


@pytest.mark.parametrize("batch", [3, 2])  # 2: the one-launch bridge
def test_round_gate_bias_matches_oracle(batch):
    case = Hn.Case(SMALL_BF16.with_(batch=batch), seed=4, gate_bias=True, max_ctx_rows=128)
    case.fill_rings()
    rep = Hn.compare_round(case, case.run_gpu(), case.run_oracle(), tol=TOL)
    assert rep["ok"], rep


@pytest.mark.parametrize("batch", [3, 2])  # 2: the one-launch bridge
def test_zero_write_is_bit_exact_plain_dflash(batch):
    """With every W_l = 0 the DSpine round must equal the same round with the bridge
    disabled (code_width = 0), bit for bit."""
    geo = SMALL_BF16.with_(batch=batch)
    w = bdsynth.make_weights(geo, 5, zero_write=True)
    a = Hn.Case(geo, seed=5, weights=w, max_ctx_rows=128)
    a.fill_rings()
    ga = a.run_gpu()
    geo0 = geo.with_(code_width=0, msg_width=0)
    b = Hn.Case(geo0, seed=5, weights=w, max_ctx_rows=128)
    b.fill_rings()
    gb = b.run_gpu()
    assert torch.equal(ga["layers"], gb["layers"])
    assert torch.equal(ga["tokens"], gb["tokens"])


def test_identity_convolution_is_bit_exact_plain_dflash():
    """DFlash2 with zero delta projections and identity base coefficients (current tap 1,
    previous tap 0) must equal the same round without the convolution, bit for bit: the
    branch outputs then reach the residual through the same single fp32 addition."""
    geo = SMALL_DFLASH2
    w = bdsynth.make_weights(geo, 9)
    for lw in w["layers"]:
        for br in ("a", "m"):
            lw["conv_delta_" + br].zero_()
            lw["conv_base_" + br].zero_()
            lw["conv_base_" + br][:, 0] = 1.0
    a = Hn.Case(geo, seed=9, weights=w, max_ctx_rows=128)
    a.fill_rings()
    ga = a.run_gpu()
    geo0 = geo.with_(conv_group=0)
    b = Hn.Case(geo0, seed=9, weights=w, max_ctx_rows=128)
    b.fill_rings()
    gb = b.run_gpu()
    assert torch.equal(ga["layers"], gb["layers"])
    assert torch.equal(ga["tokens"], gb["tokens"])


@pytest.mark.parametrize("batch", [3, 2])  # 2: the one-launch bridge
def test_round_is_deterministic_and_requests_independent(batch):
    geo = SMALL_BF16.with_(batch=batch)
    case = Hn.Case(geo, seed=6, max_ctx_rows=128)
    case.fill_rings()
    g1 = case.run_gpu()
    g2 = case.run_gpu()
    assert torch.equal(g1["layers"], g2["layers"])
    assert torch.equal(g1["tokens"], g2["tokens"])
    # changing the last request's anchor must leave the others unchanged
    last = batch - 1
    case.anchors = list(case.anchors)
    case.anchors[last] = (case.anchors[last] + 17) % geo.vocab
    if case.anchors[last] == case.mask_id:
        case.anchors[last] = (case.anchors[last] + 1) % geo.vocab
    g3 = case.run_gpu()
    W = geo.W
    assert torch.equal(g3["hidden"][:last * W], g1["hidden"][:last * W])
    assert not torch.equal(g3["hidden"][last * W:], g1["hidden"][last * W:])


# batch 2: the packed round takes the one-launch bridge, the raw one the five launches
@pytest.mark.parametrize("geo", [SMALL_BF16, SMALL_BF16.with_(batch=2), bdsynth.TINY])
def test_packed_and_raw_weights_give_identical_results(geo):
    """The packed image is a permutation of the weights, except that in a bf16 config it
    stores the attention-branch, MLP and head matrices as fp16 (their products then take
    fp16 activations instead of bf16 hi+lo pairs, the context rows' K/V products fp16 c_t
    instead of bf16 c_t).  In the fp32 config materialisation, round and head are
    bit-identical with and without it.  In bf16 the stored ring values agree to one bf16
    unit, both rounds meet the oracle and agree with each other to 2e-3, tokens equal where
    the oracle's gap exceeds 1e-2."""
    a = Hn.Case(geo, seed=8, max_ctx_rows=128, packed=True)
    b = Hn.Case(geo, seed=8, max_ctx_rows=128, packed=False, weights=a.w_host)
    a.fill_rings()
    b.fill_rings()
    for l in range(geo.n_layers):
        if geo.dtype == "f32":
            assert torch.equal(a.sess.k[l], b.sess.k[l]) and torch.equal(a.sess.v[l], b.sess.v[l])
        else:
            for x, y in ((a.sess.k[l], b.sess.k[l]), (a.sess.v[l], b.sess.v[l])):
                torch.testing.assert_close(x.float(), y.float(), rtol=2.0 ** -7, atol=2.0 ** -7)
    ga, gb = a.run_gpu(), b.run_gpu()
    if geo.dtype == "f32":
        for key in ("layers", "hidden", "tokens", "max_logit"):
            assert torch.equal(ga[key], gb[key]), key
        return
    for case, g in ((a, ga), (b, gb)):
        ref = case.run_oracle()  # each path against the oracle over its own rings
        rep = Hn.compare_round(case, g, ref, tol=TOL)
        print("packed" if case is a else "raw", rep)
        assert rep["ok"], rep
    # the two paths differ in operand precision and in the rounding of their context rings
    # (c_t fp16 vs bf16), so they agree to a few 1e-3, well inside the oracle tolerance
    assert Hn.rel_err(Hn.np32(ga["hidden"]), Hn.np32(gb["hidden"])) <= 5e-3
