"""Failure detection without a GPU fault.

Every wait between CTAs in the kernels (split-tile reductions, attention splits) is bounded
by %globaltimer; a wait that gives up flags the device error word and ends, and the next
bd_sync_status reports BD_ERR_DEVICE_TIMEOUT.  bd_selftest_wait runs that same wait on a
flag nothing sets, with a short limit, so the whole path -- the wait giving up, the error
word, its report and reset, and a usable context afterwards -- is exercised without a
fault, a trap or a hang.
"""
import numpy as np
import pytest
import torch

import bdsynth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_drafter_gb300 import builder
    builder.build()


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    from block_drafter_gb300 import binding as B
    from block_drafter_gb300.session import config_of
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.sync_status()                          # nothing pending
    B.selftest_wait(flag, 2000)              # 2 ms on a flag nothing sets
    with pytest.raises(B.BdError) as err:
        B.sync_status()
    assert err.value.status == -4            # BD_ERR_DEVICE_TIMEOUT
    B.sync_status()                          # the report cleared the error word
    flag.fill_(1)
    B.selftest_wait(flag, 2000)              # satisfied at once
    B.sync_status()
    # the context is usable: a head call afterwards gives the right argmax
    geo = bdsynth.TINY.with_(hidden=256, vocab=1000, dtype="bf16")
    g = torch.Generator().manual_seed(3)
    E = (torch.randn(1000, 256, generator=g) * 0.02).to(torch.bfloat16).cuda()
    h = torch.randn(4, 256, generator=g).cuda()
    cfg = config_of(geo, 0)
    wd = {"w_feature": E, "context_norm": E, "final_norm": E, "embed_head": E, "layers": []}
    ws_struct = B.make_weights(cfg, wd)
    ws = torch.empty(B.workspace_bytes(cfg, 8, 15, 16), dtype=torch.uint8, device="cuda")
    tok = torch.empty(4, dtype=torch.int32, device="cuda")
    B.lm_head_argmax(cfg, ws_struct, h, tok, ws)
    B.sync_status()
    logits = (h.double() @ E.double().T).cpu().numpy()
    top2 = np.sort(logits, axis=1)[:, -2:]
    sel = top2[:, 1] - top2[:, 0] > 1e-3
    assert (tok.cpu().numpy()[sel] == logits.argmax(axis=1)[sel]).all()


# the block geometry of the small parity cases: batch 3 (48 rows) takes the five-launch
# bridge, batch 2 (32 rows) the one-launch bridge
_SMALL = bdsynth.Workload(
    name="small_bf16", hidden=512, n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128,
    ffn=1024, vocab=4000, n_target_layers=3, windows=(64, 0), code_width=128, msg_width=64,
    batch=3, n_masks=15, dtype="bf16", ctx_min=40, ctx_max=300, full_capacity=320)


@pytest.mark.parametrize("batch", [3, 2])
def test_out_of_range_anchor_is_reported_without_a_fault(batch):
    """An anchor id outside the vocabulary is a device-side index error: the kernels that
    read it clamp the index (no out-of-bounds access), flag the error word, and
    bd_sync_status reports BD_ERR_INVALID_ARG once; a valid round afterwards is clean and
    repeats the result of a round that never saw the bad id."""
    import harness as Hn
    from block_drafter_gb300 import binding as B
    geo = _SMALL.with_(batch=batch)
    case = Hn.Case(geo, seed=11, max_ctx_rows=128)
    case.fill_rings()
    good = case.run_gpu()
    anchors = list(case.anchors)
    case.anchors = list(anchors)
    case.anchors[batch - 1] = geo.vocab          # one past the last id
    with pytest.raises(B.BdError) as err:
        case.run_gpu()
    assert err.value.status == -1                # BD_ERR_INVALID_ARG
    B.sync_status()                              # reported once, then clear
    case.anchors = anchors
    again = case.run_gpu()
    assert torch.equal(again["layers"], good["layers"])
    assert torch.equal(again["tokens"], good["tokens"])


def test_packed_weight_beyond_fp16_range_is_reported():
    """The packed image stores the MLP matrices as fp16 in a bf16 config: a weight beyond
    +-65504 cannot be represented, so packing flags it and bd_sync_status returns
    BD_ERR_RANGE once (no fault); an in-range image afterwards reports nothing."""
    from block_drafter_gb300 import binding as B
    from block_drafter_gb300.session import DraftSession
    geo = _SMALL.with_(batch=1, n_layers=1, windows=(64,))
    w = bdsynth.make_weights(geo, seed=4, device="cuda")
    B.sync_status()
    w["layers"][0]["w_down"][7, 3] = 1.0e5        # bf16 holds it, fp16 does not
    DraftSession(geo, w, mask_id=0, b_max=1, max_ctx_rows=16)
    with pytest.raises(B.BdError) as err:
        B.sync_status()
    assert err.value.status == -6 and "65504" in str(err.value)
    B.sync_status()
    w["layers"][0]["w_down"][7, 3] = 0.5
    DraftSession(geo, w, mask_id=0, b_max=1, max_ctx_rows=16)
    B.sync_status()


def test_fp16_activation_overflow_is_reported():
    """With the packed image the SwiGLU product is stored as an fp16 operand of the down
    projection.  Scaling one layer's gate and up matrices by 1000 (still in fp16 range)
    pushes SiLU(g) * u far beyond 65504: the store would be +-inf, so the epilogue flags it
    and bd_sync_status returns BD_ERR_RANGE; the same session with its weights restored
    drafts cleanly again."""
    import harness as Hn
    from block_drafter_gb300 import binding as B
    geo = _SMALL.with_(batch=1)
    case = Hn.Case(geo, seed=12, max_ctx_rows=128)
    case.fill_rings()
    good = case.run_gpu()
    lw = case.w_dev["layers"][0]
    saved = (lw["w_gate"].clone(), lw["w_up"].clone())
    lw["w_gate"].mul_(1000.0)
    lw["w_up"].mul_(1000.0)
    B.pack_weights(case.sess.cfg, case.sess.wstruct, case.sess.packed)
    B.sync_status()                                # the scaled weights are in range
    with pytest.raises(B.BdError) as err:
        case.run_gpu()
    assert err.value.status == -6 and "activation" in str(err.value)
    B.sync_status()
    lw["w_gate"].copy_(saved[0])
    lw["w_up"].copy_(saved[1])
    B.pack_weights(case.sess.cfg, case.sess.wstruct, case.sess.packed)
    again = case.run_gpu()
    assert torch.equal(again["layers"], good["layers"])
    assert torch.equal(again["tokens"], good["tokens"])
