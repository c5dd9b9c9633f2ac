"""The workspace-free LM-head entry point (for callers that cannot allocate device memory,
e.g. a serving engine whose pool owns every device byte, or a plugin host without an
allocation hook) must return what the workspace entry point returns.

Collected last on purpose (file name), so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from block_drafter_gb300 import builder
    builder.build()
    from block_drafter_gb300 import binding
    binding.lib()
    return binding


@pytest.mark.parametrize("dtype,H,V,rows", [("bf16", 5120, 151936, 15), ("bf16", 2048, 151936, 30),
                                            ("bf16", 512, 4000, 1), ("f32", 256, 1024, 7)])
def test_noalloc_head_matches_workspace_head_twice(B, dtype, H, V, rows):
    import bdsynth
    from block_drafter_gb300.session import config_of
    geo = bdsynth.TINY.with_(hidden=H, vocab=V, dtype=dtype)
    cfg = config_of(geo, 0)
    g = torch.Generator().manual_seed(7 * H + V + rows)
    E = (torch.randn(V, H, generator=g) * 0.02).to(bdsynth.torch_dtype(dtype)).cuda()
    wd = {"w_feature": E, "context_norm": E, "final_norm": E, "embed_head": E, "layers": []}
    ws_struct = B.make_weights(cfg, wd)
    ws = torch.empty(B.workspace_bytes(cfg, 8, 15, 16), dtype=torch.uint8, device="cuda")
    tok_ref = torch.empty(rows, dtype=torch.int32, device="cuda")
    max_ref = torch.empty(rows, dtype=torch.float32, device="cuda")
    for call in range(2):  # two calls in a row, new hidden rows each time
        h = torch.randn(rows, H, generator=g).cuda()
        B.lm_head_argmax(cfg, ws_struct, h, tok_ref, ws, max_ref)
        tok = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        mx = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
        B.lm_head_argmax_noalloc(cfg, ws_struct, h, tok, mx)
        B.sync_status()
        assert torch.equal(tok, tok_ref), (call, tok, tok_ref)
        torch.testing.assert_close(mx, max_ref, rtol=2e-3, atol=2e-3)


@pytest.mark.parametrize("big", [False, True])
def test_noalloc_head_with_packed_image_matches_workspace_head_twice(B, big):
    """A caller holding the packed weight image takes the fp16 head path (fp16 head rows,
    fp16 hidden rows); both entry points must still agree on the same packed weights."""
    import bdsynth
    from block_drafter_gb300.session import DraftSession
    if big:
        geo = bdsynth.DSPINE27B_B1.with_(n_layers=1, windows=(2048,))
        rows = 15
    else:
        geo = bdsynth.TINY.with_(dtype="bf16", hidden=512, vocab=4000, n_layers=1, windows=(0,))
        rows = 9
    wd = bdsynth.make_weights(geo, seed=3, device="cuda")
    sess = DraftSession(geo, wd, mask_id=0, b_max=1, max_ctx_rows=16)
    assert sess.wstruct.packed
    g = torch.Generator().manual_seed(11 + rows)
    tok_ref = torch.empty(rows, dtype=torch.int32, device="cuda")
    max_ref = torch.empty(rows, dtype=torch.float32, device="cuda")
    for call in range(2):
        h = torch.randn(rows, geo.hidden, generator=g).cuda()
        B.lm_head_argmax(sess.cfg, sess.wstruct, h, tok_ref, sess.workspace, max_ref)
        tok = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
        mx = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
        B.lm_head_argmax_noalloc(sess.cfg, sess.wstruct, h, tok, mx)
        B.sync_status()
        assert torch.equal(tok, tok_ref), (call, tok, tok_ref)
        torch.testing.assert_close(mx, max_ref, rtol=2e-3, atol=2e-3)


def test_noalloc_head_rejects_sizes_beyond_its_scratch(B):
    import bdsynth
    from block_drafter_gb300.session import config_of
    cfg = config_of(bdsynth.TINY.with_(hidden=256, vocab=1024, dtype="bf16"), 0)
    E = torch.zeros(1024, 256, dtype=torch.bfloat16, device="cuda")
    ws_struct = B.make_weights(cfg, {"w_feature": E, "context_norm": E, "final_norm": E,
                                     "embed_head": E, "layers": []})
    h = torch.zeros(33, 256, device="cuda")
    tok = torch.empty(33, dtype=torch.int32, device="cuda")
    with pytest.raises(B.BdError, match="rows <= 32"):
        B.lm_head_argmax_noalloc(cfg, ws_struct, h, tok)
    # a configuration the other entry points reject is rejected here too
    bad = config_of(bdsynth.TINY.with_(hidden=256, vocab=1024, dtype="bf16"), 0)
    bad.n_layers = 99
    with pytest.raises(B.BdError, match="n_layers"):
        B.lm_head_argmax_noalloc(bad, ws_struct, h[:4], tok[:4])
