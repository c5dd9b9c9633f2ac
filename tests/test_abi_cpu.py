"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports
every symbol include/blockdrafter.h declares, sizes workspaces, and rejects invalid
arguments before enqueuing anything."""
import ctypes as C
import os
import re

import pytest

import bdsynth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from block_drafter_gb300 import builder as bld
    bld.build()
    from block_drafter_gb300 import binding
    binding.lib()
    return binding


def header_symbols():
    src = open(os.path.join(ROOT, "include", "blockdrafter.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_three_entry_points():
    syms = header_symbols()
    for s in ("bd_ctx_kv_materialize", "bd_draft_round", "bd_lm_head_argmax"):
        assert s in syms


def test_library_exports_every_declared_symbol(B):
    L = B.lib()
    for s in header_symbols():
        assert hasattr(L, s), s
    assert set(B.EXPORTS) <= set(header_symbols())
    hdr = open(os.path.join(ROOT, "include", "blockdrafter.h")).read()
    assert B.abi_version() == int(re.search(r"#define BD_ABI_VERSION (\d+)", hdr).group(1))


def cfg_of(w, **kw):
    from block_drafter_gb300.session import config_of
    c = config_of(w, bdsynth.mask_token_id(w, 0))
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("name", list(bdsynth.WORKLOADS))
def test_workspace_bytes_positive_for_every_workload(B, name):
    w = bdsynth.WORKLOADS[name]
    c = cfg_of(w)
    n = B.lib().bd_workspace_bytes(C.byref(c), w.batch, w.n_masks, 2048)
    assert n > 0
    assert n < 8 << 30


def test_workspace_bytes_rejects_bad_sizes(B):
    c = cfg_of(bdsynth.TINY)
    L = B.lib()
    assert L.bd_workspace_bytes(C.byref(c), 0, 7, 16) == 0
    assert L.bd_workspace_bytes(C.byref(c), 9, 7, 16) == 0
    assert L.bd_workspace_bytes(C.byref(c), 1, 16, 16) == 0
    bad = cfg_of(bdsynth.TINY, head_dim=96)
    assert L.bd_workspace_bytes(C.byref(bad), 1, 7, 16) == 0
    bad = cfg_of(bdsynth.TINY, n_q_heads=3)
    assert L.bd_workspace_bytes(C.byref(bad), 1, 7, 16) == 0
    bad = cfg_of(bdsynth.TINY, mask_token_id=1024)
    assert L.bd_workspace_bytes(C.byref(bad), 1, 7, 16) == 0
    for gw in (-4, 6, 3, 512):   # the convolution group must be a multiple of 4 dividing H
        bad = cfg_of(bdsynth.TINY, conv_group=gw)
        assert L.bd_workspace_bytes(C.byref(bad), 1, 7, 16) == 0, gw
    ok = cfg_of(bdsynth.TINY, conv_group=16)
    assert L.bd_workspace_bytes(C.byref(ok), 1, 7, 16) >= L.bd_workspace_bytes(C.byref(c), 1, 7, 16)


def _fake_weights(B, c, n_layers):
    w = B.Weights()
    p = 0x10000
    for k in ("w_feature", "context_norm", "final_norm", "embed_head", "codebook", "g_recv",
              "g_pred", "a_val"):
        setattr(w, k, p)
    for l in range(n_layers):
        for k in B.LAYER_FIELDS:
            setattr(w.layer[l], k, p)
    return w


def test_entry_points_reject_invalid_arguments_on_host(B):
    L = B.lib()
    c = cfg_of(bdsynth.TINY)
    w = _fake_weights(B, c, c.n_layers)
    kv = B.KvCache()
    for l in range(c.n_layers):
        kv.k[l] = 0x10000
        kv.v[l] = 0x10000
    kv.b_max = 1
    ws = 0x100000
    # B out of range
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 9, 7, 0x10000,
                          None, None, None, None, ws, 1 << 30, None)
    assert st == -1 and b"B must be" in L.bd_last_error()
    # K out of range
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 16, 0x10000,
                          None, None, None, None, ws, 1 << 30, None)
    assert st == -1
    # misaligned weight
    w.layer[1].wq = 0x10008
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 7, 0x10000,
                          None, None, None, None, ws, 1 << 30, None)
    assert st == -1 and b"layer 1" in L.bd_last_error()
    w.layer[1].wq = 0x10000
    # more requests than ring rows
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 2, 7, 0x10000,
                          None, None, None, None, ws, 1 << 30, None)
    assert st == -1 and b"b_max" in L.bd_last_error()
    # misaligned workspace
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 7, 0x10000,
                          None, None, None, None, ws + 16, 1 << 30, None)
    assert st == -5
    # pending catch-up rows: more than 16 per request, missing arrays, misaligned features
    for pd in (B.Pending(0x10000, 0x10000, 0x10000, 17), B.Pending(None, 0x10000, 0x10000, 1),
               B.Pending(0x10000, None, 0x10000, 1), B.Pending(0x10008, 0x10000, 0x10000, 1),
               B.Pending(0x10000, 0x10000, 0x10000, -1)):
        st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 7, 0x10000,
                              None, None, None, C.byref(pd), ws, 1 << 30, None)
        assert st == -1 and b"pending" in L.bd_last_error()
    # head: rows out of range
    st = L.bd_lm_head_argmax(C.byref(c), C.byref(w), 0x10000, 121, 0x10000, None, ws, 1 << 30, None)
    assert st == -1
    # top-k head: k out of range, rows out of range, misaligned workspace
    for k in (0, 17):
        st = L.bd_lm_head_topk(C.byref(c), C.byref(w), 0x10000, 4, k, 0x10000, None, ws, 1 << 30, None)
        assert st == -1 and b"k must be" in L.bd_last_error()
    st = L.bd_lm_head_topk(C.byref(c), C.byref(w), 0x10000, 0, 16, 0x10000, None, ws, 1 << 30, None)
    assert st == -1
    st = L.bd_lm_head_topk(C.byref(c), C.byref(w), 0x10000, 4, 16, 0x10000, None, ws + 16, 1 << 30,
                           None)
    assert st == -5
    # FP8 retrieval: fp32 config unsupported; k, n_cand, rows, image alignment checked
    st = L.bd_lm_head_topk_fp8(C.byref(c), C.byref(w), 0x10000, 0x10000, 4, 128, 16, 0x10000, None,
                               ws, 1 << 30, None)
    assert st == -2 and b"bf16" in L.bd_last_error()
    assert L.bd_head_fp8_bytes(C.byref(c)) == 0
    cb = cfg_of(bdsynth.DSPINE27B_B1)
    wb = _fake_weights(B, cb, cb.n_layers)
    assert L.bd_head_fp8_bytes(C.byref(cb)) == 151936 * 5120 + 151936 * 4
    for (k, nc, rows) in ((0, 128, 4), (17, 128, 4), (16, 8, 4), (16, 257, 4), (16, 128, 0),
                          (16, 128, 121)):
        st = L.bd_lm_head_topk_fp8(C.byref(cb), C.byref(wb), 0x10000, 0x10000, rows, nc, k,
                                   0x10000, None, ws, 1 << 30, None)
        assert st == -1, (k, nc, rows)
    st = L.bd_lm_head_topk_fp8(C.byref(cb), C.byref(wb), 0x10010, 0x10000, 4, 128, 16, 0x10000,
                               None, ws, 1 << 30, None)
    assert st == -1 and b"1024-byte" in L.bd_last_error()
    st = L.bd_pack_head_fp8(C.byref(cb), C.byref(wb), 0x10000, 1024, None)
    assert st == -1 and b"smaller" in L.bd_last_error()
    # failure-path self-test: flag and limit checked on the host
    assert L.bd_selftest_wait(None, 1000, None) == -1
    assert L.bd_selftest_wait(0x10000, 0, None) == -1
    assert L.bd_selftest_wait(0x10002, 1000, None) == -1
    # refinement: K < 2, kc out of range, missing inputs
    st = L.bd_refine_tail(C.byref(c), C.byref(w), 0x10000, 0x10000, 0x10000, 1, 1, 16, 0x10000,
                          None, None, ws, 1 << 30, None)
    assert st == -1 and b"n_masks" in L.bd_last_error()
    for kc in (0, 17):
        st = L.bd_refine_tail(C.byref(c), C.byref(w), 0x10000, 0x10000, 0x10000, 1, 7, kc, 0x10000,
                              None, None, ws, 1 << 30, None)
        assert st == -1 and b"kc" in L.bd_last_error()
    st = L.bd_refine_tail(C.byref(c), C.byref(w), None, 0x10000, 0x10000, 1, 7, 16, 0x10000,
                          None, None, ws, 1 << 30, None)
    assert st == -1
    # materialise: no rows
    st = L.bd_ctx_kv_materialize(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 0x10000,
                                 0x10000, 0, ws, 1 << 30, None)
    assert st == -1
    # bridge on, bridge weights missing
    w.g_pred = None
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 7, 0x10000,
                          None, None, None, None, ws, 1 << 30, None)
    assert st == -1 and b"bridge" in L.bd_last_error()


def test_noalloc_head_checks_the_whole_config_on_host(B):
    """The no-allocation head applies the same configuration checks as the other entry
    points (the packed image's head offset depends on every layer's sizes), then its own
    size limits."""
    L = B.lib()
    c = cfg_of(bdsynth.TINY)
    w = _fake_weights(B, c, c.n_layers)
    for field, val, msg in (("n_layers", 99, b"n_layers"), ("head_dim", 96, b"head_dim"),
                            ("ffn", 3, b"ffn"), ("n_target_layers", 0, b"n_target_layers"),
                            ("mask_token_id", 5000, b"mask_token_id")):
        bad = cfg_of(bdsynth.TINY, **{field: val})
        st = L.bd_lm_head_argmax_noalloc(C.byref(bad), C.byref(w), 0x10000, 4, 0x10000, None, None)
        assert st == -1 and msg in L.bd_last_error(), field
    st = L.bd_lm_head_argmax_noalloc(C.byref(c), C.byref(w), 0x10000, 33, 0x10000, None, None)
    assert st == -1 and b"rows <= 32" in L.bd_last_error()


def test_timing_hook_checks_its_arguments_on_host(B):
    L = B.lib()
    ev = (C.c_void_p * 2)(0x1000, 0x2000)
    null = (C.c_void_p * 2)(0x1000, None)
    assert L.bd_set_timing_events(99, ev, ev, 2) == -1
    assert L.bd_set_timing_events(4, ev, ev, 0) == -1
    assert L.bd_set_timing_events(4, ev, ev, 33) == -1
    assert L.bd_set_timing_events(4, ev, null, 2) == -1
    assert L.bd_set_timing_events(4, None, ev, 2) == -1
    assert L.bd_set_timing_events(0, None, None, 0) == 0


def test_unsupported_geometry_is_an_error_not_a_fallback(B):
    L = B.lib()
    # bf16 with 8 query heads per KV head and W = 16 -> 128 query rows per KV head
    c = cfg_of(bdsynth.DSPINE27B_B1, n_kv_heads=4)
    w = _fake_weights(B, c, c.n_layers)
    kv = B.KvCache()
    for l in range(c.n_layers):
        kv.k[l] = kv.v[l] = 0x10000
    kv.b_max = 1
    st = L.bd_draft_round(C.byref(c), C.byref(w), C.byref(kv), 0x10000, 0x10000, 1, 15, 0x10000,
                          None, None, None, None, 0x100000, 1 << 34, None)
    assert st == -2


def test_ring_capacity_must_hold_the_window(B):
    c = cfg_of(bdsynth.DSPINE27B_B1)
    c.ring_capacity[2] = 100
    assert B.lib().bd_workspace_bytes(C.byref(c), 1, 15, 16) == 0


def test_packed_bytes_cover_every_matrix(B):
    """The packed image holds each projection matrix once (plus tile padding)."""
    for name in ("dspine_b16_27b_b1", "dflash_35b_a3b_b8", "tiny_fp32", "dflash2_27b_b1"):
        w = bdsynth.WORKLOADS[name]
        c = cfg_of(w)
        n = B.lib().bd_packed_bytes(C.byref(c))
        el = 2 if w.dtype == "bf16" else 4
        H, QD, KD = w.hidden, w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
        mats = H * w.n_target_layers * H + w.vocab * H + w.n_layers * (QD * H + 2 * KD * H + H * QD + 3 * H * w.ffn)
        if w.code_width:
            mats += 3 * w.msg_width * w.code_width + w.n_layers * (w.code_width * H + H * w.msg_width)
        if w.conv_group:
            mats += w.n_layers * 2 * (4 * H // w.conv_group) * H
        assert n >= mats * el
        assert n < mats * el * 1.05 + (16 << 20)
