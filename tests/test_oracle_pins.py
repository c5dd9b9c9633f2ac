"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself: a value the
pages print (tests/golden/page_numbers.json), a closed form worked by hand, a
textbook identity, an invariant, or a brute-force loop on tiny inputs.  Each is
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a mis-scaled softmax) fails at least one of them.
"""
import cmath
import copy
import json
import math
import os

import numpy as np
import pytest

from oracle import dspine_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
rng = np.random.default_rng(1234)


class Geo:
    """A small geometry object with the fields the oracle reads."""

    def __init__(self, **kw):
        d = dict(hidden=16, n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=24,
                 vocab=40, n_target_layers=2, windows=(0, 0), code_width=8, msg_width=4,
                 eps=1e-6, rope_theta=1e4, block_causal=False, full_capacity=64)
        d.update(kw)
        self.__dict__.update(d)

    def capacity(self, l):
        s = self.windows[l]
        return s if s > 0 else self.full_capacity


def add_conv(w, g, seed=1, gw=4, identity=False):
    """DFlash2 convolution weights for every layer of ``w`` (group width gw)."""
    r = np.random.default_rng(seed)
    H = g.hidden
    for lw in w["layers"]:
        for br in ("a", "m"):
            if identity:
                base = np.zeros((2, 2, H))
                base[:, 0] = 1.0
                lw["conv_delta_" + br] = np.zeros((4 * H // gw, H))
            else:
                base = r.normal(0, 0.3, (2, 2, H))
                base[:, 0] += 1.0
                lw["conv_delta_" + br] = r.normal(0, 0.3, (4 * H // gw, H))
            lw["conv_base_" + br] = base
    return w


def rand_weights(g, seed=0, zero_write=False, gate_bias=False):
    r = np.random.default_rng(seed)
    H, D = g.hidden, g.head_dim

    def m(*s):
        return r.normal(0, 0.3, s)

    def gain(n):
        return 1.0 + r.normal(0, 0.1, n)

    w = {"w_feature": m(H, g.n_target_layers * H), "context_norm": gain(H),
         "final_norm": gain(H), "embed_head": m(g.vocab, H), "layers": []}
    if g.code_width:
        cb = r.normal(0, 1, (g.vocab, g.code_width))
        w["codebook"] = cb / np.linalg.norm(cb, axis=1, keepdims=True)
        w["g_recv"], w["g_pred"], w["a_val"] = (m(g.msg_width, g.code_width) for _ in range(3))
        w["gate_bias"] = r.normal(0, 0.3, g.msg_width) if gate_bias else None
    for _ in range(g.n_layers):
        lw = {"in_norm": gain(H), "wq": m(g.n_q_heads * D, H), "wk": m(g.n_kv_heads * D, H),
              "wv": m(g.n_kv_heads * D, H), "q_norm": gain(D), "k_norm": gain(D),
              "wo": m(H, g.n_q_heads * D), "post_norm": gain(H), "w_gate": m(g.ffn, H),
              "w_up": m(g.ffn, H), "w_down": m(H, g.ffn)}
        if g.code_width:
            lw["r_read"] = m(g.code_width, H)
            lw["w_write"] = np.zeros((H, g.msg_width)) if zero_write else m(H, g.msg_width)
        w["layers"].append(lw)
    return w


def rand_rings(g, B, frontiers, seed=5):
    r = np.random.default_rng(seed)
    rings = {"k": [], "v": []}
    for l in range(g.n_layers):
        cap = g.capacity(l)
        rings["k"].append(r.normal(0, 1, (B, g.n_kv_heads, cap, g.head_dim)))
        rings["v"].append(r.normal(0, 1, (B, g.n_kv_heads, cap, g.head_dim)))
    return rings


# ----------------------------------------------------------------- plain_rmsnorm
def test_rmsnorm_constant_vector_closed_form():
    # x = c * 1: mean(x^2) = c^2, so out = w * c / sqrt(c^2 + eps)  (eps INSIDE the root)
    for c, eps in [(3.0, 1e-6), (0.5, 1.0), (-2.0, 0.25)]:
        x = np.full(6, c)
        w = np.array([1.0, 2.0, 0.5, -1.0, 3.0, 0.0])
        np.testing.assert_allclose(O.plain_rmsnorm(x, w, eps), w * c / math.sqrt(c * c + eps),
                                   rtol=1e-15)


def test_rmsnorm_hand_value():
    # x = [3, 4], eps = 0: mean square 12.5, so x / 3.5355339... = [0.84852814, 1.13137085]
    out = O.plain_rmsnorm(np.array([3.0, 4.0]), np.array([1.0, 0.5]), 0.0)
    np.testing.assert_allclose(out, [0.848528137423857, 0.565685424949238], rtol=1e-14)


def test_rmsnorm_unit_gain_has_rms_one():
    x = rng.normal(0, 5, (7, 33))
    y = O.plain_rmsnorm(x, np.ones(33), 1e-6)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-6)
    assert np.linalg.norm(y[0]) == pytest.approx(math.sqrt(33), rel=1e-6)


def test_head_rmsnorm_normalises_each_head_separately():
    x = np.concatenate([rng.normal(0, 1, 8), 100 * rng.normal(0, 1, 8)])[None, :]
    y = O.plain_head_rmsnorm(x, np.ones(8), 0.0, 8).reshape(2, 8)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), [1.0, 1.0], rtol=1e-13)


# ----------------------------------------------------------------- RoPE
def test_rope_hand_value_split_half():
    # D = 4, theta = 100: inv_freq = [1, 0.1]. pos 1 rotates pair (x0, x2) by 1 rad.
    x = np.array([[1.0, 0.0, 0.0, 0.0]])
    out = O.rope_1d(x, [1], 4, 100.0)
    np.testing.assert_allclose(out, [[0.5403023058681398, 0.0, 0.8414709848078965, 0.0]],
                               atol=1e-15)
    x = np.array([[0.0, 1.0, 0.0, 0.0]])     # pair (x1, x3) rotates by 0.1 rad
    out = O.rope_1d(x, [1], 4, 100.0)
    np.testing.assert_allclose(out, [[0.0, 0.9950041652780258, 0.0, 0.09983341664682815]],
                               atol=1e-15)


def test_rope_equals_complex_rotation():
    # (x_j + i x_{j+D/2}) * exp(i * pos * theta^(-2j/D)) for every head and j.
    D, theta = 16, 1e7
    x = rng.normal(0, 1, (3, 2 * D))
    pos = [0, 7, 4093]
    out = O.rope_1d(x, pos, D, theta)
    for t in range(3):
        for h in range(2):
            for j in range(D // 2):
                z = complex(x[t, h * D + j], x[t, h * D + j + D // 2])
                z *= cmath.exp(1j * pos[t] * theta ** (-2.0 * j / D))
                assert out[t, h * D + j] == pytest.approx(z.real, abs=1e-12)
                assert out[t, h * D + j + D // 2] == pytest.approx(z.imag, abs=1e-12)


def test_rope_position_zero_identity_and_norm():
    D = 128
    x = rng.normal(0, 1, (4, 3 * D))
    np.testing.assert_array_equal(O.rope_1d(x, [0, 0, 0, 0], D, 1e7), x)
    y = O.rope_1d(x, [1, 100, 5000, 123456], D, 1e7)
    np.testing.assert_allclose(np.linalg.norm(y.reshape(4, 3, D), axis=-1),
                               np.linalg.norm(x.reshape(4, 3, D), axis=-1), rtol=1e-12)


def test_rope_relative_position():
    D = 64
    q, k = rng.normal(0, 1, (1, D)), rng.normal(0, 1, (1, D))
    dots = [float((O.rope_1d(q, [m], D, 1e7) @ O.rope_1d(k, [n], D, 1e7).T)[0, 0])
            for m, n in [(10, 3), (1010, 1003), (40000, 39993)]]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ----------------------------------------------------------------- context
def test_context_fusion_hand_case():
    # W_feature = [I I] sums the two captured layers; then plain_rmsnorm.
    H = 2
    W = np.concatenate([np.eye(H), np.eye(H)], axis=1)
    s = np.array([[1.0, 2.0, 2.0, 2.0]])          # layer0 = [1,2], layer1 = [2,2] -> [3,4]
    c = O.context_fusion(s, W, np.ones(H), 0.0)
    np.testing.assert_allclose(c, [[0.848528137423857, 1.131370849898476]], rtol=1e-14)


def test_context_kv_position_independence_and_chunking():
    g = Geo(windows=(5, 0), full_capacity=32)
    w = rand_weights(g)
    n = 12
    feats = rng.normal(0, 1, (n, g.n_target_layers * g.hidden))
    pos = np.arange(3, 3 + n)
    full = O.materialize(g, w, feats, pos, 3 + n)
    # one position at a time, ascending, with the same final frontier
    one = None
    for t in range(n):
        one = O.materialize(g, w, feats[t:t + 1], pos[t:t + 1], 3 + n, rings=one)
    # two uneven chunks
    ch = O.materialize(g, w, feats[:7], pos[:7], 3 + n)
    ch = O.materialize(g, w, feats[7:], pos[7:], 3 + n, rings=ch)
    # (BLAS may sum a batched product in another order than a single row: 1e-12)
    for l in range(g.n_layers):
        for key in ("k", "v"):
            np.testing.assert_allclose(full[key][l], one[key][l], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(full[key][l], ch[key][l], rtol=1e-12, atol=1e-13)


def test_materialize_stores_only_final_window():
    g = Geo(windows=(4, 0), full_capacity=32)
    w = rand_weights(g)
    n = 11
    feats = rng.normal(0, 1, (n, g.n_target_layers * g.hidden))
    pos = np.arange(n)
    rings = O.materialize(g, w, feats, pos, n)
    # Local ring (S=4) holds exactly positions 7..10 at slots p mod 4.
    c = O.context_fusion(feats, w["w_feature"], w["context_norm"], g.eps)
    k, v = O.context_kv(c, pos, w["layers"][0]["wk"], w["layers"][0]["wv"],
                        w["layers"][0]["k_norm"], g.eps, g.head_dim, g.rope_theta)
    for p in range(7, 11):
        np.testing.assert_array_equal(rings["k"][0][0, :, p % 4, :],
                                      k[p].reshape(g.n_kv_heads, g.head_dim))
    # the full-context ring holds every position
    k1, _ = O.context_kv(c, pos, w["layers"][1]["wk"], w["layers"][1]["wv"],
                         w["layers"][1]["k_norm"], g.eps, g.head_dim, g.rope_theta)
    for p in range(11):
        np.testing.assert_array_equal(rings["k"][1][0, :, p, :],
                                      k1[p].reshape(g.n_kv_heads, g.head_dim))
    # storing only the tail chunk gives the same local ring
    tail = O.materialize(g, w, feats[7:], pos[7:], n)
    np.testing.assert_allclose(tail["k"][0], rings["k"][0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(tail["v"][0], rings["v"][0], rtol=1e-12, atol=1e-13)
    assert O.ring_live_interval(11, 4) == (7, 11)
    assert O.ring_live_interval(3, 4) == (0, 3)
    assert O.ring_slot(4097, 2048) == 1


# ----------------------------------------------------------------- attention
def _att_inputs(W, n_ctx, Hq, Hkv, D, seed):
    r = np.random.default_rng(seed)
    return (r.normal(0, 1, (W, Hq * D)), r.normal(0, 1, (W, Hkv * D)),
            r.normal(0, 1, (W, Hkv * D)), r.normal(0, 1, (n_ctx, Hkv, D)),
            r.normal(0, 1, (n_ctx, Hkv, D)))


@pytest.mark.parametrize("window,causal", [(0, False), (0, True), (3, False), (5, True),
                                           (5, False), (2, True)])
def test_attention_matches_bruteforce(window, causal):
    W, F, Hq, Hkv, D = 4, 9, 4, 2, 4
    q, kb, vb, kc, vc = _att_inputs(W, F, Hq, Hkv, D, window * 10 + causal)
    pos = np.arange(F)
    a = O.block_attention(q, kb, vb, kc, vc, pos, F, window, causal, Hq, Hkv, D)
    b = O.block_attention_bruteforce(q, kb, vb, kc, vc, pos, F, window, causal, Hq, Hkv, D)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_attention_softmax_scale_hand_value():
    # D=4, one context key and one block key; scores 2*1/sqrt(4) = 1 and 0.
    D = 4
    q = np.array([[2.0, 0, 0, 0]])
    kc = np.array([[[1.0, 0, 0, 0]]])             # [n_ctx=1, Hkv=1, D]
    vc = np.array([[[1.0, 0, 0, 0]]])
    kb = np.zeros((1, D))
    vb = np.array([[0.0, 1.0, 0, 0]])
    out = O.block_attention(q, kb, vb, kc, vc, [0], 1, 0, False, 1, 1, D)
    e = math.e
    np.testing.assert_allclose(out, [[e / (1 + e), 1 / (1 + e), 0, 0]], rtol=1e-14)


def _visible_sets(W, F, S, causal):
    """With q = 0 every visible key gets the same weight; one-hot values make the
    output row the indicator of the visible keys divided by their count."""
    n_ctx = F
    D = n_ctx + W
    q = np.zeros((W, D))
    kb = np.zeros((W, D))
    kc = np.zeros((n_ctx, 1, D))
    vc = np.eye(D)[:n_ctx][:, None, :]
    vb = np.eye(D)[n_ctx:]
    out = O.block_attention(q, kb, vb, kc, vc, np.arange(n_ctx), F, S, causal, 1, 1, D)
    return out > 1e-12


def test_window_endpoints_and_visible_counts():
    for case in GOLD["visible_context_full_left"]["cases"]:
        S, F, W = case["S"], case["F"], case["W"]
        vis = _visible_sets(W, F, S, False)
        for i in range(W):
            ctx = np.nonzero(vis[i, :F])[0]
            assert len(ctx) == max(0, S - 1 - i)         # page-printed count
            if S - 1 - i > 0:
                assert ctx.min() == F + i - (S - 1)      # distance S-1 visible
            if F + i - S >= 0:
                assert not vis[i, F + i - S]             # distance S hidden
            np.testing.assert_array_equal(vis[i, F:], [abs(j - i) < S for j in range(W)])


def test_block_causal_mask():
    W, F = 5, 6
    vis = _visible_sets(W, F, 0, True)
    for i in range(W):
        assert vis[i, :F].all()
        np.testing.assert_array_equal(vis[i, F:], [j <= i for j in range(W)])


def test_local_equals_full_when_window_covers_everything():
    W, F, Hq, Hkv, D = 4, 10, 4, 2, 8
    q, kb, vb, kc, vc = _att_inputs(W, F, Hq, Hkv, D, 7)
    a = O.block_attention(q, kb, vb, kc, vc, np.arange(F), F, F + W, False, Hq, Hkv, D)
    b = O.block_attention(q, kb, vb, kc, vc, np.arange(F), F, 0, False, Hq, Hkv, D)
    np.testing.assert_array_equal(a, b)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    W, F, Hq, Hkv, D = 3, 7, 4, 2, 8
    q, kb, vb, kc, vc = _att_inputs(W, F, Hq, Hkv, D, 9)
    a = O.block_attention(q, kb, vb, kc, vc, np.arange(F), F, 4, False, Hq, Hkv, D)
    rep = lambda t: np.repeat(t.reshape(t.shape[0], Hkv, D), Hq // Hkv, axis=1)
    b = O.block_attention(q, rep(kb).reshape(W, -1), rep(vb).reshape(W, -1), rep(kc), rep(vc),
                          np.arange(F), F, 4, False, Hq, Hq, D)
    np.testing.assert_allclose(a, b, rtol=1e-14)


# ----------------------------------------------------------------- layer
def test_silu_and_sigmoid_values():
    np.testing.assert_allclose(O.sigmoid(np.array([0.0, 1.0])), [0.5, 0.7310585786300049])
    np.testing.assert_allclose(O.silu(np.array([0.0, 1.0, -1.0])),
                               [0.0, 0.7310585786300049, -0.2689414213699951])


def _identity_layer_geo():
    return Geo(hidden=2, n_q_heads=1, n_kv_heads=1, head_dim=2, ffn=2, eps=0.0,
               code_width=0, msg_width=0, windows=(0, 0), n_layers=1)


def test_layer_swiglu_hand_value():
    # Attention output removed (W_o = 0); W_gate = I, W_up = 2I, W_down = I, unit gains.
    # y = x = [1, 1]: m = [1, 1]; x_next = y + SiLU(m) * 2m = 1 + 2 * 0.7310585786
    g = _identity_layer_geo()
    lw = {"in_norm": np.ones(2), "wq": np.eye(2), "wk": np.eye(2), "wv": np.eye(2),
          "q_norm": np.ones(2), "k_norm": np.ones(2), "wo": np.zeros((2, 2)),
          "post_norm": np.ones(2), "w_gate": np.eye(2), "w_up": 2 * np.eye(2),
          "w_down": np.eye(2)}
    x = np.array([[1.0, 1.0]])
    out, _, _ = O.dflash_layer(x, lw, g, np.array([5]), np.zeros((0, 1, 2)),
                               np.zeros((0, 1, 2)), np.zeros(0, np.int64), 5, 0)
    np.testing.assert_allclose(out, [[2.4621171572600098, 2.4621171572600098]], rtol=1e-14)


def test_layer_attention_residual_hand_value():
    # W_q = W_k = 0 -> q = k = 0 -> uniform weights over the visible keys.
    # Context values [2, 0] and [0, 4]; the block's own value W_v n with W_v = 0.
    # a = mean([2,0],[0,4],[0,0]) = [2/3, 4/3]; W_o = I; MLP removed (W_down = 0).
    # (eps > 0 so that the head norm of the all-zero q and k is 0, not 0/0.)
    g = _identity_layer_geo()
    g.eps = 1e-6
    lw = {"in_norm": np.ones(2), "wq": np.zeros((2, 2)), "wk": np.zeros((2, 2)),
          "wv": np.zeros((2, 2)), "q_norm": np.ones(2), "k_norm": np.ones(2),
          "wo": np.eye(2), "post_norm": np.ones(2), "w_gate": np.eye(2), "w_up": np.eye(2),
          "w_down": np.zeros((2, 2))}
    x = np.array([[1.0, -1.0]])
    kc = np.zeros((2, 1, 2))
    vc = np.array([[[2.0, 0.0]], [[0.0, 4.0]]])
    out, _, _ = O.dflash_layer(x, lw, g, np.array([2]), kc, vc, np.arange(2), 2, 0)
    np.testing.assert_allclose(out, [[1 + 2 / 3, -1 + 4 / 3]], rtol=1e-14)


# ----------------------------------------------------------------- bridge
def test_bridge_read_hand_value_and_norm():
    # x = [3, 4], R = I (Rc = 2), eps = 0: c = sqrt(2) * [0.6, 0.8]; r = sqrt(12.5)
    c, r = O.bridge_read(np.array([[3.0, 4.0]]), np.eye(2), 2, 0.0)
    np.testing.assert_allclose(c, [[math.sqrt(2) * 0.6, math.sqrt(2) * 0.8]], rtol=1e-14)
    np.testing.assert_allclose(r, [math.sqrt(12.5)], rtol=1e-15)
    x = rng.normal(0, 3, (5, 40))
    R = rng.normal(0, 1, (16, 40))
    c, _ = O.bridge_read(x, R, 16, 1e-6)
    np.testing.assert_allclose(np.linalg.norm(c, axis=-1), 4.0, rtol=1e-6)
    c2, _ = O.bridge_read(7.5 * x, R, 16, 1e-6)
    np.testing.assert_allclose(c2, c, rtol=1e-6)


def test_anchor_code_exact():
    row = rng.normal(0, 1, 64)
    row /= np.linalg.norm(row)
    np.testing.assert_array_equal(O.anchor_code(row, 64), 8.0 * row)
    assert np.linalg.norm(O.anchor_code(row, 1024)) == pytest.approx(32.0, rel=1e-12)


def _scalar_inject(G, Gp, A, Wl, x, c, b=None):
    one = lambda v: np.array([[v]])
    return O.inject(np.array(x, float)[:, None], np.array(c, float)[:, None],
                    np.abs(np.array(x, float)), one(G), one(Gp), one(A), one(Wl),
                    None if b is None else np.array([b]))[:, 0]


def test_inject_hand_values():
    # H = Rc = Mc = 1.  x = [2, 3] so r_1 = 3; predecessor code c_0 = 2, receiver c_1 = 1.
    # Gate 0 everywhere: g = 1/2, m = A c_0 / 2 = 1, write = r_1 * W m = 3.
    np.testing.assert_allclose(_scalar_inject(0, 0, 1, 1, [2, 3], [2, 1]), [2, 6])
    # Predecessor gate drives g -> 1: write = 3 * 2 = 6.
    np.testing.assert_allclose(_scalar_inject(0, 50, 1, 1, [2, 3], [2, 1]), [2, 9])
    # Receiver gate drives g -> 0: no write.
    np.testing.assert_allclose(_scalar_inject(-50, 0, 1, 1, [2, 3], [2, 1]), [2, 3])
    # The value comes from the predecessor's code (c_0), not the receiver's.
    np.testing.assert_allclose(_scalar_inject(0, 0, 1, 1, [2, 3], [0, 1]), [2, 3])
    # Bias enters the gate: b = +50 -> g = 1.
    np.testing.assert_allclose(_scalar_inject(0, 0, 1, 1, [2, 3], [2, 1], b=50), [2, 9])
    # Sign of the write follows W and A: W = -1 gives 3 - 3 = 0.
    np.testing.assert_allclose(_scalar_inject(0, 0, 1, -1, [2, 3], [2, 1]), [2, 0])
    # A negative receiver state scales by its RMS |x| (positive).
    np.testing.assert_allclose(_scalar_inject(0, 0, 1, 1, [2, -3], [2, 1]), [2, 0])


def test_inject_anchor_untouched_zero_write_identity_and_locality():
    W, H, Rc, Mc = 6, 10, 8, 4
    x = rng.normal(0, 1, (W, H))
    c = rng.normal(0, 1, (W, Rc))
    r = np.sqrt(np.mean(x * x, axis=-1))
    G, Gp, A = (rng.normal(0, 1, (Mc, Rc)) for _ in range(3))
    Wl = rng.normal(0, 1, (H, Mc))
    out = O.inject(x, c, r, G, Gp, A, Wl)
    np.testing.assert_array_equal(out[0], x[0])
    np.testing.assert_array_equal(O.inject(x, c, r, G, Gp, A, np.zeros((H, Mc))), x)
    for j in range(W):
        c2 = c.copy()
        c2[j] += 1.0
        diff = np.any(O.inject(x, c2, r, G, Gp, A, Wl) != out, axis=1)
        expect = np.zeros(W, bool)
        if j >= 1:
            expect[j] = True           # receiver gate term G c_j
        if j + 1 < W:
            expect[j + 1] = True       # predecessor terms G_p c_j and A c_j
        np.testing.assert_array_equal(diff, expect)


def test_inject_positive_homogeneity():
    W, H, Rc, Mc = 5, 12, 8, 4
    x = rng.normal(0, 1, (W, H))
    R = rng.normal(0, 1, (Rc, H))
    G, Gp, A = (rng.normal(0, 1, (Mc, Rc)) for _ in range(3))
    Wl = rng.normal(0, 1, (H, Mc))

    def step(xx):
        c, r = O.bridge_read(xx, R, Rc, 0.0)
        return O.inject(xx, c, r, G, Gp, A, Wl)

    np.testing.assert_allclose(step(3.0 * x), 3.0 * step(x), rtol=1e-12)


# ----------------------------------------------------------------- head
def test_argmax_bruteforce_and_ties():
    logits = rng.normal(0, 1, (6, 50))
    logits[2, 7] = logits[2, 31] = logits[2].max() + 1.0      # tie -> 7
    got = O.argmax_lowest(logits)
    for i in range(6):
        best, bi = -np.inf, -1
        for v in range(50):
            if logits[i, v] > best:
                best, bi = logits[i, v], v
        assert got[i] == bi
    assert got[2] == 7
    gap = O.top2_gap(logits)
    assert gap[2] == 0.0


def _topk_by_repeated_max(row, k):
    """Selection written out: k times, take the largest remaining score, scanning ids in
    ascending order so the lowest id wins a tie; remove it."""
    left = list(range(len(row)))
    ids = []
    for _ in range(k):
        best = None
        for v in left:
            if best is None or row[v] > row[best]:
                best = v
        ids.append(best)
        left.remove(best)
    return ids


def test_topk_bruteforce_with_ties():
    logits = rng.normal(0, 1, (5, 40))
    logits[1, [3, 20, 33]] = logits[1].max() + 0.5          # three-way tie at the top
    logits[3, [8, 9]] = np.sort(logits[3])[-5]               # a tie inside the top 16
    logits[4] = np.round(logits[4], 1)                        # many ties
    for k in (1, 5, 16, 40):
        ids, sc = O.lm_head_topk(logits, k)
        for i in range(5):
            ref = _topk_by_repeated_max(list(logits[i]), k)
            assert list(ids[i]) == ref, (k, i)
            assert list(sc[i]) == [logits[i, v] for v in ref]
    ids, _ = O.lm_head_topk(logits, 3)
    assert list(ids[1]) == [3, 20, 33]


def test_topk_first_is_argmax_and_scores_are_dot_products():
    h = rng.normal(0, 1, (4, 24))
    E = rng.normal(0, 1, (300, 24))
    E[77] = E[5]                                             # duplicate row: equal scores
    logits = O.lm_head_logits(h, E)
    ids, sc = O.lm_head_topk(logits, 16)
    assert (ids[:, 0] == O.argmax_lowest(logits)).all()
    for i in range(4):
        np.testing.assert_allclose(sc[i], [float(E[v] @ h[i]) for v in ids[i]], rtol=1e-12)
        assert (np.diff(sc[i]) <= 0).all()
        if 5 in ids[i] and 77 in ids[i]:
            assert list(ids[i]).index(5) < list(ids[i]).index(77)
    # every score outside the top 16 is <= the 16th
    for i in range(4):
        rest = np.delete(logits[i], ids[i])
        assert rest.max() <= sc[i, -1]


# ----------------------------------------------------------------- FP8 retrieval
def test_e4m3_rounding_matches_torch_float8_e4m3fn():
    """The oracle's e4m3 rounding against PyTorch's float8_e4m3fn conversion (a library
    routine) on a dense sweep with exact ties, subnormals and the largest finite value."""
    torch = pytest.importorskip("torch")
    x = rng.normal(0, 40, 100000).astype(np.float32)
    grid = np.array([0.0] + [m * 2.0 ** -9 for m in range(1, 8)] +
                    [(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)])
    grid = grid[grid <= 448]
    mids = (grid[1:] + grid[:-1]) / 2                    # exact ties between neighbours
    x = np.concatenate([x, grid, -grid, mids, -mids, np.float32([448.0, 460.0, -460.0])])
    x = x.astype(np.float32)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(O.e4m3_round(x), ref)


def test_e4m3_grid_closed_forms():
    """126 positive finite values, the largest 448 = 1.75 * 2^8, the smallest subnormal 2^-9,
    the smallest normal 2^-6; halves go to the even neighbour; large values clamp to 448."""
    pos = np.unique(O.e4m3_round(np.linspace(1e-4, 460, 2000000)))
    pos = pos[pos > 0]
    assert len(pos) == 126 and pos.max() == 448.0 and pos.min() == 2.0 ** -9
    assert 2.0 ** -6 in pos and (2.0 ** -6 - 2.0 ** -9) in pos
    np.testing.assert_array_equal(O.e4m3_round([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 1e6]),
                                  [1.0, 1.25, 0.0, 2.0 ** -8, 448.0])


def test_fp8_row_code_scales_and_codes():
    M = rng.normal(0, 0.02, (6, 64)).astype(np.float32)
    q, sc = O.fp8_row_code(M)
    np.testing.assert_array_equal(np.max(np.abs(q), axis=1), 448.0)  # the row's max maps to 448
    # scaling a row by a power of two scales its scale and leaves its codes
    q2, s2 = O.fp8_row_code(M * np.float32(8.0))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_allclose(s2, 8 * sc, rtol=0)
    # codes times scale approximate the row within half an e4m3 step (relative 2^-4)
    assert np.all(np.abs(q * sc[:, None] - M) <= np.abs(M) * 2.0 ** -4 + sc[:, None] * 2.0 ** -10)


def test_fp8_retrieval_with_every_candidate_is_the_exact_head():
    E = rng.normal(0, 0.02, (300, 32))
    h = rng.normal(0, 1, (3, 32))
    ids, sc, _ = O.lm_head_topk_fp8(h, E, n_cand=300, k=16, tile=128, per_tile=128)
    ref_ids, ref_sc = O.lm_head_topk(O.lm_head_logits(h, E), 16)
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_allclose(sc, ref_sc, rtol=1e-12)


def test_fp8_retrieval_finds_the_exact_top16_on_random_heads():
    E = rng.normal(0, 0.02, (4096, 256)).astype(np.float32)
    h = rng.normal(0, 1, (4, 256)).astype(np.float32)
    ids, sc, cand = O.lm_head_topk_fp8(h, E, n_cand=128, k=16)
    ref_ids, ref_sc = O.lm_head_topk(O.lm_head_logits(h, E), 16)
    for r in range(4):
        assert set(ref_ids[r]) <= set(cand[r])
    np.testing.assert_array_equal(ids, ref_ids)
    np.testing.assert_allclose(sc, ref_sc, rtol=1e-12)


def test_fp8_retrieval_keeps_16_per_tile():
    """A tile holding 20 of the best rows contributes only its 16 best."""
    H = 16
    E = rng.normal(0, 0.01, (512, H))
    h = np.ones((1, H))
    E[128:148] = 0.5 + 0.01 * np.arange(20)[:, None]   # tile 1 holds the 20 best rows
    _, _, cand = O.lm_head_topk_fp8(h, E, n_cand=32, k=4)
    in_tile = [c for c in cand[0] if 128 <= c < 148]
    assert sorted(in_tile) == list(range(132, 148))      # its 16 best, not all 20


def test_lm_head_chunking_matches_product():
    h = rng.normal(0, 1, (3, 16))
    E = rng.normal(0, 1, (100, 16))
    np.testing.assert_allclose(O.lm_head_logits(h, E, chunk=7), h @ E.T, rtol=1e-13)


# ----------------------------------------------------------------- full round
def _round(g, w, B=2, F=(9, 13), seed=3, mask_id=0, anchors=None, **kw):
    rings = rand_rings(g, B, F, seed)
    anchors = anchors or [5, 17][:B]
    return O.draft_round(g, w, rings, anchors, list(F)[:B], mask_id, 5, **kw), rings


def test_round_zero_write_equals_plain_dflash():
    g = Geo(windows=(6, 0))
    w = rand_weights(g, zero_write=True)
    a, _ = _round(g, w)
    g0 = Geo(windows=(6, 0), code_width=0, msg_width=0)
    b, _ = _round(g0, w)
    for key in ("x_layers", "h", "logits"):
        np.testing.assert_array_equal(a[key], b[key])


def test_round_requests_are_isolated_and_permutable():
    g = Geo(windows=(5, 0))
    w = rand_weights(g, gate_bias=True)
    rings = rand_rings(g, 2, (9, 13))
    ab = O.draft_round(g, w, rings, [5, 17], [9, 13], 0, 5)
    sw = {"k": [k[::-1].copy() for k in rings["k"]], "v": [v[::-1].copy() for v in rings["v"]]}
    ba = O.draft_round(g, w, sw, [17, 5], [13, 9], 0, 5)
    np.testing.assert_array_equal(ab["x_layers"][:, 0], ba["x_layers"][:, 1])
    np.testing.assert_array_equal(ab["tokens"][1], ba["tokens"][0])
    # changing request 1's ring leaves request 0 unchanged
    rings2 = {"k": [k.copy() for k in rings["k"]], "v": [v.copy() for v in rings["v"]]}
    rings2["k"][0][1] += 1.0
    c = O.draft_round(g, w, rings2, [5, 17], [9, 13], 0, 5)
    np.testing.assert_array_equal(c["h"][0], ab["h"][0])
    assert np.any(c["h"][1] != ab["h"][1])


# ----------------------------------------------------------------- DFlash2 convolution
def test_conv_with_zero_delta_is_a_causal_two_tap_filter_per_channel():
    """delta = 0 leaves a static depthwise filter: channel c of Conv_s(X) equals the
    causal FIR filter [base[s,0,c], base[s,1,c]] applied down the block rows (numpy's
    convolution, truncated to W rows).  Pins the tap order and the row direction."""
    W, H, gw = 6, 12, 4
    X = rng.normal(0, 1, (W, H))
    base = rng.normal(0, 1, (2, 2, H))
    delta = np.zeros((W, 2, 2, H // gw))
    for side in (0, 1):
        out = O.grouped_conv(X, base, delta, side)
        for c in range(H):
            ref = np.convolve(X[:, c], [base[side, 0, c], base[side, 1, c]])[:W]
            np.testing.assert_allclose(out[:, c], ref, rtol=1e-13, atol=1e-14)


def test_conv_delta_is_shared_by_the_channels_of_its_group():
    """A dynamic increment of group g changes exactly the gw channels g*gw .. g*gw+gw-1,
    all by the same multiple of X (current tap) and of the previous row (previous tap)."""
    W, H, gw = 5, 12, 4
    X = rng.normal(0, 1, (W, H))
    base = rng.normal(0, 1, (2, 2, H))
    delta = np.zeros((W, 2, 2, H // gw))
    ref = O.grouped_conv(X, base, delta, 1)
    d = delta.copy()
    d[3, 1, 0, 1] = 0.5          # row 3, side 1, current tap, group 1
    d[3, 1, 1, 1] = -2.0         # row 3, side 1, previous tap, group 1
    d[2, 0, 0, 2] = 7.0          # side 0 entries do not act on side 1
    out = O.grouped_conv(X, base, d, 1)
    diff = out - ref
    assert np.all(diff[[0, 1, 2, 4]] == 0)
    assert np.all(diff[3, :4] == 0) and np.all(diff[3, 8:] == 0)
    np.testing.assert_allclose(diff[3, 4:8], 0.5 * X[3, 4:8] - 2.0 * X[2, 4:8], rtol=1e-13)


def test_conv_row_zero_has_no_preceding_tap_and_rows_couple_only_to_the_next():
    W, H, gw = 7, 8, 4
    X = rng.normal(0, 1, (W, H))
    base = rng.normal(0, 1, (2, 2, H))
    delta = rng.normal(0, 1, (W, 2, 2, H // gw))
    ref = O.grouped_conv(X, base, delta, 0)
    np.testing.assert_allclose(ref[0], (base[0, 0] + np.repeat(delta[0, 0, 0], gw)) * X[0],
                               rtol=1e-13)
    Y = X.copy()
    Y[3] += 1.0
    changed = np.nonzero(np.any(O.grouped_conv(Y, base, delta, 0) != ref, axis=1))[0]
    assert list(changed) == [3, 4]


def test_conv_delta_projection_layout():
    """W_delta rows are ordered (side, tap, group): row s*2G + t*G + g feeds delta[i,s,t,g]."""
    W, H, G = 3, 8, 2
    X = rng.normal(0, 1, (W, H))
    Wd = np.zeros((4 * G, H))
    Wd[1 * 2 * G + 0 * G + 1] = 1.0      # side 1, tap 0, group 1 <- sum of X
    d = O.conv_delta(X, Wd)
    np.testing.assert_allclose(d[:, 1, 0, 1], X.sum(axis=1), rtol=1e-13)
    assert np.count_nonzero(d) == np.count_nonzero(X.sum(axis=1))


def test_dflash2_layer_with_identity_conv_is_the_dflash_layer():
    g = Geo(windows=(5, 0), code_width=0, msg_width=0)
    w = rand_weights(g)
    w2 = add_conv(copy.deepcopy(w), g, identity=True)
    a, _ = _round(g, w)
    b, _ = _round(g, w2)
    for key in ("x_layers", "h", "logits"):
        np.testing.assert_array_equal(a[key], b[key])


def test_dflash2_conv_acts_on_both_branches_and_keeps_requests_isolated():
    g = Geo(windows=(5, 0), code_width=0, msg_width=0)
    w = add_conv(rand_weights(g), g)
    base, rings = _round(g, w)
    # each of the four convolutions changes the result
    for br in ("a", "m"):
        for side in (0, 1):
            w2 = copy.deepcopy(w)
            for lw in w2["layers"]:
                lw["conv_base_" + br][side, 1] += 0.5
            res, _ = _round(g, w2)
            assert np.abs(res["h"] - base["h"]).max() > 1e-6, (br, side)
    # the convolution has no history across requests: request 1's anchor leaves request 0
    other = O.draft_round(g, w, rings, [5, 18], [9, 13], 0, 5)
    np.testing.assert_array_equal(other["h"][0], base["h"][0])


def _materialize_requests(g, w, feats, rows_of, frontiers):
    """Rings for len(frontiers) requests, request b holding positions rows_of[b]."""
    rings = {"k": [np.zeros((len(frontiers), g.n_kv_heads, g.capacity(l), g.head_dim))
                   for l in range(g.n_layers)],
             "v": [np.zeros((len(frontiers), g.n_kv_heads, g.capacity(l), g.head_dim))
                   for l in range(g.n_layers)]}
    for b, pos in enumerate(rows_of):
        if len(pos):
            O.materialize(g, w, feats[b][pos], pos, frontiers[b], rings=rings, request=b)
    return rings


def test_catch_up_round_equals_round_on_fully_materialised_context():
    """[Frontier]: a round that first catches up its pending rows sees the same context
    as a round whose context was materialised up to F beforehand (R-catch)."""
    g = Geo(windows=(5, 0), full_capacity=32)
    w = rand_weights(g, gate_bias=True)
    F, n_pend = (9, 13), (3, 1)
    feats = [rng.normal(0, 1, (f, g.n_target_layers * g.hidden)) for f in F]
    full = _materialize_requests(g, w, feats, [np.arange(f) for f in F], F)
    early = [f - n for f, n in zip(F, n_pend)]
    part = _materialize_requests(g, w, feats, [np.arange(e) for e in early], early)
    # pending rows in interleaved request order
    rows = [(1, 12), (0, 6), (0, 7), (0, 8)]
    pf = np.stack([feats[b][p] for b, p in rows])
    pend = (pf, [b for b, _ in rows], [p for _, p in rows])
    a = O.draft_round(g, w, full, [5, 17], list(F), 0, 5)
    b = O.draft_round(g, w, part, [5, 17], list(F), 0, 5, pending=pend)
    for key in ("x_layers", "h", "logits"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])
    # the caught-up rings hold the same live interval as the fully materialised ones
    for l in range(g.n_layers):
        cap = g.capacity(l)
        for r in range(2):
            lo, hi = O.ring_live_interval(F[r], cap)
            sl = np.arange(lo, hi) % cap
            for key in ("k", "v"):
                np.testing.assert_allclose(part[key][l][r][:, sl], full[key][l][r][:, sl],
                                           rtol=1e-12, atol=1e-13)


def test_catch_up_touches_only_its_requests():
    g = Geo(windows=(4, 0), full_capacity=32)
    w = rand_weights(g)
    F = (10, 11)
    rings = rand_rings(g, 2, F)
    feats = rng.normal(0, 1, (2, g.n_target_layers * g.hidden))
    base = O.draft_round(g, w, {k: [a.copy() for a in v] for k, v in rings.items()},
                         [5, 17], list(F), 0, 5)
    got = O.draft_round(g, w, rings, [5, 17], list(F), 0, 5,
                        pending=(feats, [1, 1], [9, 10]))
    np.testing.assert_array_equal(got["h"][0], base["h"][0])
    assert np.any(got["h"][1] != base["h"][1])


def test_round_block_rows_sit_at_frontier_plus_i_with_head_norm_before_rope():
    """[DFlash-notes] draft input table (anchor at position F, mask i at F + i) and per-layer
    equations (q = rope(head_rmsnorm(W_q n))), worked out by hand on a D = 2 geometry.

    One layer, one head, W_q = W_k = I, W_v = 0, W_o = I, no MLP, unit norms except a
    non-uniform query head-norm gain g = (2, 1/2), eps = 0.  Both embedding rows are
    e = (1, 0), so n = head_rmsnorm(e) = (sqrt 2, 0) and, head norm first, then RoPE
    (D = 2: angle = position), a row at position P has
        q = 2 sqrt2 (cos P, sin P),   k = sqrt2 (cos P, sin P).
    Every context key is (0, 1) (the rings hold rotated keys), so a query at P scores
    q.(0,1)/sqrt2 = 2 sin P on each of them; against a block row at P' it scores
    4 cos(P - P')/sqrt2.  Block-causal: row i sees the context and rows 0..i.  The block
    values are 0, so x_i' = e + sum_p w_p v_p over the context values v_p.
    RoPE after the head norm gives 0.5 sin P on the context instead; block positions
    0..W-1 or F-1+i shift P: each such reading changes the values below."""
    g = Geo(hidden=2, n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=2, ffn=2, vocab=4,
            windows=(0,), code_width=0, msg_width=0, eps=0.0, rope_theta=1e4,
            block_causal=True, full_capacity=8)
    I2, Z2 = np.eye(2), np.zeros((2, 2))
    w = {"w_feature": np.zeros((2, 4)), "context_norm": np.ones(2), "final_norm": np.ones(2),
         "embed_head": np.array([[1.0, 0.0], [1.0, 0.0], [0.0, 1.0], [0.0, -1.0]]),
         "layers": [{"in_norm": np.ones(2), "wq": I2, "wk": I2, "wv": Z2,
                     "q_norm": np.array([2.0, 0.5]), "k_norm": np.ones(2), "wo": I2,
                     "post_norm": np.ones(2), "w_gate": Z2, "w_up": Z2, "w_down": Z2}]}
    F, K = 3, 2
    vals = [(1.0, -2.0), (0.5, 3.0), (-4.0, 1.0)]                 # context values, positions 0..2
    rings = {"k": [np.zeros((1, 1, 8, 2))], "v": [np.zeros((1, 1, 8, 2))]}
    for p in range(F):
        rings["k"][0][0, 0, p] = (0.0, 1.0)
        rings["v"][0][0, 0, p] = vals[p]
    res = O.draft_round(g, w, rings, [1], [F], 0, K, with_head=False)
    r2 = math.sqrt(2.0)
    for i in range(K + 1):
        P = F + i
        ctx = [math.exp(2.0 * math.sin(P))] * F
        blk = [math.exp(4.0 * math.cos(P - (F + j)) / r2) for j in range(i + 1)]
        tot = sum(ctx) + sum(blk)
        want = [1.0 + sum(c * v[0] for c, v in zip(ctx, vals)) / tot,
                sum(c * v[1] for c, v in zip(ctx, vals)) / tot]
        np.testing.assert_allclose(res["x_layers"][0][0, i], want, rtol=1e-13, atol=1e-14)


def test_context_kv_head_norm_before_rope_hand_value():
    """[DFlash-notes] context K/V: k = rope(head_rmsnorm(W_k c), t).  With W_k = I,
    c = (1, 0), key gain (2, 1/2), eps = 0 and D = 2 (angle = t):
    head_rmsnorm(c) = (sqrt 2, 0), times the gain (2 sqrt2, 0), rotated by t:
    k = 2 sqrt2 (cos t, sin t).  Rotating first would give (2 sqrt2 cos t, sin t / sqrt2)."""
    for t in (0, 3, 7):
        k, v = O.context_kv(np.array([[1.0, 0.0]]), [t], np.eye(2), np.eye(2),
                            np.array([2.0, 0.5]), 0.0, 2, 1e4)
        np.testing.assert_allclose(k[0], 2 * math.sqrt(2.0) * np.array([math.cos(t), math.sin(t)]),
                                   rtol=1e-14, atol=1e-15)
        np.testing.assert_array_equal(v[0], [1.0, 0.0])


def test_round_is_invariant_to_shifting_every_position():
    """RoPE scores depend only on position differences and the window rule only on
    distances ([DFlash-notes] local-window attention rule), so materialising the same
    features at positions D..F+D-1 and drafting at frontier F+D must reproduce the
    round at frontier F: the block must move with the frontier.  (Local layers only: a
    full-context layer attends from position 0, so it has no shift symmetry.)"""
    g = Geo(windows=(5, 4), full_capacity=40)
    w = rand_weights(g, gate_bias=True)
    F, shift = 9, 13
    feats = rng.normal(0, 1, (F, g.n_target_layers * g.hidden))
    a_r = O.materialize(g, w, feats, np.arange(F), F)
    b_r = O.materialize(g, w, feats, np.arange(F) + shift, F + shift)
    a = O.draft_round(g, w, a_r, [5], [F], 0, 6)
    b = O.draft_round(g, w, b_r, [5], [F + shift], 0, 6)
    for key in ("x_layers", "h", "logits"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-9, atol=1e-11)
    np.testing.assert_array_equal(a["tokens"], b["tokens"])


def test_round_with_no_layer_updates_is_embedding_nearest_row():
    # W_o = 0, W_down = 0, W_write = 0: every layer is the identity, so the final state is
    # the embedding rows and each mask row's proposal is argmax_v E_v . rmsnorm(E_MASK).
    g = Geo(windows=(0, 0))
    w = rand_weights(g)
    for lw in w["layers"]:
        lw["wo"][:] = 0
        lw["w_down"][:] = 0
        lw["w_write"][:] = 0
    res, _ = _round(g, w, mask_id=11)
    E = w["embed_head"]
    n2 = sum(E[11][d] ** 2 for d in range(g.hidden)) / g.hidden
    hm = [w["final_norm"][d] * E[11][d] / math.sqrt(n2 + g.eps) for d in range(g.hidden)]
    best = max(range(g.vocab), key=lambda v: (sum(E[v][d] * hm[d] for d in range(g.hidden)), -v))
    assert (res["tokens"] == best).all()
    np.testing.assert_allclose(res["x_layers"][-1][0, 0], E[5], rtol=0, atol=0)


def test_round_injection_changes_only_successors_of_the_anchor_row():
    g = Geo(windows=(0, 0), n_layers=1)
    w = rand_weights(g)
    res, _ = _round(g, w, B=1, F=(9,))
    w0 = rand_weights(g, zero_write=True)
    ref, _ = _round(g, w0, B=1, F=(9,))
    # anchor row: identical with or without the write (its incoming write is zero)
    np.testing.assert_array_equal(res["x_layers"][0][0, 0], ref["x_layers"][0][0, 0])
    assert np.all(np.any(res["x_layers"][0][0, 1:] != ref["x_layers"][0][0, 1:], axis=-1))


# ----------------------------------------------------------------- page-printed numbers
def test_kv_bytes_per_position_and_windows():
    gd = GOLD["kv_bytes_per_position"]
    geo = gd["geometry"]
    per = O.kv_bytes_per_position(geo["n_layers"], geo["n_kv_heads"], geo["head_dim"],
                                  geo["k_bytes"], geo["v_bytes"])
    assert per == gd["value"]
    assert per * GOLD["kv_bytes_window_8192_mib"]["capacity"] == \
        GOLD["kv_bytes_window_8192_mib"]["value"] * 2 ** 20
    assert per * GOLD["kv_bytes_131072_gib"]["capacity"] == \
        GOLD["kv_bytes_131072_gib"]["value"] * 2 ** 30


def test_ring_image_40mib():
    gd = GOLD["ring_image_27b_dflash2_mib"]
    g = gd["geometry"]
    assert O.ring_image_bytes(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["capacity"],
                              g["k_bytes"], g["v_bytes"]) == gd["value"] * 2 ** 20


def test_injection_parameter_count_pins_shared_and_per_layer_maps():
    gd = GOLD["injection_params_qwen3_8b_millions"]
    g = gd["geometry"]
    n = O.injection_param_count(g["hidden"], g["n_layers"], g["code_width"], g["msg_width"])
    assert round(n / 1e6) == gd["value"]
    assert n == 33_030_144
    # Per-layer gate maps (instead of shared) would give about 41M; a second per-layer
    # read matrix about 54M: both miss the page's ~33M.
    assert round((n + 4 * 3 * g["msg_width"] * g["code_width"]) / 1e6) != gd["value"]
    assert round((n + g["n_layers"] * g["code_width"] * g["hidden"]) / 1e6) != gd["value"]


def test_codebook_and_table_sizes():
    gd = GOLD["codebook_mib"]
    assert gd["shape"][0] * gd["shape"][1] * gd["elem_bytes"] / 2 ** 20 == pytest.approx(gd["value"], abs=0.5)
    gd = GOLD["greedy_tail_tables_mib"]
    tot = sum(a * b for a, b in gd["shapes"]) * gd["elem_bytes"] / 2 ** 20
    assert tot == pytest.approx(gd["value"], abs=0.05)


def test_27b_block_geometry():
    gd = GOLD["block_27b"]
    import bdsynth
    w = bdsynth.DSPINE27B_B1
    assert w.W == gd["W"] and w.n_masks == gd["masks"]
    assert w.n_q_heads * w.head_dim == gd["q_proj_width"] and w.hidden == gd["hidden"]
    assert w.mask_token_id == GOLD["qwen3_mask_token_id"]["value"]


# ----------------------------------------------------------------- last-write refinement
def _cands(res, b, k):
    ids, _ = O.lm_head_topk(res["logits"][b], k)
    return ids


def test_refining_row_one_with_the_anchor_reproduces_the_round():
    g = Geo(windows=(6, 0))
    w = rand_weights(g, gate_bias=True)
    res, _ = _round(g, w)
    for b, a in enumerate([5, 17]):
        h1 = O.refine_state(g, w, res["tail"][b], 1, a)
        np.testing.assert_allclose(h1, res["h"][b, 1], rtol=1e-12, atol=1e-12)


def test_refining_with_the_predicted_code_reproduces_every_row():
    # Give token t the round's predicted (unit-scaled) code of row i - 1: refining row i
    # with t must then redo exactly the round's last injection into row i.
    g = Geo(windows=(6, 0))
    w = rand_weights(g)
    res, _ = _round(g, w, B=1, F=(9,))
    tail = res["tail"][0]
    for i in range(2, 6):
        w2 = dict(w)
        cb = np.array(w["codebook"], dtype=np.float64)
        cb[3] = tail["c"][i - 1] / math.sqrt(g.code_width)
        w2["codebook"] = cb
        np.testing.assert_allclose(O.refine_state(g, w2, tail, i, 3), res["h"][0, i],
                                   rtol=1e-12, atol=1e-12)


def test_zero_write_tables_do_not_depend_on_the_predecessor():
    g = Geo(windows=(6, 0))
    w = rand_weights(g, zero_write=True)
    res, _ = _round(g, w, B=1, F=(9,))
    cand = _cands(res, 0, 4)
    s1, tables, picks, tokens = O.refine_tail(g, w, res["tail"][0], 5, cand)
    for t in tables:
        assert np.allclose(t, t[0][None, :], rtol=1e-12, atol=1e-12)
    # every row then picks its best candidate, which is the round's own argmax
    assert (tokens == res["tokens"][0]).all() and (picks == 0).all()
    np.testing.assert_allclose(s1, res["logits"][0, 0, cand[0]], rtol=1e-12)


def test_walk_follows_the_previous_choice_and_tables_are_local():
    g = Geo(windows=(6, 0))
    w = rand_weights(g, seed=2)
    res, _ = _round(g, w, B=1, F=(9,))
    cand = _cands(res, 0, 4)
    s1, tables, picks, tokens = O.refine_tail(g, w, res["tail"][0], 5, cand)
    assert picks[0] == int(np.argmax(s1))
    for i in range(2, 6):
        row = tables[i - 2][picks[i - 2]]
        assert picks[i - 1] == int(np.argmax(row))
        assert tokens[i - 1] == cand[i - 1][picks[i - 1]]
    # table entry (i, p, j) by its definition: refine row i with candidate p of row i-1,
    # score candidate j of row i
    for i, p, j in ((2, 0, 1), (4, 3, 2), (5, 1, 0)):
        h = O.refine_state(g, w, res["tail"][0], i, int(cand[i - 2][p]))
        assert abs(tables[i - 2][p, j] - float(np.asarray(w["embed_head"])[cand[i - 1][j]] @ h)) < 1e-12
    # changing row 3's pre-injection state changes table 3 only
    t2 = {k: np.array(v, copy=True) for k, v in res["tail"][0].items()}
    t2["u"][3] *= 1.5
    _, tables2, _, _ = O.refine_tail(g, w, t2, 5, cand)
    changed = [not np.allclose(tables2[t], tables[t]) for t in range(4)]
    assert changed == [False, True, False, False]
