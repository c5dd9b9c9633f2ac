"""Plain fp64 CPU oracle of one DFlash/DSpine block-drafter proposal round.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this module.
The CUDA library never calls it and shares no code with it.

Everything is NumPy float64, written step by step in the order the pages state the
method, with no blocking, fusion or reordering.  Inputs are bf16- or fp32-valued
arrays (any NumPy float dtype); they are widened to float64 on use and never rounded.

Sources (cited by page title and section throughout):
  [DFlash-notes]  NInfer maintainer page "dflash.md" (DFlash / DFlash2 backends):
                  the conditioning equations, the context K/V projection, the draft
                  input table, the local-window attention rule, the per-layer equations,
                  the proposal head and the ring storage paragraph.
  [Bridge]        "DSpine for Qwen3.8-27B: Causal Features Through Depth", section
                  "The bridge: read 1,024 features, write through rank 512".
  [Cache]         same page, section "An attention window is not a cache-size guarantee".
  [Transfer]      "DSpine 完全拆解", section "统一转移空间" (unified transfer space).
  [Gate]          "DSpine 完全拆解", section "相邻因果注入" / "门控与写回" (gate and write).
  [BlockCausal]   "DSpine 完全拆解", section "块因果注意力" (block-causal attention).
  [Backbone]      "DSpark, every bolt and rivet", section 5.1 "The parallel backbone".
  [Refine]        "DSpine for Qwen3.8-27B: Causal Features Through Depth", section "The
                  last write is refined using discrete candidates" (16 candidates per
                  proposal row; the fallback path scores with the BF16 vocabulary head).
  [Tail]          "DSpine 完全拆解", section "前驱条件解码与 transition cache"
                  (last-write refinement, the K x K transition table, greedy walk).
  [Conv]          "dflash.md", the DFlash2 paragraphs on the dynamic grouped convolution
                  around the attention and MLP branches and the per-layer DFlash2 equations.
  [Frontier]      "dflash.md", the paragraph on the processed-token frontier F: committed
                  target feature rows that the drafter has not yet converted are
                  materialised before the block is proposed, so the context reaches F.

Readings taken where the pages are schematic or garbled:
  R-gate   g = sigmoid(G c_t + G_p c_{t-1} + b), m = g * (A c_{t-1}); b absent means 0.
  R-eps    the bridge floor epsilon is the config's RMSNorm eps; r itself has no eps.
  R-scale  the code scale is sqrt(Rc); anchor code = sqrt(Rc) * codebook[anchor].
  R-read   one read matrix R_l per layer, applied to every row of the block.
  R-anchor row 0 of each request's block takes the anchor code in every layer and
           receives no write; all writes use the pre-injection codes of that layer.
  R-rms    the write scale r is the RMS of the pre-injection receiver state, no eps.
  R-last   every layer, including the last, is followed by its injection.
  R-rope   split-half rotation: (x_j, x_{j+D/2}) -> (x_j cos - x_{j+D/2} sin,
           x_{j+D/2} cos + x_j sin), angle = pos * theta^(-2j/D).
  R-gqa    query head h reads KV head h // (Hq / Hkv).
  R-mask   a key at position p is visible from a query at position P iff |P - p| < S
           for a local layer (every populated position for a full layer); the
           block-causal flag additionally hides block keys j > i.
  R-tie    argmax ties go to the lowest token id; only the K mask rows are scored.
  R-catch  a round given pending rows first materialises them exactly as a separate
           materialisation would (each request's rows into its own rings, stored only
           inside the final live window of the frontier they complete), then drafts.
  R-conv   DFlash2 grouped convolution (layers with conv weights): per branch,
           delta = W_delta X reshaped [W, 2 sides, 2 taps, H/gw groups] from the branch's
           normalised input X; Conv_s(X)[i, c] = (base[s,0,c] + delta[i,s,0,c//gw]) X[i, c]
           + [i >= 1] (base[s,1,c] + delta[i,s,1,c//gw]) X[i-1, c] with i the block row
           (row 0, the anchor, has no preceding tap; no history across requests or
           rounds).  Side 0 prepares the branch input, side 1 finishes the branch output
           with the same delta; base is stored [2 sides][2 taps][H].
  R-fp8    FP8 retrieval ([Refine]: row-scaled FP8 scores over the whole vocabulary, 128
           candidates, BF16 rescoring, 16 kept).  Row scale s = max|row| / 448 and codes
           q = e4m3(row / s) (round to nearest even, largest finite 448), both computed in
           fp32 like the kernel; the hidden row is coded the same way.  Approximate score of
           vocabulary row v = s_v * (q_v . q_h) (the hidden row's scale is common to a row
           and left out).  Candidates: each 128-row vocabulary tile keeps its 16 best
           approximate scores, and the row keeps the n_cand best of those (a tile holding
           more than 16 of the n_cand best loses its excess); ties go to the lower id.  The
           candidates are rescored with the exact head and the k best kept (R-topk order).
  R-topk   a row's k candidates are its k largest exact logits over the whole
           vocabulary, by descending score; equal scores keep the lower token id first.
  R-tail   last-write refinement of block row i with predecessor token s: the last
           layer's injection into row i is redone from its pre-injection state u_i, its
           receiver code c_i and RMS r_i, with the predecessor code replaced by
           sqrt(Rc) * codebook[s]; the result goes through the final norm and the tied
           head.  Row 1's predecessor is the anchor, whose code the round already used,
           so row 1 keeps the round's scores; rows i >= 2 get the table
           T_i[p, j] = score of candidate j of row i after refinement with candidate p of
           row i - 1.  The greedy walk takes, row by row, the lowest-rank argmax of the
           table row of the previous choice.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------- norms
def plain_rmsnorm(x, w, eps: float) -> np.ndarray:
    """w * x / sqrt(mean(x^2) + eps) over the last axis.  [DFlash-notes], conditioning."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return _f64(w) * x / np.sqrt(ms + eps)


def plain_head_rmsnorm(x, w, eps: float, head_dim: int) -> np.ndarray:
    """plain_rmsnorm applied to each head_dim-wide head of the last axis.
    [DFlash-notes], per-layer equations (query/key normalisation)."""
    x = _f64(x)
    shp = x.shape
    xh = x.reshape(shp[:-1] + (shp[-1] // head_dim, head_dim))
    return plain_rmsnorm(xh, w, eps).reshape(shp)


# --------------------------------------------------------------------------- rope
def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2j/D) for j < D/2 (R-rope)."""
    j = np.arange(head_dim // 2, dtype=F64)
    return theta ** (-2.0 * j / head_dim)


def rope_1d(x, positions, head_dim: int, theta: float) -> np.ndarray:
    """Full-head split-half rotary embedding at absolute scalar positions.

    x: [T, n_heads * head_dim]; positions: [T].  [DFlash-notes] (scalar RoPE,
    full-head split-half) with the reading R-rope."""
    x = _f64(x)
    T = x.shape[0]
    half = head_dim // 2
    ang = _f64(positions)[:, None] * rope_inv_freq(head_dim, theta)[None, :]   # [T, half]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    xh = x.reshape(T, -1, head_dim)
    x1, x2 = xh[..., :half], xh[..., half:]
    out = np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)
    return out.reshape(x.shape)


# --------------------------------------------------------------------------- context
def context_fusion(s, w_feature, context_norm, eps: float) -> np.ndarray:
    """c_t = plain_rmsnorm(W_feature s_t, context_norm); W_feature is bias-free.
    s: [T, n_tgt * H] (the captured residuals concatenated in recorded order).
    [DFlash-notes], conditioning; [Backbone] context feature extraction."""
    return plain_rmsnorm(_f64(s) @ _f64(w_feature).T, context_norm, eps)


def context_kv(c, positions, wk, wv, k_norm, eps: float, head_dim: int, theta: float):
    """One draft layer's context K/V from the common c_t:
    k = rope_1d(plain_head_rmsnorm(W_k c, key_norm), t);  v = W_v c.
    Raw k is normalised without any intermediate rounding.  [DFlash-notes], context K/V."""
    c = _f64(c)
    k = rope_1d(plain_head_rmsnorm(c @ _f64(wk).T, k_norm, eps, head_dim), positions,
                head_dim, theta)
    v = c @ _f64(wv).T
    return k, v


def ring_slot(position: int, capacity: int) -> int:
    """Absolute position p lives in slot p mod S of a ring of capacity S.
    [DFlash-notes], ring storage."""
    return position % capacity


def ring_live_interval(frontier: int, capacity: int):
    """[max(0, F - S), F): the positions a ring of capacity S holds at frontier F.
    [DFlash-notes], ring storage."""
    return max(0, frontier - capacity), frontier


def materialize(geo, weights, feats, positions, frontier_after: int, rings=None,
                request: int = 0) -> Dict[str, list]:
    """Store one request's context K/V for the given positions into per-layer rings.

    feats: [n, n_tgt*H] captured residual rows for ``positions`` (ascending).  Only
    positions in each ring's final live interval [F - S, F) (F = ``frontier_after``)
    are stored; the frontier still covers the whole chunk.  [DFlash-notes], context
    prefill and ring storage.

    rings: {"k": [L arrays [B, Hkv, cap, D]], "v": [...]} (created if None, B = 1).
    """
    L, Hkv, D = geo.n_layers, geo.n_kv_heads, geo.head_dim
    if rings is None:
        rings = {"k": [np.zeros((1, Hkv, geo.capacity(l), D)) for l in range(L)],
                 "v": [np.zeros((1, Hkv, geo.capacity(l), D)) for l in range(L)]}
    positions = np.asarray(positions, dtype=np.int64)
    c = context_fusion(feats, weights["w_feature"], weights["context_norm"], geo.eps)
    for l in range(L):
        lw = weights["layers"][l]
        k, v = context_kv(c, positions, lw["wk"], lw["wv"], lw["k_norm"], geo.eps, D,
                          geo.rope_theta)
        cap = geo.capacity(l)
        lo, hi = ring_live_interval(frontier_after, cap)
        for t, p in enumerate(positions):
            if lo <= p < hi:
                s = ring_slot(int(p), cap)
                rings["k"][l][request, :, s, :] = k[t].reshape(Hkv, D)
                rings["v"][l][request, :, s, :] = v[t].reshape(Hkv, D)
    return rings


# --------------------------------------------------------------------------- attention
def key_visible(p_query: int, p_key: int, window: int) -> bool:
    """|p_key - p_query| < S for a local layer (S = window > 0); always for a full
    layer (window == 0).  [DFlash-notes], local-window attention rule."""
    return window <= 0 or abs(p_key - p_query) < window


def block_attention(q, k_blk, v_blk, k_ctx, v_ctx, ctx_positions, frontier: int,
                    window: int, block_causal: bool, n_q_heads: int, n_kv_heads: int,
                    head_dim: int) -> np.ndarray:
    """softmax(q K^T / sqrt(D) + mask) V over concat(context, block) for one request.

    q: [W, Hq*D] (block rows at positions F..F+W-1); k_blk, v_blk: [W, Hkv*D];
    k_ctx, v_ctx: [n_ctx, Hkv, D] at ``ctx_positions`` (all < F).  Returns [W, Hq*D].
    [DFlash-notes] per-layer equations and window rule; [BlockCausal] for the flag.
    Explicit max-subtracted softmax."""
    W = q.shape[0]
    D = head_dim
    G = n_q_heads // n_kv_heads
    qh = _f64(q).reshape(W, n_q_heads, D)
    kb = _f64(k_blk).reshape(W, n_kv_heads, D)
    vb = _f64(v_blk).reshape(W, n_kv_heads, D)
    kc = _f64(k_ctx)
    vc = _f64(v_ctx)
    ctx_positions = np.asarray(ctx_positions, dtype=np.int64)
    n_ctx = kc.shape[0]
    out = np.zeros((W, n_q_heads, D))
    scale = 1.0 / math.sqrt(D)
    for i in range(W):
        pq = frontier + i
        vis_ctx = np.array([key_visible(pq, int(p), window) for p in ctx_positions], bool)
        vis_blk = np.array([key_visible(pq, frontier + j, window) and
                            (not block_causal or j <= i) for j in range(W)], bool)
        for h in range(n_q_heads):
            g = h // G
            keys = np.concatenate([kc[:, g, :], kb[:, g, :]], axis=0)      # [n_ctx+W, D]
            vals = np.concatenate([vc[:, g, :], vb[:, g, :]], axis=0)
            vis = np.concatenate([vis_ctx, vis_blk])
            s = keys @ qh[i, h] * scale
            s = np.where(vis, s, -np.inf)
            s = s - np.max(s)
            p = np.exp(s)
            p = p / np.sum(p)
            out[i, h] = p @ vals
    return out.reshape(W, n_q_heads * D)


def block_attention_bruteforce(q, k_blk, v_blk, k_ctx, v_ctx, ctx_positions, frontier,
                               window, block_causal, n_q_heads, n_kv_heads, head_dim):
    """The same attention as a per-(query, key) double loop with scalar arithmetic.
    Used only to check ``block_attention`` on tiny inputs."""
    W = q.shape[0]
    D = head_dim
    G = n_q_heads // n_kv_heads
    q = _f64(q).reshape(W, n_q_heads, D)
    kb = _f64(k_blk).reshape(W, n_kv_heads, D)
    vb = _f64(v_blk).reshape(W, n_kv_heads, D)
    kc, vc = _f64(k_ctx), _f64(v_ctx)
    keys_pos = [int(p) for p in ctx_positions] + [frontier + j for j in range(W)]
    out = np.zeros((W, n_q_heads, D))
    for i in range(W):
        for h in range(n_q_heads):
            g = h // G
            scores, vals = [], []
            for kk, pk in enumerate(keys_pos):
                is_blk = kk >= len(ctx_positions)
                j = kk - len(ctx_positions)
                if window > 0 and abs(pk - (frontier + i)) >= window:
                    continue
                if is_blk and block_causal and j > i:
                    continue
                kvec = kb[j, g] if is_blk else kc[kk, g]
                vvec = vb[j, g] if is_blk else vc[kk, g]
                dot = 0.0
                for d in range(D):
                    dot += q[i, h, d] * kvec[d]
                scores.append(dot / math.sqrt(D))
                vals.append(vvec)
            mx = max(scores)
            ws = [math.exp(s - mx) for s in scores]
            tot = sum(ws)
            acc = np.zeros(D)
            for wgt, vv in zip(ws, vals):
                acc += (wgt / tot) * vv
            out[i, h] = acc
    return out.reshape(W, n_q_heads * D)


# --------------------------------------------------------------------------- layer
def silu(x):
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def conv_delta(X, w_delta) -> np.ndarray:
    """delta = W_delta X per block row, as [W, 2 sides, 2 taps, groups].  [Conv], R-conv."""
    X = _f64(X)
    return (X @ _f64(w_delta).T).reshape(X.shape[0], 2, 2, -1)


def grouped_conv(X, base, delta, side: int) -> np.ndarray:
    """Conv_side(X) over the block rows of one request ([Conv], R-conv): channel c of
    group g = c // gw takes (base[side,0,c] + delta[i,side,0,g]) X[i,c], plus, for i >= 1,
    (base[side,1,c] + delta[i,side,1,g]) X[i-1,c]."""
    X = _f64(X)
    W, H = X.shape
    b = _f64(base).reshape(2, 2, H)
    gw = H // delta.shape[-1]
    cur = b[side, 0] + np.repeat(delta[:, side, 0, :], gw, axis=1)     # [W, H]
    prev = b[side, 1] + np.repeat(delta[:, side, 1, :], gw, axis=1)
    out = cur * X
    out[1:] += prev[1:] * X[:-1]
    return out


def dflash_layer(x, lw, geo, positions, k_ctx, v_ctx, ctx_positions, frontier: int,
                 layer: int):
    """One draft layer for one request's block (no injection).  [DFlash-notes]:
        n = plain_rmsnorm(x, input_norm)
        q = rope(head_rmsnorm(W_q n)), k = rope(head_rmsnorm(W_k n)), v = W_v n
        a = attention(q, [K_ctx; k], [V_ctx; v]) ; y = x + W_o a
        m = plain_rmsnorm(y, post_attention_norm)
        x_next = y + W_down(SiLU(W_gate m) * (W_up m))
    With DFlash2 convolution weights in ``lw`` ([Conv], R-conv) each branch's normalised
    input is prepared by Conv_0 and its output finished by Conv_1 before the residual add:
        d_a = delta(n);  q, k, v from Conv_0(n);  y = x + Conv_1(W_o a)
        d_m = delta(m);  z = W_down(SiLU(W_gate p) * (W_up p)), p = Conv_0(m)
        x_next = y + Conv_1(z)
    Returns (x_next, block k, block v)."""
    D, eps, th = geo.head_dim, geo.eps, geo.rope_theta
    conv = "conv_delta_a" in lw
    x = _f64(x)
    n = plain_rmsnorm(x, lw["in_norm"], eps)
    if conv:
        d_a = conv_delta(n, lw["conv_delta_a"])
        n = grouped_conv(n, lw["conv_base_a"], d_a, 0)
    q = rope_1d(plain_head_rmsnorm(n @ _f64(lw["wq"]).T, lw["q_norm"], eps, D), positions, D, th)
    k = rope_1d(plain_head_rmsnorm(n @ _f64(lw["wk"]).T, lw["k_norm"], eps, D), positions, D, th)
    v = n @ _f64(lw["wv"]).T
    a = block_attention(q, k, v, k_ctx, v_ctx, ctx_positions, frontier, geo.windows[layer],
                        geo.block_causal, geo.n_q_heads, geo.n_kv_heads, D)
    o = a @ _f64(lw["wo"]).T
    y = x + (grouped_conv(o, lw["conv_base_a"], d_a, 1) if conv else o)
    m = plain_rmsnorm(y, lw["post_norm"], eps)
    if conv:
        d_m = conv_delta(m, lw["conv_delta_m"])
        m = grouped_conv(m, lw["conv_base_m"], d_m, 0)
    z = (silu(m @ _f64(lw["w_gate"]).T) * (m @ _f64(lw["w_up"]).T)) @ _f64(lw["w_down"]).T
    x_next = y + (grouped_conv(z, lw["conv_base_m"], d_m, 1) if conv else z)
    return x_next, k, v


# --------------------------------------------------------------------------- bridge
def bridge_read(x, r_read, code_width: int, eps: float):
    """DSpine code read for every row:  r = sqrt(mean x^2),  z = R_l x / (r + eps),
    c = sqrt(Rc) z / (||z|| + eps).  Returns (c [W, Rc], r [W]).
    [Bridge] read equations; [Transfer] (one learned projection per layer)."""
    x = _f64(x)
    r = np.sqrt(np.mean(x * x, axis=-1))
    z = (x / (r + eps)[:, None]) @ _f64(r_read).T
    c = math.sqrt(code_width) * z / (np.linalg.norm(z, axis=-1) + eps)[:, None]
    return c, r


def anchor_code(codebook_row, code_width: int) -> np.ndarray:
    """Anchor rows use sqrt(Rc) times the anchor token's stored code.  [Bridge];
    [Transfer] (a known token enters the space as r C_x)."""
    return math.sqrt(code_width) * _f64(codebook_row)


def inject(x, c, r, g_recv, g_pred, a_val, w_write, gate_bias=None) -> np.ndarray:
    """Adjacent gated causal injection for one request's block (R-gate, R-anchor, R-rms):
        for i >= 1: g = sigmoid(G c_i + G_p c_{i-1} + b),  m = g * (A c_{i-1}),
                    x'_i = x_i + r_i W_l m
        x'_0 = x_0 (the anchor receives no write)
    All codes are the pre-injection codes of this layer.  [Bridge]; [Gate]."""
    x = _f64(x)
    c = _f64(c)
    b = np.zeros(_f64(g_recv).shape[0]) if gate_bias is None else _f64(gate_bias)
    G, Gp, A, Wl = _f64(g_recv), _f64(g_pred), _f64(a_val), _f64(w_write)
    out = x.copy()
    for i in range(1, x.shape[0]):
        g = sigmoid(G @ c[i] + Gp @ c[i - 1] + b)
        m = g * (A @ c[i - 1])
        out[i] = x[i] + r[i] * (Wl @ m)
    return out


# --------------------------------------------------------------------------- head
def lm_head_logits(h, embed_head, chunk: int = 16384) -> np.ndarray:
    """logits = E h with the tied [V, H] head, computed in vocabulary chunks to bound
    memory (a plain matrix product; chunking does not change any value)."""
    h = _f64(h)
    E = embed_head
    V = E.shape[0]
    out = np.empty((h.shape[0], V))
    for v0 in range(0, V, chunk):
        out[:, v0:v0 + chunk] = h @ _f64(E[v0:v0 + chunk]).T
    return out


def argmax_lowest(logits) -> np.ndarray:
    """Per-row argmax; ties resolve to the lowest token id (R-tie)."""
    return np.argmax(_f64(logits), axis=-1)


def lm_head_topk(logits, k: int):
    """[Refine]: the k candidate tokens of each row and their scores -- the k largest
    logits of the full vocabulary, by descending score, equal scores by ascending token
    id (R-topk).  A stable sort of the negated logits gives exactly that order."""
    logits = _f64(logits)
    ids = np.argsort(-logits, axis=-1, kind="stable")[:, :k]
    return ids, np.take_along_axis(logits, ids, axis=-1)


# --------------------------------------------------------------------------- FP8 retrieval
E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 (OCP FP8 E4M3FN) value, ties to even, magnitudes above the
    largest finite value 448 clamped to it.  E4M3 has 3 mantissa bits, exponent bias 7 and
    no infinities: normal values are (1 + m/8) 2^e for e >= -6, subnormals m 2^-9."""
    x = _f64(x)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                      # below 2^-6 the spacing stays 2^-9
    step = np.exp2(e - 3.0)
    r = np.rint(a / step) * step                 # np.rint rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.sign(x) * r


def fp8_row_code(M):
    """Row-scaled FP8 code of each row of M (R-fp8): scale s = max|row| / 448 and codes
    e4m3(row / s), both in fp32.  Returns (codes as float64 values, scales)."""
    M32 = np.asarray(M, dtype=np.float32)
    mx = np.max(np.abs(M32), axis=-1)
    s = (mx / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = e4m3_round((M32 / s[..., None]).astype(np.float32))
    return q, s.astype(np.float64)


def lm_head_topk_fp8(hidden, embed_head, n_cand: int, k: int, tile: int = 128,
                     per_tile: int = 16):
    """[Refine] FP8 retrieval then BF16 rescoring (R-fp8).  Returns (ids [rows, k], exact
    scores [rows, k], candidate ids [rows, n_cand] in approximate-score order)."""
    qE, sE = fp8_row_code(embed_head)
    qh, _ = fp8_row_code(hidden)
    approx = (qh @ qE.T) * sE[None, :]                       # [rows, V]
    rows, V = approx.shape
    pool_ids = []
    for t0 in range(0, V, tile):
        blk = approx[:, t0:t0 + tile]
        ids = np.argsort(-blk, axis=-1, kind="stable")[:, :per_tile] + t0
        pool_ids.append(ids)
    pool = np.concatenate(pool_ids, axis=1)                  # [rows, tiles * per_tile]
    pool_sc = np.take_along_axis(approx, pool, axis=1)
    order = np.lexsort((pool, -pool_sc), axis=-1)[:, :n_cand]  # score desc, id asc
    cand = np.take_along_axis(pool, order, axis=1)
    E = _f64(embed_head)
    exact = np.einsum("rkh,rh->rk", E[cand], _f64(hidden))
    sel = np.lexsort((cand, -exact), axis=-1)[:, :k]
    return (np.take_along_axis(cand, sel, axis=1), np.take_along_axis(exact, sel, axis=1), cand)


def top2_gap(logits) -> np.ndarray:
    s = np.sort(_f64(logits), axis=-1)
    return s[:, -1] - s[:, -2]


# --------------------------------------------------------------------------- round
def ring_context(rings, layer: int, request: int, frontier: int, capacity: int):
    """The context K/V a request's ring holds for one layer: positions of the live
    interval in ascending order, read from slot p mod S."""
    lo, hi = ring_live_interval(frontier, capacity)
    pos = np.arange(lo, hi, dtype=np.int64)
    slots = pos % capacity
    k = _f64(rings["k"][layer][request])[:, slots, :].transpose(1, 0, 2)   # [n, Hkv, D]
    v = _f64(rings["v"][layer][request])[:, slots, :].transpose(1, 0, 2)
    return k, v, pos


def draft_request(geo, weights, rings, request: int, anchor: int, frontier: int,
                  mask_id: int, n_masks: int) -> Dict[str, np.ndarray]:
    """One request's block through every draft layer (plus injection when the
    geometry has a code width), then the final norm.  [DFlash-notes] draft input
    table and per-layer equations; [Bridge] and [Gate] for the injection."""
    W = n_masks + 1
    E = weights["embed_head"]
    ids = [anchor] + [mask_id] * n_masks
    x = _f64(np.stack([np.asarray(E[i]) for i in ids]))                 # [W, H]
    positions = frontier + np.arange(W, dtype=np.int64)
    inj = geo.code_width > 0
    layers_x = []
    for l in range(geo.n_layers):
        lw = weights["layers"][l]
        k_ctx, v_ctx, cpos = ring_context(rings, l, request, frontier, geo.capacity(l))
        x, _, _ = dflash_layer(x, lw, geo, positions, k_ctx, v_ctx, cpos, frontier, l)
        tail = None
        if inj:
            c, r = bridge_read(x, lw["r_read"], geo.code_width, geo.eps)
            c[0] = anchor_code(weights["codebook"][anchor], geo.code_width)
            tail = {"u": x.copy(), "c": c, "r": r}
            x = inject(x, c, r, weights["g_recv"], weights["g_pred"], weights["a_val"],
                       lw["w_write"], weights.get("gate_bias"))
        layers_x.append(x.copy())
    h = plain_rmsnorm(x, weights["final_norm"], geo.eps)
    out = {"x_layers": np.stack(layers_x), "h": h}
    if inj:
        out["tail"] = tail  # the last layer's pre-injection state, codes and RMS
    return out


def catch_up(geo, weights, rings, frontiers: Sequence[int], feats, requests, positions):
    """Materialise pending context rows before a round (R-catch, [Frontier]): row t
    (features feats[t], request requests[t], position positions[t]) goes into its
    request's rings; ``frontiers[b]`` is the frontier the rows complete.  The rings are
    updated in place and returned."""
    requests = np.asarray(requests, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    for b in sorted(set(requests.tolist())):
        sel = np.nonzero(requests == b)[0]
        materialize(geo, weights, _f64(feats)[sel], positions[sel], int(frontiers[b]),
                    rings=rings, request=b)
    return rings


def draft_round(geo, weights, rings, anchors: Sequence[int], frontiers: Sequence[int],
                mask_id: int, n_masks: int, with_head: bool = True,
                pending=None) -> Dict[str, np.ndarray]:
    """The whole proposal round for B independent requests.
    Returns x_layers [L, B, W, H], h [B, W, H] and, with the head, the mask rows'
    logits [B, K, V], argmax tokens [B, K] and top-2 gaps [B, K].
    [DFlash-notes] proposal head: only the K mask columns are scored.
    pending = (feats, requests, positions): rows caught up into ``rings`` first
    (catch_up)."""
    if pending is not None:
        catch_up(geo, weights, rings, frontiers, *pending)
    outs = [draft_request(geo, weights, rings, b, int(anchors[b]), int(frontiers[b]),
                          mask_id, n_masks) for b in range(len(anchors))]
    res = {"x_layers": np.stack([o["x_layers"] for o in outs], axis=1),
           "h": np.stack([o["h"] for o in outs])}
    if geo.code_width > 0:
        res["tail"] = [o["tail"] for o in outs]
    if with_head:
        B = len(anchors)
        hm = res["h"][:, 1:, :].reshape(B * n_masks, -1)
        logits = lm_head_logits(hm, weights["embed_head"])
        res["logits"] = logits.reshape(B, n_masks, -1)
        res["tokens"] = argmax_lowest(logits).reshape(B, n_masks)
        res["gap"] = top2_gap(logits).reshape(B, n_masks)
    return res


# --------------------------------------------------------------------------- tail
def refine_state(geo, weights, tail, i: int, s: int) -> np.ndarray:
    """Last-write refinement of block row i (>= 1) with predecessor token s (R-tail):
        c_pred = sqrt(Rc) C_s,  g = sigmoid(G c_i + G_p c_pred + b),  m = g * (A c_pred),
        x' = u_i + r_i W_L m,   h' = plain_rmsnorm(x', final_norm).
    [Tail] last-write refinement; [Gate] for the injection it redoes."""
    lw = weights["layers"][geo.n_layers - 1]
    u, c, r = _f64(tail["u"][i]), _f64(tail["c"][i]), float(tail["r"][i])
    b = np.zeros(_f64(weights["g_recv"]).shape[0]) if weights.get("gate_bias") is None \
        else _f64(weights["gate_bias"])
    c_pred = anchor_code(weights["codebook"][s], geo.code_width)
    g = sigmoid(_f64(weights["g_recv"]) @ c + _f64(weights["g_pred"]) @ c_pred + b)
    m = g * (_f64(weights["a_val"]) @ c_pred)
    x = u + r * (_f64(lw["w_write"]) @ m)
    return plain_rmsnorm(x[None, :], weights["final_norm"], geo.eps)[0]


def refine_tail(geo, weights, tail, anchor: int, cand):
    """Transition tables and greedy walk of one request's block (R-tail).
    cand [K, k]: candidate token ids of block rows 1..K (row i at cand[i - 1]).
    Returns (scores1 [k], tables [K-1, k, k], picks [K] candidate indices, tokens [K]);
    tables[i - 2][p, j] = E[cand[i-1][j]] . refine_state(i, cand[i-2][p]).
    [Tail]: the K x K pair scores, then the left-to-right lookup."""
    E = weights["embed_head"]
    K, k = cand.shape
    h1 = refine_state(geo, weights, tail, 1, anchor)
    scores1 = np.array([float(_f64(E[v]) @ h1) for v in cand[0]])
    tables = np.zeros((K - 1, k, k))
    for i in range(2, K + 1):
        for p in range(k):
            h = refine_state(geo, weights, tail, i, int(cand[i - 2][p]))
            tables[i - 2, p] = [float(_f64(E[v]) @ h) for v in cand[i - 1]]
    picks = np.zeros(K, dtype=np.int64)
    picks[0] = int(np.argmax(scores1))             # lowest rank on ties
    for i in range(2, K + 1):
        picks[i - 1] = int(np.argmax(tables[i - 2, picks[i - 2]]))
    tokens = np.array([cand[i][picks[i]] for i in range(K)])
    return scores1, tables, picks, tokens


# --------------------------------------------------------------------------- sizes
def kv_bytes_per_position(n_layers: int, n_kv_heads: int, head_dim: int,
                          k_bytes: int, v_bytes: int) -> int:
    """Draft K/V bytes one retained position occupies over all layers.  [Cache]."""
    return n_layers * n_kv_heads * head_dim * (k_bytes + v_bytes)


def ring_image_bytes(n_layers: int, n_kv_heads: int, head_dim: int, capacity: int,
                     k_bytes: int = 2, v_bytes: int = 2) -> int:
    """Bytes of all local rings of one request.  [DFlash-notes], ring storage."""
    return kv_bytes_per_position(n_layers, n_kv_heads, head_dim, k_bytes, v_bytes) * capacity


def injection_param_count(hidden: int, n_layers: int, code_width: int, msg_width: int) -> int:
    """Per layer one read R_l [Rc, H] and one write W_l [H, Mc]; the receiver gate,
    predecessor gate and value maps [Mc, Rc] are shared by all layers (R-read).
    [Bridge]; [Gate]; [Transfer] (about 33M extra parameters at Qwen3-8B geometry)."""
    return n_layers * (code_width * hidden + hidden * msg_width) + 3 * msg_width * code_width


def round_weight_bytes(geo, elem_bytes: int = 2) -> int:
    """Weight bytes one round streams: every draft layer's projections (and the
    bridge's, when present), the shared gate maps and the tied head."""
    H, D, L = geo.hidden, geo.head_dim, geo.n_layers
    per_layer = (H * geo.n_q_heads * D + 2 * H * geo.n_kv_heads * D + geo.n_q_heads * D * H
                 + 3 * H * geo.ffn + 4 * H + 2 * D)
    if geo.code_width > 0:
        per_layer += geo.code_width * H + H * geo.msg_width
    total = L * per_layer + geo.vocab * H + H
    if geo.code_width > 0:
        total += 3 * geo.msg_width * geo.code_width
    return total * elem_bytes
