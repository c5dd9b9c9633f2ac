"""Full-size parity: the benchmark geometries, in the launch configuration bench.py times.

Round parity uses the oracle in its second mode (it reads the GPU's context rings), so
these checks are independent of the materialisation check.  Requests are independent,
so at B=8 the oracle recomputes sampled requests one by one.  Tolerances as in
test_gpu_parity: hidden states max|gpu-ref|/max|ref| <= 2e-2, tokens exact where the
oracle's top-2 gap exceeds 1e-2.
"""
import json

import numpy as np
import pytest
import torch

import bdsynth
import harness as Hn
from oracle import dspine_oracle as O

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 2e-2


def record(name, rep):
    """Print the case's error report (pytest shows it with -s or on failure)."""
    print(json.dumps({"case": name, **rep}))


@pytest.fixture(scope="module", autouse=True)
def built():
    from block_drafter_gb300 import builder
    builder.build()


def run_case(geo, requests, seed=0):
    case = Hn.Case(geo, seed=seed, gen_device="cuda", max_ctx_rows=2048)
    case.fill_rings()
    gpu = case.run_gpu()
    ref = case.run_oracle(requests)
    rep = Hn.compare_round(case, gpu, ref, requests=requests, tol=TOL)
    rep = {k: (v if not isinstance(v, float) else round(v, 6)) for k, v in rep.items()}
    rep["requests"] = requests
    rep["frontiers"] = [case.frontiers[b] for b in requests]
    return rep


def test_dspine_27b_b1_full_round():
    rep = run_case(bdsynth.DSPINE27B_B1, [0])
    record("dspine_b16_27b_b1", rep)
    print(rep)
    assert rep["ok"], rep


def test_dflash2_27b_b1_full_round():
    rep = run_case(bdsynth.DFLASH2_27B_B1, [0])
    record("dflash2_27b_b1", rep)
    print(rep)
    assert rep["ok"], rep


def test_dspine_27b_b8_sampled_requests():
    rep = run_case(bdsynth.DSPINE27B_B8, [0, 4, 7])
    record("dspine_b16_27b_b8", rep)
    print(rep)
    assert rep["ok"], rep


def test_dflash_35b_b8_sampled_requests():
    rep = run_case(bdsynth.DFLASH35B_B8, [2, 5])
    record("dflash_35b_a3b_b8", rep)
    print(rep)
    assert rep["ok"], rep


def test_ctx_materialize_27b_sampled_positions():
    """The 2048-row prefill chunk (positions 0..2047): every layer's stored K and V at
    sampled positions against the oracle's per-position projection."""
    geo = bdsynth.CTX27B
    case = Hn.Case(geo, seed=0, gen_device="cuda", max_ctx_rows=2048)
    used = case.fill_rings()
    (c0, feats), = used[0]
    assert c0 == 0 and feats.shape[0] == 2048
    pos = np.array([0, 1, 2, 511, 1024, 1500, 2046, 2047])
    wnp = Hn.weights_to_np(case.w_host)
    rings = O.materialize(geo, wnp, Hn.np32(feats[torch.as_tensor(pos, device=feats.device)]),
                          pos, 2048)
    worst = 0.0
    for l in range(geo.n_layers):
        for key, ring in (("k", case.sess.k[l]), ("v", case.sess.v[l])):
            got = Hn.np32(ring[0])[:, pos % geo.capacity(l)]
            ref = rings[key][l][0][:, pos % geo.capacity(l)]
            err = Hn.rel_err(got, ref)
            worst = max(worst, err)
            assert err <= TOL, (l, key, err)
    record("ctx_materialize_27b", {"positions": pos.tolist(), "max_rel_err": round(worst, 6)})


def test_materialize_chunking_and_final_window_on_gpu():
    """Splitting a chunk across calls stores identical rings (bit for bit), and a chunk
    longer than the ring stores exactly its final window."""
    geo = bdsynth.DSPINE27B_B1.with_(n_layers=2, windows=(64, 64), hidden=512, ffn=1024,
                                     vocab=2048, code_width=128, msg_width=64, n_q_heads=8,
                                     n_kv_heads=2, n_target_layers=3, mask_token_id=-1)
    a = Hn.Case(geo, seed=9, frontiers=[200], max_ctx_rows=256)
    b = Hn.Case(geo, seed=9, frontiers=[200], max_ctx_rows=256, weights=a.w_host)
    feats = a.features(0, 0, 200, 0).cuda()
    front = torch.tensor([200], dtype=torch.int64, device="cuda")
    req = torch.zeros(200, dtype=torch.int32, device="cuda")
    pos = torch.arange(200, dtype=torch.int64, device="cuda")
    a.sess.materialize(feats, req, pos, front)                   # one 200-row call
    b.sess.materialize(feats[:77], req[:77], pos[:77], front)    # three uneven calls
    b.sess.materialize(feats[77:150], req[77:150], pos[77:150], front)
    b.sess.materialize(feats[150:], req[150:], pos[150:], front)
    torch.cuda.synchronize()
    for l in range(geo.n_layers):
        assert torch.equal(a.sess.k[l], b.sess.k[l]) and torch.equal(a.sess.v[l], b.sess.v[l])
    # only the final window [136, 200) was stored; the ring holds nothing else
    c = Hn.Case(geo, seed=9, frontiers=[200], max_ctx_rows=256, weights=a.w_host)
    c.sess.materialize(feats[136:], req[136:], pos[136:], front)
    torch.cuda.synchronize()
    for l in range(geo.n_layers):
        assert torch.equal(a.sess.k[l], c.sess.k[l]) and torch.equal(a.sess.v[l], c.sess.v[l])
