"""The one-launch bridge evaluates the code read in a factored order: z' = R_l x before the
row norm is applied, then c = sqrt(Rc) z' / (|z'| + eps (r + eps)), with that per-row scale
applied after the gate/value products (G c = s G z').  These identities tie the order to
the oracle's reading (z = R_l x / (r + eps), c = sqrt(Rc) z / (|z| + eps)) in exact
arithmetic; they are checked here in fp64 on random rows, including rows whose norm is tiny
or large enough for eps to matter.  (Arithmetic check of the kernel's formula; the kernel
itself is checked against the oracle by the GPU parity tests.)"""
import math

import numpy as np

from oracle import dspine_oracle as O


def _factored(x, R, Rc, eps):
    r = np.sqrt(np.mean(x * x, axis=-1))
    zp = x @ R.T                                   # z' = R x, no normalisation yet
    s = math.sqrt(Rc) / (np.linalg.norm(zp, axis=-1) + eps * (r + eps))
    return zp, s, r


def test_factored_code_equals_the_oracle_reading():
    rng = np.random.default_rng(7)
    H, Rc, eps = 96, 32, 1e-6
    R = rng.normal(0.0, 0.1, (Rc, H))
    x = rng.normal(0.0, 1.0, (6, H)) * np.array([1e-7, 1e-4, 1.0, 3.0, 1e3, 1e5])[:, None]
    c_ref, r_ref = O.bridge_read(x, R, Rc, eps)
    zp, s, r = _factored(x, R, Rc, eps)
    np.testing.assert_allclose(r, r_ref, rtol=1e-14)
    np.testing.assert_allclose(zp * s[:, None], c_ref, rtol=1e-12, atol=1e-300)


def test_scale_after_the_product_equals_the_product_of_the_code():
    rng = np.random.default_rng(8)
    H, Rc, Mc, eps = 64, 32, 16, 1e-6
    R = rng.normal(0.0, 0.1, (Rc, H))
    G = rng.normal(0.0, 0.1, (Mc, Rc))
    x = rng.normal(0.0, 1.0, (5, H))
    c_ref, _ = O.bridge_read(x, R, Rc, eps)
    zp, s, _ = _factored(x, R, Rc, eps)
    np.testing.assert_allclose((zp @ G.T) * s[:, None], c_ref @ G.T, rtol=1e-12, atol=1e-15)


def test_a_wrong_floor_term_is_detected():
    """The floor is eps (r + eps), not eps: with eps the size of |z'| the two differ."""
    rng = np.random.default_rng(9)
    H, Rc, eps = 64, 16, 1e-2
    R = rng.normal(0.0, 0.1, (Rc, H))
    x = rng.normal(0.0, 1.0, (3, H)) * 1e-3
    c_ref, _ = O.bridge_read(x, R, Rc, eps)
    zp = x @ R.T
    wrong = math.sqrt(Rc) * zp / (np.linalg.norm(zp, axis=-1) + eps)[:, None]
    assert not np.allclose(wrong, c_ref, rtol=1e-6)
