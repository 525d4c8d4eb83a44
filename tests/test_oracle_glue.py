"""Pins of the float64 forward-pass glue (oracle/glue.py) against closed forms
and invariants that a dropped term, a wrong sign or a swapped half would
break. CPU only."""
import math

import numpy as np

from oracle import glue

rng = np.random.default_rng(7)


def bf16(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_rmsnorm_constant_row_is_sign_times_gamma():
    g = bf16(rng.uniform(0.5, 1.5, 64))
    for c in (3.0, -0.25):
        out = glue.rmsnorm(np.full((1, 64), c), g, 0.0)
        assert np.allclose(out[0], math.copysign(1.0, c) * glue._f64_of_bf16(g), rtol=0, atol=1e-15)


def test_rmsnorm_scale_invariance_and_unit_mean_square():
    x = rng.standard_normal((3, 256))
    g = bf16(np.ones(256))
    a = glue.rmsnorm(x, g, 0.0)
    assert np.allclose(glue.rmsnorm(7.5 * x, g, 0.0), a, atol=1e-14)
    assert np.allclose(np.mean(a * a, axis=1), 1.0, atol=1e-14)
    # eps enters under the root: a row of zeros stays zero, a tiny row is damped
    assert np.all(glue.rmsnorm(np.zeros((1, 8)), bf16(np.ones(8)), 1e-5) == 0)
    small = glue.rmsnorm(np.full((1, 4), 1e-3), bf16(np.ones(4)), 1e-6)
    assert np.allclose(small, 1e-3 / math.sqrt(1e-6 + 1e-6))


def test_rope_identity_at_zero_norms_and_composition():
    x = rng.standard_normal((2, 3, 128))
    assert np.allclose(glue.rope(x, [0, 0], 1e4), x, atol=0)
    r = glue.rope(x, [5, 1234], 1e4)
    pair = lambda y: y[..., :64] ** 2 + y[..., 64:] ** 2  # noqa: E731
    assert np.allclose(pair(r), pair(x), rtol=1e-12)
    assert np.allclose(glue.rope(glue.rope(x, [5, 1234], 1e4), [7, 100], 1e4), glue.rope(x, [12, 1334], 1e4),
                       atol=1e-10)


def test_rope_hand_values():
    # pair 0 turns by p radians (frequency theta^0 = 1); pair 32 by p / sqrt(theta)
    e0 = np.zeros((1, 1, 128))
    e0[0, 0, 0] = 1.0
    r = glue.rope(e0, [3], 10000.0)[0, 0]
    assert np.isclose(r[0], math.cos(3.0)) and np.isclose(r[64], math.sin(3.0))
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2
    e32 = np.zeros((1, 1, 128))
    e32[0, 0, 32 + 64] = 1.0  # b of pair 32: (0, 1) -> (-sin, cos)
    r = glue.rope(e32, [10], 10000.0)[0, 0]
    ang = 10 / math.sqrt(10000.0)
    assert np.isclose(r[32], -math.sin(ang)) and np.isclose(r[96], math.cos(ang))


def test_rope_split_heads_and_positions():
    Hq, Hkv = 4, 2
    qkv = rng.standard_normal((6, (Hq + 2 * Hkv) * 128))
    q, k, v = glue.rope_split(qkv, Hq, Hkv, 100, 3, 5e5)
    h = qkv.reshape(6, Hq + 2 * Hkv, 128)
    assert np.array_equal(v, h[:, Hq + Hkv:])
    assert np.allclose(q[3], glue.rope(h[3:4, :Hq], [100], 5e5)[0])  # row 3 is position 100 again
    assert np.allclose(k[5], glue.rope(h[5:6, Hq:Hq + Hkv], [102], 5e5)[0])


def test_silu_mul_closed_forms():
    gu = np.array([[0.0, math.log(3.0), 40.0, -40.0, 2.0, 2.0, 2.0, 2.0]])
    out = glue.silu_mul(gu)[0]
    assert out[0] == 0.0
    assert np.isclose(out[1], 0.75 * math.log(3.0) * 2.0)  # sigmoid(ln 3) = 3/4
    assert np.isclose(out[2], 80.0) and abs(out[3]) < 1e-15


def test_argmax_ties_and_nan():
    lg = np.array([[1.0, 5.0, 5.0, -1.0], [np.nan, 2.0, 7.0, 7.0], [-np.inf, -np.inf, -3.0, -np.inf]])
    assert list(glue.argmax(lg)) == [1, 2, 2]


def test_embed_rows():
    table = bf16(rng.standard_normal((10, 8)))
    out = glue.embed([3, 3, 9], table)
    assert np.array_equal(out[0], glue._f64_of_bf16(table[3])) and np.array_equal(out[2], glue._f64_of_bf16(table[9]))
