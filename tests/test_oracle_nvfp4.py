"""Pins of the oracle's NVFP4 quantiser and of the NVFP4-weight layer: golden E2M1 codes
from the format definition, an exhaustive nearest-even search over the E2M1 values, closed
forms of the matrix scale, block properties, and the quantisation axis of every weight."""
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_codes.txt")


def e2m1_table():
    """Every E2M1 code's value from the bit fields (sign, exponent with bias 1, mantissa)."""
    vals = {}
    for c in range(16):
        s = -1.0 if c & 8 else 1.0
        e, m = (c >> 1) & 3, c & 1
        vals[c] = s * (0.5 * m if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    return vals


def test_e2m1_golden_codes():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 15
    for v, code in rows:
        q = O.e2m1_round(np.array([float(v)]))
        assert O.e2m1_encode(q)[0] == int(code, 16), (v, code)
        assert O.e2m1_decode(np.array([int(code, 16)], np.uint8))[0] == float(v)


def test_e2m1_round_matches_exhaustive_nearest_even():
    table = e2m1_table()
    pos = sorted((v, c) for c, v in table.items() if v >= 0 and c < 8)
    rng = np.random.default_rng(0)
    samples = np.concatenate([rng.uniform(0, 7, 4000), 2.0 ** rng.uniform(-6, 3, 2000),
                              np.array([v for v, _ in pos]),
                              np.array([(pos[i][0] + pos[i + 1][0]) / 2 for i in range(len(pos) - 1)])])
    for a in samples:
        want = 6.0 if a > 6 else min(pos, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))[0]
        assert O.e2m1_round(np.array([a]))[0] == want, a
        assert O.e2m1_round(np.array([-a]))[0] == -want
    for c, v in table.items():
        if c == 8:       # negative zero encodes as code 8 only from -0.0
            continue
        assert O.e2m1_encode(np.array([v]))[0] == c


def test_matrix_scale_closed_form():
    assert O.nv_matrix_scale(448.0 * 6.0) == 1.0
    assert O.nv_matrix_scale(448.0 * 6.0 * (1 + 2 ** -30)) == 2.0
    assert O.nv_matrix_scale(448.0 * 6.0 / 2) == 0.5
    assert O.nv_matrix_scale(0.0) == 1.0
    for a in 2.0 ** np.random.default_rng(1).uniform(-40, 40, 500):
        g = O.nv_matrix_scale(a)
        assert a <= 2688.0 * g < 2 * a and np.log2(g) == np.round(np.log2(g))


def test_nv_block_properties():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 48)) * 2.0 ** rng.integers(-6, 6, (1, 48))
    codes, scales, g = O.nv_quantize(v, 0)
    assert codes.shape == (64, 48) and scales.shape == (4, 48) and codes.max() < 16
    assert g == O.nv_matrix_scale(np.abs(v).max())
    deq = O.nv_dequantize(codes, scales, g, 0)
    blk = np.abs(v).reshape(4, 16, 48)
    s = O.e4m3_decode(scales)
    # every block scale is the E4M3 value nearest to amax / (6 g)
    np.testing.assert_array_equal(s, O.e4m3_round(blk.max(axis=1) / (6 * g)))
    # elements are E2M1 values at most 6; the block maximum lands within one E2M1 step of 6
    assert (np.abs(O.e2m1_decode(codes)) <= 6).all()
    e = np.abs(deq - v).reshape(4, 16, 48)
    assert (e <= (blk.max(axis=1, keepdims=True) / 6) * 1.07 + 1e-300).all()   # half of the largest step, 2 units, plus scale rounding
    # a block of E2M1 values times one power of two (with a 6 in it) is exact
    u = rng.choice(np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6.0]), (32, 8))
    u[0] = 6.0
    w = u * 2.0 ** rng.integers(-4, 4, (1, 8))
    np.testing.assert_array_equal(O.nv_roundtrip(w, 0), w)
    # zeros quantise to code 0 and scale 0; the axis argument is honoured
    c0, s0, _ = O.nv_quantize(np.zeros((16, 3)), 0)
    assert (c0 == 0).all() and (s0 == 0).all()
    cT, sT, gT = O.nv_quantize(v.T, 1)
    np.testing.assert_array_equal(cT, codes.T)
    np.testing.assert_array_equal(sT, scales.T)


def _nv_structured(rng, shape, axis):
    """E2M1 values times a power of two constant along `axis` (each 16-block holds a 6) and
    either 1 or 2^-4 across it: exact under NVFP4 along `axis`, not across it."""
    u = rng.choice(np.array([0, 0.5, 1, 1.5, 2, 3, 4, -0.5, -1, -1.5, -2, -3, -4.0]), shape)
    u = np.moveaxis(u, axis, 0)
    u[::16] = 6.0
    u = np.moveaxis(u, 0, axis)
    other = 1 - axis
    c = 2.0 ** -rng.choice(np.array([0, 4]), shape[other])
    return u * (c[None, :] if other == 1 else c[:, None])


def test_nvfp4_layer_quantises_each_weight_along_its_contraction_axis():
    # W1, W3 along H and W2 along F: weights exact along their contraction axis (and not
    # across it) make the NVFP4 layer equal to the float64 layer element for element; a
    # wrong axis for any of them, or a missing matrix scale, breaks the equality
    rng = np.random.default_rng(31)
    T, H, F, E, k = 40, 64, 64, 4, 2
    x = rng.standard_normal((T, H))
    W1 = np.stack([_nv_structured(rng, (H, F), 0) for _ in range(E)]) * 0.01
    W3 = np.stack([_nv_structured(rng, (H, F), 0) for _ in range(E)]) * 2.0 ** -7
    W2 = np.stack([_nv_structured(rng, (F, H), 0) for _ in range(E)]) * 2.0 ** -6
    W1 = W1 / 0.01 * 2.0 ** -7                     # powers of two keep the structure exact
    Wr = rng.standard_normal((H, E)) * 0.3
    assert (O.nv_roundtrip(W1[0], 0) == W1[0]).all() and (O.nv_roundtrip(W1[0], 1) != W1[0]).any()
    assert (O.nv_roundtrip(W2[0], 0) == W2[0]).all() and (O.nv_roundtrip(W2[0], 1) != W2[0]).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k)
    fnv = O.forward(x, Wr, None, W1, W3, W2, k, precision="nvfp4")
    np.testing.assert_allclose(fnv["out"], f64["out"], rtol=1e-12, atol=1e-300)
    # each weight that is not exact shows its own rounding (none of the three is left unquantised)
    for i in range(3):
        Ws = [W1, W3, W2]
        Ws[i] = Ws[i] * 1.3
        got = O.forward(x, Wr, None, *Ws, k, precision="nvfp4")["out"]
        assert O.max_abs_rel(got, O.forward(x, Wr, None, *Ws, k)["out"]) > 1e-3, i
