"""Pins of the oracle's MXFP8 quantiser: golden E4M3 codes from the OCP MX
specification, an exhaustive nearest-value search over all 256 codes, closed
forms for the shared scale, and the error bound of the emulated layer."""
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def load_golden():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            v, c = line.split()
            rows.append((float(v), int(c, 16)))
    return rows


def test_e4m3_golden_codes():
    for v, code in load_golden():
        q = O.e4m3_round(np.array([v]))
        assert O.e4m3_encode(q)[0] == code, (v, hex(code), hex(O.e4m3_encode(q)[0]))


def e4m3_table():
    """All finite E4M3 values, built from the bit-field definition."""
    vals = {}
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 0xF and m == 7:
            continue
        vals[c] = s * ((m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return vals


def test_e4m3_round_matches_exhaustive_nearest_even():
    table = e4m3_table()
    pos = sorted((v, c) for c, v in table.items() if v >= 0 and not (v == 0 and c == 0x80))
    rng = np.random.default_rng(0)
    samples = np.concatenate([
        rng.uniform(0, 460, 3000), 2.0 ** rng.uniform(-12, 9, 3000),
        np.array([v for v, _ in pos]),
        np.array([(pos[i][0] + pos[i + 1][0]) / 2 for i in range(len(pos) - 1)]),  # exact ties
    ])
    for a in samples:
        if a > 448:
            want = 448.0
        else:
            best = min(pos, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))   # nearest, tie -> even code
            want = best[0]
        got = O.e4m3_round(np.array([a]))[0]
        assert got == want, (a, got, want)
        assert O.e4m3_round(np.array([-a]))[0] == -want
    for c, v in table.items():
        if c == 0x80:
            continue
        assert O.e4m3_encode(np.array([v]))[0] == c
        assert O.e4m3_decode(np.array([c], np.uint8))[0] == v


def test_scale_exponent_closed_form():
    # smallest s with amax <= 448 * 2^s
    assert O.mx_scale_exponent(np.array([448.0]))[0] == 0
    assert O.mx_scale_exponent(np.array([448.0 * (1 + 2 ** -20)]))[0] == 1
    assert O.mx_scale_exponent(np.array([1.0]))[0] == -8          # 1 <= 448*2^-8 = 1.75
    assert O.mx_scale_exponent(np.array([1.75]))[0] == -8
    assert O.mx_scale_exponent(np.array([1.76]))[0] == -7
    assert O.mx_scale_exponent(np.array([0.0]))[0] == -127
    assert O.mx_scale_exponent(np.array([2.0 ** -140]))[0] == -127    # clamp
    for a in 2.0 ** np.random.default_rng(1).uniform(-30, 30, 500):
        s = O.mx_scale_exponent(np.array([a]))[0]
        assert a <= 448 * 2.0 ** s and a > 448 * 2.0 ** (s - 1)


def test_mx_block_properties():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((6, 128)) * 2.0 ** rng.integers(-10, 10, (6, 1))
    codes, scales = O.mx_quantize(v, 1)
    assert codes.shape == (6, 128) and scales.shape == (6, 4)
    deq = O.mx_dequantize(codes, scales, 1)
    blk = np.abs(v).reshape(6, 4, 32)
    # the block maximum maps to a finite code <= 448 (never saturates)
    q = O.e4m3_decode(codes).reshape(6, 4, 32)
    assert np.abs(q).max() <= 448 and np.isfinite(q).all()
    # normal-range elements carry at most half an E4M3 ulp: relative error <= 2^-4
    big = blk >= blk.max(axis=2, keepdims=True) * 2.0 ** -6
    rel = np.abs(deq.reshape(6, 4, 32) - v.reshape(6, 4, 32)) / np.where(big, blk, 1)
    assert rel[big].max() <= 2.0 ** -4
    # a block of powers of two is exact
    p2 = 2.0 ** rng.integers(-5, 5, (2, 64)).astype(float) * rng.choice([-1, 1], (2, 64))
    np.testing.assert_array_equal(O.mx_roundtrip(p2, 1), p2)
    # an all-zero block -> scale byte 0, code 0
    c0, s0 = O.mx_quantize(np.zeros((1, 32)), 1)
    assert (c0 == 0).all() and (s0 == 0).all()
    # quantisation follows the requested axis
    cT, sT = O.mx_quantize(v.T, 0)
    np.testing.assert_array_equal(cT, codes.T)
    np.testing.assert_array_equal(sT, scales.T)


def test_roundtrip_equals_dequantised_codes():
    # mx_roundtrip forms the represented values directly; they must be exactly what the
    # bytes of mx_quantize decode to, over the whole exponent range, zeros and both axes
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 256)) * 2.0 ** rng.integers(-135, 130, (64, 256))
    v[3] = 0.0
    v[5, :32] = 448.0 * 2.0 ** 7
    for axis in (0, 1):
        c, s = O.mx_quantize(v, axis)
        np.testing.assert_array_equal(O.mx_roundtrip(v, axis), O.mx_dequantize(c, s, axis))


def test_segmented_token_blocks_do_not_cross_segments():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((50, 32))
    v[20:30] *= 1000.0            # a loud segment must not coarsen its neighbours
    got = O.mx_roundtrip_segments(v, [0, 20, 30], [20, 30, 50])
    np.testing.assert_array_equal(got[0:20], O.mx_roundtrip(np.vstack([v[0:20], np.zeros((12, 32))]), 0)[:20])
    np.testing.assert_array_equal(got[30:50], O.mx_roundtrip(np.vstack([v[30:50], np.zeros((12, 32))]), 0)[:20])
    assert O.max_abs_rel(got[0:20], v[0:20]) < 2.0 ** -3


def test_mxfp8_layer_within_format_error_of_exact():
    from tests.test_oracle_ffn_grad import rand_layer
    x, Wr, W1, W3, W2 = rand_layer(9, 40, 64, 4, 64, wstd=0.1)
    f64 = O.forward(x, Wr, None, W1, W3, W2, 2)
    fmx = O.forward(x, Wr, None, W1, W3, W2, 2, precision="mxfp8")
    err = O.max_abs_rel(fmx["out"], f64["out"])
    assert 1e-4 < err < 0.1
    dout = np.random.default_rng(1).standard_normal(x.shape)
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(fmx, dout, x, Wr, W1, W3, W2)
    for key in ("dx", "dW1", "dW3", "dW2", "dWr"):
        e = O.max_abs_rel(gmx[key], g64[key])
        assert 1e-5 < e < 0.15, (key, e)


def _axis_structured(rng, shape, axis):
    """Entries u * c with u in {0, +-1/4, +-1/2, +-1, +-2} and a power-of-two scale c that is
    constant along `axis` (the contraction axis) but spans 2^0 .. 2^-20 along the other one:
    MX blocks along `axis` hold one scale (exact in E4M3), blocks across it do not."""
    u = rng.choice(np.array([0.0, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0, 2.0, -2.0]), shape)
    other = 1 - axis
    c = 2.0 ** -rng.choice(np.array([0, 20]), shape[other])
    return u * (c[None, :] if other == 1 else c[:, None])


def test_mxfp8_forward_quantises_each_operand_along_its_contraction_axis():
    # x along H, W1/W3 along H, h along F, W2 along F: with operands whose blocks are exact along
    # their contraction axis (and inexact across it), the emulated MXFP8 forward must equal the
    # float64 forward with only h rounded, blockwise along F, before GEMM2. A wrong axis for any
    # operand, or a missing / extra quantisation point, breaks the equality.
    rng = np.random.default_rng(11)
    T, H, F, E, k = 64, 64, 64, 4, 2
    x = _axis_structured(rng, (T, H), 1)
    W1 = np.stack([_axis_structured(rng, (H, F), 0) for _ in range(E)])
    W3 = np.stack([_axis_structured(rng, (H, F), 0) for _ in range(E)])
    W2 = np.stack([_axis_structured(rng, (F, H), 0) for _ in range(E)])
    Wr = rng.standard_normal((H, E)) * 0.3
    # the structure is what makes the test sensitive
    assert (O.mx_roundtrip(x, 1) == x).all() and (O.mx_roundtrip(x, 0) != x).any()
    assert (O.mx_roundtrip(W1[0], 0) == W1[0]).all() and (O.mx_roundtrip(W1[0], 1) != W1[0]).any()
    assert (O.mx_roundtrip(W2[0], 0) == W2[0]).all() and (O.mx_roundtrip(W2[0], 1) != W2[0]).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k)
    fmx = O.forward(x, Wr, None, W1, W3, W2, k, precision="mxfp8")
    np.testing.assert_array_equal(fmx["ids"], f64["ids"])
    # exact operands: GEMM1's pre-activations are the float64 ones, element for element
    np.testing.assert_array_equal(fmx["a"], f64["a"])
    np.testing.assert_array_equal(fmx["b"], f64["b"])
    h = f64["h"]
    assert (O.mx_roundtrip(h, 1) != h).any()
    Y = np.zeros((T * k, H))
    for e, s0, s1 in O.expert_segments(f64):
        Y[s0:s1] = O.mx_roundtrip(h[s0:s1], 1) @ W2[e]
    s2s = f64["slot_to_sorted"].reshape(T, k)
    want = sum(f64["w"][:, j:j + 1] * Y[s2s[:, j]] for j in range(k))
    np.testing.assert_allclose(fmx["out"], want, rtol=1e-12, atol=1e-300)
    assert O.max_abs_rel(fmx["out"], f64["out"]) > 1e-6      # h's rounding is visible


def test_mxfp8_backward_dgrads_quantise_along_their_contraction_axes():
    # The backward's MXFP8 points on the dx path: dY rows and W2 along H (GEMM2 dgrad, K = H), da,
    # db and W1, W3 along F (GEMM1 dgrad, K = F). The forward is run in float64 and only the
    # backward emulates MXFP8, so with dY, W2 exact along H and W1, W3 exact along F (each inexact
    # across), da and db must equal the float64 ones exactly and dx must equal the float64
    # composition with only da and db rounded blockwise along F.
    rng = np.random.default_rng(13)
    T, H, F, E, k = 64, 64, 64, 4, 2
    x = rng.standard_normal((T, H))
    W1 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W3 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W2 = np.stack([_axis_structured(rng, (F, H), 1) for _ in range(E)])
    Wr = rng.standard_normal((H, E)) * 0.3
    dout = _axis_structured(rng, (T, H), 1)
    assert (O.mx_roundtrip(W1[0], 1) == W1[0]).all() and (O.mx_roundtrip(W1[0], 0) != W1[0]).any()
    assert (O.mx_roundtrip(W2[0], 1) == W2[0]).all() and (O.mx_roundtrip(W2[0], 0) != W2[0]).any()
    assert (O.mx_roundtrip(dout, 1) == dout).all() and (O.mx_roundtrip(dout, 0) != dout).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k)
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(dict(f64, precision="mxfp8"), dout, x, Wr, W1, W3, W2)
    np.testing.assert_array_equal(gmx["da"], g64["da"])
    np.testing.assert_array_equal(gmx["db"], g64["db"])
    np.testing.assert_array_equal(gmx["dlogits"], g64["dlogits"])
    da, db = g64["da"], g64["db"]
    assert (O.mx_roundtrip(da, 1) != da).any()
    dX = np.zeros((T * k, H))
    for e, s0, s1 in O.expert_segments(f64):
        dX[s0:s1] = O.mx_roundtrip(da[s0:s1], 1) @ W1[e].T + O.mx_roundtrip(db[s0:s1], 1) @ W3[e].T
    s2s = f64["slot_to_sorted"].reshape(T, k)
    want = sum(dX[s2s[:, j]] for j in range(k)) + g64["dlogits"] @ Wr.T
    np.testing.assert_allclose(gmx["dx"], want, rtol=1e-12, atol=1e-300)
    assert O.max_abs_rel(gmx["dx"], g64["dx"]) > 1e-6      # da, db rounding is visible


def _runs(fwd):
    """Per expert, the (start, end) of its runs of sorted rows, in macrobatch order."""
    runs = {}
    for e, s0, s1 in O.expert_segments(fwd):
        runs.setdefault(e, []).append((s0, s1))
    return runs


def _token_blocks(v, s0, s1):
    """v's rows s0..s1 (one run) rounded in 32-row blocks along the token axis that start
    at the run's first row."""
    return O.mx_roundtrip_segments(v[s0:s1], [0], [s1 - s0])


@pytest.mark.parametrize("macro", [0, 24])
def test_mxfp8_weight_gradient_quantises_along_the_token_axis(macro):
    # dW1 = X^T da contracts over each expert's rows: both operands are rounded in 32-row blocks
    # along the token axis that start at each (macrobatch, expert) run and never cross it. With X
    # exact along the tokens (inexact across) and the dgrad operands exact as above, dW1 must equal
    # the sum over the expert's runs of X_run^T times da_run rounded in the run's own blocks.
    # macro = 24 gives three macrobatches, so experts have several runs whose lengths are not
    # multiples of 32: a block that starts anywhere but the run's first row changes the result.
    rng = np.random.default_rng(17)
    T, H, F, E, k = 64, 64, 64, 4, 2
    x = _axis_structured(rng, (T, H), 0)
    W1 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W3 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W2 = np.stack([_axis_structured(rng, (F, H), 1) for _ in range(E)])
    Wr = rng.standard_normal((H, E)) * 0.3
    dout = _axis_structured(rng, (T, H), 1)
    f64 = O.forward(x, Wr, None, W1, W3, W2, k, macrobatch_tokens=macro)
    Xs = f64["Xs"]
    assert (O.mx_roundtrip(Xs, 1) != Xs).any()                 # rows of Xs are not exact along H
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(dict(f64, precision="mxfp8"), dout, x, Wr, W1, W3, W2)
    da = g64["da"]
    runs = _runs(f64)
    if macro:
        assert max(len(r) for r in runs.values()) >= 2
        assert any((s1 - s0) % 32 for r in runs.values() for s0, s1 in r)
    want = np.zeros_like(g64["dW1"])
    for e, rr in runs.items():
        for s0, s1 in rr:
            want[e] += Xs[s0:s1].T @ _token_blocks(da, s0, s1)
    np.testing.assert_allclose(gmx["dW1"], want, rtol=1e-12, atol=1e-300)
    assert O.max_abs_rel(gmx["dW1"], g64["dW1"]) > 1e-6


def _sorted_row_weights(fwd):
    return fwd["w"].reshape(-1)[fwd["sorted_to_slot"].astype(np.int64)]


def test_mxfp8_dW2_rounds_hw_along_the_token_axis():
    # dW2 = (w h)^T dY contracts over each expert's rows. With dout exact along the tokens (one
    # power-of-two scale per column, inexact across the columns), the dY operand is unchanged by
    # its token-axis rounding, so dW2 must equal the sum over runs of (w h)_run rounded in the
    # run's 32-row blocks, transposed, times dY_run.
    rng = np.random.default_rng(19)
    T, H, F, E, k = 64, 64, 64, 4, 2
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, H, F)) * 0.2
    W3 = rng.standard_normal((E, H, F)) * 0.2
    W2 = rng.standard_normal((E, F, H)) * 0.2
    Wr = rng.standard_normal((H, E)) * 0.3
    dout = _axis_structured(rng, (T, H), 0)
    assert (O.mx_roundtrip(dout, 0) == dout).all() and (O.mx_roundtrip(dout, 1) != dout).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k, macrobatch_tokens=24)
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(dict(f64, precision="mxfp8"), dout, x, Wr, W1, W3, W2)
    hw = _sorted_row_weights(f64)[:, None] * f64["h"]
    Gin = dout[f64["tok"]]
    want = np.zeros_like(g64["dW2"])
    for e, rr in _runs(f64).items():
        for s0, s1 in rr:
            assert (_token_blocks(Gin, s0, s1) == Gin[s0:s1]).all()
            want[e] += _token_blocks(hw, s0, s1).T @ Gin[s0:s1]
    np.testing.assert_allclose(gmx["dW2"], want, rtol=1e-12, atol=1e-300)
    assert O.max_abs_rel(gmx["dW2"], g64["dW2"]) > 1e-6      # the h.w rounding is visible


def test_mxfp8_dW2_rounds_dy_along_the_token_axis():
    # The other operand of dW2. A layer built so that h.w is exact along the tokens: k = 1
    # (w = 1); x[t] = c_t e_0 + e_(1 + chosen expert) with c_t in {1, 2, 4}; W1 and W3 read only
    # x[:, 0], with W1[e][0, :] = 64 so a = 64 c_t and sigmoid(a) rounds to exactly 1 in
    # float64 (silu(a) = a); W3[e][0, f] a signed power of two; so h[t, f] = 64 c_t^2 W3[e][0, f]
    # and every column of h within a run holds powers of two at most 16x apart (exact at one
    # scale). The router reads only the one-hot part. dout is exact along H and inexact along the
    # tokens, so dW2 must equal (w h)_run^T times dY_run rounded in the run's 32-row blocks.
    rng = np.random.default_rng(23)
    T, H, F, E, k = 96, 64, 64, 4, 1
    c = rng.choice(np.array([1.0, 2.0, 4.0]), T)
    chosen = rng.integers(0, E, T)
    x = np.zeros((T, H))
    x[:, 0] = c
    x[np.arange(T), 1 + chosen] = 1.0
    Wr = np.zeros((H, E))
    Wr[1 + np.arange(E), np.arange(E)] = 10.0
    W1 = np.zeros((E, H, F)); W3 = np.zeros((E, H, F))
    W1[:, 0, :] = 64.0
    W3[:, 0, :] = rng.choice(np.array([-1.0, 1.0]), (E, F)) * 2.0 ** rng.integers(-3, 4, (E, F))
    W2 = rng.standard_normal((E, F, H)) * 0.2
    dout = _axis_structured(rng, (T, H), 1)
    assert (O.mx_roundtrip(dout, 1) == dout).all() and (O.mx_roundtrip(dout, 0) != dout).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k, macrobatch_tokens=40)
    np.testing.assert_array_equal(f64["ids"][:, 0], chosen)
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(dict(f64, precision="mxfp8"), dout, x, Wr, W1, W3, W2)
    hw = _sorted_row_weights(f64)[:, None] * f64["h"]
    Gin = dout[f64["tok"]]
    runs = _runs(f64)
    assert max(len(r) for r in runs.values()) >= 2
    want = np.zeros_like(g64["dW2"])
    for e, rr in runs.items():
        for s0, s1 in rr:
            assert (_token_blocks(hw, s0, s1) == hw[s0:s1]).all()    # the structure holds
            want[e] += hw[s0:s1].T @ _token_blocks(Gin, s0, s1)
    np.testing.assert_allclose(gmx["dW2"], want, rtol=1e-12, atol=1e-300)
    # the dY rounding is visible (the rows scaled by 2^-20 lose most of their bits)
    assert O.max_abs_rel(gmx["dW2"], g64["dW2"]) > 1e-8


def test_mxfp8_backward_rounds_dy_along_H():
    # The GEMM2 dgrad reads dY quantised along H. With W2 exact along H, that is the only
    # rounding before da, db and dlogits, so with a dout that is NOT exact along H the emulated
    # backward must give exactly what the float64 backward gives for dout rounded along H first
    # (and visibly not what it gives for the unrounded dout).
    rng = np.random.default_rng(29)
    T, H, F, E, k = 64, 64, 64, 4, 2
    x = rng.standard_normal((T, H))
    W1 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W3 = np.stack([_axis_structured(rng, (H, F), 1) for _ in range(E)])
    W2 = np.stack([_axis_structured(rng, (F, H), 1) for _ in range(E)])
    Wr = rng.standard_normal((H, E)) * 0.3
    dout = rng.standard_normal((T, H))
    dq = O.mx_roundtrip(dout, 1)
    assert (dq != dout).any()
    f64 = O.forward(x, Wr, None, W1, W3, W2, k)
    gq = O.backward(f64, dq, x, Wr, W1, W3, W2)
    g64 = O.backward(f64, dout, x, Wr, W1, W3, W2)
    gmx = O.backward(dict(f64, precision="mxfp8"), dout, x, Wr, W1, W3, W2)
    for key in ("da", "db", "dlogits"):
        np.testing.assert_array_equal(gmx[key], gq[key], err_msg=key)
    assert O.max_abs_rel(g64["da"], gq["da"]) > 1e-6
