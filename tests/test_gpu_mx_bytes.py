"""MXFP8 activation bytes made on the GPU, compared with the oracle's quantiser
(run on a GB300).

The quantised copies of the dispatched x rows (the gather inside GEMM1), of dY
along H (the reverse combine) and of every token-axis operand of the weight
gradients come from bf16 values the test also has, so their E4M3 codes and
E8M0 scales must equal the oracle's byte for byte. GEMM1's h and the GEMM2
dgrad's da, db are quantised from fp32 values the GPU computed; the test
rebuilds them in float64 from the GPU's own saved inputs and requires the
oracle's bytes wherever that reference decides them (a value not within its
error bound of a rounding or scale boundary)."""
import numpy as np
import pytest
import torch

import workloads as WL
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    assert torch.cuda.is_available()


def G():
    import tests.gpu_common as g
    return g


def _padded_rows(src64, row_slot, k):
    """The expert-sorted padded rows of a token tensor: row r holds src[slot // k], padding 0."""
    out = np.zeros((len(row_slot), src64.shape[1]))
    real = row_slot >= 0
    out[real] = src64[row_slot[real] // k]
    return out


@pytest.mark.parametrize("T", [300, 1000])
def test_mxfp8_activation_bytes_match_oracle_quantiser(T):
    g = G()
    w = WL.Workload("mx_bytes", T=T, H=512, E=8, k=2, F=512, precision="mxfp8", zipf_s=0.8)
    inp = WL.make_inputs(w)
    d = g.device_inputs(inp)
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, "mxfp8")
    assert layer.plan.num_macrobatches == 1
    layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    out, ids, wts = layer.forward(d["x"], d["Wr"], d["bias"], d["W1"], d["W3"], d["W2"])
    layer.status()
    H, F, E, k = w.H, w.F, w.E, w.k
    rp = layer.plan.rows_padded_max
    offp = g.u8(layer.buffer("PADDED_OFFSETS")).view(np.int32)
    end = int(offp[E])
    row_slot = g.u8(layer.buffer("ROW_SLOT")).view(np.int32)[:end]
    x64, dout64 = O.bf16_to_f64(inp["x"]), O.bf16_to_f64(inp["dout"])
    Xpad = _padded_rows(x64, row_slot, k)

    # the gather's x rows along H (ring row = padded row: one macrobatch)
    codes = g.u8(layer.buffer("RING_X"))[:end * H].reshape(end, H)
    sf = g.atoms_to_rows(g.u8(layer.buffer("RING_X_SCALES")), end, H)
    rc, rs = O.mx_quantize(Xpad, 1)
    np.testing.assert_array_equal(sf, rs, err_msg="x scales")
    np.testing.assert_array_equal(codes, rc, err_msg="x codes")

    # GEMM1's h along F, from the GPU's saved bf16 a, b
    a = g.bf16_blocks(layer.buffer("A"), rp, F, end)
    b = g.bf16_blocks(layer.buffer("B"), rp, F, end)
    h64 = O.silu(a) * b
    hc = g.u8(layer.buffer("RING_H"))[:end * F].reshape(end, F)
    hs = g.atoms_to_rows(g.u8(layer.buffer("RING_H_SCALES")), end, F)
    und = g.check_mx_decided(hc, hs, h64, 1, rel=1e-5)
    assert und[1] < 0.05 * h64.size, und

    dx, dWr, dW1, dW3, dW2 = layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"])
    layer.status()
    Dpad = _padded_rows(dout64, row_slot, k)

    # dY rows along H (the GEMM2 dgrad's A operand)
    rc, rs = O.mx_quantize(Dpad, 1)
    np.testing.assert_array_equal(g.atoms_to_rows(g.u8(layer.buffer("DY_ROWS_SCALES")), end, H), rs)
    np.testing.assert_array_equal(g.u8(layer.buffer("DY_ROWS"))[:end * H].reshape(end, H), rc)

    # token-axis operands x and dY, gathered from the inputs: blocks of 32 rows start at every
    # run (runs start at multiples of 128)
    def tokens(name, C):
        c = g.u8(layer.buffer(name)).reshape(C, rp)[:, :end]
        s = g.atoms_to_rows(g.u8(layer.buffer(name + "_SCALES")), C, rp)[:, :end // 32]
        return c, s

    for name, ref in (("X_TOKENS", Xpad), ("DY_TOKENS", Dpad)):
        c, s = tokens(name, ref.shape[1])
        rc, rs = O.mx_quantize(ref, 0)
        np.testing.assert_array_equal(s, rs.T, err_msg=name + " scales")
        np.testing.assert_array_equal(c, rc.T, err_msg=name + " codes")

    # the GEMM2 dgrad epilogue's da, db along F: G = dY (quantised along H) times W2 (quantised
    # along H) accumulated in fp32 on the GPU; the reference forms it in float64
    W2 = O.bf16_to_f64(inp["W2"])
    wslot = g.dev_to_np(wts).reshape(-1)
    wrow = np.where(row_slot >= 0, wslot[np.maximum(row_slot, 0)], 0.0)
    Gq = O.mx_roundtrip(Dpad, 1)
    Gm = np.zeros((end, F))
    for e in range(E):
        s0, s1 = int(offp[e]), int(offp[e + 1])
        if s1 > s0:
            Gm[s0:s1] = Gq[s0:s1] @ O.mx_roundtrip(W2[e], 1).T
    sg = O.sigmoid(a)
    dh = wrow[:, None] * Gm
    da = dh * b * sg * (1.0 + a * (1.0 - sg))
    db = dh * O.silu(a)
    for name, ref in (("DA_ROWS", da), ("DB_ROWS", db)):
        c = g.u8(layer.buffer(name))[:end * F].reshape(end, F)
        s = g.atoms_to_rows(g.u8(layer.buffer(name + "_SCALES")), end, F)
        # fp32 accumulation over H on the GPU: a looser bound than h's, so more values sit near a
        # midpoint; at least 85 % of the codes are still decided and compared exactly
        und = g.check_mx_decided(c, s, ref, 1, rel=1e-4)
        assert und[1] < 0.15 * ref.size, (name, und)
    # the same epilogue's da, db rounded to bf16 and quantised along the padded rows (blocks of
    # 32 rows: a warp's rows), the dW1/dW3 operands
    for name, ref in (("DA_TOKENS", da), ("DB_TOKENS", db)):
        c, s = tokens(name, F)
        und = g.check_mx_decided(c.T, s.T, ref, 0, rel=1e-4, bf16_values=True)
        assert und[1] < 0.2 * ref.size, (name, und)
    # and h.w, the dW2 operand: h = bf16(silu(a) b) recomputed from the saved a, b in fp32 (within
    # 1e-5 of float64), w h rounded to bf16
    dlt = 1e-5 * np.abs(h64)
    wcol = wrow[:, None]
    hw_lo = g.bf16_round(wcol * g.bf16_round(h64 - dlt))
    hw_hi = g.bf16_round(wcol * g.bf16_round(h64 + dlt))
    c, s = tokens("HW_TOKENS", F)
    und = g.check_mx_interval(c.T, s.T, hw_lo, hw_hi, 0)
    assert und[1] < 0.05 * hw_lo.size, ("HW_TOKENS", und)
