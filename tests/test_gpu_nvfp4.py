"""NVFP4 expert weights on a GB300: the quantised bytes against the oracle's quantiser (bit
exact), and the few-token forward that streams them against the oracle run with the same
NVFP4 weights."""
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


TILE = 4096 + 512   # one 128-column x 64-K tile: [128 rows][32 B] codes, then [128 rows][4 B] scales


def _unpack(buf, E, H, F):
    """(name, K, N, codes [E][N/128][K/64][128][32], scales [E][N/128][K/64][128][4]) of W1, W3, W2
    and the byte offset of the matrix scales, read from the NVFP4 buffer: W1 and W3 interleaved
    per 128-K stage ([E][F/128][H/128][W1 k, W1 k+64, W3 k, W3 k+64]), then W2
    ([E][H/128][F/128][k, k+64]), each part 1 KB aligned."""
    a1024 = lambda v: -(-v // 1024) * 1024
    tiles = E * (H // 64) * (F // 128)
    w13 = buf[:2 * tiles * TILE].reshape(E, F // 128, H // 128, 2, 2, TILE)
    o = a1024(2 * tiles * TILE)
    w2 = buf[o:o + tiles * TILE].reshape(E, H // 128, F // 64, TILE)
    gs = a1024(o + tiles * TILE)
    out = []
    for name, K, N, t in (("W1", H, F, w13[:, :, :, 0].reshape(E, F // 128, H // 64, TILE)),
                          ("W3", H, F, w13[:, :, :, 1].reshape(E, F // 128, H // 64, TILE)),
                          ("W2", F, H, w2)):
        codes = t[..., :4096].reshape(E, N // 128, K // 64, 128, 32)
        scales = t[..., 4096:].reshape(E, N // 128, K // 64, 128, 4)
        out.append((name, K, N, codes, scales))
    return out, gs


def test_nvfp4_weights_bit_exact():
    w = WL.Workload("nv_small", T=64, H=256, E=4, k=2, F=512, precision="nvfp4")
    inp = WL.make_inputs(w)
    d = G().device_inputs(inp)
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, "nvfp4")
    layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    layer.status()
    buf = layer.qweights.cpu().numpy()
    buf = buf[(-layer.qweights.data_ptr()) % 1024:]
    mats, gs_off = _unpack(buf, w.E, w.H, w.F)
    g_all = buf[gs_off:gs_off + 12 * w.E].view(np.float32).reshape(3, w.E)
    for mi, (name, K, N, packed, sc) in enumerate(mats):
        W = O.bf16_to_f64(inp[name])
        nib = np.stack([packed & 15, packed >> 4], axis=-1).reshape(w.E, N // 128, K // 64, 128, 64)
        codes = nib.transpose(0, 2, 4, 1, 3).reshape(w.E, K, N)          # [e][k][n]
        scales = sc.transpose(0, 2, 4, 1, 3).reshape(w.E, K // 16, N)
        for e in range(w.E):
            rc, rs, rg = O.nv_quantize(W[e], 0)
            assert g_all[mi, e] == rg, (name, e)
            np.testing.assert_array_equal(scales[e], rs, err_msg=f"{name} scales e={e}")
            np.testing.assert_array_equal(codes[e], rc, err_msg=f"{name} codes e={e}")


@pytest.mark.parametrize("T", [1, 16, 64, 128])
def test_nvfp4_decode_forward_matches_oracle(T):
    import mixture_experts_layer_sum_gb300.moe as M
    base = WL.BALANCED
    w = base.with_(T=T, precision="nvfp4")
    inp = WL.make_inputs(base, tokens=T)
    M.moe_profile_begin()
    gpu = G().run_gpu(w, inp, backward=False)
    names = {n for n, _, _ in M.moe_profile_end()}
    assert "decode_ffn_nvfp4" in names, names
    errs = G().check_layer(w, inp, gpu, backward=False)
    print("nvfp4 decode", T, errs)


def test_nvfp4_limits():
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    with pytest.raises(M.MoeError) as e:
        MoeLayer(200, 256, 512, 4, 2, "nvfp4")             # more tokens than the decode kernel takes
    assert e.value.status == M.MOE_ERR_UNSUPPORTED
    w = WL.Workload("nv_small", T=32, H=256, E=4, k=2, F=512, precision="nvfp4")
    inp = WL.make_inputs(w)
    d = G().device_inputs(inp)
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, "nvfp4")
    layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    layer.forward(d["x"], d["Wr"], None, d["W1"], d["W3"], d["W2"])
    with pytest.raises(M.MoeError) as e:
        layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"])
    assert e.value.status == M.MOE_ERR_UNSUPPORTED
    layer.status()
