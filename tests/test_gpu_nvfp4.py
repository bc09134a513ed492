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


def _matrices(E, H, F):
    """(name, K, N) of the three quantised matrix sets and their byte offsets, in buffer order."""
    a1024 = lambda v: -(-v // 1024) * 1024
    out, o = [], 0
    for name, K, N in (("W1", H, F), ("W3", H, F), ("W2", F, H)):
        n = E * K * N
        codes = o
        o = a1024(o + n // 2)
        scales = o
        o = a1024(o + n // 16)
        out.append((name, K, N, codes, scales))
    return out, o


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
    mats, gs_off = _matrices(w.E, w.H, w.F)
    g_all = buf[gs_off:gs_off + 12 * w.E].view(np.float32).reshape(3, w.E)
    for mi, (name, K, N, co, so) in enumerate(mats):
        W = O.bf16_to_f64(inp[name])
        n = w.E * K * N
        packed = buf[co:co + n // 2].reshape(w.E, N // 128, K // 64, 128, 32)
        nib = np.stack([packed & 15, packed >> 4], axis=-1).reshape(w.E, N // 128, K // 64, 128, 64)
        codes = nib.transpose(0, 2, 4, 1, 3).reshape(w.E, K, N)          # [e][k][n]
        sc = buf[so:so + n // 16].reshape(w.E, N // 128, K // 64, 128, 4)
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
