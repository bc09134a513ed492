"""GPU parity of the MXFP8 path (run on a GB300).

- moe_quantize_weights: E4M3 codes and E8M0 scales of all six weight copies
  are bit-exact against the oracle's quantiser (same blocks, same rounding).
- forward + backward against the oracle run with the same MXFP8 quantisation
  emulated at the same points: max-abs-relative error below 6e-2."""
import os

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


def atoms_to_rows(sf_bytes, rows, K):
    return G().atoms_to_rows(sf_bytes, rows, K)


def test_quantize_weights_bit_exact():
    w = WL.Workload("mx_small", T=64, H=256, E=4, k=2, F=512, precision="mxfp8")
    inp = WL.make_inputs(w)
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    d = G().device_inputs(inp)
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, "mxfp8")
    layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    layer.status()
    qw = layer.qweights.cpu().numpy()
    E, H, F = w.E, w.H, w.F
    n = E * H * F
    # layout: six (codes, scales) pairs, each region 1024-aligned, base aligned inside the buffer
    ptr = layer.qweights.data_ptr()
    start = (-ptr) % 1024
    offs = []
    o = 0
    for _ in range(6):
        c = o; o = -(-(o + n) // 1024) * 1024
        s_ = o; o = -(-(o + n // 32) // 1024) * 1024
        offs.append((start + c, start + s_))
    W = {k: O.bf16_to_f64(inp[k]) for k in ("W1", "W3", "W2")}
    cases = [("W1", True, H, F), ("W3", True, H, F), ("W2", True, F, H),
             ("W2", False, F, H), ("W1", False, H, F), ("W3", False, H, F)]
    for i, (name, transposed, R, C) in enumerate(cases):
        codes = qw[offs[i][0]:offs[i][0] + n]
        sf = qw[offs[i][1]:offs[i][1] + n // 32]
        for e in range(E):
            if transposed:      # stored [C][R], blocks along R
                ref_c, ref_s = O.mx_quantize(W[name][e].T, 1)
                got_c = codes[e * C * R:(e + 1) * C * R].reshape(C, R)
                got_s = atoms_to_rows(sf[e * C * R // 32:(e + 1) * C * R // 32], C, R)
            else:               # stored [R][C], blocks along C
                ref_c, ref_s = O.mx_quantize(W[name][e], 1)
                got_c = codes[e * R * C:(e + 1) * R * C].reshape(R, C)
                got_s = atoms_to_rows(sf[e * R * C // 32:(e + 1) * R * C // 32], R, C)
            np.testing.assert_array_equal(got_s, ref_s, err_msg=f"{name} scales e={e} transposed={transposed}")
            np.testing.assert_array_equal(got_c, ref_c, err_msg=f"{name} codes e={e} transposed={transposed}")


@pytest.mark.parametrize("T,macro", [(300, 0), (300, 100), (1, 0)])
def test_mxfp8_fwd_bwd_small(T, macro):
    w = WL.Workload("mx_small", T=T, H=512, E=8, k=2, F=512, precision="mxfp8", zipf_s=0.8)
    inp = WL.make_inputs(w)
    gpu = G().run_gpu(w, inp, macrobatch_tokens=macro)
    errs = G().check_layer(w, inp, gpu, macrobatch_tokens=macro)
    print("mxfp8 small", T, macro, errs)


def test_mxfp8_workload_shape_reduced_tokens():
    # H=7168, F=2048 (the pages' shape), E=16, k=8, Zipf(0.8) skew, first 256 tokens
    w = WL.MXFP8
    inp = WL.make_inputs(w, tokens=256)
    w = w.with_(T=256)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("mxfp8 7168x2048 T=256", errs)


def test_mxfp8_deterministic():
    w = WL.Workload("mx_small", T=200, H=512, E=8, k=2, F=512, precision="mxfp8")
    inp = WL.make_inputs(w)
    a = G().run_gpu(w, inp)
    b = G().run_gpu(w, inp)
    for key in ("out", "dx", "dWr", "dW1", "dW3", "dW2"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def _check_sampled_tokens(w, inp, gpu, n, seed):
    # out and dx of a token depend only on that token's rows: its x and dout rows
    # are quantised along H, its routed rows' h, da, db along F, and the weight
    # copies are fixed, so the oracle (same quantisation emulated) runs on the sample
    sample = np.sort(np.random.default_rng(seed).choice(w.T, n, replace=False))
    sub = {k: (v[sample] if k in ("x", "dout") else v) for k, v in inp.items()}
    oi = G().oracle_inputs(sub)
    args = (oi["x"], oi["Wr"], oi["bias"], oi["W1"], oi["W3"], oi["W2"], w.k)
    r = O.router(oi["x"], oi["Wr"], oi["bias"], w.k)   # ids checked against the router alone
    ids, _ = G().reconcile_ids(gpu["ids"][sample].astype(np.int32), r, w.k)
    wc = G().weight_caches(w)
    f = O.forward(*args, precision="mxfp8", ids=ids, weight_cache=wc[0])
    errs = {"out": O.max_abs_rel(gpu["out"][sample], f["out"])}
    g = O.backward(f, oi["dout"], oi["x"], oi["Wr"], oi["W1"], oi["W3"], oi["W2"], weight_cache=wc[1])
    errs["dx"] = O.max_abs_rel(gpu["dx"][sample], g["dx"])
    assert errs["out"] < G().MX_TOL and errs["dx"] < G().MX_TOL, errs
    return errs


_INPUTS = {}


def _inputs(w):
    # the full-size workloads' inputs are drawn once per test session (about 10^9 samples each)
    if w.name not in _INPUTS:
        _INPUTS.clear()
        _INPUTS[w.name] = WL.make_inputs(w)
    return _INPUTS[w.name]


def test_mxfp8_full_size_every_output():
    # the MXFP8 workload at full size (T=8192, H=7168, E=16, k=8, F=2048) in the launch
    # configuration the bench times: out, dx, dW_r and the three weight gradients element by
    # element against the oracle run with the same quantisation emulated; sampled tokens too
    w = WL.MXFP8
    inp = _inputs(w)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("mxfp8 full size", errs)
    errs = _check_sampled_tokens(w, inp, gpu, 48, 3)
    print("mxfp8 full size, sampled", errs)


def test_ring_full_size_sampled_tokens():
    # T=16384 through the 256 MiB ring: many macrobatches through the one ring, minibatch at
    # the wave rule; forward and dx of sampled tokens
    w = WL.RING
    inp = _inputs(w)
    gpu = G().run_gpu(w, inp, ring_bytes=w.ring_bytes)
    assert gpu["layer"].plan.num_macrobatches > 2
    errs = _check_sampled_tokens(w, inp, gpu, 48, 4)
    print("ring full size, sampled", gpu["layer"].plan.num_macrobatches, "macrobatches", errs)


def test_ring_minibatch_sizes_bitwise_equal():
    # the ring workload's forward at every minibatch size of its sweep and at the wave rule:
    # the minibatch only decides when a GEMM1 tile may start, never a row's arithmetic, so out
    # (and the router's ids and weights) must be identical bytes
    w = WL.RING
    inp = _inputs(w)
    d = G().device_inputs({k: inp[k] for k in ("x", "Wr", "W1", "W3", "W2", "bias")})
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    ref = None
    for mb in (0,) + tuple(w.minibatch_rows):
        layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, "mxfp8", ring_bytes=w.ring_bytes, minibatch_rows=mb)
        layer.quantize_weights(d["W1"], d["W3"], d["W2"])
        out, ids, wts = layer.forward(d["x"], d["Wr"], d["bias"], d["W1"], d["W3"], d["W2"])
        layer.status()
        got = (out.view(torch.int16).cpu(), ids.cpu(), wts.cpu())
        if ref is None:
            ref = got
            assert layer.plan.num_macrobatches > 2
        else:
            for a, b in zip(ref, got):
                assert torch.equal(a, b), mb
        del layer
        torch.cuda.empty_cache()


def _host_memory_gb():
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES") / 1e9
    except (ValueError, OSError, AttributeError):
        return 0.0


@pytest.mark.skipif(bool(os.environ.get("MOE_SKIP_SLOW_TESTS")) or _host_memory_gb() < 150,
                    reason="needs about 100 GB of host memory for the float64 oracle (MOE_SKIP_SLOW_TESTS unset)")
def test_ring_full_size_every_output():
    # the ring workload with every output compared element by element against the oracle run
    # with the same quantisation emulated (its float64 arrays take about 100 GB of host memory;
    # about four minutes on a 16-core host)
    w = WL.RING
    inp = _inputs(w)
    gpu = G().run_gpu(w, inp, ring_bytes=w.ring_bytes)
    Mb = gpu["layer"].plan.macrobatch_tokens
    errs = G().check_layer(w, inp, gpu, macrobatch_tokens=Mb)
    print("ring full size", gpu["layer"].plan.num_macrobatches, "macrobatches", errs)
