"""GPU parity of the CUDA layer against the float64 oracle (run on a GB300).

Indices are bit-exact (schedule) or equal up to near-ties (router); floats are
within max-abs-relative 1e-2 (forward) and 2e-2 (backward) of the oracle; the
combine and every gradient are bit-reproducible run to run."""
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


def test_tiny_forward_backward():
    w = WL.TINY
    inp = WL.make_inputs(w)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("tiny", errs)


@pytest.mark.parametrize("T", [1, 5, 77, 130])
def test_ragged_token_counts(T):
    w = WL.TINY
    inp = WL.make_inputs(w, tokens=T)
    gpu = G().run_gpu(w, inp)
    G().check_layer(w, inp, gpu)


def test_zero_tokens():
    w = WL.TINY
    inp = WL.make_inputs(w, tokens=0)
    d = G().device_inputs(inp)
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    layer = MoeLayer(0, w.H, w.F, w.E, w.k)
    layer.forward(d["x"], d["Wr"], None, d["W1"], d["W3"], d["W2"])
    dx, dWr, dW1, dW3, dW2 = layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"])
    layer.status()
    for t in (dWr, dW1, dW3, dW2):
        assert torch.count_nonzero(t).item() == 0


def test_macrobatches_match_single_pass():
    w = WL.TINY
    inp = WL.make_inputs(w)
    one = G().run_gpu(w, inp)
    many = G().run_gpu(w, inp, macrobatch_tokens=100)     # 3 macrobatches, last one ragged
    assert many["layer"].plan.num_macrobatches == 3
    # rows do not depend on the partition and the combine order is fixed: bitwise equal
    np.testing.assert_array_equal(one["out"], many["out"])
    np.testing.assert_array_equal(one["dx"], many["dx"])
    G().check_layer(w, inp, many, macrobatch_tokens=100)


def test_accumulate_adds_into_gradients():
    w = WL.TINY
    inp = WL.make_inputs(w)
    base = G().run_gpu(w, inp)
    init = {k: torch.full(s, 0.5, device="cuda") for k, s in
            (("dWr", (w.H, w.E)), ("dW1", (w.E, w.H, w.F)), ("dW3", (w.E, w.H, w.F)), ("dW2", (w.E, w.F, w.H)))}
    acc = G().run_gpu(w, inp, accumulate_into=init)
    for key in ("dWr", "dW1", "dW3", "dW2"):
        np.testing.assert_allclose(acc[key], base[key] + 0.5, rtol=0, atol=1e-6)


def test_single_expert_hot_and_empty_experts():
    # a huge bias on expert 3 and a large negative one elsewhere: experts with no rows
    w = WL.TINY.with_(zipf_s=None)
    inp = WL.make_inputs(w)
    inp["bias"] = np.full(w.E, -30.0, np.float32)
    inp["bias"][3] = 30.0
    inp["bias"][5] = 29.0
    gpu = G().run_gpu(w, inp)
    assert set(np.unique(gpu["ids"])) == {3, 5}
    G().check_layer(w, inp, gpu)
    for e in (0, 1, 2, 4, 6, 7):
        assert np.abs(gpu["dW1"][e]).max() == 0 and np.abs(gpu["dW2"][e]).max() == 0


def test_determinism_bitwise():
    w = WL.TINY.with_(T=200)
    inp = WL.make_inputs(w)
    a = G().run_gpu(w, inp)
    b = G().run_gpu(w, inp)
    for key in ("out", "ids", "w", "dx", "dWr", "dW1", "dW3", "dW2"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_schedule_bit_exact():
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    rng = np.random.default_rng(0)
    # the last three fit one macrobatch of at most eight 256-slot chunks: the one-block schedule
    for T, E, k, Mb in [(4096, 32, 4, 0), (1000, 64, 8, 300), (3, 8, 2, 0), (16384, 16, 8, 2000), (2049, 7, 3, 0),
                        (64, 32, 4, 0), (100, 7, 3, 0), (256, 64, 8, 0)]:
        # skewed ids: each token picks k distinct experts, Zipf-weighted
        pr = (np.arange(1, E + 1) ** -1.2); pr /= pr.sum()
        ids = np.stack([rng.choice(E, size=k, replace=False, p=pr) for _ in range(T)]).astype(np.int32)
        layer = MoeLayer(T, 256, 256, E, k, macrobatch_tokens=Mb)
        c, off, s2s, s2r = layer.schedule(torch.from_numpy(ids).cuda())
        layer.status()
        ref = O.schedule(ids, E, Mb)
        np.testing.assert_array_equal(c.cpu().numpy().reshape(ref["counts"].shape), ref["counts"])
        np.testing.assert_array_equal(off.cpu().numpy().reshape(ref["offsets"].shape), ref["offsets"])
        np.testing.assert_array_equal(s2s.cpu().numpy(), ref["sorted_to_slot"])
        np.testing.assert_array_equal(s2r.cpu().numpy(), ref["slot_to_sorted"])


def test_balanced_fwd_bwd_full_size():
    # the balanced workload at full size (T=4096, H=2048, E=32, k=4, F=1024) in the launch
    # configuration the bench times: out, dx and every weight gradient element by element
    w = WL.BALANCED
    inp = WL.make_inputs(w)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("balanced", errs)


def test_skewed_fwd_bwd_reduced_tokens():
    # the skewed-routing shape (E=64, k=8, H=4096, F=1536) on its first 1024 tokens:
    # every tile path, ragged experts, full oracle comparison of every gradient
    w = WL.SKEWED
    inp = WL.make_inputs(w, tokens=1024)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("skewed-1024", errs)


def test_skewed_fwd_bwd_full_size():
    # full T=8192 (65,536 routed rows, the hottest expert near the 8x-of-mean cap): out, dx and
    # every weight gradient element by element against the float64 oracle
    w = WL.SKEWED
    inp = WL.make_inputs(w)
    gpu = G().run_gpu(w, inp)
    errs = G().check_layer(w, inp, gpu)
    print("skewed full size", errs)
    counts = np.bincount(gpu["ids"].ravel(), minlength=w.E)
    assert counts.max() / counts.mean() > 4      # the skew really is skewed


@pytest.mark.parametrize("mb", [128, 384, 1 << 20])
def test_minibatch_sizes_bitwise_equal(mb):
    # the fused dispatch publishes rows minibatch by minibatch; no row's arithmetic
    # depends on the partition, so every minibatch size gives identical bytes
    w = WL.TINY
    inp = WL.make_inputs(w)
    base = G().run_gpu(w, inp, backward=False)
    other = G().run_gpu(w, inp, backward=False, minibatch_rows=mb, macrobatch_tokens=100)
    np.testing.assert_array_equal(base["out"], other["out"])
