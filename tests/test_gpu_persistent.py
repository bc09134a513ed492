"""The persistent forward against the one-launch-per-stage forward (run on a GB300).

Both forwards do the same arithmetic on the same rows in the same order (the
persistent one only changes when a tile may start), so out, the router's ids
and weights, and every backward result computed from each forward's saved
context must be identical bytes; the persistent forward is also compared with
the oracle by every other GPU test, which runs it by default."""
import numpy as np
import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    assert torch.cuda.is_available()


def G():
    import tests.gpu_common as g
    return g


def both_modes(w, inp, backward=True, **kw):
    import mixture_experts_layer_sum_gb300.moe as M
    out = []
    for mode in (M.MOE_FORWARD_PERSISTENT, M.MOE_FORWARD_PER_STAGE):
        M.moe_profile_begin()
        r = G().run_gpu(w, inp, backward=backward, forward_mode=mode, **kw)
        names = {n for n, _, _ in M.moe_profile_end()}
        out.append((r, names))
    (p, pn), (s, sn) = out
    assert "forward_persistent" in pn and "grouped_gemm_fwd1_swiglu" not in pn, pn
    assert "grouped_gemm_fwd1_swiglu" in sn and "forward_persistent" not in sn, sn
    keys = ("out", "ids", "w") + (("dx", "dWr", "dW1", "dW3", "dW2") if backward else ())
    for key in keys:
        np.testing.assert_array_equal(p[key], s[key], err_msg=key)
    return p


@pytest.mark.parametrize("macro", [0, 100, 33])
def test_persistent_equals_per_stage_bf16(macro):
    w = WL.TINY
    inp = WL.make_inputs(w)
    p = both_modes(w, inp, macrobatch_tokens=macro)
    G().check_layer(w, inp, p, macrobatch_tokens=macro)


@pytest.mark.parametrize("macro", [0, 100])
def test_persistent_equals_per_stage_mxfp8(macro):
    w = WL.Workload("mx_small", T=300, H=512, E=8, k=2, F=512, precision="mxfp8", zipf_s=0.8)
    inp = WL.make_inputs(w)
    p = both_modes(w, inp, macrobatch_tokens=macro)
    G().check_layer(w, inp, p, macrobatch_tokens=macro)


def test_persistent_equals_per_stage_balanced_full_size():
    w = WL.BALANCED
    both_modes(w, WL.make_inputs(w), backward=False)


def test_persistent_equals_per_stage_ring_full_size():
    # four macrobatches through the 256 MiB token ring: every hand-off between macrobatches
    w = WL.RING
    p = both_modes(w, WL.make_inputs(w), backward=False, ring_bytes=w.ring_bytes)
    assert p["layer"].plan.num_macrobatches > 2
