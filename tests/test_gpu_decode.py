"""Decode-shaped forward (few bf16 tokens) on a GB300.

With T <= 128 tokens in one macrobatch the forward runs the decode kernel: the
weights are the M operand and each expert's routed rows (at most T) the N
operand, so every expert's weights stream from HBM once. Checked against the
float64 oracle: out (forward) and, through the generic backward that reads the
decode forward's saved context, every gradient."""
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


def run_profiled(w, inp, **kw):
    import mixture_experts_layer_sum_gb300.moe as M
    M.moe_profile_begin()
    gpu = G().run_gpu(w, inp, **kw)
    names = {n for n, _, _ in M.moe_profile_end()}
    return gpu, names


@pytest.mark.parametrize("base,T", [(WL.BALANCED, 1), (WL.BALANCED, 8), (WL.BALANCED, 64), (WL.BALANCED, 128),
                                    (WL.TINY, 64), (WL.SKEWED, 64)])
def test_decode_forward_matches_oracle(base, T):
    w = base.with_(T=T)
    inp = WL.make_inputs(base, tokens=T)      # the workload's first T tokens
    gpu, names = run_profiled(w, inp)
    assert "decode_ffn" in names and "grouped_gemm_fwd1_swiglu" not in names, names
    errs = G().check_layer(w, inp, gpu)
    print("decode", base.name, T, errs)


def test_decode_equals_grouped_path_within_rounding():
    # the same 64 tokens through the grouped GEMMs (two macrobatches force that path): both are
    # within the forward tolerance of the oracle and of each other
    w = WL.BALANCED.with_(T=64)
    inp = WL.make_inputs(WL.BALANCED, tokens=64)
    dec, n1 = run_profiled(w, inp, backward=False)
    grp, n2 = run_profiled(w, inp, backward=False, macrobatch_tokens=32)
    assert "decode_ffn" in n1 and "decode_ffn" not in n2
    np.testing.assert_array_equal(dec["ids"], grp["ids"])
    assert O.max_abs_rel(dec["out"], grp["out"]) < 1e-2


def test_decode_deterministic():
    w = WL.BALANCED.with_(T=64)
    inp = WL.make_inputs(WL.BALANCED, tokens=64)
    a = G().run_gpu(w, inp)
    b = G().run_gpu(w, inp)
    for key in ("out", "dx", "dWr", "dW1", "dW3", "dW2"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


@pytest.mark.parametrize("base", [WL.BALANCED, WL.SKEWED])
def test_router_does_not_depend_on_batch_size(base):
    # a batch of a few router blocks loads four steps ahead, a full one a single step; the MMAs
    # run in the same order, so the first 64 tokens get bitwise the same ids and weights
    small = G().run_gpu(base.with_(T=64), WL.make_inputs(base, tokens=64), backward=False)
    full = G().run_gpu(base, WL.make_inputs(base), backward=False)
    np.testing.assert_array_equal(small["ids"], full["ids"][:64])
    np.testing.assert_array_equal(small["w"], full["w"][:64])
