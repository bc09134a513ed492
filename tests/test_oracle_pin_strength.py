"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a scratch copy of oracle/moe_oracle.py (a
dropped term, a wrong sign, index or axis, a swapped operand), loads the copy
as its own module, points the pin that should notice it at the copy, and
requires the pin to fail (a failed check, or an error the mistake provokes).
The unmodified copy must pass the same pins, so a failure comes from the
planted mistake and nothing else."""
import importlib.util
import os

import pytest

from tests import test_oracle_ffn_grad as FG
from tests import test_oracle_mxfp8 as MX
from tests import test_oracle_nvfp4 as NV
from tests import test_oracle_router_schedule as RS

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "moe_oracle.py")

SCHED_CASES = [(1, 1, 1, 0), (37, 5, 2, 0), (64, 8, 3, 10), (50, 4, 4, 7), (33, 16, 1, 0), (30, 6, 2, 100)]


def _pins(module, *names):
    def run():
        for n in names:
            fn = getattr(module, n)
            if n == "test_schedule_matches_bruteforce":
                for case in SCHED_CASES:
                    fn(*case)
            elif n in ("test_forward_equals_dense_masked", "test_gradients_match_central_differences"):
                for macro in (0, 3):
                    fn(macro)
            elif n == "test_mxfp8_weight_gradient_quantises_along_the_token_axis":
                for macro in (0, 24):
                    fn(macro)
            else:
                fn()
    return module, run


ROUTER = _pins(RS, "test_router_zero_weights_pins_tie_break", "test_router_bias_only_closed_form",
               "test_router_two_expert_closed_form", "test_router_k_equals_E_weights_are_probs")
SCHED = _pins(RS, "test_schedule_matches_bruteforce")
FFN = _pins(FG, "test_forward_equals_dense_masked")
GRAD = _pins(FG, "test_gradients_match_central_differences")
MXF = _pins(MX, "test_mxfp8_forward_quantises_each_operand_along_its_contraction_axis")
MXB = _pins(MX, "test_mxfp8_backward_dgrads_quantise_along_their_contraction_axes")
MXW = _pins(MX, "test_mxfp8_weight_gradient_quantises_along_the_token_axis")
MXW2H = _pins(MX, "test_mxfp8_dW2_rounds_hw_along_the_token_axis")
MXW2G = _pins(MX, "test_mxfp8_dW2_rounds_dy_along_the_token_axis")
MXDY = _pins(MX, "test_mxfp8_backward_rounds_dy_along_H")
MXRT = _pins(MX, "test_roundtrip_equals_dequantised_codes")
NVQ = _pins(NV, "test_e2m1_golden_codes", "test_e2m1_round_matches_exhaustive_nearest_even",
            "test_matrix_scale_closed_form", "test_nv_block_properties")
NVL = _pins(NV, "test_nvfp4_layer_quantises_each_weight_along_its_contraction_axis")

# (what the mistake is, text in the oracle, its replacement, the pins that must notice it)
MUTATIONS = [
    ("top-k ties to the higher index", 'order = np.argsort(-p, axis=1, kind="stable")',
     'order = np.argsort(p, axis=1, kind="stable")[:, ::-1]', ROUTER),
    ("weights not renormalised", "w = psel / psel.sum(axis=1, keepdims=True)", "w = psel", ROUTER),
    ("bias subtracted", "logits = logits + np.asarray(bias, np.float64)[None, :]",
     "logits = logits - np.asarray(bias, np.float64)[None, :]", ROUTER),
    ("silu with the wrong sign", "return a / (1.0 + np.exp(-a))", "return a / (1.0 + np.exp(a))", FFN),
    ("gate on the wrong branch", "h[s0:s1] = silu(a[s0:s1]) * b[s0:s1]", "h[s0:s1] = silu(b[s0:s1]) * a[s0:s1]", FFN),
    ("combine weight of slot 0 for every slot", 'out += r["w"][:, j:j + 1] * Y[s2s[:, j]]',
     'out += r["w"][:, 0:1] * Y[s2s[:, j]]', FFN),
    ("dispatched token index wrong", 'tok = sch["sorted_to_slot"].astype(np.int64) // k',
     'tok = sch["sorted_to_slot"].astype(np.int64) % k', FFN),
    ("dw from a instead of h", "dwrow[s0:s1] = np.sum(G * he, axis=1)", "dwrow[s0:s1] = np.sum(G * ae, axis=1)", GRAD),
    ("dh without the routing weight", "dh = wrow[s0:s1, None] * G", "dh = G", GRAD),
    ("sign flip in da", "da = dh * be * sg * (1.0 + ae * (1.0 - sg))", "da = dh * be * sg * (1.0 - ae * (1.0 - sg))", GRAD),
    ("db without sigmoid", "db = dh * ae * sg", "db = dh * ae", GRAD),
    ("dW2 from da instead of h.w", "dW2[e] = hwe.T @ Ge", "dW2[e] = dae.T @ Ge", GRAD),
    ("reverse dispatch sums slot 0 only", "dx += dX[s2s[:, j]]", "dx += dX[s2s[:, 0]]", GRAD),
    ("router backward without 1/S", "dpsel = (dw - np.sum(wsel * dw, axis=1, keepdims=True)) / S",
     "dpsel = (dw - np.sum(wsel * dw, axis=1, keepdims=True))", GRAD),
    ("schedule order reversed within a key", 'sorted_to_slot = np.argsort(key, kind="stable")',
     "sorted_to_slot = np.argsort(key * R + (R - 1 - slot))", SCHED),
    ("macrobatch from the slot, not the token", "m = (slot // k) // Mb", "m = slot // Mb", SCHED),
    ("expert-major schedule key", "key = m * E + ids.reshape(-1).astype(np.int64)",
     "key = ids.reshape(-1).astype(np.int64) * nM + m", SCHED),
    ("run end off by one", "offsets[mm, E] = flat[(mm + 1) * E]", "offsets[mm, E] = flat[(mm + 1) * E] - 1", SCHED),
    ("MXFP8: W1 along F in the forward", "W1e = mx_roundtrip(W1e, 0)", "W1e = mx_roundtrip(W1e, 1)", MXF),
    ("MXFP8: W2 along H in the forward", "W2e = mx_roundtrip(W2e, 0)", "W2e = mx_roundtrip(W2e, 1)", MXF),
    ("MXFP8: h not rounded", "he = mx_roundtrip(h[s0:s1], 1) if mx else h[s0:s1]", "he = h[s0:s1]", MXF),
    ("MXFP8: x along the tokens", "Xe = mx_roundtrip(Xe, 1)", "Xe = mx_roundtrip(Xe.T.copy(), 1).T", MXF),
    ("MXFP8: W2 along F in the dgrad", "W2e = mx_roundtrip(W2e, 1)     # K = H", "W2e = mx_roundtrip(W2e, 0)     # K = H", MXB),
    ("MXFP8: da not rounded for dX", "dX[s0:s1] = mx_roundtrip(da, 1) @", "dX[s0:s1] = da @", MXB),
    ("MXFP8: W3 along H in the dgrad", "W3e = mx_roundtrip(W3e, 1)     # K = F",
     "W3e = mx_roundtrip(W3e, 0)     # K = F", MXB),
    ("MXFP8: da not rounded for dW1", "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), q(hwe), q(Ge)",
     "Xe, dae, dbe, hwe, Ge = q(Xe), dae, q(dbe), q(hwe), q(Ge)", MXW),
    ("MXFP8: X along H for dW1", "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), q(hwe), q(Ge)",
     "Xe, dae, dbe, hwe, Ge = mx_roundtrip(Xe, 1), q(dae), q(dbe), q(hwe), q(Ge)", MXW),
    ("weight gradients from each expert's first run only",
     "idx = np.concatenate([np.arange(s0, s1) for s0, s1 in es])",
     "idx = np.concatenate([np.arange(s0, s1) for s0, s1 in es[:1]])", GRAD),
    ("MXFP8: h.w not rounded for dW2", "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), q(hwe), q(Ge)",
     "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), hwe, q(Ge)", MXW2H),
    ("MXFP8: dY not rounded for dW2", "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), q(hwe), q(Ge)",
     "Xe, dae, dbe, hwe, Ge = q(Xe), q(dae), q(dbe), q(hwe), Ge", MXW2G),
    ("MXFP8: token-axis blocks start at the expert's first run, not at each run",
     "starts.append(pos); pos += s1 - s0; ends.append(pos)",
     "starts.append(0); pos += s1 - s0; ends.append(pos)", MXW),
    ("MXFP8: dY not rounded along H for the GEMM2 dgrad", "G = mx_roundtrip(Ge, 1) @ W2e.T",
     "G = Ge @ W2e.T", MXDY),
    ("NVFP4: E2M1 ties away from zero", "q = np.minimum(np.round(a / quantum) * quantum, E2M1_MAX)",
     "q = np.minimum(np.floor(a / quantum + 0.5) * quantum, E2M1_MAX)", NVQ),
    ("NVFP4: E2M1 spacing of 1 from 1.5 on", "quantum = np.where(a < 2.0, 0.5,", "quantum = np.where(a < 1.5, 0.5,", NVQ),
    ("NVFP4: no saturation at 6", "q = np.minimum(np.round(a / quantum) * quantum, E2M1_MAX)",
     "q = np.round(a / quantum) * quantum", NVQ),
    ("NVFP4: matrix scale rounded down", "return math.ldexp(1.0, ex - 1) if mant == 0.5 else math.ldexp(1.0, ex)",
     "return math.ldexp(1.0, ex - 1)", NVQ),
    ("NVFP4: block scale without the matrix scale", "s = e4m3_round(np.abs(blk).max(axis=-1) / (E2M1_MAX * g))",
     "s = e4m3_round(np.abs(blk).max(axis=-1) / E2M1_MAX)", NVQ),
    ("NVFP4: blocks of 32", "NV_BLOCK = 16", "NV_BLOCK = 32", NVQ),
    ("NVFP4: W1 along F", "W1e = nv_roundtrip(W1e, 0)", "W1e = nv_roundtrip(W1e, 1)", NVL),
    ("NVFP4: W2 along H", "W2e = nv_roundtrip(W2e, 0)", "W2e = nv_roundtrip(W2e, 1)", NVL),
    ("NVFP4: W3 not quantised", "W3e = nv_roundtrip(W3e, 0)", "W3e = W3e", NVL),
    ("MXFP8: round trip without the block scale", "out = (e4m3_round(blk / scale) * scale).reshape(v.shape)",
     "out = e4m3_round(blk).reshape(v.shape)", MXRT),
]


def _load(tmp_path, name, text):
    path = tmp_path / f"{name}.py"
    path.write_text(text)
    spec = importlib.util.spec_from_file_location(name, str(path))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("what,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pin_catches_planted_mistake(tmp_path, monkeypatch, what, old, new, pins):
    src = open(ORACLE).read()
    assert src.count(old) >= 1, f"the oracle no longer contains: {old}"
    module, run = pins
    monkeypatch.setattr(module, "O", _load(tmp_path, "oracle_copy", src))
    run()                                                     # the unmodified copy passes
    monkeypatch.setattr(module, "O", _load(tmp_path, "oracle_mutant", src.replace(old, new, 1)))
    with pytest.raises(Exception):                           # a failed check, or a crash
        run()
