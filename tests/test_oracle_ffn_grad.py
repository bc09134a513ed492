"""Pins of the oracle's forward (expert FFN + combine) and backward:
a dense evaluation of every expert masked by routing, textbook special cases
(E=1 dense SwiGLU via torch's own silu, identical experts, zero input,
linearity in W2) and central finite differences of every gradient."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def rand_layer(seed, T, H, E, F, wstd=0.3, rstd=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    Wr = rng.standard_normal((H, E)) * rstd
    W1 = rng.standard_normal((E, H, F)) * wstd
    W3 = rng.standard_normal((E, H, F)) * wstd
    W2 = rng.standard_normal((E, F, H)) * wstd
    return x, Wr, W1, W3, W2


def dense_masked(x, Wr, bias, W1, W3, W2, k):
    """Every expert on every token; weight = renormalised prob if selected, else 0."""
    T = x.shape[0]
    E = Wr.shape[1]
    xt = torch.from_numpy(x)
    out = torch.zeros_like(xt)
    logits = xt @ torch.from_numpy(Wr)
    if bias is not None:
        logits = logits + torch.from_numpy(bias)
    p = torch.softmax(logits, dim=1)
    for t in range(T):
        chosen = sorted(range(E), key=lambda e: (-p[t, e].item(), e))[:k]
        S = sum(p[t, e].item() for e in chosen)
        for e in range(E):
            g = p[t, e].item() / S if e in chosen else 0.0
            hid = torch.nn.functional.silu(xt[t] @ torch.from_numpy(W1[e])) * (xt[t] @ torch.from_numpy(W3[e]))
            out[t] += g * (hid @ torch.from_numpy(W2[e]))
    return out.numpy()


@pytest.mark.parametrize("macro", [0, 3])
def test_forward_equals_dense_masked(macro):
    x, Wr, W1, W3, W2 = rand_layer(0, 11, 8, 5, 12)
    bias = np.linspace(-0.5, 0.5, 5)
    f = O.forward(x, Wr, bias, W1, W3, W2, 2, macrobatch_tokens=macro)
    ref = dense_masked(x, Wr, bias, W1, W3, W2, 2)
    np.testing.assert_allclose(f["out"], ref, rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu_ffn():
    x, Wr, W1, W3, W2 = rand_layer(1, 9, 16, 1, 24)
    f = O.forward(x, Wr, None, W1, W3, W2, 1)
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0])) * (xt @ torch.from_numpy(W3[0]))) @ torch.from_numpy(W2[0])
    np.testing.assert_allclose(f["out"], ref.numpy(), rtol=1e-12, atol=1e-13)
    assert (f["w"] == 1.0).all()


def test_identical_experts_reduce_to_dense_ffn():
    x, Wr, W1, W3, W2 = rand_layer(2, 10, 8, 6, 16)
    W1[:] = W1[0]; W3[:] = W3[0]; W2[:] = W2[0]
    f = O.forward(x, Wr, None, W1, W3, W2, 3)
    xt = torch.from_numpy(x)
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0])) * (xt @ torch.from_numpy(W3[0]))) @ torch.from_numpy(W2[0])
    np.testing.assert_allclose(f["out"], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_zero_input_gives_zero_output():
    x, Wr, W1, W3, W2 = rand_layer(3, 6, 8, 4, 8)
    f = O.forward(np.zeros_like(x), Wr, None, W1, W3, W2, 2)
    assert np.abs(f["out"]).max() == 0.0


def test_linear_in_W2():
    x, Wr, W1, W3, W2 = rand_layer(4, 6, 8, 4, 8)
    _, _, _, _, W2b = rand_layer(5, 6, 8, 4, 8)
    f1 = O.forward(x, Wr, None, W1, W3, W2, 2)["out"]
    f2 = O.forward(x, Wr, None, W1, W3, W2b, 2)["out"]
    f3 = O.forward(x, Wr, None, W1, W3, 2.0 * W2 - 3.0 * W2b, 2)["out"]
    np.testing.assert_allclose(f3, 2.0 * f1 - 3.0 * f2, rtol=1e-11, atol=1e-12)


def loss(x, Wr, bias, W1, W3, W2, k, dout, ids, macro=0):
    return float(np.sum(dout * O.forward(x, Wr, bias, W1, W3, W2, k, ids=ids, macrobatch_tokens=macro)["out"]))


@pytest.mark.parametrize("macro", [0, 3])
def test_gradients_match_central_differences(macro):
    # macro = 3 splits the 6 tokens into two macrobatches, so experts have one run of
    # sorted rows in each and the weight gradients must contract over both runs
    T, H, E, F, k = 6, 8, 4, 16, 2
    x, Wr, W1, W3, W2 = rand_layer(6, T, H, E, F, wstd=0.4, rstd=1.0)
    bias = np.array([0.3, -0.2, 0.1, 0.0])
    dout = np.random.default_rng(7).standard_normal((T, H))
    f = O.forward(x, Wr, bias, W1, W3, W2, k, macrobatch_tokens=macro)
    assert O.topk_margin(f["logits"], k).min() > 1e-3      # selection stays fixed under perturbation
    if macro:
        runs = np.bincount([e for e, _, _ in O.expert_segments(f)], minlength=E)
        assert runs.max() >= 2                              # some expert really has two runs
    g = O.backward(f, dout, x, Wr, W1, W3, W2)
    ids = f["ids"]
    eps = 1e-6
    params = {"x": x, "Wr": Wr, "W1": W1, "W3": W3, "W2": W2}
    grads = {"x": g["dx"], "Wr": g["dWr"], "W1": g["dW1"], "W3": g["dW3"], "W2": g["dW2"]}
    for name, P in params.items():
        num = np.zeros_like(P)
        it = np.nditer(P, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = P[i]
            P[i] = old + eps
            lp = loss(params["x"], params["Wr"], bias, params["W1"], params["W3"], params["W2"], k, dout, ids, macro)
            P[i] = old - eps
            lm = loss(params["x"], params["Wr"], bias, params["W1"], params["W3"], params["W2"], k, dout, ids, macro)
            P[i] = old
            num[i] = (lp - lm) / (2 * eps)
        scale = max(np.abs(num).max(), 1e-3)
        assert np.abs(num - grads[name]).max() / scale < 1e-6, name


def test_router_weight_gradient_vanishes_when_k_equals_E_and_experts_identical():
    # with k = E the weights are p and sum to one; identical experts make the
    # output independent of p, so dWr must be exactly the zero matrix (up to rounding)
    x, Wr, W1, W3, W2 = rand_layer(8, 5, 8, 3, 8)
    W1[:] = W1[0]; W3[:] = W3[0]; W2[:] = W2[0]
    f = O.forward(x, Wr, None, W1, W3, W2, 3)
    g = O.backward(f, np.ones((5, 8)), x, Wr, W1, W3, W2)
    assert np.abs(g["dWr"]).max() < 1e-12


def test_max_abs_rel_metric():
    assert O.max_abs_rel(np.array([1.0, 2.0]), np.array([1.0, 4.0])) == 0.5
    assert O.max_abs_rel(np.zeros(3), np.zeros(3)) == 0.0
