"""Failure detection on the GPU without a GPU fault (run on a GB300).

A host-injected failure (config fault_mask MOE_FAULT_GEMM1_READY: the first
minibatch's ready counter is set so that it never reaches its target) makes
GEMM1's bounded wait run out. The device status word must report
MOE_ERR_TIMEOUT, every kernel must return (each wait is bounded and gives up
once the status word is set), the query clears the word, and the same CUDA
context must then run the layer correctly."""
import time

import pytest
import torch

import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("mode", [0, 1])   # the persistent forward, one launch per stage
def test_gemm1_wait_runs_out_and_context_survives(mode):
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    import tests.gpu_common as G
    w = WL.TINY
    inp = WL.make_inputs(w)
    d = G.device_inputs(inp)
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, timeout_ms=100, fault_mask=M.MOE_FAULT_GEMM1_READY,
                     forward_mode=mode)
    assert layer.plan.num_macrobatches == 1 and layer.plan.minibatch_rows >= w.T * w.k   # one minibatch
    t0 = time.time()
    layer.forward(d["x"], d["Wr"], d["bias"], d["W1"], d["W3"], d["W2"])
    with pytest.raises(M.MoeError) as err:
        layer.status()
    assert err.value.status == M.MOE_ERR_TIMEOUT
    assert time.time() - t0 < 30.0          # bounded: 100 ms per wait, then every role leaves
    layer.status()                          # the query cleared the status word
    # same process and CUDA context: a fresh layer still matches the oracle
    gpu = G.run_gpu(w, inp)
    G.check_layer(w, inp, gpu)


def test_schedule_reports_out_of_range_ids():
    # expert ids outside [0, E) passed to moe_schedule: the schedule's own check skips their
    # slots (no access depends on them) and reports MOE_ERR_INTERNAL; the valid slots are counted
    import numpy as np
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    T, E, k = 300, 8, 2
    rng = np.random.default_rng(5)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    for t, j, v in [(3, 0, E), (17, 1, -1), (250, 0, E + 100)]:
        ids[t, j] = v
    layer = MoeLayer(T, 256, 256, E, k)
    counts, _, _, _ = layer.schedule(torch.from_numpy(ids).cuda())
    with pytest.raises(M.MoeError) as err:
        layer.status()
    assert err.value.status == M.MOE_ERR_INTERNAL
    valid = ids[(ids >= 0) & (ids < E)]
    np.testing.assert_array_equal(counts.cpu().numpy().reshape(-1), np.bincount(valid, minlength=E))
    layer.status()                          # cleared by the query


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
@pytest.mark.parametrize("which,bad", [("ROW_SLOT", 1 << 30), ("ROW_SLOT", -7), ("SLOT_ROW", 1 << 30),
                                       ("SLOT_ROW", -3)])
def test_corrupted_saved_index_maps_are_reported(precision, which, bad):
    # the forward's row<->slot maps in the saved context overwritten between forward and backward
    # with indices outside their ranges: every backward kernel that follows them (the reverse
    # combine gathers, the GEMM2 dgrad epilogue, the router backward, the reverse dispatch) checks
    # the index, skips the access and reports MOE_ERR_INTERNAL; the same context then still runs
    # the layer correctly
    import numpy as np
    import mixture_experts_layer_sum_gb300.moe as M
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    import tests.gpu_common as G
    w = WL.TINY if precision == "bf16" else WL.Workload("mx_small", T=300, H=512, E=8, k=2, F=512,
                                                            precision="mxfp8", zipf_s=0.8)
    inp = WL.make_inputs(w)
    d = G.device_inputs(inp)
    layer = MoeLayer(w.T, w.H, w.F, w.E, w.k, w.precision)
    if precision == "mxfp8":
        layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    layer.forward(d["x"], d["Wr"], d["bias"], d["W1"], d["W3"], d["W2"])
    layer.status()
    torch.cuda.synchronize()
    offp = layer.buffer("PADDED_OFFSETS").view(torch.int32).cpu().numpy()
    m = layer.buffer(which).view(torch.int32)
    if which == "ROW_SLOT":
        e = int(np.nonzero(np.diff(offp[:w.E + 1]) > 0)[0][0])   # a run with rows
        targets = [int(offp[e]), int(offp[e]) + 1]                 # its first two rows (real slots)
    else:
        targets = [0, w.T * w.k - 1]
    for r in targets:
        m[r] = bad
    torch.cuda.synchronize()
    layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"])
    with pytest.raises(M.MoeError) as err:
        layer.status()
    assert err.value.status == M.MOE_ERR_INTERNAL
    layer.status()                          # cleared by the query
    del layer
    gpu = G.run_gpu(w, inp)
    G.check_layer(w, inp, gpu)
