"""moe_schedule_static, the schedule entry point for callers that cannot
allocate device memory (its scratch is a static device array inside the
library), must give exactly what moe_schedule gives with a caller workspace.
Two calls in a row with different routings check that what one call leaves in
the shared array does not leak into the next. Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    import mixture_experts_layer_sum_gb300.moe as m
    assert torch.cuda.is_available()
    return m


def routed_ids(seed, T, E, k):
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def run_both(m, T, E, k, Mb, seed):
    cfg = m.make_config(T, 256, 256, E, k, macrobatch_tokens=Mb)
    plan = m.moe_plan(cfg)
    ids = torch.from_numpy(routed_ids(seed, T, E, k)).cuda()
    R = T * k
    outs = []
    for static in (False, True):
        counts = torch.full((plan.num_macrobatches * E,), -7, dtype=torch.int32, device="cuda")
        offsets = torch.full((plan.num_macrobatches * (E + 1),), -7, dtype=torch.int32, device="cuda")
        s2s = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        s2r = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        if static:
            st = m.library().moe_schedule_static(ctypes.byref(cfg), ids.data_ptr(), counts.data_ptr(),
                                                 offsets.data_ptr(), s2s.data_ptr(), s2r.data_ptr(), None)
            assert st == m.MOE_OK, m.moe_last_error_string()
        else:
            ws = torch.empty(m.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
            m.moe_schedule(cfg, ids, counts, offsets, s2s, s2r, ws, stream=0)
            m.moe_query_status(ws, stream=0)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy() for t in (counts, offsets, s2s, s2r)])
    return outs


def test_static_schedule_matches_workspace_schedule_twice(moe):
    # first call: many macrobatches and 64 experts; second call: a different,
    # smaller routing, so stale histograms from the first would show
    for T, E, k, Mb, seed in [(3000, 64, 8, 700, 1), (513, 8, 2, 0, 2)]:
        ref, got = run_both(moe, T, E, k, Mb, seed)
        for a, b in zip(ref, got):
            np.testing.assert_array_equal(a, b)
        assert ref[0].sum() == T * k


def test_static_schedule_rejects_shapes_beyond_capacity(moe):
    # 65536 tokens x 8 slots in macrobatches of 32 tokens: 2048 macrobatches x 64 experts
    # need about 393 k words of scratch, over the 262 k the 1 MiB array holds. Every buffer
    # is real and sized for the call, so a regression in the capacity check shows up as a
    # wrong status, not as a stray access.
    T, E, k, Mb = 65536, 64, 8, 32
    cfg = moe.make_config(T, 256, 256, E, k, macrobatch_tokens=Mb)
    plan = moe.moe_plan(cfg)
    assert plan.num_macrobatches == T // Mb
    ids = torch.from_numpy(routed_ids(5, 64, E, k)).cuda().repeat(T // 64, 1).contiguous()
    counts = torch.zeros(plan.num_macrobatches * E, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(plan.num_macrobatches * (E + 1), dtype=torch.int32, device="cuda")
    s2s = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    s2r = torch.zeros(T * k, dtype=torch.int32, device="cuda")
    st = moe.library().moe_schedule_static(ctypes.byref(cfg), ids.data_ptr(), counts.data_ptr(),
                                           offsets.data_ptr(), s2s.data_ptr(), s2r.data_ptr(), None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert "1 MiB" in moe.moe_last_error_string()
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(s2s.abs().sum()) == 0    # nothing ran
