"""Host-only checks of the C-ABI library: it builds, loads, exports every
function include/moe.h declares, plans sizes (the minibatch floor is pinned to
the figure the pages print) and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_sum_gb300 import build_ext
    build_ext.build()
    import mixture_experts_layer_sum_gb300.moe as m
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(moe):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_abi_version(moe):
    assert moe.moe_abi_version() == 3


def test_minibatch_floor_matches_pages_golden(moe):
    path = os.path.join(ROOT, "tests", "golden", "minibatch_floor.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    for sms, H, F, want in rows:
        cfg = moe.make_config(4096, int(H), int(F), 16, 8, num_sms=int(sms))
        assert moe.moe_plan(cfg).minibatch_rows == int(want)


def test_plan_sizes_and_ring(moe):
    cfg = moe.make_config(16384, 7168, 2048, 16, 8, num_sms=152, ring_bytes=256 << 20)
    p = moe.moe_plan(cfg)
    assert p.num_macrobatches > 1
    assert p.ring_bytes <= 256 << 20
    assert p.macrobatch_tokens * p.num_macrobatches >= 16384
    assert p.workspace_bytes == moe.moe_workspace_size(cfg)
    assert p.saved_bytes == moe.moe_saved_size(cfg)
    full = moe.make_config(16384, 7168, 2048, 16, 8, num_sms=152)
    pf = moe.moe_plan(full)
    assert pf.num_macrobatches == 1 and pf.macrobatch_tokens == 16384
    # padded rows bound: every (macrobatch, expert) run padded to 128 rows
    assert pf.rows_padded_max >= 16384 * 8 and pf.rows_padded_max % 128 == 0


def test_saved_keeps_dispatched_rows_for_bf16(moe):
    # bf16: the forward's expert-sorted x rows [rows_padded_max, H] bf16 live in the saved context
    # for any number of macrobatches (GEMM1 reads them there, then the backward's dW1/dW3); MXFP8
    # keeps the same context without them (its weight gradient needs x along the tokens)
    a1024 = lambda v: -(-v // 1024) * 1024
    T, H, F, E, k = 4096, 2048, 1024, 32, 4
    for Mb in (0, 1024):
        bf = moe.make_config(T, H, F, E, k, macrobatch_tokens=Mb, num_sms=152)
        mx = moe.make_config(T, H, F, E, k, "mxfp8", macrobatch_tokens=Mb, num_sms=152)
        p = moe.moe_plan(bf)
        assert p.num_macrobatches == (1 if Mb == 0 else 4)
        assert moe.moe_saved_size(bf) - moe.moe_saved_size(mx) == a1024(2 * p.rows_padded_max * H)


@pytest.mark.parametrize("kw,status", [
    (dict(T=16, H=250, F=512, E=4, k=2), 2),    # H not a multiple of 256
    (dict(T=16, H=256, F=500, E=4, k=2), 2),
    (dict(T=16, H=256, F=512, E=65, k=2), 2),   # too many experts
    (dict(T=16, H=256, F=512, E=4, k=5), 1),    # k > E
    (dict(T=-1, H=256, F=512, E=4, k=2), 1),
    (dict(T=16, H=256, F=512, E=4, k=0), 1),
])
def test_bad_shapes_rejected(moe, kw, status):
    cfg = moe.make_config(num_sms=148, **kw)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_plan(cfg)
    assert ei.value.status == status
    assert moe.moe_workspace_size(cfg) == 0


def test_null_pointers_rejected_without_gpu(moe):
    cfg = moe.make_config(64, 256, 512, 8, 2, num_sms=148)
    lib = moe.library()
    st = lib.moe_forward(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None,
                         None, 0, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert "null" in moe.moe_last_error_string()
    st = lib.moe_backward(ctypes.byref(cfg), None, None, None, None, None, None, None, None, None, None,
                          None, None, None, 0, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = lib.moe_schedule(ctypes.byref(cfg), None, None, None, None, None, None, 0, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_small_buffers_rejected_without_gpu(moe):
    cfg = moe.make_config(64, 256, 512, 8, 2, num_sms=148)
    lib = moe.library()
    fake = 1 << 20   # never dereferenced: the size check fails first
    ws = moe.moe_workspace_size(cfg)
    st = lib.moe_forward(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, None, fake, fake, fake,
                         fake, moe.moe_saved_size(cfg) - 1025, fake, ws, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = lib.moe_forward(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, None, fake, fake, fake,
                         fake, moe.moe_saved_size(cfg), fake, ws - 1025, None)
    assert st == moe.MOE_ERR_WORKSPACE
    # an unaligned workspace base costs up to 1023 bytes of the slack
    st = lib.moe_forward(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, None, fake, fake, fake,
                         fake, moe.moe_saved_size(cfg), fake + 1, ws - 2, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = lib.moe_forward(ctypes.byref(cfg), fake + 8, fake, None, fake, fake, fake, None, fake, fake, fake,
                         fake, moe.moe_saved_size(cfg), fake, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG      # misaligned x


def test_library_does_not_reference_oracle():
    pkg = os.path.join(ROOT, "mixture_experts_layer_sum_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower(), f


def test_buffer_locations_lie_inside_their_buffers(moe):
    for prec in ("bf16", "mxfp8"):
        for Mb in (0, 700):
            cfg = moe.make_config(3000, 512, 512, 16, 4, prec, macrobatch_tokens=Mb, num_sms=152)
            p = moe.moe_plan(cfg)
            for name in moe.BUFFERS:
                mx_only = name.endswith("_SCALES") or name.endswith("_ROWS") or name.endswith("_TOKENS")
                bf16_only = name in ("DA", "DB", "HW")   # MXFP8 quantises them straight from the epilogue
                if (prec == "bf16" and mx_only) or (prec == "mxfp8" and bf16_only):
                    with pytest.raises(moe.MoeError) as e:
                        moe.moe_buffer_location(cfg, name)
                    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
                    continue
                in_saved, off, nb = moe.moe_buffer_location(cfg, name)
                limit = (p.saved_bytes if in_saved else p.workspace_bytes) - 1024
                assert nb > 0 and off % 1024 == 0 and off + nb <= limit, (prec, name)
    # an unknown buffer and null outputs are rejected
    cfg = moe.make_config(64, 256, 256, 4, 2, num_sms=152)
    i, o, n = ctypes.c_int(), ctypes.c_size_t(), ctypes.c_size_t()
    lib = moe.library()
    assert lib.moe_buffer_location(ctypes.byref(cfg), len(moe.BUFFERS), ctypes.byref(i), ctypes.byref(o),
                                   ctypes.byref(n)) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_buffer_location(ctypes.byref(cfg), 0, None, None, None) == moe.MOE_ERR_INVALID_ARG


def test_ring_holds_one_macrobatch(moe):
    # the macrobatch is the largest token count whose padded rows of dispatched tokens (MXFP8:
    # E4M3 along H plus scales; bf16: 2H bytes), in whole 128-row tiles, fit the ring once
    # (less 8 KiB for buffer alignment); a kernel never overlaps its predecessor on the stream,
    # so one macrobatch is in flight at a time
    H, F, E, k = 7168, 2048, 16, 8
    pad = 127 * E
    for prec, row in (("mxfp8", H + H // 32), ("bf16", 2 * H)):
        cfg = moe.make_config(16384, H, F, E, k, prec, ring_bytes=256 << 20, num_sms=152)
        p = moe.moe_plan(cfg)
        cap = ((256 << 20) - 8192) // row // 128 * 128
        assert p.macrobatch_tokens * k + pad <= cap < (p.macrobatch_tokens + 1) * k + pad, prec
        assert p.ring_bytes <= 256 << 20
        assert p.num_macrobatches == -(-16384 // p.macrobatch_tokens)


def test_nvfp4_weight_buffer_holds_the_stage_layout(moe):
    # W1 and W3 interleaved per 128-K stage, then W2, then the matrix scales and the quantiser's
    # maxima, each part 1 KB aligned; a tile (128 columns x 64 K) is 4096 code and 512 scale bytes
    a1024 = lambda v: -(-v // 1024) * 1024
    for E, H, F in [(32, 2048, 1024), (4, 256, 512), (64, 7168, 2048)]:
        tiles = E * (H // 64) * (F // 128)
        w2 = a1024(2 * tiles * 4608)
        gscale = a1024(w2 + tiles * 4608)
        end = a1024(a1024(gscale + 12 * E) + 12 * E)
        size = moe.moe_qweights_size(moe.make_config(64, H, F, E, 4, "nvfp4"))
        assert end <= size <= end + 1024, (E, H, F, size, end)
