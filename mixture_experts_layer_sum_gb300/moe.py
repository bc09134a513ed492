"""Python binding of the GB300 MoE layer library (libmoe_gb300.so).

Thin ctypes marshalling over the C ABI in include/moe.h: every function has the
C name and takes torch tensors (device memory) or raw integer pointers. All
arithmetic runs in the library's CUDA kernels; if the library is missing the
import of this module fails instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from .build_ext import LIB as LIB_PATH  # noqa: E402

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_INTERNAL = 6
MOE_FAULT_GEMM1_READY = 1   # config fault_mask bit (failure-detection tests)
MOE_PRECISION_BF16 = 0
MOE_PRECISION_MXFP8 = 1
MOE_PRECISION_NVFP4 = 2
MOE_FORWARD_PERSISTENT = 0
MOE_FORWARD_PER_STAGE = 1

EXPORTED = (
    "moe_abi_version", "moe_plan", "moe_workspace_size", "moe_saved_size", "moe_qweights_size",
    "moe_schedule", "moe_schedule_static", "moe_quantize_weights", "moe_forward", "moe_backward", "moe_query_status",
    "moe_reset_status", "moe_last_error_string", "moe_profile_begin", "moe_profile_end", "moe_buffer_location",
)

# moe_buffer_t (include/moe.h): intermediate buffers moe_buffer_location can locate
BUFFERS = (
    "PADDED_OFFSETS", "ROW_SLOT", "A", "B", "RING_X", "RING_X_SCALES", "RING_H", "RING_H_SCALES",
    "DA", "DB", "HW", "DY_ROWS", "DY_ROWS_SCALES", "DA_ROWS", "DA_ROWS_SCALES", "DB_ROWS", "DB_ROWS_SCALES",
    "X_TOKENS", "X_TOKENS_SCALES", "DY_TOKENS", "DY_TOKENS_SCALES", "HW_TOKENS", "HW_TOKENS_SCALES",
    "DA_TOKENS", "DA_TOKENS_SCALES", "DB_TOKENS", "DB_TOKENS_SCALES", "SLOT_ROW",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"moe status {status}: {message}")
        self.status = status


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("H", ctypes.c_int), ("F", ctypes.c_int), ("E", ctypes.c_int),
                ("k", ctypes.c_int), ("precision", ctypes.c_int), ("minibatch_rows", ctypes.c_int),
                ("macrobatch_tokens", ctypes.c_int), ("ring_bytes", ctypes.c_size_t),
                ("timeout_ms", ctypes.c_uint), ("num_sms", ctypes.c_int), ("fault_mask", ctypes.c_uint),
                ("forward_mode", ctypes.c_int)]


class moe_kernel_time_t(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class moe_plan_t(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int), ("minibatch_rows", ctypes.c_int),
                ("macrobatch_tokens", ctypes.c_int), ("num_macrobatches", ctypes.c_int),
                ("rows_padded_max", ctypes.c_int), ("ring_rows", ctypes.c_int),
                ("ring_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("saved_bytes", ctypes.c_size_t), ("qweights_bytes", ctypes.c_size_t)]


def make_config(T, H, F, E, k, precision="bf16", minibatch_rows=0, macrobatch_tokens=0, ring_bytes=0,
                timeout_ms=0, num_sms=0, fault_mask=0, forward_mode=0) -> moe_config_t:
    p = {"bf16": MOE_PRECISION_BF16, "mxfp8": MOE_PRECISION_MXFP8, "nvfp4": MOE_PRECISION_NVFP4}.get(precision, precision)
    return moe_config_t(T, H, F, E, k, p, minibatch_rows, macrobatch_tokens, ring_bytes, timeout_ms, num_sms,
                        fault_mask, forward_mode)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m mixture_experts_layer_sum_gb300.build_ext` "
            "(the MoE layer has no non-CUDA implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    cfgp = ctypes.POINTER(moe_config_t)
    sig = {
        "moe_abi_version": ([], ctypes.c_int),
        "moe_plan": ([cfgp, ctypes.POINTER(moe_plan_t)], ctypes.c_int),
        "moe_workspace_size": ([cfgp], ctypes.c_size_t),
        "moe_saved_size": ([cfgp], ctypes.c_size_t),
        "moe_qweights_size": ([cfgp], ctypes.c_size_t),
        "moe_schedule": ([cfgp, P, P, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
        "moe_schedule_static": ([cfgp, P, P, P, P, P, P], ctypes.c_int),
        "moe_quantize_weights": ([cfgp, P, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
        "moe_forward": ([cfgp, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t, P],
                        ctypes.c_int),
        "moe_backward": ([cfgp, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_int, P, ctypes.c_size_t, P],
                         ctypes.c_int),
        "moe_query_status": ([P, P], ctypes.c_int),
        "moe_reset_status": ([P, P], ctypes.c_int),
        "moe_last_error_string": ([], ctypes.c_char_p),
        "moe_profile_begin": ([], ctypes.c_int),
        "moe_profile_end": ([ctypes.POINTER(moe_kernel_time_t), ctypes.c_int], ctypes.c_int),
        "moe_buffer_location": ([cfgp, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t),
                                 ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def library():
    return _lib


def _ptr(t):
    """Device pointer of a torch tensor (or an int / None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(s):
    if s is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int):
    if st != MOE_OK:
        raise MoeError(st, moe_last_error_string())
    return st


def moe_abi_version() -> int:
    return _lib.moe_abi_version()


def moe_last_error_string() -> str:
    return (_lib.moe_last_error_string() or b"").decode()


def moe_plan(cfg: moe_config_t) -> moe_plan_t:
    plan = moe_plan_t()
    _check(_lib.moe_plan(ctypes.byref(cfg), ctypes.byref(plan)))
    return plan


def moe_workspace_size(cfg: moe_config_t) -> int:
    return _lib.moe_workspace_size(ctypes.byref(cfg))


def moe_saved_size(cfg: moe_config_t) -> int:
    return _lib.moe_saved_size(ctypes.byref(cfg))


def moe_qweights_size(cfg: moe_config_t) -> int:
    return _lib.moe_qweights_size(ctypes.byref(cfg))


def moe_schedule(cfg, topk_ids, counts, offsets, sorted_to_slot, slot_to_sorted, workspace, stream=None):
    return _check(_lib.moe_schedule(ctypes.byref(cfg), _ptr(topk_ids), _ptr(counts), _ptr(offsets),
                                    _ptr(sorted_to_slot), _ptr(slot_to_sorted), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream)))


def moe_schedule_static(cfg, topk_ids, counts, offsets, sorted_to_slot, slot_to_sorted, stream=None):
    """moe_schedule without a workspace (scratch in the library's static device array)."""
    return _check(_lib.moe_schedule_static(ctypes.byref(cfg), _ptr(topk_ids), _ptr(counts), _ptr(offsets),
                                           _ptr(sorted_to_slot), _ptr(slot_to_sorted), _stream(stream)))


def moe_quantize_weights(cfg, W1, W3, W2, qweights, stream=None):
    return _check(_lib.moe_quantize_weights(ctypes.byref(cfg), _ptr(W1), _ptr(W3), _ptr(W2), _ptr(qweights),
                                            _nbytes(qweights) if qweights is not None else 0, _stream(stream)))


def moe_forward(cfg, x, W_r, bias, W1, W3, W2, qweights, out, topk_ids, topk_w, saved, workspace, stream=None):
    return _check(_lib.moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(W_r), _ptr(bias), _ptr(W1), _ptr(W3),
                                   _ptr(W2), _ptr(qweights), _ptr(out), _ptr(topk_ids), _ptr(topk_w),
                                   _ptr(saved), _nbytes(saved), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream)))


def moe_backward(cfg, dout, x, W_r, W1, W3, W2, qweights, saved, dx, dW_r, dW1, dW3, dW2, accumulate,
                 workspace, stream=None):
    return _check(_lib.moe_backward(ctypes.byref(cfg), _ptr(dout), _ptr(x), _ptr(W_r), _ptr(W1), _ptr(W3),
                                    _ptr(W2), _ptr(qweights), _ptr(saved), _ptr(dx), _ptr(dW_r), _ptr(dW1),
                                    _ptr(dW3), _ptr(dW2), int(accumulate), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream)))


def moe_query_status(workspace, stream=None):
    return _check(_lib.moe_query_status(_ptr(workspace), _stream(stream)))


def moe_reset_status(workspace, stream=None):
    return _check(_lib.moe_reset_status(_ptr(workspace), _stream(stream)))


def moe_profile_begin():
    return _check(_lib.moe_profile_begin())


def moe_profile_end(max_entries: int = 64):
    """Returns [(kernel name, launches, total ms)] recorded since moe_profile_begin."""
    buf = (moe_kernel_time_t * max_entries)()
    n = _lib.moe_profile_end(buf, max_entries)
    if n < 0:
        raise MoeError(-n, moe_last_error_string())
    return [(buf[i].name.decode(), buf[i].launches, buf[i].total_ms) for i in range(min(n, max_entries))]


def moe_buffer_location(cfg, name):
    """(in_saved, offset, bytes) of an intermediate buffer, by its moe_buffer_t name without the
    MOE_BUF_ prefix (a test and debugging aid; see include/moe.h)."""
    in_saved, off, nb = ctypes.c_int(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.moe_buffer_location(ctypes.byref(cfg), BUFFERS.index(name), ctypes.byref(in_saved),
                                    ctypes.byref(off), ctypes.byref(nb)))
    return bool(in_saved.value), off.value, nb.value
