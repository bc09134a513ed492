"""MoeLayer: the user-facing Python object over the C ABI.

It only owns device buffers (workspace, forward->backward context, outputs)
allocated with PyTorch and passes pointers to libmoe_gb300.so; every step of
the layer runs in the library's CUDA kernels.
"""
from __future__ import annotations

import torch

from . import moe as _m


class MoeLayer:
    def __init__(self, T, H, F, E, k, precision="bf16", *, device="cuda", ring_bytes=0, macrobatch_tokens=0,
                 minibatch_rows=0, timeout_ms=0, fault_mask=0, forward_mode=0):
        self.shape = dict(T=T, H=H, F=F, E=E, k=k)
        self.device = torch.device(device)
        self.cfg = _m.make_config(T, H, F, E, k, precision, minibatch_rows, macrobatch_tokens, ring_bytes,
                                  timeout_ms, 0, fault_mask, forward_mode)
        self.plan = _m.moe_plan(self.cfg)
        self.workspace = torch.empty(self.plan.workspace_bytes, dtype=torch.uint8, device=self.device)
        self.saved = torch.empty(self.plan.saved_bytes, dtype=torch.uint8, device=self.device)
        self.qweights = None
        if precision in ("mxfp8", "nvfp4"):
            self.qweights = torch.empty(_m.moe_qweights_size(self.cfg), dtype=torch.uint8, device=self.device)
        _m.moe_reset_status(self.workspace)

    def quantize_weights(self, W1, W3, W2, stream=None):
        """MXFP8 or NVFP4 copies of the bf16 weights (run once per weight update)."""
        _m.moe_quantize_weights(self.cfg, W1, W3, W2, self.qweights, stream)

    def forward(self, x, Wr, bias, W1, W3, W2, out=None, topk_ids=None, topk_w=None, stream=None):
        T, H, k = self.shape["T"], self.shape["H"], self.shape["k"]
        dev = self.device
        out = out if out is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        topk_ids = topk_ids if topk_ids is not None else torch.empty(T, k, dtype=torch.int32, device=dev)
        topk_w = topk_w if topk_w is not None else torch.empty(T, k, dtype=torch.float32, device=dev)
        _m.moe_forward(self.cfg, x, Wr, bias, W1, W3, W2, self.qweights, out, topk_ids, topk_w, self.saved,
                       self.workspace, stream)
        return out, topk_ids, topk_w

    def backward(self, dout, x, Wr, W1, W3, W2, dx=None, dWr=None, dW1=None, dW3=None, dW2=None,
                 accumulate=False, stream=None):
        T, H, F, E = self.shape["T"], self.shape["H"], self.shape["F"], self.shape["E"]
        dev = self.device
        dx = dx if dx is not None else torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        dWr = dWr if dWr is not None else torch.empty(H, E, dtype=torch.float32, device=dev)
        dW1 = dW1 if dW1 is not None else torch.empty(E, H, F, dtype=torch.float32, device=dev)
        dW3 = dW3 if dW3 is not None else torch.empty(E, H, F, dtype=torch.float32, device=dev)
        dW2 = dW2 if dW2 is not None else torch.empty(E, F, H, dtype=torch.float32, device=dev)
        _m.moe_backward(self.cfg, dout, x, Wr, W1, W3, W2, self.qweights, self.saved, dx, dWr, dW1, dW3, dW2,
                        accumulate, self.workspace, stream)
        return dx, dWr, dW1, dW3, dW2

    def schedule(self, topk_ids, macrobatch_tokens=None, stream=None):
        """Counts, offsets and both permutations of the stable (macrobatch, expert) sort."""
        p = self.plan
        E = self.shape["E"]
        R = topk_ids.numel()
        dev = self.device
        counts = torch.empty(p.num_macrobatches * E, dtype=torch.int32, device=dev)
        offsets = torch.empty(p.num_macrobatches * (E + 1), dtype=torch.int32, device=dev)
        s2s = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        s2sorted = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        _m.moe_schedule(self.cfg, topk_ids, counts, offsets, s2s, s2sorted, self.workspace, stream)
        return counts, offsets, s2s[:R], s2sorted[:R]

    def buffer(self, name):
        """A uint8 view of one intermediate buffer inside the saved buffer or the workspace
        (moe_buffer_location; a test and debugging aid)."""
        in_saved, off, nb = _m.moe_buffer_location(self.cfg, name)
        base = self.saved if in_saved else self.workspace
        start = (-base.data_ptr()) % 1024          # the library's 1024-byte-aligned base
        return base[start + off:start + off + nb]

    def status(self, stream=None):
        """Synchronises and raises MoeError if a device-side check failed."""
        return _m.moe_query_status(self.workspace, stream)
