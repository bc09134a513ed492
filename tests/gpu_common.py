"""Helpers of the GPU parity tests: run the CUDA layer on seeded inputs and
compare it with the float64 oracle on the same bf16 bytes."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
import workloads as WL

FWD_TOL = 1e-2     # max-abs-relative, forward (BF16)
BWD_TOL = 2e-2     # max-abs-relative, backward (BF16)
MX_TOL = 6e-2      # max-abs-relative, MXFP8, against the oracle with the same quantisation emulated
NEAR_TIE = 1e-4    # logit gap below which GPU and oracle may pick different experts


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev_to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


def device_inputs(inp):
    d = {k: bf16_dev(v) for k, v in inp.items() if k != "bias" and v is not None}
    d["bias"] = torch.from_numpy(inp["bias"]).cuda() if inp.get("bias") is not None else None
    return d


def oracle_inputs(inp):
    o = {k: O.bf16_to_f64(v) for k, v in inp.items() if k != "bias" and v is not None}
    o["bias"] = None if inp.get("bias") is None else inp["bias"].astype(np.float64)
    return o


def run_gpu(w: WL.Workload, inp, backward=True, accumulate_into=None, **layer_kw):
    from mixture_experts_layer_sum_gb300.layer import MoeLayer
    d = device_inputs(inp)
    T = inp["x"].shape[0]
    layer = MoeLayer(T, w.H, w.F, w.E, w.k, w.precision, **layer_kw)
    if w.precision in ("mxfp8", "nvfp4"):
        layer.quantize_weights(d["W1"], d["W3"], d["W2"])
    out, ids, wts = layer.forward(d["x"], d["Wr"], d["bias"], d["W1"], d["W3"], d["W2"])
    res = {"out": out, "ids": ids, "w": wts}
    if backward:
        kw = {}
        if accumulate_into is not None:
            kw = {k: v.clone() for k, v in accumulate_into.items()}
        dx, dWr, dW1, dW3, dW2 = layer.backward(d["dout"], d["x"], d["Wr"], d["W1"], d["W3"], d["W2"],
                                                accumulate=accumulate_into is not None, **kw)
        res.update(dx=dx, dWr=dWr, dW1=dW1, dW3=dW3, dW2=dW2)
    layer.status()
    torch.cuda.synchronize()
    res = {k: dev_to_np(v) for k, v in res.items()}
    res["layer"] = layer
    return res


def reconcile_ids(gpu_ids, oracle_fwd, k):
    """GPU ids must equal the oracle's except on near-tie tokens. Returns the ids
    to feed the oracle (the GPU's), after checking every difference is a near tie."""
    logits = oracle_fwd["logits"]
    diff = np.nonzero((np.sort(gpu_ids, axis=1) != np.sort(oracle_fwd["ids"], axis=1)).any(axis=1))[0]
    if len(diff):
        srt = -np.sort(-logits[diff], axis=1)
        gap = srt[:, k - 1] - srt[:, k]
        assert (gap < NEAR_TIE * (1 + np.abs(srt[:, k - 1]))).all(), f"non-tie id mismatch at tokens {diff[:10]}"
    same_set = np.setdiff1d(np.arange(gpu_ids.shape[0]), diff)
    # on agreeing tokens the slot order (descending probability) must agree too,
    # except where two chosen experts are themselves near-tied
    bad = same_set[(gpu_ids[same_set] != oracle_fwd["ids"][same_set]).any(axis=1)]
    for t in bad:
        l = logits[t, gpu_ids[t]]
        assert np.min(np.abs(np.diff(np.sort(l)))) < NEAR_TIE * (1 + np.abs(l).max()), t
    return gpu_ids, len(diff)


_WEIGHT_CACHES = {}


def weight_caches(w):
    """The oracle's weight-copy caches (forward, dgrad) for a workload's weights: workloads with
    the same seed and weight shapes draw the same weights, so one session quantises them once."""
    key = (w.seed, w.E, w.H, w.F, w.weight_std, w.precision)
    if key not in _WEIGHT_CACHES:
        _WEIGHT_CACHES.clear()
        _WEIGHT_CACHES[key] = ({}, {})
    return _WEIGHT_CACHES[key]


def check_layer(w, inp, gpu, backward=True, macrobatch_tokens=0):
    oi = oracle_inputs(inp)
    wc = weight_caches(w)
    f = O.forward(oi["x"], oi["Wr"], oi["bias"], oi["W1"], oi["W3"], oi["W2"], w.k,
                  precision=w.precision, macrobatch_tokens=macrobatch_tokens, weight_cache=wc[0])
    ids, nties = reconcile_ids(gpu["ids"].astype(np.int32), f, w.k)
    if nties or (ids != f["ids"]).any():
        f = O.forward(oi["x"], oi["Wr"], oi["bias"], oi["W1"], oi["W3"], oi["W2"], w.k,
                      precision=w.precision, macrobatch_tokens=macrobatch_tokens, ids=ids, weight_cache=wc[0])
    errs = {"w": float(np.abs(gpu["w"] - f["w"]).max()) if f["w"].size else 0.0,
            "out": O.max_abs_rel(gpu["out"], f["out"])}
    # NVFP4: the weights are exact on both sides (the same quantisation); activations as in bf16
    ftol, btol = (MX_TOL, MX_TOL) if w.precision == "mxfp8" else (FWD_TOL, BWD_TOL)
    assert errs["w"] < 1e-4, errs
    assert errs["out"] < ftol, errs
    if backward:
        g = O.backward(f, oi["dout"], oi["x"], oi["Wr"], oi["W1"], oi["W3"], oi["W2"], weight_cache=wc[1])
        for key in ("dx", "dWr", "dW1", "dW3", "dW2"):
            errs[key] = O.max_abs_rel(gpu[key], g[key])
            assert errs[key] < btol, (key, errs)
    return errs


# ---------------------------------------------------------------- raw buffers of the library


def atoms_to_rows(sf_bytes, rows, K):
    """Scale atoms (512 B per 128 rows x 128 elements of K) -> [rows, K/32] scale bytes."""
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    off = ((r // 128) * (K // 128) + (kb * 32) // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
    return np.asarray(sf_bytes)[off]


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def bf16_rows(t: torch.Tensor, rows, cols) -> np.ndarray:
    """A uint8 device view holding bf16 [rows][cols] row-major -> float64."""
    return O.bf16_to_f64(u8(t)[:2 * rows * cols].view(np.uint16).reshape(rows, cols))


def bf16_blocks(t: torch.Tensor, rows, cols, keep=None) -> np.ndarray:
    """bf16 [rows][cols] stored in 32 x 32 blocks of 2 KB (block (r/32, c/32) row-major; element
    (r, c) at ((c % 32) / 8 * 32 + r % 32) * 8 + c % 8 inside it) -> float64 [keep, cols] (the
    first keep rows, default all; rows past the written ones are never converted)."""
    v = u8(t)[:2 * rows * cols].view(np.uint16).reshape(rows // 32, cols // 32, 4, 32, 8)
    # axes: block row, block col, c/8 within block, r within block, c%8
    keep = rows if keep is None else keep
    return O.bf16_to_f64(v.transpose(0, 3, 1, 2, 4).reshape(rows, cols)[:keep])


def bf16_round(v) -> np.ndarray:
    """float64 -> bf16 values as float64, through fp32 (each step to nearest even; monotone)."""
    return WL.bf16_bits_to_f32(WL.f32_to_bf16_bits(np.asarray(v, np.float32))).astype(np.float64)


def check_mx_decided(codes, scales, ref, axis, rel, bf16_values=False):
    """MXFP8 bytes the GPU made from values that agree with the float64 `ref` to within `rel`
    of their block maximum (its own arithmetic differs in rounding only). Where the block
    maximum is farther than rel from a scale boundary, the scale byte must be the oracle
    quantiser's; at the GPU's scale, an element whose value cannot cross a rounding midpoint
    within that error must carry the oracle's code; an element that can must lie between the
    roundings of the two ends of its error interval (rounding is monotone). bf16_values: the
    GPU rounded its values to bf16 before quantising them, so the interval ends are rounded the
    same way and the scale test allows the bf16 step too. Returns (undecided scales, undecided
    codes) counts."""
    rc, rs = O.mx_quantize(ref, axis)
    mv = lambda a: np.moveaxis(np.asarray(a), axis, -1)
    refm, gc, gs, rsm = mv(ref), mv(codes), mv(scales).astype(np.int64), mv(rs).astype(np.int64)
    n = refm.shape[-1]
    blk = refm.reshape(refm.shape[:-1] + (n // 32, 32))
    amax = np.abs(blk).max(-1)
    s = rsm - 127
    hi, lo = 448.0 * np.exp2(s), 448.0 * np.exp2(s - 1)
    rs_ = rel + (2.0 ** -8 if bf16_values else 0.0)
    near = (np.abs(amax - hi) <= rs_ * hi) | (np.abs(amax - lo) <= rs_ * lo)
    near &= amax > 0
    assert (gs[~near] == rsm[~near]).all(), "scale bytes differ away from a scale boundary"
    gscale = np.exp2(gs.astype(np.float64) - 127)[..., None]
    scaled = blk / gscale
    dev = (rel * amax)[..., None] / gscale
    pre = bf16_round if bf16_values else (lambda a: a)
    q_lo, q_hi = O.e4m3_round(pre(scaled - dev)), O.e4m3_round(pre(scaled + dev))
    got = O.e4m3_decode(gc.reshape(blk.shape))
    decided = q_lo == q_hi
    assert (got[decided] == q_lo[decided]).all(), "codes differ where the reference decides them"
    assert ((got >= q_lo) & (got <= q_hi)).all(), "a code lies outside the reference's interval"
    return int(near.sum()), int((~decided).sum())


def check_mx_interval(codes, scales, lo, hi, axis):
    """MXFP8 bytes of values known only to lie in [lo, hi] elementwise (lo <= hi, both float64,
    every rounding the GPU applies before quantising already taken into the ends). Where every
    value of the interval gives one scale byte, the GPU's must be it, and it must lie between
    the bytes of the interval's smallest and largest block maxima; at the GPU's scale every code
    must lie between the roundings of its interval's ends (rounding is monotone). Returns
    (undecided scales, undecided codes) counts."""
    mv = lambda a: np.moveaxis(np.asarray(a), axis, -1)
    lo_m, hi_m, gc, gs = mv(lo), mv(hi), mv(codes), mv(scales).astype(np.int64)
    n = lo_m.shape[-1]
    shp = lo_m.shape[:-1] + (n // 32, 32)
    lo_b, hi_b = lo_m.reshape(shp), hi_m.reshape(shp)
    assert (lo_b <= hi_b).all()
    same_sign = (lo_b > 0) | (hi_b < 0)
    mag_lo = np.where(same_sign, np.minimum(np.abs(lo_b), np.abs(hi_b)), 0.0).max(-1)
    mag_hi = np.maximum(np.abs(lo_b), np.abs(hi_b)).max(-1)
    s_lo, s_hi = O.mx_scale_exponent(mag_lo), O.mx_scale_exponent(mag_hi)
    gsx = gs - 127
    assert ((gsx >= s_lo) & (gsx <= s_hi)).all(), "a scale byte lies outside its interval"
    gscale = np.exp2(gsx.astype(np.float64))[..., None]
    q_lo, q_hi = O.e4m3_round(lo_b / gscale), O.e4m3_round(hi_b / gscale)
    got = O.e4m3_decode(gc.reshape(shp))
    assert ((got >= q_lo) & (got <= q_hi)).all(), "a code lies outside its interval"
    return int((s_lo != s_hi).sum()), int((q_lo != q_hi).sum())
