"""Seeded synthetic inputs for the MoE layer (shared by the oracle tests, the GPU
tests and the benchmark).

This module only draws random numbers and stores them as bfloat16 bit patterns.
It holds none of the layer's arithmetic: no router, no schedule, no expert FFN.
Both the CPU oracle and the CUDA library consume the exact same bf16 bytes.

Workloads (the pages print no model dimensions except the hidden size 7168 and
the expert intermediate size 2048 of the "Kimi 2.5" shape in the minibatch
discussion, Mixture-of-Kittens article (kucoin.com), section 02):

  name                          T      H     E   k    F    precision  router skew
  tiny_T256_H256_E8_k2_F512     256    256   8   2    512  bf16       none
  balanced_T4096_H2048_E32_k4   4096   2048  32  4    1024 bf16       none
  skewed_T8192_H4096_E64_k8     8192   4096  64  8    1536 bf16       Zipf s=1.2 bias
  mxfp8_T8192_H7168_E16_k8      8192   7168  16  8    2048 mxfp8      Zipf s=0.8 bias
  ring_T16384_H7168_E16_k8      16384  7168  16  8    2048 mxfp8      Zipf s=1.0 bias, 256 MiB ring

Distributions: x and the upstream gradient dout ~ N(0, 1); W1, W3, W2 and the
router weight W_r ~ N(0, 0.02); the optional router bias is
bias_e = ln z_(e+1) with z_r proportional to r^-s (a Zipf pmf over expert rank).

Every tensor has its own Philox stream keyed by (seed, tensor name), drawn in
float32 and rounded to bfloat16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Optional

import numpy as np

MIB = 1 << 20


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    F: int
    precision: str = "bf16"          # "bf16" or "mxfp8"
    zipf_s: Optional[float] = None   # router bias skew, None = no bias
    backward: bool = True
    ring_bytes: int = 0              # 0 = ring sized to hold every routed row
    minibatch_rows: tuple = ()       # sweep values (ring workload only)
    seed: int = 0
    weight_std: float = 0.02

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_T256_H256_E8_k2_F512", 256, 256, 8, 2, 512),
        Workload("balanced_T4096_H2048_E32_k4_F1024", 4096, 2048, 32, 4, 1024),
        Workload("skewed_T8192_H4096_E64_k8_F1536", 8192, 4096, 64, 8, 1536, zipf_s=1.2),
        Workload("mxfp8_T8192_H7168_E16_k8_F2048", 8192, 7168, 16, 8, 2048,
                 precision="mxfp8", zipf_s=0.8),
        Workload("ring_T16384_H7168_E16_k8_F2048", 16384, 7168, 16, 8, 2048,
                 precision="mxfp8", zipf_s=1.0, ring_bytes=256 * MIB,
                 minibatch_rows=(512, 1024, 1536, 2048, 2560, 3072)),
    ]
}

TINY = WORKLOADS["tiny_T256_H256_E8_k2_F512"]
BALANCED = WORKLOADS["balanced_T4096_H2048_E32_k4_F1024"]
SKEWED = WORKLOADS["skewed_T8192_H4096_E64_k8_F1536"]
MXFP8 = WORKLOADS["mxfp8_T8192_H7168_E16_k8_F2048"]
RING = WORKLOADS["ring_T16384_H7168_E16_k8_F2048"]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.
    Inputs here are finite normal samples, so no NaN handling is needed."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _stream(seed: int, name: str) -> np.random.Generator:
    key = (int(seed) << 32) | zlib.crc32(name.encode())
    return np.random.Generator(np.random.Philox(key=key))


def normal_bf16(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) samples as bf16 bits, one Philox stream per tensor name."""
    n = int(np.prod(shape))
    g = _stream(seed, name)
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 26
    for s in range(0, n, chunk):
        v = g.standard_normal(min(chunk, n - s), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:s + len(v)] = f32_to_bf16_bits(v)
    return out.reshape(shape)


def zipf_bias(E: int, s: Optional[float]) -> Optional[np.ndarray]:
    """Per-expert router logit bias ln(pmf) of a Zipf(s) law over rank e+1."""
    if s is None:
        return None
    r = np.arange(1, E + 1, dtype=np.float64)
    pmf = r ** (-s)
    pmf /= pmf.sum()
    return np.log(pmf).astype(np.float32)


def make_inputs(w: Workload, tokens: Optional[int] = None, need=("x", "Wr", "W1", "W3", "W2", "dout")):
    """Returns a dict of host arrays: bf16 bit tensors (uint16) and the fp32 bias.

    x [T,H], Wr [H,E], W1 [E,H,F], W3 [E,H,F], W2 [E,F,H], dout [T,H], bias [E] or None.
    `tokens` truncates x/dout to their first rows (same values as the full draw)."""
    T = w.T
    out = {"bias": zipf_bias(w.E, w.zipf_s)}
    shapes = {
        "x": ((T, w.H), 1.0),
        "Wr": ((w.H, w.E), w.weight_std),
        "W1": ((w.E, w.H, w.F), w.weight_std),
        "W3": ((w.E, w.H, w.F), w.weight_std),
        "W2": ((w.E, w.F, w.H), w.weight_std),
        "dout": ((T, w.H), 1.0),
    }
    for name in need:
        shape, std = shapes[name]
        a = normal_bf16(w.seed, name, shape, std)
        if tokens is not None and name in ("x", "dout"):
            a = a[:tokens]
        out[name] = a
    return out
