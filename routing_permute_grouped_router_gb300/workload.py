"""Seeded synthetic workloads for the mixture-of-experts layer step.

This module only draws inputs. It holds none of the layer's arithmetic, and it
is shared by the parity tests (which hand the same arrays to the CPU oracle and
to the CUDA library) and by ``bench.py``.

The five workloads restate the layer configurations that the expert-parallel
training step is measured on ("The step timeline: dispatch, expert GEMM,
combine" on the gpu_expert_parallel page; capacity factor and top-k from the
"Expert Parallelism" section of the distributed-training tutorial):

==================  =====  ====  ====  ==  =  ========  =====  ===========
name                T      d     f     E   k  capacity  dtype  router bias
==================  =====  ====  ====  ==  =  ========  =====  ===========
switch_tiny_f32       256    64   128   4  1  cf 1.25   f32    0
top2_e8_bf16         4096  1024  4096   8  2  cf 1.25   bf16   0
zipf_e64_bf16       16384  2048  2048  64  2  cf 1.0    bf16   log-Zipf 1.1
dropless_e32_bf16   32768  4096  1536  32  4  none      bf16   log-Zipf 1.3
train_e16_bf16       8192  2048  4096  16  2  cf 1.25   bf16   0  (x4 micro-batches, fwd+bwd)
==================  =====  ====  ====  ==  =  ========  =====  ===========

Recipe (all draws from numpy's PCG64):

* expert and router weights from ``default_rng([seed, 0])`` in the order
  W_r [d,E] ~ N(0, 1/d), W1 [E,d,f] ~ N(0, 1/d), W3 [E,d,f] ~ N(0, 1/d),
  W2 [E,f,d] ~ N(0, 1/f);
* micro-batch m draws x [T,d] ~ N(0,1) and then dY [T,d] ~ N(0,1) from
  ``default_rng([seed, 1, m])``;
* the router bias is b_e = -s * ln(e + 1) for the Zipf workloads (the softmax
  of the bias alone is then proportional to (e+1)^-s), zero otherwise;
* for bf16 workloads x, W1, W3, W2 and dY are rounded to bf16
  (round-to-nearest-even); W_r and b stay fp32;
* margin filter: any token whose sorted router logits have a gap below
  ``margin`` (1e-3) among the top min(k+1, E) is redrawn from
  ``default_rng([seed, 2, m, attempt])`` until none is left.  The filter only
  selects inputs; nothing it computes is handed to either side.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Sizes of one mixture-of-experts layer workload."""

    name: str
    T: int
    d_model: int
    d_ff: int
    E: int
    k: int
    capacity_factor: float  # <= 0 means dropless
    dtype: str
    zipf_s: float = 0.0
    micro_batches: int = 1
    backward: bool = False
    capacity: int = -1  # >= 0 overrides the capacity factor

    def replace(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "switch_tiny_f32": LayerShape("switch_tiny_f32", 256, 64, 128, 4, 1, 1.25, F32),
    "top2_e8_bf16": LayerShape("top2_e8_bf16", 4096, 1024, 4096, 8, 2, 1.25, BF16),
    "zipf_e64_bf16": LayerShape("zipf_e64_bf16", 16384, 2048, 2048, 64, 2, 1.0, BF16, zipf_s=1.1),
    "dropless_e32_bf16": LayerShape("dropless_e32_bf16", 32768, 4096, 1536, 32, 4, 0.0, BF16, zipf_s=1.3),
    "train_e16_bf16": LayerShape("train_e16_bf16", 8192, 2048, 4096, 16, 2, 1.25, BF16,
                                 micro_batches=4, backward=True),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the raw uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_widen(bits: np.ndarray) -> np.ndarray:
    """Exact float32 values of raw bfloat16 bits."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


class Tensor:
    """One input array: the exact float32 values and, for bf16, the raw bits to upload."""

    def __init__(self, values32: np.ndarray, dtype: str):
        if dtype == BF16:
            self.bits = bf16_bits(values32)
            self.f32 = bf16_widen(self.bits)
        else:
            self.bits = None
            self.f32 = np.ascontiguousarray(values32, dtype=np.float32)
        self.dtype = dtype

    def set_rows(self, rows: np.ndarray, values32: np.ndarray) -> None:
        """Replace the given leading-axis rows (used by the margin redraw)."""
        if self.dtype == BF16:
            self.bits[rows] = bf16_bits(values32)
            self.f32[rows] = bf16_widen(self.bits[rows])
        else:
            self.f32[rows] = values32

    @property
    def shape(self):
        return self.f32.shape

    def f64(self) -> np.ndarray:
        return self.f32.astype(np.float64)

    def torch(self, device="cpu"):
        """The array as a torch tensor in the workload dtype (bf16 from the exact bits)."""
        import torch

        if self.dtype == BF16:
            t = torch.from_numpy(self.bits.view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(self.f32)
        return t.to(device)


@dataclasses.dataclass
class Workload:
    shape: LayerShape
    W_r: np.ndarray  # [d, E] float32
    bias: Optional[np.ndarray]  # [E] float32 or None
    W1: Tensor  # [E, d, f]
    W3: Tensor  # [E, d, f]
    W2: Tensor  # [E, f, d]
    x: List[Tensor]  # per micro-batch [T, d]
    dy: List[Tensor]  # per micro-batch [T, d] (empty unless backward)
    redrawn: int = 0


def _normal(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def zipf_bias(E: int, s: float) -> np.ndarray:
    """b_e = -s ln(e+1): softmax of the bias alone is proportional to (e+1)^-s."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def _rows_failing_margin(x32: np.ndarray, W_r: np.ndarray, bias, k: int, margin: float) -> np.ndarray:
    """Token indices whose top-min(k+1,E) sorted logits have a gap below ``margin``."""
    s = x32.astype(np.float64) @ W_r.astype(np.float64)
    if bias is not None:
        s += bias.astype(np.float64)
    E = s.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-s, axis=1)[:, :m]
    if m < 2:
        return np.zeros(0, dtype=np.int64)
    gaps = top[:, :-1] - top[:, 1:]
    return np.nonzero((gaps < margin).any(axis=1))[0]


def make(shape: LayerShape, seed: int = 0, margin: float = 1e-3, micro_batches: Optional[int] = None,
         with_dy: Optional[bool] = None) -> Workload:
    """Draw one workload following the recipe in the module docstring."""
    T, d, f, E, k = shape.T, shape.d_model, shape.d_ff, shape.E, shape.k
    nmb = shape.micro_batches if micro_batches is None else micro_batches
    want_dy = shape.backward if with_dy is None else with_dy
    wr = np.random.default_rng([seed, 0])
    W_r = _normal(wr, (d, E), 1.0 / math.sqrt(d))
    W1 = Tensor(_normal(wr, (E, d, f), 1.0 / math.sqrt(d)), shape.dtype)
    W3 = Tensor(_normal(wr, (E, d, f), 1.0 / math.sqrt(d)), shape.dtype)
    W2 = Tensor(_normal(wr, (E, f, d), 1.0 / math.sqrt(f)), shape.dtype)
    bias = zipf_bias(E, shape.zipf_s) if shape.zipf_s > 0 else None
    xs, dys = [], []
    redrawn = 0
    for m in range(nmb):
        rm = np.random.default_rng([seed, 1, m])
        x32 = _normal(rm, (T, d), 1.0)
        dy32 = _normal(rm, (T, d), 1.0) if want_dy else None
        x = Tensor(x32, shape.dtype)
        if margin > 0:
            attempt = 0
            bad = _rows_failing_margin(x.f32, W_r, bias, k, margin)
            while bad.size:
                if attempt > 1000:
                    raise RuntimeError("margin filter did not converge")
                rr = np.random.default_rng([seed, 2, m, attempt])
                x.set_rows(bad, _normal(rr, (bad.size, d), 1.0))
                redrawn += bad.size
                bad = bad[_rows_failing_margin(x.f32[bad], W_r, bias, k, margin)]
                attempt += 1
        xs.append(x)
        if want_dy:
            dys.append(Tensor(dy32, shape.dtype))
    return Workload(shape, W_r, bias, W1, W3, W2, xs, dys, redrawn)
