"""Seeded synthetic workloads for the packed (bi)LSTM.

This module only draws numbers: sequence lengths, input frames, weights and
the fixed upstream gradient.  It holds none of the LSTM arithmetic, so both
the CPU oracle and the CUDA path can consume its output without sharing any
of the method's code.

The five workloads follow the shapes the pages describe for variable-length
recognition data (line and word strips in "No Padding Please", Sec. VII;
filterbank-like speech frames in the RETURNN paper, Sec. 6), which are not
available here:

    id  shape                                    lengths
    1   uni,  1 layer, D=16,  H=32,   fp32, B=8    uniform int [5, 40]
    2   bi,   1 layer, D=40,  H=256,  fp32, B=32   log-normal, median 300, clamp [50, 1500]
    3   bi,   5 layers, D=40, H=512,  bf16, B=64   log-normal, median 600, clamp [100, 2000]
    4   bi,   1 layer, D=64,  H=256,  fp32, B=128  uniform int [100, 1000]
    5   bi,   3 layers, D=64, H=1024, bf16, B=256  uniform int [20, 120]

Draw order from ``numpy.random.default_rng(seed)``: lengths, x, then per
layer and per direction (W, R, b, p_i, p_f, p_o), then G.  Weights use the
layout the library expects: ``W[ndir, 4H, D]``, ``R[ndir, 4H, H]``,
``b[ndir, 4H]``, ``peep[ndir, 3, H]`` (rows p_i, p_f, p_o), gate blocks in
the order (i, f, z, o) along the 4H axis.  ``x`` and ``G`` are given in the
caller's order: sequences concatenated frame after frame.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    num_directions: int
    num_layers: int
    input_size: int
    hidden_size: int
    dtype: str              # "f32" or "bf16": the GEMM operand type
    batch: int
    lengths: tuple          # ("uniform", lo, hi) or ("lognormal", median, sigma, lo, hi)
    x_dist: str             # "normal" or "uniform01"
    weight_range: float
    forget_bias: float = 0.0


WORKLOADS = {
    1: WorkloadSpec("uni-1x32-d16-b8", 1, 1, 16, 32, "f32", 8,
                    ("uniform", 5, 40), "normal", 0.1, 1.0),
    2: WorkloadSpec("bi-1x256-d40-b32", 2, 1, 40, 256, "f32", 32,
                    ("lognormal", 300.0, 0.5, 50, 1500), "normal", 0.08),
    3: WorkloadSpec("bi-5x512-d40-b64-bf16", 2, 5, 40, 512, "bf16", 64,
                    ("lognormal", 600.0, 0.5, 100, 2000), "normal", 0.05),
    4: WorkloadSpec("bi-1x256-d64-b128", 2, 1, 64, 256, "f32", 128,
                    ("uniform", 100, 1000), "uniform01", 0.1),
    5: WorkloadSpec("bi-3x1024-d64-b256-bf16", 2, 3, 64, 1024, "bf16", 256,
                    ("uniform", 20, 120), "normal", 0.03),
}


def default_seed(workload_id: int) -> int:
    return 1000 + int(workload_id)


def draw_lengths(rng: np.random.Generator, spec_lengths: tuple, batch: int) -> np.ndarray:
    kind = spec_lengths[0]
    if kind == "uniform":
        lo, hi = spec_lengths[1], spec_lengths[2]
        return rng.integers(lo, hi + 1, size=batch).astype(np.int32)   # inclusive both ends
    if kind == "lognormal":
        median, sigma, lo, hi = spec_lengths[1:]
        raw = rng.lognormal(mean=math.log(median), sigma=sigma, size=batch)
        return np.rint(np.clip(raw, lo, hi)).astype(np.int32)
    if kind == "fixed":
        return np.asarray(spec_lengths[1], dtype=np.int32)
    raise ValueError(f"unknown length distribution {kind!r}")


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bfloat16 (ties to even); result is float32."""
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    bits = a32.view(np.uint32).astype(np.uint64)
    rounding = ((bits >> 16) & 1) + 0x7FFF
    out = ((bits + rounding) >> 16) << 16
    res = out.astype(np.uint32).view(np.float32)
    # NaN stays NaN (never produced by these generators, kept for completeness)
    return np.where(np.isnan(a32), a32, res)


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    lengths: np.ndarray          # int32 [B]
    x: np.ndarray                # float32 [N, D] caller order (bf16-representable for bf16 specs)
    layers: list                 # per layer: dict W, R, b, peep (float32; W/R bf16-representable for bf16)
    G: np.ndarray                # float32 [N, ndir*H] upstream gradient of the top layer, caller order

    @property
    def N(self) -> int:
        return int(self.lengths.sum())

    @property
    def T(self) -> int:
        return int(self.lengths.max()) if len(self.lengths) else 0

    def layer_input_size(self, layer: int) -> int:
        return self.spec.input_size if layer == 0 else self.spec.num_directions * self.spec.hidden_size


def make_workload(spec: WorkloadSpec, seed: int, lengths: np.ndarray | None = None) -> Workload:
    """Draw one workload.  ``lengths`` overrides the length draw (used for edge cases)."""
    rng = np.random.default_rng(seed)
    drawn = draw_lengths(rng, spec.lengths, spec.batch)
    if lengths is not None:
        drawn = np.asarray(lengths, dtype=np.int32)
    n = int(drawn.sum())
    D, H, nd = spec.input_size, spec.hidden_size, spec.num_directions
    if spec.x_dist == "normal":
        x = rng.standard_normal((n, D))
    elif spec.x_dist == "uniform01":
        x = rng.uniform(0.0, 1.0, size=(n, D))
    else:
        raise ValueError(spec.x_dist)
    x = x.astype(np.float32)
    a = spec.weight_range
    layers = []
    for layer in range(spec.num_layers):
        Dl = D if layer == 0 else nd * H
        W = np.empty((nd, 4 * H, Dl), np.float32)
        R = np.empty((nd, 4 * H, H), np.float32)
        b = np.empty((nd, 4 * H), np.float32)
        peep = np.empty((nd, 3, H), np.float32)
        for d in range(nd):
            W[d] = rng.uniform(-a, a, size=(4 * H, Dl))
            R[d] = rng.uniform(-a, a, size=(4 * H, H))
            b[d] = rng.uniform(-a, a, size=4 * H)
            peep[d, 0] = rng.uniform(-a, a, size=H)
            peep[d, 1] = rng.uniform(-a, a, size=H)
            peep[d, 2] = rng.uniform(-a, a, size=H)
            b[d, H:2 * H] += np.float32(spec.forget_bias)
        if spec.dtype == "bf16":
            W = round_bf16(W)
            R = round_bf16(R)
        layers.append({"W": W, "R": R, "b": b, "peep": peep})
    if spec.dtype == "bf16":
        x = round_bf16(x)
    G = rng.standard_normal((n, nd * H)).astype(np.float32)
    return Workload(spec=spec, seed=seed, lengths=drawn, x=x, layers=layers, G=G)


def workload(workload_id: int, seed: int | None = None, batch: int | None = None,
             lengths: np.ndarray | None = None) -> Workload:
    """The named workload, optionally with a smaller batch (same distributions)."""
    spec = WORKLOADS[int(workload_id)]
    if batch is not None:
        spec = dataclasses.replace(spec, batch=int(batch))
    return make_workload(spec, default_seed(workload_id) if seed is None else seed, lengths)


def custom(num_directions: int, num_layers: int, input_size: int, hidden_size: int,
           lengths, seed: int, dtype: str = "f32", weight_range: float = 0.1,
           x_dist: str = "normal", forget_bias: float = 0.0) -> Workload:
    """A small ad-hoc workload with explicit lengths (edge cases, ragged tails)."""
    lengths = np.asarray(lengths, dtype=np.int32)
    spec = WorkloadSpec("custom", num_directions, num_layers, input_size, hidden_size, dtype,
                        len(lengths), ("fixed", tuple(int(v) for v in lengths)), x_dist,
                        weight_range, forget_bias)
    return make_workload(spec, seed)


# --------------------------------------------------------------------------- 2-D (MDLSTM) workloads
#
# "No Padding Please", Sec. VII: word strips (IAM words, batch 200 with packing)
# and line strips (IAM lines, batch 12 with packing) feed MDLSTM layers of 2 to 100
# units after block-strided convolutions.  The page gives no image-size
# distribution; these stand-ins draw heights and widths uniformly in ranges of the
# feature maps such strips give after the model's first 4x down-sampling, one
# MDLSTM layer with its four scan directions.
#
#   name    images  height   width     D   H
#   words   200     [8, 24]  [8, 96]   16  32
#   lines   12      [12, 20] [200, 600] 16 32
#
# Draw order from ``numpy.random.default_rng(seed)``: heights, widths, x, then per
# direction (W, U1, U2, b, peep), then G; the named workloads then add a forget bias of -1
# to both forget gates' biases.  Layouts: W[ndir, 5H, D], U1/U2[ndir, 5H, H],
# b[ndir, 5H], peep[ndir, 6, H] (p_i1, p_i2, p_f1, p_f2, p_o1, p_o2), gate blocks in
# the order (i, f1, f2, z, o); x[N, D] and G[N, ndir*H] in caller order (images back to
# back, each row by row).


@dataclasses.dataclass(frozen=True)
class MdSpec:
    name: str
    num_directions: int
    input_size: int
    hidden_size: int
    batch: int
    heights: tuple          # ("uniform", lo, hi)
    widths: tuple
    x_dist: str
    weight_range: float
    forget_bias: float = -1.0


# forget bias -1 on both forget gates: f1 + f2 stays near 0.5 instead of 1, the regime in which
# the 2-D state does not grow along the scan (Sec. III: with the two forget gates summing to
# more than one the state norm grows, the instability the page's stable cells address)
MD_WORKLOADS = {
    "words": MdSpec("md-4x32-d16-words-b200", 4, 16, 32, 200, ("uniform", 8, 24), ("uniform", 8, 96),
                    "uniform01", 0.1),
    "lines": MdSpec("md-4x32-d16-lines-b12", 4, 16, 32, 12, ("uniform", 12, 20), ("uniform", 200, 600),
                    "uniform01", 0.1),
}


@dataclasses.dataclass
class MdWorkload:
    name: str
    heights: np.ndarray
    widths: np.ndarray
    x: np.ndarray
    layer: dict
    G: np.ndarray
    num_directions: int
    input_size: int
    hidden_size: int

    @property
    def N(self) -> int:
        return int((self.heights.astype(np.int64) * self.widths).sum())


def md_custom(num_directions: int, input_size: int, hidden_size: int, heights, widths, seed: int,
              weight_range: float = 0.1, x_dist: str = "normal", name: str = "md-custom",
              forget_bias: float = -1.0) -> MdWorkload:
    rng = np.random.default_rng(seed)
    hs = np.asarray(heights, dtype=np.int32)
    ws = np.asarray(widths, dtype=np.int32)
    return _md_draw(rng, name, num_directions, input_size, hidden_size, hs, ws, weight_range, x_dist, forget_bias)


def _md_draw(rng, name, nd, D, H, hs, ws, wr, x_dist, forget_bias=0.0) -> MdWorkload:
    N = int((hs.astype(np.int64) * ws).sum())
    if x_dist == "uniform01":
        x = rng.uniform(0.0, 1.0, (N, D))
    else:
        x = rng.standard_normal((N, D))
    keys = ("W", "U1", "U2", "b", "peep")
    shapes = {"W": (5 * H, D), "U1": (5 * H, H), "U2": (5 * H, H), "b": (5 * H,), "peep": (6, H)}
    per = {k: [] for k in keys}
    for _ in range(nd):
        for k in keys:
            per[k].append(rng.uniform(-wr, wr, shapes[k]))
    layer = {k: np.stack(v) for k, v in per.items()}
    layer["b"][:, H:3 * H] += forget_bias              # the two forget gates' blocks
    layer = {k: v.astype(np.float32) for k, v in layer.items()}
    G = rng.standard_normal((N, nd * H))
    return MdWorkload(name, hs, ws, x.astype(np.float32), layer, G.astype(np.float32), nd, D, H)


def md_workload(name: str = "words", seed: int | None = None, batch: int | None = None) -> MdWorkload:
    spec = MD_WORKLOADS[name]
    rng = np.random.default_rng(4242 if seed is None else seed)
    n = spec.batch if batch is None else int(batch)
    hs = rng.integers(spec.heights[1], spec.heights[2] + 1, n).astype(np.int32)
    ws = rng.integers(spec.widths[1], spec.widths[2] + 1, n).astype(np.int32)
    return _md_draw(rng, spec.name, spec.num_directions, spec.input_size, spec.hidden_size, hs, ws,
                    spec.weight_range, spec.x_dist, spec.forget_bias)
