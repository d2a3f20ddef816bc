"""Shared helpers of the GPU parity tests: run a workload through the C ABI
and through the oracle, and compare.

Error metric.  The required bars are a maximum relative error of 1e-4 (fp32
path) and 2e-2 (bf16-operand path); the pages define neither term.  Reading:
the relative error of an output tensor is its largest absolute deviation
relative to its largest magnitude,

    err = max_i |g_i - r_i| / max_i |r_i| .

An element-by-element ratio is ill-posed here: gradients are sums of many
signed terms and have entries near zero by cancellation, and the bf16 path's
own defined arithmetic (h and the gate errors rounded to bf16 before each
product) already moves such entries by more than 100% of their value while
moving no entry by more than ~3e-3 of the tensor's scale (measured on the
oracle alone, with and without that rounding).  The element-wise ratio with
a floor of 1e-3 of the tensor's scale is still computed and recorded as a
diagnostic (``elementwise``).

For the bf16 path a second, tighter comparison runs against the oracle in
its bf16-product mode (the same roundings as the kernels), so that a wrong
kernel cannot hide inside the 2e-2 allowance for rounding.
"""
from __future__ import annotations

import json
import os

import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2
# bf16 path vs the oracle doing the same roundings: what remains is fp32
# accumulation order and the rare operand that rounds to the other bf16
# neighbour (one bf16 ulp, 2^-8 relative) because the fp32 values differ.
TOL_BF16_EMULATED = 5e-3


def rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    peak = float(np.abs(ref).max())
    dev = float(np.abs(got - ref).max())
    return dev / peak if peak > 0 else dev


def elementwise_err(got, ref, floor=1e-3) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    peak = float(np.abs(ref).max())
    denom = np.maximum(np.abs(ref), max(floor * peak, 1e-300))
    return float(np.max(np.abs(got - ref) / denom))


def device_layers(w, device="cuda"):
    import torch
    bf16 = w.spec.dtype == "bf16"
    wdt = torch.bfloat16 if bf16 else torch.float32
    out = []
    for lay in w.layers:
        out.append({"W": torch.from_numpy(lay["W"]).to(device=device, dtype=wdt).contiguous(),
                    "R": torch.from_numpy(lay["R"]).to(device=device, dtype=wdt).contiguous(),
                    "b": torch.from_numpy(lay["b"]).to(device=device, dtype=torch.float32).contiguous(),
                    "peep": torch.from_numpy(lay["peep"]).to(device=device, dtype=torch.float32).contiguous()})
    return out


def run_gpu(w, padded: bool = False, device="cuda", ctas: int = 0, engine: int = 0, stepwise: bool = False,
            variant: int = -1):
    """pack -> all layers forward -> all layers backward -> unpack, through the C ABI."""
    import torch
    from padding_free_variable_gb300 import ops
    bf16 = w.spec.dtype == "bf16"
    plan = ops.Plan(w.lengths, padded=padded)
    if ctas:
        plan.set_ctas_per_direction(ctas)
    if variant >= 0:
        plan.debug_cluster_variant(variant)
    if engine:
        plan.set_gemm_engine(engine)
    stack = ops.PackedLSTMStack(plan, device_layers(w, device), w.spec.input_size, w.spec.hidden_size,
                                w.spec.num_directions, bf16, device, stepwise=stepwise)
    x = torch.from_numpy(w.x).to(device=device, dtype=torch.bfloat16 if bf16 else torch.float32)
    G = torch.from_numpy(w.G).to(device)
    y_cat, dx_cat = stack.step(x, G)
    torch.cuda.synchronize()
    status = plan.poll()
    assert status == 0, f"device status {status}"
    res = {"y": y_cat.cpu().numpy(), "dx": dx_cat.cpu().numpy(),
           "h_n": stack.h_n.cpu().numpy(), "c_n": stack.c_n.cpu().numpy(),
           "grads": [{k: v.cpu().numpy() for k, v in g.items()} for g in stack.grads],
           "plan": plan, "stack": stack}
    return res


def run_oracle(w, seqs=None, nthreads=None, bf16_products=False):
    """The oracle on the whole workload, or on the sequences `seqs` only."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    lengths, x, G = w.lengths, w.x, w.G
    if seqs is not None:
        st = np.concatenate([[0], np.cumsum(w.lengths)])
        lengths = w.lengths[seqs]
        x = np.concatenate([w.x[st[s]:st[s + 1]] for s in seqs])
        G = np.concatenate([w.G[st[s]:st[s + 1]] for s in seqs])
    return oracle.lstm_stack(lengths, x, w.layers, w.spec.num_directions, w.spec.hidden_size, G=G,
                             nthreads=nthreads, bf16_products=bf16_products)


def select_rows(w, seqs, arr):
    st = np.concatenate([[0], np.cumsum(w.lengths)])
    return np.concatenate([arr[st[s]:st[s + 1]] for s in seqs])


def _pairs(gpu, ref, grads):
    out = [("y", gpu["y"], ref["y"]), ("dx", gpu["dx"], ref["dx"]),
           ("h_n", gpu["h_n"], ref["h_n"]), ("c_n", gpu["c_n"], ref["c_n"])]
    if grads:
        for l, (g, r) in enumerate(zip(gpu["grads"], ref["grads"])):
            for k in ("W", "R", "b", "peep"):
                out.append((f"L{l}.d{k}", g[k], r[k]))
    return out


def record(label, kind, errs, elem):
    path = os.environ.get("PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, "against": kind, "max_rel": errs, "elementwise_1e-3": elem}) + "\n")


def compare_all(gpu, ref, tol, grads=True, label="", against="oracle"):
    pairs = _pairs(gpu, ref, grads)
    errs = {k: rel_err(g, r) for k, g, r in pairs}
    elem = {k: elementwise_err(g, r) for k, g, r in pairs}
    record(label, against, errs, elem)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label} vs {against} over tolerance {tol}: {bad} (all: {errs})"
    return errs
