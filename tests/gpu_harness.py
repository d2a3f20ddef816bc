"""Shared helpers of the GPU parity tests: run a workload through the C ABI
and through the oracle, and compare.

Error metrics.  The required bars are a maximum relative error of 1e-4 (fp32
path) and 2e-2 (bf16-operand path); the pages define neither term.  Two
readings are computed for every output tensor:

    normwise     err = max_i |g_i - r_i| / max_i |r_i|
    element-wise err = max_i |g_i - r_i| / max(|r_i|, 1e-3 max_j |r_j|)

The fp32 path is gated on BOTH: the normwise error at 1e-4, and the
element-wise error (floor 1e-3 of the tensor's scale) at TOL_F32_ELEMENTWISE.
That second bar is set from what plain fp32 arithmetic reaches on these
cases: the CUDA-core engine (FFMA products, fp32 accumulation) measured up
to 1.0e-3 element-wise against the fp64 oracle on the same inputs (workload
2's dpeep; workload 4's dW 9.2e-4; the small cases 1.5e-4 to 5.0e-4), so
no fp32 implementation meets 1e-4 element-wise on every entry near the
floor.  2e-3 is twice that worst case, and 2-9x below what the products
reached when each term kept only 2^-17 of its value (a two-piece bf16
split: 3.5e-3 to 1.7e-2 on workloads 2 and 4).

The bf16 path is gated normwise only.  Its own defined arithmetic (h and the
gate errors rounded to bf16 before each product) moves gradient entries near
zero by more than 100% of their value while moving no entry by more than
~3e-3 of the tensor's scale (measured on the oracle alone, with and without
that rounding), so an element-wise ratio would reject every correct bf16
implementation; it is still recorded (``elementwise``).  A second, tighter
comparison runs against the oracle in its bf16-product mode (the same
roundings as the kernels), so that a wrong kernel cannot hide inside the
2e-2 allowance for rounding.
"""
from __future__ import annotations

import json
import os

import numpy as np

TOL_F32 = 1e-4
TOL_F32_ELEMENTWISE = 2e-3
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
    from padding_free_variable_gb300 import ops
    return ops.device_layers(w.layers, w.spec.dtype == "bf16", device)


def run_gpu(w, padded: bool = False, device="cuda", ctas: int = 0, engine: int = 0, stepwise: bool = False,
            variant: int = -1, group_slots: int = 0, states=None):
    """pack -> all layers forward -> all layers backward -> unpack, through the C ABI.
    states: optional dict of numpy h0, c0, dh_n, dc_n [layers][ndir][B][H] (lstm_fwd_state /
    lstm_bwd_state); the result then holds dh0 and dc0 too."""
    import torch
    from padding_free_variable_gb300 import ops
    bf16 = w.spec.dtype == "bf16"
    plan = ops.Plan(w.lengths, padded=padded)
    if ctas:
        plan.set_ctas_per_direction(ctas)
    if variant >= 0:
        plan.debug_cluster_variant(variant)
    if group_slots:
        plan.debug_sequence_groups(group_slots)
    if engine:
        plan.set_gemm_engine(engine)
    stack = ops.PackedLSTMStack(plan, device_layers(w, device), w.spec.input_size, w.spec.hidden_size,
                                w.spec.num_directions, bf16, device, stepwise=stepwise)
    if states is not None:
        dev = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device))
               for k, v in states.items()}
        stack.set_states(dev.get("h0"), dev.get("c0"), dev.get("dh_n"), dev.get("dc_n"))
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
    if states is not None:
        res["dh0"] = stack.dh0.cpu().numpy()
        res["dc0"] = stack.dc0.cpu().numpy()
    return res


def run_oracle(w, seqs=None, nthreads=None, bf16_products=False, states=None):
    """The oracle on the whole workload, or on the sequences `seqs` only (optionally from
    initial states, with final-state errors: a dict of h0, c0, dh_n, dc_n)."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    lengths, x, G = w.lengths, w.x, w.G
    if seqs is not None:
        st = np.concatenate([[0], np.cumsum(w.lengths)])
        lengths = w.lengths[seqs]
        x = np.concatenate([w.x[st[s]:st[s + 1]] for s in seqs])
        G = np.concatenate([w.G[st[s]:st[s + 1]] for s in seqs])
    st = states or {}
    return oracle.lstm_stack(lengths, x, w.layers, w.spec.num_directions, w.spec.hidden_size, G=G,
                             nthreads=nthreads, bf16_products=bf16_products, h0=st.get("h0"), c0=st.get("c0"),
                             dh_n=st.get("dh_n"), dc_n=st.get("dc_n"))


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
        for k in ("dh0", "dc0"):
            if k in gpu:
                out.append((k, gpu[k], ref[k]))
    return out


def record(label, kind, errs, elem):
    path = os.environ.get("PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, "against": kind, "max_rel": errs, "elementwise_1e-3": elem}) + "\n")


def compare_all(gpu, ref, tol, grads=True, label="", against="oracle", elem_tol=None):
    """Normwise gate at `tol`; element-wise gate at `elem_tol` (default: TOL_F32_ELEMENTWISE
    for the fp32 bar, none for the bf16 bars)."""
    if elem_tol is None and tol == TOL_F32:
        elem_tol = TOL_F32_ELEMENTWISE
    pairs = _pairs(gpu, ref, grads)
    errs = {k: rel_err(g, r) for k, g, r in pairs}
    elem = {k: elementwise_err(g, r) for k, g, r in pairs}
    record(label, against, errs, elem)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label} vs {against} over tolerance {tol}: {bad} (all: {errs})"
    if elem_tol is not None:
        bad = {k: v for k, v in elem.items() if not v <= elem_tol}
        assert not bad, f"{label} vs {against} element-wise over {elem_tol}: {bad} (all: {elem})"
    return errs
