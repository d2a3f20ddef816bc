"""Python-side use of the C ABI: plans, per-layer calls and a layer stack.

PyTorch is used for device memory and streams only; every step of the path
(pack, products, recurrence, BPTT, unpack) runs in liblstm_packed.so.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import LayerGrads, LayerParams, LayerShape, State, StateGrads, check


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class Plan:
    """Packing plan of one batch of sequence lengths: packed (default), the padded layout,
    a segment plan (``segments=(chunk, step)``: lstm_plan_create_segments) or a window plan
    (``window=(start, width)``: lstm_plan_create_window)."""

    def __init__(self, lengths, padded: bool = False, segments=None, window=None):
        lib = _lib.load()
        lens = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
        self.lengths = lens
        self.padded = padded
        h = ctypes.c_void_p()
        lp = lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        if segments is not None:
            check(lib.lstm_plan_create_segments(lp, int(lens.size), int(segments[0]), int(segments[1]),
                                                ctypes.byref(h)), "lstm_plan_create_segments")
        elif window is not None:
            check(lib.lstm_plan_create_window(lp, int(lens.size), int(window[0]), int(window[1]), ctypes.byref(h)),
                  "lstm_plan_create_window")
        else:
            fn = lib.lstm_plan_create_padded if padded else lib.lstm_plan_create
            check(fn(lp, int(lens.size), ctypes.byref(h)), "lstm_plan_create")
        self.handle = h
        rows, frames = ctypes.c_int64(), ctypes.c_int64()
        steps, batch = ctypes.c_int32(), ctypes.c_int32()
        check(lib.lstm_plan_info(h, ctypes.byref(rows), ctypes.byref(steps), ctypes.byref(batch),
                                 ctypes.byref(frames)), "lstm_plan_info")
        self.rows, self.steps, self.batch, self.frames = rows.value, steps.value, batch.value, frames.value

    def tables(self):
        """(batch_sizes[T], offsets[T+1], perm[B], slot_len[B]) as numpy copies."""
        lib = _lib.load()
        p = [ctypes.POINTER(ctypes.c_int32)() for _ in range(4)]
        check(lib.lstm_plan_tables(self.handle, *[ctypes.byref(q) for q in p]), "lstm_plan_tables")
        T, B = self.steps, self.batch
        return (np.ctypeslib.as_array(p[0], (T,)).copy() if T else np.zeros(0, np.int32),
                np.ctypeslib.as_array(p[1], (T + 1,)).copy(),
                np.ctypeslib.as_array(p[2], (B,)).copy(),
                np.ctypeslib.as_array(p[3], (B,)).copy())

    def set_wait_limit(self, ns: int):
        check(_lib.load().lstm_plan_set_wait_limit(self.handle, int(ns)), "lstm_plan_set_wait_limit")

    def set_ctas_per_direction(self, ctas: int):
        check(_lib.load().lstm_plan_set_ctas_per_direction(self.handle, int(ctas)),
              "lstm_plan_set_ctas_per_direction")

    def enable_timing(self, on: bool = True):
        check(_lib.load().lstm_plan_enable_timing(self.handle, int(bool(on))), "lstm_plan_enable_timing")

    def read_timing(self) -> dict:
        """{kind: (milliseconds, timed calls)} summed since timing was enabled."""
        n = len(_lib.KERNEL_KINDS)
        ms = (ctypes.c_double * n)()
        calls = (ctypes.c_int64 * n)()
        check(_lib.load().lstm_plan_read_timing(self.handle, ms, calls), "lstm_plan_read_timing")
        return {k: (ms[i], calls[i]) for i, k in enumerate(_lib.KERNEL_KINDS)}

    def launch_count(self) -> int:
        return int(_lib.load().lstm_plan_launch_count(self.handle))

    def recurrent_config(self, backward: bool = False) -> dict:
        """Configuration of the last forward (or backward) recurrent launch."""
        k, g, m, v = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        check(_lib.load().lstm_plan_recurrent_config(self.handle, int(bool(backward)), ctypes.byref(k),
                                                     ctypes.byref(g), ctypes.byref(m), ctypes.byref(v)),
              "lstm_plan_recurrent_config")
        kind = ("none", "grid", "cluster", "step_launches", "persistent_wide")[k.value]
        out = {"kernel": kind, "ctas_per_direction": g.value, "product": ("cuda_cores", "mma_sync", "tcgen05")[m.value]}
        if kind == "persistent_wide":
            out["cluster_size"] = v.value            # CTAs sharing each operand tile by multicast
        else:
            out.update({"exchange": "bulk" if v.value & 1 else "barrier", "tma_tiles": bool(v.value & 2)})
        return out

    def recurrent_groups(self, backward: bool = False) -> tuple:
        """(sequence groups, sorted slots per group) of the last forward (or backward) recurrent launch."""
        g, r = ctypes.c_int32(), ctypes.c_int32()
        check(_lib.load().lstm_plan_recurrent_groups(self.handle, int(bool(backward)), ctypes.byref(g),
                                                     ctypes.byref(r)), "lstm_plan_recurrent_groups")
        return g.value, r.value

    def debug_wide_recurrence(self, mode: int):
        """bf16 layers with H > 512: -1 automatic, 0 per-step launches, 1 the persistent kernel."""
        check(_lib.load().lstm_debug_wide_recurrence(self.handle, int(mode)), "lstm_debug_wide_recurrence")

    def debug_wide_stages(self, max_stages: int = -1) -> tuple:
        """Cap the persistent wide kernels' operand-ring depth (0 none, -1 unchanged); returns the
        depths (forward, backward) the last persistent launches used."""
        f, b = ctypes.c_int32(), ctypes.c_int32()
        check(_lib.load().lstm_debug_wide_stages(self.handle, int(max_stages), ctypes.byref(f), ctypes.byref(b)),
              "lstm_debug_wide_stages")
        return f.value, b.value

    def debug_sequence_groups(self, slots: int):
        """Force the cluster kernels' slots per sequence group (0 = automatic)."""
        check(_lib.load().lstm_debug_sequence_groups(self.handle, int(slots)), "lstm_debug_sequence_groups")

    def trace_steps(self, buffer, steps: int):
        """Phase stamps into `buffer` (int64 device tensor of 2*ndir*steps*8), or off with steps=0."""
        check(_lib.load().lstm_debug_trace_steps(self.handle, _ptr(buffer), int(steps)), "lstm_debug_trace_steps")

    def set_gemm_engine(self, engine: int):
        """0 = tensor cores for bf16 operands (default), 1 = CUDA cores."""
        check(_lib.load().lstm_plan_set_gemm_engine(self.handle, int(engine)), "lstm_plan_set_gemm_engine")

    def debug_skip_arrival(self, cta: int):
        check(_lib.load().lstm_debug_skip_arrival(self.handle, int(cta)), "lstm_debug_skip_arrival")

    def debug_cluster_variant(self, variant: int):
        """Restrict the cluster recurrent kernels to one variant (-1 automatic; bit 0 bulk, bit 1 TMA tiles)."""
        check(_lib.load().lstm_debug_cluster_variant(self.handle, int(variant)), "lstm_debug_cluster_variant")

    def poll(self, stream=None) -> int:
        """Synchronise and return (and clear) the device status code."""
        return int(_lib.load().lstm_status_poll(self.handle, _stream(stream)))

    def pack(self, x_cat: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        width = x_cat.shape[1]
        if out is None:
            out = torch.empty((self.rows, width), dtype=x_cat.dtype, device=x_cat.device)
        check(_lib.load().lstm_pack(self.handle, _ptr(x_cat), width, x_cat.element_size(), _ptr(out),
                                    _stream(stream)), "lstm_pack")
        return out

    def unpack(self, y_packed: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        width = y_packed.shape[1]
        if out is None:
            out = torch.empty((self.frames, width), dtype=y_packed.dtype, device=y_packed.device)
        check(_lib.load().lstm_unpack(self.handle, _ptr(y_packed), width, y_packed.element_size(),
                                      _ptr(out), _stream(stream)), "lstm_unpack")
        return out

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            _lib.load().lstm_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def segments_host(lengths, chunk: int, step: int):
    """(sequence, start, length) arrays of lstm_plan_create_segments' segments (host only)."""
    lib = _lib.load()
    lens = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
    lp = lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    n = ctypes.c_int32()
    check(lib.lstm_segments_host(lp, int(lens.size), int(chunk), int(step), ctypes.byref(n), None, None, None, 0),
          "lstm_segments_host")
    out = [np.zeros(n.value, np.int32) for _ in range(3)]
    ptrs = [o.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) for o in out]
    check(lib.lstm_segments_host(lp, int(lens.size), int(chunk), int(step), ctypes.byref(n), *ptrs, n.value),
          "lstm_segments_host")
    return tuple(out)


def form_batches(lengths, budget: int, padded_budget: bool = False) -> np.ndarray:
    """Batch index of each sequence under a frame budget (lstm_form_batches; host only)."""
    lib = _lib.load()
    lens = np.ascontiguousarray(np.asarray(lengths, dtype=np.int32))
    out = np.zeros(lens.size, np.int32)
    nb = ctypes.c_int32()
    check(lib.lstm_form_batches(lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(lens.size), int(budget),
                                1 if padded_budget else 0, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                ctypes.byref(nb)), "lstm_form_batches")
    return out


def device_layers(layers, bf16: bool, device="cuda") -> list:
    """Per-layer parameter dicts (numpy W, R, b, peep in the header's layout) as device tensors:
    W and R in the layer's operand type (bf16 or fp32), b and peep fp32."""
    wdt = torch.bfloat16 if bf16 else torch.float32
    out = []
    for lay in layers:
        out.append({"W": torch.from_numpy(np.ascontiguousarray(lay["W"])).to(device=device, dtype=wdt).contiguous(),
                    "R": torch.from_numpy(np.ascontiguousarray(lay["R"])).to(device=device, dtype=wdt).contiguous(),
                    "b": torch.from_numpy(np.ascontiguousarray(lay["b"])).to(device=device, dtype=torch.float32),
                    "peep": torch.from_numpy(np.ascontiguousarray(lay["peep"])).to(device=device,
                                                                                   dtype=torch.float32)})
    return out


def layer_shape(input_size, hidden_size, num_directions, bf16: bool) -> LayerShape:
    return LayerShape(int(input_size), int(hidden_size), int(num_directions),
                      _lib.LSTM_BF16 if bf16 else _lib.LSTM_F32)


def workspace_bytes(plan: Plan, shape: LayerShape) -> int:
    return int(_lib.load().lstm_workspace_bytes(plan.handle, ctypes.byref(shape)))


def scratch_bytes(plan: Plan, shape: LayerShape) -> int:
    return int(_lib.load().lstm_scratch_bytes(plan.handle, ctypes.byref(shape)))


def _params(layer: dict) -> LayerParams:
    return LayerParams(layer["W"].data_ptr(), layer["R"].data_ptr(), layer["b"].data_ptr(),
                       layer["peep"].data_ptr())


def input_projection(plan: Plan, shape: LayerShape, layer: dict, x_packed, out, stream=None):
    check(_lib.load().lstm_debug_input_projection(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)),
                                                  _ptr(x_packed), _ptr(out), _stream(stream)),
          "lstm_debug_input_projection")


def layer_forward(plan: Plan, shape: LayerShape, layer: dict, x_packed, y_packed, y_lo, h_n, c_n,
                  workspace, stream=None):
    check(_lib.load().lstm_fwd(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)),
                               _ptr(x_packed), _ptr(y_packed), _ptr(y_lo), _ptr(h_n), _ptr(c_n),
                               _ptr(workspace), _stream(stream)), "lstm_fwd")


def layer_backward(plan: Plan, shape: LayerShape, layer: dict, x_packed, y_packed, workspace, dy_packed,
                   dx_packed, grads: dict, scratch, stream=None):
    g = LayerGrads(grads["W"].data_ptr(), grads["R"].data_ptr(), grads["b"].data_ptr(),
                   grads["peep"].data_ptr())
    check(_lib.load().lstm_bwd(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)),
                               _ptr(x_packed), _ptr(y_packed), _ptr(workspace), _ptr(dy_packed),
                               _ptr(dx_packed), ctypes.byref(g), _ptr(scratch), _stream(stream)),
          "lstm_bwd")


def state_scratch_bytes(plan: Plan, shape: LayerShape) -> int:
    return int(_lib.load().lstm_state_scratch_bytes(plan.handle, ctypes.byref(shape)))


def layer_forward_state(plan: Plan, shape: LayerShape, layer: dict, h0, c0, x_packed, y_packed, y_lo, h_n, c_n,
                        workspace, state_scratch, stream=None):
    """lstm_fwd_state: the layer starting from h0 / c0 ([ndir][B][H] fp32 device tensors or None)."""
    st = State(0 if h0 is None else h0.data_ptr(), 0 if c0 is None else c0.data_ptr())
    check(_lib.load().lstm_fwd_state(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)), ctypes.byref(st),
                                     _ptr(x_packed), _ptr(y_packed), _ptr(y_lo), _ptr(h_n), _ptr(c_n),
                                     _ptr(workspace), _ptr(state_scratch), _stream(stream)), "lstm_fwd_state")


def layer_backward_state(plan: Plan, shape: LayerShape, layer: dict, h0, c0, x_packed, y_packed, workspace, dy_packed,
                         dx_packed, grads: dict, dh_n, dc_n, dh0, dc0, scratch, state_scratch, stream=None):
    """lstm_bwd_state: also takes dL/dh_n, dL/dc_n and returns dL/dh0, dL/dc0 (any may be None)."""
    st = State(0 if h0 is None else h0.data_ptr(), 0 if c0 is None else c0.data_ptr())
    sg = StateGrads(*[0 if t is None else t.data_ptr() for t in (dh_n, dc_n, dh0, dc0)])
    g = LayerGrads(grads["W"].data_ptr(), grads["R"].data_ptr(), grads["b"].data_ptr(), grads["peep"].data_ptr())
    check(_lib.load().lstm_bwd_state(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)), ctypes.byref(st),
                                     _ptr(x_packed), _ptr(y_packed), _ptr(workspace), _ptr(dy_packed),
                                     _ptr(dx_packed), ctypes.byref(g), ctypes.byref(sg), _ptr(scratch),
                                     _ptr(state_scratch), _stream(stream)), "lstm_bwd_state")


def stepwise_scratch_bytes(plan: Plan, shape: LayerShape) -> int:
    return int(_lib.load().lstm_stepwise_scratch_bytes(plan.handle, ctypes.byref(shape)))


def layer_forward_stepwise(plan: Plan, shape: LayerShape, layer: dict, x_packed, y_packed, y_lo, h_n, c_n,
                           workspace, scratch, stream=None):
    check(_lib.load().lstm_fwd_stepwise(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)),
                                        _ptr(x_packed), _ptr(y_packed), _ptr(y_lo), _ptr(h_n), _ptr(c_n),
                                        _ptr(workspace), _ptr(scratch), _stream(stream)), "lstm_fwd_stepwise")


def layer_backward_stepwise(plan: Plan, shape: LayerShape, layer: dict, x_packed, y_packed, workspace,
                            dy_packed, dx_packed, grads: dict, scratch, stream=None):
    g = LayerGrads(grads["W"].data_ptr(), grads["R"].data_ptr(), grads["b"].data_ptr(),
                   grads["peep"].data_ptr())
    check(_lib.load().lstm_bwd_stepwise(plan.handle, ctypes.byref(shape), ctypes.byref(_params(layer)),
                                        _ptr(x_packed), _ptr(y_packed), _ptr(workspace), _ptr(dy_packed),
                                        _ptr(dx_packed), ctypes.byref(g), _ptr(scratch), _stream(stream)),
          "lstm_bwd_stepwise")


class PackedLSTMStack:
    """A stack of (bi)LSTM layers run through the C ABI on one packed batch.

    ``layers``: per layer a dict of device tensors W, R (fp32, or bf16 when
    ``bf16``), b and peep (fp32) in the header's layout.  Buffers for every
    layer's activations, workspace and gradients are allocated once, so
    ``forward``/``backward`` allocate nothing and may be replayed.
    ``stepwise=True`` runs the per-step-launch comparator path instead of the
    persistent recurrent kernels.
    """

    def __init__(self, plan: Plan, layers: list, input_size: int, hidden_size: int,
                 num_directions: int, bf16: bool, device="cuda", stepwise: bool = False):
        self.plan, self.layers, self.stepwise = plan, layers, bool(stepwise)
        self.D0, self.H, self.nd, self.bf16 = int(input_size), int(hidden_size), int(num_directions), bool(bf16)
        dev = torch.device(device)
        rows, H, nd = plan.rows, self.H, self.nd
        xdt = torch.bfloat16 if self.bf16 else torch.float32
        self.shapes = [layer_shape(self.D0 if l == 0 else nd * H, H, nd, self.bf16) for l in range(len(layers))]
        self.x_packed = torch.empty((rows, self.D0), dtype=xdt, device=dev)
        self.y = [torch.empty((rows, nd * H), dtype=torch.float32, device=dev) for _ in layers]
        # bf16 copies of every layer output but the last feed the next layer's products
        self.y_lo = [torch.empty((rows, nd * H), dtype=torch.bfloat16, device=dev)
                     if (self.bf16 and l + 1 < len(layers)) else None for l in range(len(layers))]
        self.h_n = torch.empty((len(layers), nd, plan.batch, H), dtype=torch.float32, device=dev)
        self.c_n = torch.empty_like(self.h_n)
        self.ws = [torch.empty(max(1, workspace_bytes(plan, s)), dtype=torch.uint8, device=dev)
                   for s in self.shapes]
        need = max((stepwise_scratch_bytes if self.stepwise else scratch_bytes)(plan, s) for s in self.shapes)
        self.scratch = torch.empty(max(1, need), dtype=torch.uint8, device=dev)
        # initial states / final-state errors ([layers][ndir][B][H] fp32, caller order) when set;
        # dh0 / dc0 are filled by backward_packed then
        self.h0 = self.c0 = self.dh_n = self.dc_n = None
        self.dh0 = self.dc0 = None
        self.state_scratch = None
        self.dy_packed = torch.empty((rows, nd * H), dtype=torch.float32, device=dev)
        self.dx = [torch.empty((rows, s.input_size), dtype=torch.float32, device=dev) for s in self.shapes]
        self.grads = [{"W": torch.empty(tuple(lay["W"].shape), dtype=torch.float32, device=dev),
                       "R": torch.empty(tuple(lay["R"].shape), dtype=torch.float32, device=dev),
                       "b": torch.empty(tuple(lay["b"].shape), dtype=torch.float32, device=dev),
                       "peep": torch.empty(tuple(lay["peep"].shape), dtype=torch.float32, device=dev)}
                      for lay in layers]

    def set_states(self, h0=None, c0=None, dh_n=None, dc_n=None):
        """Initial states and final-state errors of every layer ([layers][ndir][B][H] fp32 device tensors,
        caller order; None = zero).  Afterwards forward_packed / backward_packed run through
        lstm_fwd_state / lstm_bwd_state, and backward_packed fills self.dh0 / self.dc0."""
        self.h0, self.c0, self.dh_n, self.dc_n = h0, c0, dh_n, dc_n
        dev = self.y[0].device
        shape = (len(self.layers), self.nd, self.plan.batch, self.H)
        self.dh0 = torch.empty(shape, dtype=torch.float32, device=dev)
        self.dc0 = torch.empty(shape, dtype=torch.float32, device=dev)
        need = max(state_scratch_bytes(self.plan, s) for s in self.shapes)
        self.state_scratch = torch.empty(max(1, need), dtype=torch.uint8, device=dev)

    def _st(self, t, l):
        return None if t is None else t[l]

    def layer_input(self, l):
        return self.x_packed if l == 0 else (self.y_lo[l - 1] if self.bf16 else self.y[l - 1])

    def forward_packed(self, stream=None):
        for l, lay in enumerate(self.layers):
            if self.state_scratch is not None:
                layer_forward_state(self.plan, self.shapes[l], lay, self._st(self.h0, l), self._st(self.c0, l),
                                    self.layer_input(l), self.y[l], self.y_lo[l], self.h_n[l], self.c_n[l],
                                    self.ws[l], self.state_scratch, stream)
            elif self.stepwise:
                layer_forward_stepwise(self.plan, self.shapes[l], lay, self.layer_input(l), self.y[l],
                                       self.y_lo[l], self.h_n[l], self.c_n[l], self.ws[l], self.scratch, stream)
            else:
                layer_forward(self.plan, self.shapes[l], lay, self.layer_input(l), self.y[l], self.y_lo[l],
                              self.h_n[l], self.c_n[l], self.ws[l], stream)
        return self.y[-1]

    def backward_packed(self, stream=None):
        dy = self.dy_packed
        back = layer_backward_stepwise if self.stepwise else layer_backward
        for l in range(len(self.layers) - 1, -1, -1):
            if self.state_scratch is not None:
                layer_backward_state(self.plan, self.shapes[l], self.layers[l], self._st(self.h0, l),
                                     self._st(self.c0, l), self.layer_input(l), self.y[l], self.ws[l], dy, self.dx[l],
                                     self.grads[l], self._st(self.dh_n, l), self._st(self.dc_n, l), self.dh0[l],
                                     self.dc0[l], self.scratch, self.state_scratch, stream)
            else:
                back(self.plan, self.shapes[l], self.layers[l], self.layer_input(l), self.y[l],
                     self.ws[l], dy, self.dx[l], self.grads[l], self.scratch, stream)
            dy = self.dx[l]
        return self.dx[0]

    def step(self, x_cat, G_cat, stream=None):
        """pack -> forward of every layer -> backward of every layer -> unpack."""
        self.plan.pack(x_cat, self.x_packed, stream)
        self.plan.pack(G_cat, self.dy_packed, stream)
        self.forward_packed(stream)
        self.backward_packed(stream)
        return self.plan.unpack(self.y[-1], stream=stream), self.plan.unpack(self.dx[0], stream=stream)


class TruncatedBPTT:
    """Truncated back-propagation through time over windows of `window` frames ("Single Stream
    Parallelization...", Sec. 4, BPTT(h; h') with h = h'): window k of every sequence runs
    lstm_fwd_state from window k-1's final states (carry=True; the forward direction only -- the
    reverse direction cannot see the frames after its window and starts each window from zero)
    and lstm_bwd_state with the window's own errors, so no error crosses a window boundary.
    Each window is one window plan (lstm_plan_create_window) over the caller's full tensors.
    carry=False gives RETURNN-style independent chunks (every window from the zero state)."""

    def __init__(self, lengths, layers: list, input_size: int, hidden_size: int, num_directions: int,
                 bf16: bool, window: int, device="cuda", carry: bool = True):
        lens = np.asarray(lengths, dtype=np.int32)
        T = int(lens.max()) if lens.size else 0
        self.window, self.carry = int(window), bool(carry)
        self.frames = int(lens.sum())
        self.plans = [Plan(lens, window=(k * self.window, self.window)) for k in range(max(1, -(-T // self.window)))]
        self.stacks = [PackedLSTMStack(p, layers, input_size, hidden_size, num_directions, bf16, device)
                       for p in self.plans]
        for st in self.stacks:
            st.set_states()
        self.nd, self.H, self.D0 = int(num_directions), int(hidden_size), int(input_size)

    def step(self, x_cat, G_cat, stream=None):
        """All windows in order; returns (y_cat, dx_cat, per-window gradients).  y and dx are the
        caller's full tensors (every frame written by its window); window k's weight gradients
        are those of its own frames' errors (one mini-batch of BPTT(h'; h'))."""
        dev = x_cat.device
        y_cat = torch.zeros((self.frames, self.nd * self.H), dtype=torch.float32, device=dev)
        dx_cat = torch.zeros((self.frames, self.D0), dtype=torch.float32, device=dev)
        grads = []
        h = c = None
        for plan, st in zip(self.plans, self.stacks):
            st.h0, st.c0 = (h, c) if self.carry else (None, None)
            plan.pack(x_cat, st.x_packed, stream)
            plan.pack(G_cat, st.dy_packed, stream)
            st.forward_packed(stream)
            st.backward_packed(stream)
            plan.unpack(st.y[-1], y_cat, stream)
            plan.unpack(st.dx[0], dx_cat, stream)
            grads.append([{k: v.clone() for k, v in g.items()} for g in st.grads])
            h, c = st.h_n.clone(), st.c_n.clone()
            if self.nd == 2:               # the reverse direction restarts every window from zero
                h[:, 1].zero_()
                c[:, 1].zero_()
        return y_cat, dx_cat, grads


# --------------------------------------------------------------------------- 2-D (MDLSTM) layers

def md_compute_host(heights, widths, row_width: int = 0, num_directions: int = 1, schedule: int = 0) -> dict:
    """The 2-D packing and schedule computed on the host (lstm_md_plan_compute_host)."""
    lib = _lib.load()
    hs = np.ascontiguousarray(np.asarray(heights, dtype=np.int32))
    ws = np.ascontiguousarray(np.asarray(widths, dtype=np.int32))
    n = int(hs.size)
    N = int((hs.astype(np.int64) * ws).sum())
    cells = N * int(num_directions)
    pi = ctypes.POINTER(ctypes.c_int32)
    info = np.zeros(4, dtype=np.int32)
    y0 = np.zeros(max(n, 1), dtype=np.int32)
    x0 = np.zeros(max(n, 1), dtype=np.int32)
    # the step count is only known afterwards: ask for it first
    check(lib.lstm_md_plan_compute_host(hs.ctypes.data_as(pi), ws.ctypes.data_as(pi), n, int(row_width),
                                        int(num_directions), int(schedule), info.ctypes.data_as(pi), None, None,
                                        None, None, None, None, None, None), "lstm_md_plan_compute_host")
    steps = int(info[0])
    step_off = np.zeros(num_directions * (steps + 1), dtype=np.int64)
    t = {k: np.zeros(max(cells, 1), dtype=np.int32) for k in ("src", "pred1", "pred2", "succ1", "succ2")}
    check(lib.lstm_md_plan_compute_host(hs.ctypes.data_as(pi), ws.ctypes.data_as(pi), n, int(row_width),
                                        int(num_directions), int(schedule), info.ctypes.data_as(pi),
                                        y0.ctypes.data_as(pi), x0.ctypes.data_as(pi),
                                        step_off.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                        *[t[k].ctypes.data_as(pi) for k in ("src", "pred1", "pred2", "succ1",
                                                                            "succ2")]),
          "lstm_md_plan_compute_host")
    out = {"steps": steps, "height": int(info[1]), "width": int(info[2]), "rows": int(info[3]),
           "y0": y0[:n], "x0": x0[:n], "step_off": step_off.reshape(num_directions, steps + 1)}
    out.update({k: v[:cells] for k, v in t.items()})
    return out


class MdPlan:
    """Example-packing plan of a list of images for one MDLSTM layer's scan directions.
    schedule 1 (default): every image from step 0 along its own anti-diagonals; 0: the
    page's canvas, a cell at its skewed canvas column (same results, more steps)."""

    def __init__(self, heights, widths, row_width: int = 0, num_directions: int = 4, schedule: int = 1):
        lib = _lib.load()
        self.heights = np.ascontiguousarray(np.asarray(heights, dtype=np.int32))
        self.widths = np.ascontiguousarray(np.asarray(widths, dtype=np.int32))
        self.num_directions = int(num_directions)
        h = ctypes.c_void_p()
        pi = ctypes.POINTER(ctypes.c_int32)
        check(lib.lstm_md_plan_create(self.heights.ctypes.data_as(pi), self.widths.ctypes.data_as(pi),
                                      int(self.heights.size), int(row_width), self.num_directions, int(schedule),
                                      ctypes.byref(h)), "lstm_md_plan_create")
        self.handle = h
        px, st, ch, cw, rows = (ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(),
                                ctypes.c_int32())
        check(lib.lstm_md_plan_info(h, ctypes.byref(px), ctypes.byref(st), ctypes.byref(ch), ctypes.byref(cw),
                                    ctypes.byref(rows)), "lstm_md_plan_info")
        self.pixels, self.steps = px.value, st.value
        self.canvas = (ch.value, cw.value)
        self.rows = rows.value

    def placement(self):
        n = int(self.heights.size)
        y0 = np.zeros(max(n, 1), dtype=np.int32)
        x0 = np.zeros(max(n, 1), dtype=np.int32)
        pi = ctypes.POINTER(ctypes.c_int32)
        check(_lib.load().lstm_md_plan_placement(self.handle, y0.ctypes.data_as(pi), x0.ctypes.data_as(pi)),
              "lstm_md_plan_placement")
        return y0[:n], x0[:n]

    def step_cells(self) -> np.ndarray:
        so = np.zeros(self.num_directions * (self.steps + 1), dtype=np.int64)
        check(_lib.load().lstm_md_plan_step_cells(self.handle, so.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))),
              "lstm_md_plan_step_cells")
        return so.reshape(self.num_directions, self.steps + 1)

    def set_wait_limit(self, ns: int):
        check(_lib.load().lstm_md_plan_set_wait_limit(self.handle, int(ns)), "lstm_md_plan_set_wait_limit")

    def poll(self, stream=None) -> int:
        return int(_lib.load().lstm_md_status_poll(self.handle, _stream(stream)))

    def debug_skip_arrival(self, cta: int):
        check(_lib.load().lstm_md_debug_skip_arrival(self.handle, int(cta)), "lstm_md_debug_skip_arrival")

    def launch_count(self) -> int:
        return int(_lib.load().lstm_md_plan_launch_count(self.handle))

    def enable_timing(self, on: bool = True):
        check(_lib.load().lstm_md_plan_enable_timing(self.handle, 1 if on else 0), "lstm_md_plan_enable_timing")

    def read_timing(self) -> dict:
        ms = (ctypes.c_double * 4)()
        calls = (ctypes.c_int64 * 4)()
        check(_lib.load().lstm_md_plan_read_timing(self.handle, ms, calls), "lstm_md_plan_read_timing")
        return {k: (ms[i], calls[i]) for i, k in enumerate(_lib.MD_KINDS)}

    def close(self):
        if getattr(self, "handle", None):
            _lib.load().lstm_md_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class MdLayer:
    """One MDLSTM layer (fp32) over an MdPlan: device weights, workspace and scratch.
    layer: W[ndir,5H,D], U1/U2[ndir,5H,H], b[ndir,5H], peep[ndir,6,H] (torch, cuda)."""

    def __init__(self, plan: MdPlan, layer: dict, input_size: int, hidden_size: int, device="cuda"):
        lib = _lib.load()
        self.plan = plan
        self.layer = {k: torch.as_tensor(v, dtype=torch.float32, device=device).contiguous() for k, v in layer.items()}
        self.shape = _lib.MdShape(int(input_size), int(hidden_size), plan.num_directions)
        ws = lib.lstm_md_workspace_bytes(plan.handle, ctypes.byref(self.shape))
        sc = lib.lstm_md_scratch_bytes(plan.handle, ctypes.byref(self.shape))
        if ws == 0 and plan.pixels > 0:
            raise ValueError("unsupported MDLSTM layer shape")
        self.workspace = torch.empty(max(int(ws), 16), dtype=torch.uint8, device=device)
        self.scratch = torch.empty(max(int(sc), 16), dtype=torch.uint8, device=device)
        self.grads = {k: torch.empty_like(v) for k, v in self.layer.items()}

    def _params(self):
        L = self.layer
        return _lib.MdParams(L["W"].data_ptr(), L["U1"].data_ptr(), L["U2"].data_ptr(), L["b"].data_ptr(),
                             L["peep"].data_ptr())

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        nd, H = self.plan.num_directions, self.shape.hidden_size
        if y is None:
            y = torch.empty((self.plan.pixels, nd * H), dtype=torch.float32, device=x.device)
        prm = self._params()
        check(_lib.load().lstm_md_fwd(self.plan.handle, ctypes.byref(self.shape), ctypes.byref(prm), _ptr(x),
                                      _ptr(y), _ptr(self.workspace), _stream(stream)), "lstm_md_fwd")
        return y

    def backward(self, x: torch.Tensor, dy: torch.Tensor, dx: torch.Tensor | None = None, stream=None):
        if dx is None:
            dx = torch.empty_like(x)
        prm = self._params()
        g = self.grads
        gr = _lib.MdGrads(g["W"].data_ptr(), g["U1"].data_ptr(), g["U2"].data_ptr(), g["b"].data_ptr(),
                          g["peep"].data_ptr())
        check(_lib.load().lstm_md_bwd(self.plan.handle, ctypes.byref(self.shape), ctypes.byref(prm), _ptr(x),
                                      _ptr(self.workspace), _ptr(dy), _ptr(dx), ctypes.byref(gr), _ptr(self.scratch),
                                      _stream(stream)), "lstm_md_bwd")
        return dx
