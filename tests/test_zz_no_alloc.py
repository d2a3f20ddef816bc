"""lstm_bwd_noalloc: the layer backward pass for callers that cannot allocate.

Some callers cannot call cudaMalloc -- a host framework whose memory pool owns
the device memory and forbids allocations from outside it, or a real-time loop
that must not allocate once it has started.  lstm_bwd_noalloc takes the
scratch that lstm_bwd needs from one fixed array inside the library instead of
from the caller.  These tests call it through the C ABI twice in a row and
check both results against lstm_bwd with a caller-allocated scratch, and check
that a layer needing more scratch than the array holds is refused up front.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


def _grads_like(layer):
    return {k: torch.full(tuple(layer[k].shape), float("nan"), dtype=torch.float32, device="cuda")
            for k in ("W", "R", "b", "peep")}


def _lgrads(g):
    from padding_free_variable_gb300._lib import LayerGrads
    return LayerGrads(g["W"].data_ptr(), g["R"].data_ptr(), g["b"].data_ptr(), g["peep"].data_ptr())


NOALLOC_CASES = [
    # ndir, D, H, lengths, bf16, CTAs per direction (0 = automatic)
    (2, 16, 64, [9, 0, 4, 13, 13, 2, 7], False, 4),     # grid kernels: the partial-product exchange
    (2, 32, 256, [60, 3, 44, 17, 60, 9, 33, 1], True, 0),   # cluster kernels + tcgen05 operands (bf16)
    (2, 32, 128, [21, 3, 14, 17, 1, 9], False, 0),      # cluster kernels + six-segment fp32 operands
]


@pytest.mark.parametrize("case", NOALLOC_CASES, ids=["grid-f32", "cluster-bf16", "cluster-f32"])
def test_noalloc_backward_matches_lstm_bwd_on_two_calls_in_a_row(case):
    """Two calls in a row give exactly lstm_bwd's results: both run the same kernels on the
    same operands, and the library is bitwise repeatable, so any difference would be a
    scratch-aliasing slip."""
    from padding_free_variable_gb300 import _lib, ops, synthetic
    from padding_free_variable_gb300._lib import LayerParams

    nd, D, H, lengths, bf16, ctas = case
    w = synthetic.custom(nd, 1, D, H, lengths, seed=2025 + H, dtype="bf16" if bf16 else "f32",
                         weight_range=0.1 if bf16 else 0.3)
    plan = ops.Plan(w.lengths)
    if ctas:
        plan.set_ctas_per_direction(ctas)
    layer = ops.device_layers(w.layers, bf16)[0]
    shape = ops.layer_shape(D, H, nd, bf16)
    assert ops.scratch_bytes(plan, shape) <= 32 * 1024 * 1024
    xdt = torch.bfloat16 if bf16 else torch.float32
    x = plan.pack(torch.from_numpy(w.x).to("cuda", dtype=xdt))
    dy = plan.pack(torch.from_numpy(w.G).cuda())
    y = torch.empty((plan.rows, nd * H), dtype=torch.float32, device="cuda")
    ws = torch.empty(ops.workspace_bytes(plan, shape), dtype=torch.uint8, device="cuda")
    ops.layer_forward(plan, shape, layer, x, y, None, None, None, ws)
    saved = ws.clone()                               # lstm_bwd overwrites the saved gates

    ref_g = _grads_like(layer)
    ref_dx = torch.empty((plan.rows, D), dtype=torch.float32, device="cuda")
    scratch = torch.empty(ops.scratch_bytes(plan, shape), dtype=torch.uint8, device="cuda")
    ops.layer_backward(plan, shape, layer, x, y, ws, dy, ref_dx, ref_g, scratch)
    torch.cuda.synchronize()
    assert plan.poll() == 0
    expect_kernel = "grid" if ctas else "cluster"
    assert plan.recurrent_config(True)["kernel"] == expect_kernel

    lib = _lib.load()
    params = LayerParams(layer["W"].data_ptr(), layer["R"].data_ptr(), layer["b"].data_ptr(),
                         layer["peep"].data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        ws.copy_(saved)
        g = _grads_like(layer)
        dx = torch.full((plan.rows, D), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.lstm_bwd_noalloc(plan.handle, ctypes.byref(shape), ctypes.byref(params),
                                  ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(dy.data_ptr()),
                                  ctypes.c_void_p(dx.data_ptr()), ctypes.byref(_lgrads(g)), stream)
        assert rc == _lib.LSTM_OK, _lib.status_string(rc)
        torch.cuda.synchronize()
        assert plan.poll() == 0
        assert plan.recurrent_config(True)["kernel"] == expect_kernel
        assert torch.equal(dx, ref_dx), f"call {call}: dx"
        for k in g:
            assert torch.equal(g[k], ref_g[k]), f"call {call}: d{k}"


def test_noalloc_refuses_a_layer_beyond_its_scratch():
    from padding_free_variable_gb300 import _lib, ops
    from padding_free_variable_gb300._lib import LayerGrads, LayerParams
    plan = ops.Plan(np.full(256, 120, dtype=np.int32))
    shape = ops.layer_shape(2048, 1024, 2, True)
    assert ops.scratch_bytes(plan, shape) > 32 * 1024 * 1024
    rc = _lib.load().lstm_bwd_noalloc(plan.handle, ctypes.byref(shape), ctypes.byref(LayerParams()),
                                      None, None, None, None, None, ctypes.byref(LayerGrads()), None)
    assert rc == _lib.LSTM_ERR_UNSUPPORTED
