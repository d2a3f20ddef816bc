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


def test_noalloc_backward_matches_lstm_bwd_on_two_calls_in_a_row():
    from padding_free_variable_gb300 import _lib, ops, synthetic
    from padding_free_variable_gb300._lib import LayerParams
    from gpu_harness import TOL_F32, device_layers, rel_err

    w = synthetic.custom(2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], seed=2025, weight_range=0.3)
    plan = ops.Plan(w.lengths)
    plan.set_ctas_per_direction(4)                  # several CTAs: the exchange buffer is used
    layer = device_layers(w)[0]
    shape = ops.layer_shape(16, 64, 2, False)
    assert ops.scratch_bytes(plan, shape) <= 32 * 1024 * 1024
    x = plan.pack(torch.from_numpy(w.x).cuda())
    dy = plan.pack(torch.from_numpy(w.G).cuda())
    y = torch.empty((plan.rows, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(ops.workspace_bytes(plan, shape), dtype=torch.uint8, device="cuda")
    ops.layer_forward(plan, shape, layer, x, y, None, None, None, ws)
    saved = ws.clone()                               # lstm_bwd overwrites the saved gates

    ref_g = _grads_like(layer)
    ref_dx = torch.empty((plan.rows, 16), dtype=torch.float32, device="cuda")
    scratch = torch.empty(ops.scratch_bytes(plan, shape), dtype=torch.uint8, device="cuda")
    ops.layer_backward(plan, shape, layer, x, y, ws, dy, ref_dx, ref_g, scratch)
    torch.cuda.synchronize()
    assert plan.poll() == 0

    lib = _lib.load()
    params = LayerParams(layer["W"].data_ptr(), layer["R"].data_ptr(), layer["b"].data_ptr(),
                         layer["peep"].data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        ws.copy_(saved)
        g = _grads_like(layer)
        dx = torch.full((plan.rows, 16), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.lstm_bwd_noalloc(plan.handle, ctypes.byref(shape), ctypes.byref(params),
                                  ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(dy.data_ptr()),
                                  ctypes.c_void_p(dx.data_ptr()), ctypes.byref(_lgrads(g)), stream)
        assert rc == _lib.LSTM_OK, _lib.status_string(rc)
        torch.cuda.synchronize()
        assert plan.poll() == 0
        assert rel_err(dx.cpu().numpy(), ref_dx.cpu().numpy()) <= TOL_F32, f"call {call}: dx"
        for k in g:
            assert rel_err(g[k].cpu().numpy(), ref_g[k].cpu().numpy()) <= TOL_F32, f"call {call}: d{k}"


def test_noalloc_refuses_a_layer_beyond_its_scratch():
    from padding_free_variable_gb300 import _lib, ops
    from padding_free_variable_gb300._lib import LayerGrads, LayerParams
    plan = ops.Plan(np.full(256, 120, dtype=np.int32))
    shape = ops.layer_shape(2048, 1024, 2, True)
    assert ops.scratch_bytes(plan, shape) > 32 * 1024 * 1024
    rc = _lib.load().lstm_bwd_noalloc(plan.handle, ctypes.byref(shape), ctypes.byref(LayerParams()),
                                      None, None, None, None, None, ctypes.byref(LayerGrads()), None)
    assert rc == _lib.LSTM_ERR_UNSUPPORTED
