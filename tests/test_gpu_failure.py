"""Failure detection without a GPU fault: one CTA of the recurrent kernel never
announces its steps (a host-set test hook), so its peers' bounded barrier
waits run out.  The launch must return, the status word must say
LSTM_ERR_TIMEOUT, and the context must stay usable for a clean rerun."""
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


def test_barrier_timeout_is_reported_and_context_survives():
    from padding_free_variable_gb300 import _lib, ops, synthetic
    from gpu_harness import device_layers
    w = synthetic.custom(2, 1, 8, 256, [30, 20, 10, 5], seed=4)
    plan = ops.Plan(w.lengths)
    plan.set_ctas_per_direction(8)           # several CTAs per direction meet at each step
    plan.set_wait_limit(200_000_000)        # 0.2 s
    layers = device_layers(w)
    stack = ops.PackedLSTMStack(plan, layers, 8, 256, 2, False)
    x = torch.from_numpy(w.x).cuda()
    stack.plan.pack(x, stack.x_packed)
    plan.debug_skip_arrival(1)
    stack.forward_packed()
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    assert plan.poll() == _lib.LSTM_OK          # cleared
    plan.debug_skip_arrival(-1)
    y1 = stack.forward_packed().clone()
    assert plan.poll() == _lib.LSTM_OK
    y2 = stack.forward_packed().clone()
    assert plan.poll() == _lib.LSTM_OK
    assert torch.equal(y1, y2)
    assert torch.isfinite(y1).all()
