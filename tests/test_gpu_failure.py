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


@pytest.mark.parametrize("variant", [-1, 0, 2], ids=["auto", "barrier", "barrier-tiles"])
def test_cluster_kernels_timeout_is_reported_and_context_survives(variant):
    """The cluster kernels' waits that can run out are the bounded waits on MMA completion
    (and, with the bulk exchange, on the peers' operands).  With the test hook one CTA
    withholds the completion signal of its first product: its wait runs out, it stops
    issuing and sending, its peers' operand waits run out in turn, every CTA still runs all
    its cluster barriers, frees its tensor memory only after its products are done, and
    reports LSTM_ERR_TIMEOUT; the context stays usable (forward and backward)."""
    from padding_free_variable_gb300 import _lib, ops, synthetic
    from gpu_harness import device_layers
    w = synthetic.custom(2, 1, 8, 64, [30, 20, 10, 5, 17], seed=4)
    layers = device_layers(w)

    def fresh():
        plan = ops.Plan(w.lengths)
        plan.debug_cluster_variant(variant)
        stack = ops.PackedLSTMStack(plan, layers, 8, 64, 2, False)
        return plan, stack

    x = torch.from_numpy(w.x).cuda()
    G = torch.from_numpy(w.G).cuda()
    ref_plan, ref_stack = fresh()
    y_ref, dx_ref = (t.clone() for t in ref_stack.step(x, G))
    assert ref_plan.poll() == _lib.LSTM_OK
    for backward in (False, True):
        cfg = ref_plan.recurrent_config(backward)
        assert cfg["kernel"] == "cluster", cfg
        if variant >= 0:
            assert (cfg["exchange"] == "bulk") == bool(variant & 1) and cfg["tma_tiles"] == bool(variant & 2), cfg

    plan, stack = fresh()
    plan.set_wait_limit(50_000_000)          # 50 ms
    plan.pack(x, stack.x_packed)
    plan.pack(G, stack.dy_packed)
    plan.debug_skip_arrival(1)
    stack.forward_packed()
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    stack.forward_packed()
    assert plan.poll() == _lib.LSTM_OK
    plan.debug_skip_arrival(1)
    stack.backward_packed()
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    y, dx = stack.step(x, G)
    assert plan.poll() == _lib.LSTM_OK
    assert torch.equal(y, y_ref) and torch.equal(dx, dx_ref)


@pytest.mark.parametrize("mode", [1, 2], ids=["clusters", "no-clusters"])
def test_wide_persistent_kernels_timeout_is_reported_and_context_survives(mode):
    """The persistent kernels of layers wider than a cluster wait at a grid barrier every step.
    With the test hook one CTA never announces its first step: the other CTAs' bounded waits
    run out, every CTA leaves through its bounded teardown (with clusters: after its peers'
    stage releases and the final cluster barrier), LSTM_ERR_TIMEOUT is reported, and a clean
    rerun in the same context gives the reference results bit for bit (forward and backward)."""
    from padding_free_variable_gb300 import _lib, ops, synthetic
    from gpu_harness import device_layers
    w = synthetic.custom(2, 1, 16, 576, [9, 4, 13, 7, 11], seed=4, dtype="bf16", weight_range=0.05)
    layers = device_layers(w)

    def fresh():
        plan = ops.Plan(w.lengths)
        plan.debug_wide_recurrence(mode)
        return plan, ops.PackedLSTMStack(plan, layers, 16, 576, 2, True)

    x = torch.from_numpy(w.x).cuda().to(torch.bfloat16)
    G = torch.from_numpy(w.G).cuda()
    ref_plan, ref_stack = fresh()
    y_ref, dx_ref = (t.clone() for t in ref_stack.step(x, G))
    assert ref_plan.poll() == _lib.LSTM_OK
    assert ref_plan.recurrent_config(False)["kernel"] == "persistent_wide"
    plan, stack = fresh()
    plan.set_wait_limit(50_000_000)          # 50 ms
    plan.pack(x, stack.x_packed)
    plan.pack(G, stack.dy_packed)
    plan.debug_skip_arrival(3)
    stack.forward_packed()
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    stack.forward_packed()
    assert plan.poll() == _lib.LSTM_OK
    plan.debug_skip_arrival(3)
    stack.backward_packed()
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    y, dx = stack.step(x, G)
    assert plan.poll() == _lib.LSTM_OK
    assert torch.equal(y, y_ref) and torch.equal(dx, dx_ref)


def test_md_layer_timeout_is_reported_and_context_survives():
    """The 2-D MDLSTM walk waits at a grid barrier between steps.  With the test hook one CTA
    never arrives at the first barrier: every CTA's bounded wait runs out, LSTM_ERR_TIMEOUT is
    reported for the forward and the backward walk, and a clean rerun in the same context
    gives the reference results bit for bit."""
    from padding_free_variable_gb300 import _lib, ops, synthetic
    w = synthetic.md_custom(4, 8, 16, [5, 9, 3, 7], [11, 4, 8, 6], seed=4, weight_range=0.3)

    def fresh():
        plan = ops.MdPlan(w.heights, w.widths, 0, 4, 0)
        return plan, ops.MdLayer(plan, w.layer, 8, 16)

    x = torch.from_numpy(w.x).cuda()
    G = torch.from_numpy(w.G).cuda()
    ref_plan, ref = fresh()
    y_ref = ref.forward(x).clone()
    dx_ref = ref.backward(x, G).clone()
    assert ref_plan.poll() == _lib.LSTM_OK
    plan, layer = fresh()
    plan.set_wait_limit(50_000_000)          # 50 ms
    plan.debug_skip_arrival(3)
    layer.forward(x)
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    layer.forward(x)
    assert plan.poll() == _lib.LSTM_OK
    plan.debug_skip_arrival(3)
    layer.backward(x, G)
    assert plan.poll() == _lib.LSTM_ERR_TIMEOUT
    plan.debug_skip_arrival(-1)
    y = layer.forward(x)
    dx = layer.backward(x, G)
    assert plan.poll() == _lib.LSTM_OK
    assert torch.equal(y, y_ref) and torch.equal(dx, dx_ref)
