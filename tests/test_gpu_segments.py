"""Segment plans (RETURNN-style chunking into possibly overlapping segments, RETURNN paper,
Sec. 4) and window plans for truncated BPTT ("Single Stream Parallelization...", Sec. 4,
BPTT(h; h')) through the C ABI, against the oracle run on the same segments / windows."""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_BF16, TOL_F32, compare_all, elementwise_err, rel_err, TOL_F32_ELEMENTWISE

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


def _close(got, ref, tol, label):
    assert rel_err(got, ref) <= tol, (label, rel_err(got, ref))
    if tol == TOL_F32:
        assert elementwise_err(got, ref) <= TOL_F32_ELEMENTWISE, (label, elementwise_err(got, ref))


@pytest.mark.parametrize("chunk,step,dtype", [(6, 6, "f32"), (7, 4, "f32"), (8, 5, "bf16"), (1, 1, "f32")])
def test_segment_plan_matches_oracle_on_segments(chunk, step, dtype):
    import oracle
    from padding_free_variable_gb300 import ops
    bf16 = dtype == "bf16"
    w = synthetic.custom(2, 2, 16, 64, [19, 0, 4, 13, 25, 2, 7], seed=chunk * 10 + step, dtype=dtype,
                         weight_range=0.1 if bf16 else 0.3)
    seq, start, length = ops.segments_host(w.lengths, chunk, step)
    plan = ops.Plan(w.lengths, segments=(chunk, step))
    assert plan.batch == len(seq) and plan.frames == w.N and plan.rows == int(length.sum())
    stack = ops.PackedLSTMStack(plan, ops.device_layers(w.layers, bf16), 16, 64, 2, bf16)
    xdt = torch.bfloat16 if bf16 else torch.float32
    x = torch.from_numpy(w.x).to("cuda", dtype=xdt)
    y = torch.zeros((w.N, 128), device="cuda")
    dx = torch.zeros((w.N, 16), device="cuda")
    plan.pack(x, stack.x_packed)
    plan.pack(torch.from_numpy(w.G).cuda(), stack.dy_packed)
    stack.forward_packed()
    stack.backward_packed()
    plan.unpack(stack.y[-1], y)
    plan.unpack(stack.dx[0], dx)
    torch.cuda.synchronize()
    assert plan.poll() == 0
    # the oracle on the segments as sequences of their own (frames read by two segments appear twice)
    cst = np.concatenate([[0], np.cumsum(w.lengths)])
    src = np.concatenate([cst[seq[u]] + start[u] + np.arange(length[u]) for u in range(len(seq))]).astype(int)
    ref = oracle.lstm_stack(length, w.x[src], w.layers, 2, 64, G=w.G[src], nthreads=4)
    tol = TOL_BF16 if bf16 else TOL_F32
    for l, (g, r) in enumerate(zip(stack.grads, ref["grads"])):
        for k in ("W", "R", "b", "peep"):
            _close(g[k].cpu().numpy(), r[k], tol, f"L{l}.d{k}")
    _close(stack.h_n.cpu().numpy(), ref["h_n"], tol, "h_n")
    # each frame comes back from the segment that owns it (up to the next segment's start)
    own = np.concatenate([np.arange(length[u]) < (step if start[u] + length[u] < w.lengths[seq[u]] else length[u])
                          for u in range(len(seq))])
    order = np.argsort(src[own], kind="stable")
    assert np.array_equal(src[own][order], np.arange(w.N))
    _close(y.cpu().numpy(), ref["y"][own][order], tol, "y")
    _close(dx.cpu().numpy(), ref["dx"][own][order], tol, "dx")


@pytest.mark.parametrize("nd,dtype,carry", [(1, "f32", True), (2, "f32", True), (2, "bf16", True), (2, "f32", False)])
def test_truncated_bptt_windows_match_oracle(nd, dtype, carry):
    """Window k of every sequence from window k-1's final states (forward direction), its own
    errors back-propagated through it alone; against the oracle doing the same per window."""
    import oracle
    from padding_free_variable_gb300 import ops
    bf16 = dtype == "bf16"
    H, D, win = 64, 16, 6
    w = synthetic.custom(nd, 2, D, H, [19, 0, 4, 13, 25, 2, 7], seed=31 + nd, dtype=dtype,
                         weight_range=0.1 if bf16 else 0.3)
    drv = ops.TruncatedBPTT(w.lengths, ops.device_layers(w.layers, bf16), D, H, nd, bf16, win, carry=carry)
    xdt = torch.bfloat16 if bf16 else torch.float32
    y, dx, grads = drv.step(torch.from_numpy(w.x).to("cuda", dtype=xdt), torch.from_numpy(w.G).cuda())
    torch.cuda.synchronize()
    cst = np.concatenate([[0], np.cumsum(w.lengths)])
    h = c = None
    y_ref = np.zeros_like(y.cpu().numpy())
    dx_ref = np.zeros_like(dx.cpu().numpy())
    tol = TOL_BF16 if bf16 else TOL_F32
    for k, g_gpu in enumerate(grads):
        L = np.clip(w.lengths - k * win, 0, win)
        src = np.concatenate([cst[b] + k * win + np.arange(L[b]) for b in range(len(L))]).astype(int)
        ref = oracle.lstm_stack(L, w.x[src], w.layers, nd, H, G=w.G[src], nthreads=4,
                                h0=h if carry else None, c0=c if carry else None)
        y_ref[src], dx_ref[src] = ref["y"], ref["dx"]
        for l, (g, r) in enumerate(zip(g_gpu, ref["grads"])):
            for key in ("W", "R", "b", "peep"):
                _close(g[key].cpu().numpy(), r[key], tol, f"window {k} L{l}.d{key}")
        h, c = ref["h_n"].copy(), ref["c_n"].copy()
        if nd == 2:
            h[:, 1] = 0.0
            c[:, 1] = 0.0
    _close(y.cpu().numpy(), y_ref, tol, "y")
    _close(dx.cpu().numpy(), dx_ref, tol, "dx")
    if carry and nd == 1 and not bf16:
        # carrying the state makes the forward pass exact: the windows' outputs are the whole
        # sequences' outputs
        full = oracle.lstm_stack(w.lengths, w.x, w.layers, 1, H)
        _close(y.cpu().numpy(), full["y"], TOL_F32, "y vs whole sequences")
