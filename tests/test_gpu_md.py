"""2-D example-packing for MDLSTM layers on the GPU, against the fp64 oracle.

Every case packs a list of images ("No Padding Please", Sec. V, App. B), runs one MDLSTM
layer forward and backward through the C ABI (lstm_md_fwd / lstm_md_bwd), and compares
y, dx and every parameter gradient with the oracle, which runs each image and scan
direction on its own.  Bars as for the fp32 1-D path: normwise 1e-4 and element-wise
2e-3 (floor 1e-3 of the tensor's scale).
"""
import numpy as np
import pytest

import oracle
from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_F32, TOL_F32_ELEMENTWISE, elementwise_err, rel_err

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


def run_md(w, schedule=0, row_width=0, G=None):
    from padding_free_variable_gb300 import ops
    plan = ops.MdPlan(w.heights, w.widths, row_width, w.num_directions, schedule)
    layer = ops.MdLayer(plan, w.layer, w.input_size, w.hidden_size)
    x = torch.from_numpy(w.x).cuda()
    y = layer.forward(x)
    dy = torch.from_numpy(w.G if G is None else G).cuda()
    dx = layer.backward(x, dy)
    torch.cuda.synchronize()
    assert plan.poll() == 0
    out = {"y": y.cpu().numpy(), "dx": dx.cpu().numpy(),
           "grads": {k: v.cpu().numpy() for k, v in layer.grads.items()}, "plan": plan}
    return out


def compare(gpu, ref, label):
    pairs = [("y", gpu["y"], ref["y"]), ("dx", gpu["dx"], ref["dx"])]
    pairs += [(k, gpu["grads"][k], ref["grads"][k]) for k in ("W", "U1", "U2", "b", "peep")]
    for name, g, r in pairs:
        e, el = rel_err(g, r), elementwise_err(g, r)
        assert e <= TOL_F32, (label, name, e)
        assert el <= TOL_F32_ELEMENTWISE, (label, name, el)


CASES = [
    # ndir, D, H, heights, widths, row width
    (4, 3, 2, [3, 2, 3, 3, 2], [5, 4, 2, 3, 7], 0),
    (1, 5, 20, list(np.random.default_rng(1).integers(1, 9, 10)), list(np.random.default_rng(2).integers(1, 20, 10)), 0),
    (4, 16, 32, list(np.random.default_rng(3).integers(1, 12, 20)), list(np.random.default_rng(4).integers(1, 30, 20)), 24),
    (1, 8, 64, [6, 5, 6], [9, 14, 3], 0),                                  # U^T resident, 2 units a lane
    (2, 8, 100, [4, 7, 3, 4], [11, 5, 8, 6], 0),                           # weights from L2, 4 units a lane
    (4, 4, 8, [0, 1, 1, 5, 3, 1], [4, 1, 9, 1, 0, 1], 0),                   # empty, 1x1, one row, one column
]


@pytest.mark.parametrize("schedule", [0, 1], ids=["canvas", "diagonal"])
@pytest.mark.parametrize("case", CASES, ids=[f"nd{c[0]}-D{c[1]}-H{c[2]}-n{len(c[3])}" for c in CASES])
def test_md_layer_matches_oracle(case, schedule):
    nd, D, H, hs, ws, rw = case
    w = synthetic.md_custom(nd, D, H, hs, ws, seed=100 + H, weight_range=0.3)
    gpu = run_md(w, schedule, rw)
    ref = oracle.md_layer(w.heights, w.widths, w.x, w.layer, w.G)
    compare(gpu, ref, f"md {case} schedule {schedule}")
    assert gpu["plan"].launch_count() > 0


def test_schedules_compute_the_same_cells():
    """Canvas and diagonal schedules run every cell from the same predecessors: y and dx (a
    product over pixels in pixel order) are bitwise equal; the weight gradients sum over the
    cells in cell order, which the schedule changes, and agree to rounding."""
    w = synthetic.md_custom(4, 16, 32, list(np.random.default_rng(7).integers(1, 14, 24)),
                            list(np.random.default_rng(8).integers(1, 40, 24)), seed=9, weight_range=0.3)
    a, b = run_md(w, 0), run_md(w, 1)
    assert a["plan"].steps > b["plan"].steps
    for k in ("y", "dx"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("W", "U1", "U2", "b", "peep"):
        assert rel_err(a["grads"][k], b["grads"][k]) <= 1e-5, k


def test_md_bitwise_repeatable():
    w = synthetic.md_custom(4, 8, 16, [5, 9, 2, 7], [13, 4, 8, 7], seed=3, weight_range=0.3)
    a, b = run_md(w), run_md(w)
    for k in ("y", "dx"):
        assert np.array_equal(a[k], b[k]), k
    for k in a["grads"]:
        assert np.array_equal(a["grads"][k], b["grads"][k]), k


@pytest.mark.parametrize("name", ["words", "lines"])
def test_md_workload_full_size_sampled(name):
    """The bench's workloads at full size, in the bench's launch configuration; the oracle
    runs only sampled images: y and dx of those images are compared, and dL/dy is zero on
    every other image so that the full-batch parameter gradients equal the oracle's on the
    sample alone."""
    w = synthetic.md_workload(name)
    rng = np.random.default_rng(0)
    n = w.heights.size
    pick = np.sort(rng.choice(n, size=min(6, n), replace=False))
    pix_off = np.concatenate([[0], np.cumsum(w.heights.astype(np.int64) * w.widths)])
    rows = np.concatenate([np.arange(pix_off[i], pix_off[i + 1]) for i in pick])
    G = np.zeros_like(w.G)
    G[rows] = w.G[rows]
    gpu = run_md(w, 1, G=G)
    ref = oracle.md_layer(w.heights[pick], w.widths[pick], w.x[rows], w.layer, w.G[rows])
    sub = {"y": gpu["y"][rows], "dx": gpu["dx"][rows], "grads": gpu["grads"]}
    compare(sub, ref, f"md workload {name}")
