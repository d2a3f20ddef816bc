"""The persistent recurrent kernels of bf16 layers wider than one cluster (H > 512): R (and
R^T) resident in the shared memory of H/16 CTAs per direction, the previous step's operand
streamed back with TMA, tcgen05 products, a grid barrier per step; the backward either splits
the gate errors over clusters of four CTAs (partial products exchanged through distributed
shared memory) or streams all of them into every CTA.  Against the oracle, and against the
per-step-launch path on the same inputs."""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_BF16, TOL_BF16_EMULATED, compare_all, rel_err, run_gpu, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


def _run(w, mode, **kw):
    import torch as _t
    from gpu_harness import device_layers
    from padding_free_variable_gb300 import ops
    plan = ops.Plan(w.lengths, padded=kw.get("padded", False))
    plan.debug_wide_recurrence(mode)
    if kw.get("stages"):
        plan.debug_wide_stages(kw["stages"])
    bf16 = True
    stack = ops.PackedLSTMStack(plan, device_layers(w), w.spec.input_size, w.spec.hidden_size,
                                w.spec.num_directions, bf16)
    if kw.get("states") is not None:
        st = {k: (None if v is None else _t.from_numpy(v).cuda()) for k, v in kw["states"].items()}
        stack.set_states(st["h0"], st["c0"], st["dh_n"], st["dc_n"])
    y, dx = stack.step(_t.from_numpy(w.x).to("cuda", dtype=_t.bfloat16), _t.from_numpy(w.G).cuda())
    _t.cuda.synchronize()
    assert plan.poll() == 0
    out = {"y": y.cpu().numpy(), "dx": dx.cpu().numpy(), "h_n": stack.h_n.cpu().numpy(),
           "c_n": stack.c_n.cpu().numpy(), "grads": [{k: v.cpu().numpy() for k, v in g.items()} for g in stack.grads],
           "plan": plan}
    if kw.get("states") is not None:
        out["dh0"], out["dc0"] = stack.dh0.cpu().numpy(), stack.dc0.cpu().numpy()
    return out


CASES = [
    # ndir, layers, D, H, lengths
    (2, 2, 24, 576, [7, 1, 12, 0, 12, 3]),
    (1, 1, 32, 640, [20, 7, 13, 1]),
    (2, 1, 64, 1024, list(np.random.default_rng(5).integers(1, 30, 40))),
    (2, 1, 16, 1024, list(np.random.default_rng(6).integers(1, 12, 200))),    # two 128-row tiles
]


@pytest.mark.parametrize("mode", [1, 2], ids=["clusters", "no-clusters"])
@pytest.mark.parametrize("case", CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-B{len(c[4])}" for c in CASES])
def test_persistent_wide_matches_oracle(case, mode):
    """Both forms of the launch: clusters of 4 CTAs (forward: sharing each operand tile by
    multicast; backward: splitting the gate errors four ways), mode 1, and no clusters (every
    CTA loads every tile it needs itself), mode 2."""
    nd, nl, D, H, lengths = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=13 + H, dtype="bf16", weight_range=0.05)
    gpu = _run(w, mode)
    for backward in (False, True):
        cfg = gpu["plan"].recurrent_config(backward)
        assert cfg["kernel"] == "persistent_wide" and cfg["ctas_per_direction"] == H // 16, cfg
        assert cfg["cluster_size"] == (4 if mode == 1 else 1), cfg
    auto = _run(w, -1)           # the automatic choice: both persistent, the backward split
    for backward in (False, True):
        assert auto["plan"].recurrent_config(backward)["kernel"] == "persistent_wide"
    assert auto["plan"].recurrent_config(True)["cluster_size"] == 4
    compare_all(auto, run_oracle(w), TOL_BF16, label=f"wide automatic {case}")
    compare_all(gpu, run_oracle(w), TOL_BF16, label=f"wide persistent {case}")
    compare_all(gpu, run_oracle(w, bf16_products=True), TOL_BF16_EMULATED, label=f"wide persistent {case}",
                against="oracle-bf16-products")
    step = _run(w, 0)
    assert step["plan"].recurrent_config(False)["kernel"] == "step_launches"
    for k in ("y", "dx", "h_n", "c_n"):
        assert rel_err(gpu[k], step[k]) <= 5e-3, (k, rel_err(gpu[k], step[k]))


def test_persistent_wide_padded_and_states():
    w = synthetic.custom(2, 1, 24, 576, [7, 1, 12, 0, 12, 3], seed=21, dtype="bf16", weight_range=0.05)
    gpu = _run(w, 1, padded=True)
    assert gpu["plan"].recurrent_config(False)["kernel"] == "persistent_wide"
    compare_all(gpu, run_oracle(w), TOL_BF16, label="wide persistent padded")
    rng = np.random.default_rng(3)
    shape = (1, 2, 6, 576)
    st = {k: rng.uniform(-0.5, 0.5, shape).astype(np.float32) for k in ("h0", "c0", "dh_n", "dc_n")}
    gpu = _run(w, 1, states=st)
    compare_all(gpu, run_oracle(w, states=st), TOL_BF16, label="wide persistent states")


@pytest.mark.parametrize("mode", [1, 2], ids=["clusters", "no-clusters"])
def test_persistent_wide_bitwise_repeatable(mode):
    w = synthetic.custom(2, 1, 32, 1024, list(np.random.default_rng(9).integers(1, 20, 30)), seed=2,
                         dtype="bf16", weight_range=0.05)
    a, b = _run(w, mode), _run(w, mode)
    for k in ("y", "dx", "h_n", "c_n"):
        assert np.array_equal(a[k], b[k]), k
    for ga, gb in zip(a["grads"], b["grads"]):
        for k in ga:
            assert np.array_equal(ga[k], gb[k]), k


def test_split_backward_against_unsplit_and_ring_depth():
    """The forward is the same arithmetic with or without multicast: bitwise equal.  The
    K-split backward (clusters) and the unsplit one (no clusters) add the same partial products
    in different orders, and the bf16 rounding of the gate errors passed between steps can
    amplify that: equal within the bf16 path's bar.  The operand ring's depth does not change
    any result bit (the product's accumulation order is fixed)."""
    w = synthetic.custom(2, 1, 32, 1024, list(np.random.default_rng(4).integers(1, 40, 160)), seed=7,
                         dtype="bf16", weight_range=0.05)
    split, unsplit = _run(w, 1), _run(w, 2)
    for k in ("y", "h_n", "c_n"):
        assert np.array_equal(split[k], unsplit[k]), k
    assert rel_err(split["dx"], unsplit["dx"]) <= 5e-3, rel_err(split["dx"], unsplit["dx"])
    for gs, gu in zip(split["grads"], unsplit["grads"]):
        for k in gs:
            assert rel_err(gs[k], gu[k]) <= 5e-3, (k, rel_err(gs[k], gu[k]))
    shallow = _run(w, 1, stages=2)
    assert shallow["plan"].debug_wide_stages(-1) == (2, 2)
    assert split["plan"].debug_wide_stages(-1)[0] >= 3
    for k in ("y", "dx", "h_n", "c_n"):
        assert np.array_equal(split[k], shallow[k]), k
    for ga, gb in zip(split["grads"], shallow["grads"]):
        for k in ga:
            assert np.array_equal(ga[k], gb[k]), k
