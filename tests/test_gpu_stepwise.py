"""The per-step-launch comparator path (one product launch per direction and
one cell launch per time step, the RETURNN paper's Sec. 4.2 design) against
the oracle, on the same seeded inputs and tolerances as the persistent path."""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_BF16, TOL_F32, compare_all, run_gpu, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


CASES = [
    # ndir, layers, D, H, lengths, dtype
    (1, 1, 8, 32, [1], "f32"),
    (1, 2, 8, 48, [5, 40, 39, 1, 2, 3, 4, 30], "f32"),
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], "f32"),
    (2, 2, 24, 136, [17, 2, 9, 33, 1, 0, 12, 33], "f32"),
    (2, 2, 16, 64, [9, 0, 4, 21, 21, 2], "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}" for c in CASES])
def test_stepwise_matches_oracle(case):
    nd, nl, D, H, lengths, dtype = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=11 + H, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, stepwise=True)
    compare_all(gpu, run_oracle(w), TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"stepwise {case}")


@pytest.mark.parametrize("wid", [1, 2])
def test_stepwise_full_workload(wid):
    w = synthetic.workload(wid)
    gpu = run_gpu(w, stepwise=True)
    compare_all(gpu, run_oracle(w), TOL_F32, label=f"stepwise workload {wid}")


def test_wide_bf16_layers_run_per_step_tensor_core_products():
    """bf16 layers whose R does not fit one cluster (H > 512) run their recurrence through
    lstm_fwd / lstm_bwd as per-step tcgen05 products plus cell launches."""
    from gpu_harness import TOL_BF16_EMULATED
    w = synthetic.custom(2, 2, 24, 520, [7, 1, 12, 0, 12, 3], seed=77, dtype="bf16", weight_range=0.1)
    gpu = run_gpu(w)
    for backward in (False, True):
        cfg = gpu["plan"].recurrent_config(backward)
        assert cfg["kernel"] == "step_launches" and cfg["product"] == "tcgen05", cfg
    compare_all(gpu, run_oracle(w), TOL_BF16, label="wide bf16 per-step")
    compare_all(gpu, run_oracle(w, bf16_products=True), TOL_BF16_EMULATED, label="wide bf16 per-step",
                against="oracle-bf16-products")


def test_wide_bf16_padded_plan_runs_the_same_per_step_kernels():
    """The zero-padded comparator of a layer wider than a cluster (H > 512) runs the same
    per-step tcgen05 products and masked cell kernels as the packed run, and gives the
    per-sequence results ("On batching variable size inputs...", Sec. 2: padding to the
    longest sequence of the batch)."""
    w = synthetic.custom(2, 2, 24, 520, [7, 1, 12, 0, 12, 3], seed=78, dtype="bf16", weight_range=0.1)
    gpu = run_gpu(w, padded=True)
    for backward in (False, True):
        cfg = gpu["plan"].recurrent_config(backward)
        assert cfg["kernel"] == "step_launches" and cfg["product"] == "tcgen05", cfg
    compare_all(gpu, run_oracle(w), TOL_BF16, label="wide bf16 padded")
    packed = run_gpu(w)
    for k in ("y", "dx", "h_n", "c_n"):
        assert np.abs(gpu[k] - packed[k]).max() <= 1e-6 * max(1.0, np.abs(packed[k]).max()), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_stepwise_padded_plan_matches_oracle(dtype):
    w = synthetic.custom(2, 2, 16, 64, [9, 0, 4, 21, 21, 2], seed=19, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, padded=True, stepwise=True)
    compare_all(gpu, run_oracle(w), TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"stepwise padded {dtype}")
