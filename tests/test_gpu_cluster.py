"""The cluster-resident recurrent kernels (one thread-block cluster per
direction, tcgen05 per-step products, DSMEM exchange) against the oracle, on
the shapes that select them (H a multiple of 32, one direction's R within a
cluster of at most 16 CTAs), and against the grid kernels on the same input."""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_BF16, TOL_BF16_EMULATED, TOL_F32, compare_all, rel_err, run_gpu, run_oracle

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
    (1, 2, 8, 32, [5, 40, 39, 1, 2, 3, 4, 30], "f32"),
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], "f32"),
    (2, 2, 24, 128, [17, 2, 9, 33, 1, 0, 12, 33], "f32"),
    (2, 1, 40, 256, list(np.random.default_rng(9).integers(1, 80, 20)), "f32"),
    (2, 2, 16, 64, [9, 0, 4, 21, 21, 2], "bf16"),
    (2, 1, 32, 256, [60, 3, 44, 17, 60, 9], "bf16"),
    # wide batches: 112 and 128 operand rows (fewer accumulator chains fit next to R in TMEM)
    (2, 1, 16, 64, list(np.random.default_rng(3).integers(1, 20, 100)), "f32"),
    (2, 1, 32, 256, list(np.random.default_rng(4).integers(1, 12, 128)), "f32"),
    # H = 512: clusters of 16 CTAs per direction
    (1, 1, 32, 512, [20, 7, 13, 1], "bf16"),
    (2, 2, 24, 512, [30, 5, 17, 30, 2, 9], "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}" for c in CASES])
def test_cluster_kernels_match_oracle(case):
    nd, nl, D, H, lengths, dtype = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=5 + H, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w)
    for backward in (False, True):
        cfg = gpu["plan"].recurrent_config(backward)
        assert (cfg["kernel"], cfg["ctas_per_direction"], cfg["product"]) == ("cluster", H // 32, "tcgen05"), cfg
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"cluster {case}")
    if dtype == "bf16":
        compare_all(gpu, run_oracle(w, bf16_products=True), TOL_BF16_EMULATED, label=f"cluster {case}",
                    against="oracle-bf16-products")
    grid = run_gpu(w, ctas=H // 32)          # an explicit CTA count selects the grid kernels
    for k in ("y", "dx", "h_n", "c_n"):
        assert rel_err(gpu[k], grid[k]) <= (TOL_BF16 if dtype == "bf16" else TOL_F32), k


VARIANT_CASES = [
    (2, 1, 16, 64, [9, 0, 4, 21, 21, 2, 7], "f32"),
    (2, 2, 24, 128, [17, 2, 9, 33, 1, 0, 12, 33], "f32"),
    (1, 1, 32, 256, list(np.random.default_rng(12).integers(1, 40, 40)), "f32"),
    (2, 1, 32, 256, [60, 3, 44, 17, 60, 9], "bf16"),
]


@pytest.mark.parametrize("variant", [0, 1, 2, 3], ids=["barrier", "bulk", "barrier-tiles", "bulk-tiles"])
@pytest.mark.parametrize("case", VARIANT_CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}" for c in VARIANT_CASES])
def test_every_cluster_variant_matches_oracle(case, variant):
    """Each exchange (DSMEM stores between barrier halves, or bulk copies into double
    buffers) with and without TMA operand tiles: the automatic choice picks by shared
    memory, so small batches alone would reach only one of them."""
    nd, nl, D, H, lengths, dtype = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=40 + H + variant, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, variant=variant)
    for backward in (False, True):
        cfg = gpu["plan"].recurrent_config(backward)
        assert cfg["kernel"] == "cluster", cfg
        assert cfg["exchange"] == ("bulk" if variant & 1 else "barrier"), cfg
        assert cfg["tma_tiles"] == bool(variant & 2), cfg
    compare_all(gpu, run_oracle(w), TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"variant {variant} {case}")


def test_cluster_kernels_padded_plan():
    w = synthetic.custom(2, 1, 12, 64, [6, 0, 2, 9, 1, 6], seed=31, weight_range=0.4)
    gpu = run_gpu(w, padded=True)
    compare_all(gpu, run_oracle(w), TOL_F32, label="cluster padded")
