"""The cluster-resident recurrent kernels (one thread-block cluster per
direction and sequence group, tcgen05 per-step products, DSMEM exchange)
against the oracle, on the shapes that select them (H a multiple of 32, one
direction's R within a cluster of at most 16 CTAs), and against the grid
kernels on the same input."""
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
    # wide batches (the automatic choice cuts them into sequence groups of a few slots)
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


GROUP_CASES = [
    # ndir, layers, D, H, lengths, dtype, slots per group
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7, 20, 1, 1, 6, 5, 0, 17, 3, 8, 8, 2, 11, 4], "f32", 8),   # ragged last group
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7, 20, 1, 1, 6, 5, 0, 17, 3, 8, 8, 2, 11, 4], "f32", 1),   # one slot each
    (2, 2, 8, 32, [12, 5, 0, 0, 0, 0, 0, 0, 0, 0], "f32", 2),        # groups whose sequences are all empty
    (1, 1, 24, 128, list(np.random.default_rng(21).integers(1, 30, 24)), "f32", 16),
    (2, 1, 32, 256, [60, 3, 44, 17, 60, 9, 33, 33, 1, 50, 12, 7], "bf16", 5),
    # one group of 112 / 128 operand rows: fewer accumulator chains fit next to R in TMEM
    (2, 1, 16, 64, list(np.random.default_rng(3).integers(1, 20, 100)), "f32", 128),
    (2, 1, 32, 256, list(np.random.default_rng(4).integers(1, 12, 128)), "bf16", 128),
]


@pytest.mark.parametrize("case", GROUP_CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}-S{c[6]}" for c in GROUP_CASES])
def test_sequence_groups_match_oracle_and_one_group(case):
    """Cutting the sorted slots into groups (one cluster per direction and group) changes
    neither the results nor their bits: each row's products and cell see the same operands."""
    nd, nl, D, H, lengths, dtype, slots = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=70 + H + slots, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, group_slots=slots)
    B = len(lengths)
    expect = (-(-B // min(slots, B)), min(slots, B))
    for backward in (False, True):
        assert gpu["plan"].recurrent_config(backward)["kernel"] == "cluster"
        assert gpu["plan"].recurrent_groups(backward) == expect
    compare_all(gpu, run_oracle(w), TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"groups {case}")
    if B <= 128:
        one = run_gpu(w, group_slots=B)
        assert one["plan"].recurrent_groups(False) == (1, B)
        for k in ("y", "dx", "h_n", "c_n"):
            assert np.array_equal(gpu[k], one[k]), k
        for ga, gb in zip(gpu["grads"], one["grads"]):
            for k in ga:
                assert np.array_equal(ga[k], gb[k]), k


def test_automatic_groups_give_every_cluster_an_sm():
    """The automatic group size: the smallest multiple of 8 slots that fits every (direction,
    group) cluster on its own SMs."""
    w = synthetic.custom(2, 1, 16, 256, list(np.random.default_rng(8).integers(1, 30, 64)), seed=3)
    gpu = run_gpu(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups, slots = gpu["plan"].recurrent_groups(False)
    assert slots % 8 == 0 and groups == -(-64 // slots)
    assert groups * 2 * 8 <= sms
    assert slots == 8 or (-(-64 // (slots - 8))) * 2 * 8 > sms
    compare_all(gpu, run_oracle(w), TOL_F32, label="automatic groups")
