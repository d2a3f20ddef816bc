"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Invariant I1 ("No Padding Please", Sec. V-B: the packed computation equals
what is obtained for each input separately): the oracle loops over each
sequence alone, the GPU runs the packed batch.
"""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import (TOL_BF16, TOL_BF16_EMULATED, TOL_F32, compare_all, rel_err, run_gpu, run_oracle,
                         select_rows)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


@pytest.mark.parametrize("wid", [1, 2])
def test_full_workload_fp32(wid):
    w = synthetic.workload(wid)
    gpu = run_gpu(w)
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_F32, label=f"workload {wid}")


@pytest.mark.slow
def test_full_workload_4_fp32():
    w = synthetic.workload(4)
    gpu = run_gpu(w)
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_F32, label="workload 4")


SMALL = [
    # ndir, layers, D, H, lengths, dtype, CTAs per direction (0 = automatic)
    (1, 1, 8, 8, [1], "f32", 0),
    (2, 1, 16, 8, [5, 0, 3, 3, 1], "f32", 2),
    (2, 2, 24, 40, [17, 2, 9, 33, 1, 0, 12], "f32", 0),
    (2, 2, 24, 40, [17, 2, 9, 33, 1, 0, 12], "f32", 3),      # 14 units per CTA, last CTA 12
    (1, 3, 8, 64, [40, 39, 1], "f32", 5),
    (2, 1, 32, 136, list(np.random.default_rng(5).integers(1, 51, 37)), "f32", 0),
    (2, 1, 4, 200, [70, 3, 70, 12, 1, 44], "f32", 76),       # 3 units per CTA, ragged last
    (2, 2, 16, 48, [9, 0, 4, 21, 21, 2], "bf16", 0),
    (2, 2, 16, 48, [9, 0, 4, 21, 21, 2], "bf16", 7),
    (2, 1, 40, 520, [30, 7, 1, 19], "bf16", 0),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"nd{c[0]}-L{c[1]}-D{c[2]}-H{c[3]}-{c[5]}-g{c[6]}" for c in SMALL])
def test_small_shapes(case):
    nd, nl, D, H, lengths, dtype, ctas = case
    # bf16 cases use weights twice the bf16 workloads' scale: at U(+-0.3) and H = 520 the bf16
    # rounding itself (oracle against oracle) already moves y by 2.6e-2 of its scale
    w = synthetic.custom(nd, nl, D, H, lengths, seed=77 + H, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, ctas=ctas)
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_BF16 if dtype == "bf16" else TOL_F32, label=str(case))
    if dtype == "bf16":
        emu = run_oracle(w, bf16_products=True)
        compare_all(gpu, emu, TOL_BF16_EMULATED, label=str(case), against="oracle-bf16-products")


@pytest.mark.parametrize("wid,batch", [(3, 6), (5, 8)])
def test_bf16_workloads_reduced_batch(wid, batch):
    """Full layer widths and depth of the bf16 workloads on a few sequences: every output
    and every gradient against the oracle fed the same bf16-rounded x, W and R."""
    w = synthetic.workload(wid, batch=batch)
    gpu = run_gpu(w)
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_BF16, label=f"workload {wid} B={batch}")
    emu = run_oracle(w, bf16_products=True)
    compare_all(gpu, emu, TOL_BF16_EMULATED, label=f"workload {wid} B={batch}", against="oracle-bf16-products")


@pytest.mark.slow
@pytest.mark.parametrize("wid", [3, 5])
def test_bf16_workloads_full_size_sampled(wid):
    """Full-size bf16 workloads (all B sequences, full depth and width) in the benchmarked
    launch configuration.  The upstream gradient G is zero on every sequence but three
    sampled ones, so the batch's weight gradients are exactly the sum over those three
    (the others pass no error); the oracle runs the three alone.  Every output and every
    gradient of every layer is compared."""
    w = synthetic.workload(wid)
    seqs = list(np.argsort(w.lengths, kind="stable")[:2]) + [int(np.argmax(w.lengths))] if wid == 5 else \
        list(np.argsort(w.lengths, kind="stable")[:2]) + [int(np.argsort(w.lengths, kind="stable")[len(w.lengths) // 2])]
    st = np.concatenate([[0], np.cumsum(w.lengths)])
    keep = np.zeros(len(w.G), dtype=bool)
    for q in seqs:
        keep[st[q]:st[q + 1]] = True
    w.G = np.where(keep[:, None], w.G, 0.0).astype(np.float32)
    gpu = run_gpu(w)
    ref = run_oracle(w, seqs=seqs, nthreads=len(seqs))
    sub = {"y": select_rows(w, seqs, gpu["y"]), "dx": select_rows(w, seqs, gpu["dx"]),
           "h_n": gpu["h_n"][:, :, seqs], "c_n": gpu["c_n"][:, :, seqs], "grads": gpu["grads"]}
    compare_all(sub, ref, TOL_BF16, label=f"workload {wid} full size, 3 sampled sequences")
    # the unsampled sequences pass no error: their input gradient is exactly zero
    assert not np.any(gpu["dx"][~keep])


ENGINE_CASES = [
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], "f32", 4),
    (2, 2, 24, 40, [17, 2, 9, 33, 1, 0, 12], "f32", 3),
    (1, 2, 8, 32, [5, 40, 39, 1, 2, 3, 4, 30], "f32", 0),
    (2, 2, 16, 48, [9, 0, 4, 21, 21, 2], "bf16", 7),
    (2, 1, 32, 256, [60, 3, 44, 17, 60, 9], "bf16", 0),
]


@pytest.mark.parametrize("engine", [0, 1], ids=["tensor-cores", "cuda-cores"])
@pytest.mark.parametrize("case", ENGINE_CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}-g{c[6]}" for c in ENGINE_CASES])
def test_both_product_engines(case, engine):
    """The tensor-core and the CUDA-core products of every kernel against the oracle."""
    nd, nl, D, H, lengths, dtype, ctas = case
    w = synthetic.custom(nd, nl, D, H, lengths, seed=11 + H, dtype=dtype,
                         weight_range=0.1 if dtype == "bf16" else 0.3)
    gpu = run_gpu(w, ctas=ctas, engine=engine)
    ref = run_oracle(w)
    compare_all(gpu, ref, TOL_BF16 if dtype == "bf16" else TOL_F32, label=f"{case} engine={engine}")
    if dtype == "bf16":
        emu = run_oracle(w, bf16_products=True)
        compare_all(gpu, emu, TOL_BF16_EMULATED, label=f"{case} engine={engine}", against="oracle-bf16-products")


def test_padded_comparator_matches_oracle():
    """Invariant I3 on the GPU: the padded, masked run gives the per-sequence results."""
    w = synthetic.custom(2, 2, 12, 24, [6, 0, 2, 9, 1, 6], seed=31, weight_range=0.4)
    for ctas in (0, 4):
        gpu = run_gpu(w, padded=True, ctas=ctas)
        ref = run_oracle(w)
        compare_all(gpu, ref, TOL_F32, label=f"padded ctas={ctas}")


def test_bitwise_repeatable():
    w = synthetic.workload(2, batch=12)
    a = run_gpu(w)
    b = run_gpu(w)
    for k in ("y", "dx", "h_n", "c_n"):
        assert np.array_equal(a[k], b[k]), k
    for ga, gb in zip(a["grads"], b["grads"]):
        for k in ga:
            assert np.array_equal(ga[k], gb[k]), k


def test_permuting_sequences_permutes_outputs():
    """Invariant I2 on the GPU: caller order in, caller order out."""
    w = synthetic.custom(2, 1, 8, 32, [5, 9, 2, 9, 7], seed=12)
    perm = np.array([3, 0, 4, 2, 1])
    st = np.concatenate([[0], np.cumsum(w.lengths)])
    w2 = synthetic.custom(2, 1, 8, 32, w.lengths[perm], seed=12)
    w2.x = np.concatenate([w.x[st[i]:st[i + 1]] for i in perm])
    w2.G = np.concatenate([w.G[st[i]:st[i + 1]] for i in perm])
    w2.layers = w.layers
    a, b = run_gpu(w), run_gpu(w2)
    np.testing.assert_array_equal(select_rows(w, perm, a["y"]), b["y"])
    np.testing.assert_array_equal(a["h_n"][:, :, perm], b["h_n"])
