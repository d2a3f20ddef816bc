"""Initial states and final-state errors through the C ABI (lstm_fwd_state / lstm_bwd_state)
against the oracle given the same h0, c0, dh_n and dc_n (RETURNN paper, Sec. 3.2: the final
state of one recurrent network passed on as the initial state of another).  Every recurrent
kernel family is reached: the cluster kernels (fp32 and bf16), the grid kernels, the per-step
tcgen05 path of layers wider than a cluster, and the CUDA-core engine."""
import numpy as np
import pytest

from padding_free_variable_gb300 import synthetic
from gpu_harness import TOL_BF16, TOL_BF16_EMULATED, TOL_F32, compare_all, run_gpu, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from padding_free_variable_gb300 import build
    build.build()


def _states(w, seed, scale=0.5, which=("h0", "c0", "dh_n", "dc_n")):
    rng = np.random.default_rng(seed)
    shape = (w.spec.num_layers, w.spec.num_directions, len(w.lengths), w.spec.hidden_size)
    return {k: (rng.uniform(-scale, scale, shape).astype(np.float32) if k in which else None)
            for k in ("h0", "c0", "dh_n", "dc_n")}


CASES = [
    # ndir, layers, D, H, lengths, dtype, ctas (0 = automatic), engine, expected recurrent kernel
    (2, 2, 16, 64, [9, 0, 4, 13, 13, 2, 7], "f32", 0, 0, "cluster"),
    (1, 1, 8, 32, [5, 40, 39, 1, 2, 3, 4, 30], "f32", 0, 0, "cluster"),
    (2, 1, 32, 256, [60, 3, 44, 17, 60, 9], "bf16", 0, 0, "cluster"),
    (2, 2, 24, 40, [17, 2, 9, 33, 1, 0, 12], "f32", 3, 0, "grid"),
    (2, 1, 16, 48, [9, 0, 4, 21, 21, 2], "bf16", 4, 0, "grid"),
    (2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], "f32", 0, 1, "grid"),
    (2, 2, 24, 520, [7, 1, 12, 0, 12, 3], "bf16", 0, 0, "step_launches"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"nd{c[0]}-L{c[1]}-H{c[3]}-{c[5]}-g{c[6]}-e{c[7]}" for c in CASES])
def test_states_match_oracle(case):
    nd, nl, D, H, lengths, dtype, ctas, engine, kernel = case
    bf16 = dtype == "bf16"
    w = synthetic.custom(nd, nl, D, H, lengths, seed=90 + H, dtype=dtype, weight_range=0.1 if bf16 else 0.3)
    st = _states(w, 7 + H)
    gpu = run_gpu(w, ctas=ctas, engine=engine, states=st)
    for backward in (False, True):
        assert gpu["plan"].recurrent_config(backward)["kernel"] == kernel
    ref = run_oracle(w, states=st)
    compare_all(gpu, ref, TOL_BF16 if bf16 else TOL_F32, label=f"states {case}")
    if bf16:
        compare_all(gpu, run_oracle(w, states=st, bf16_products=True), TOL_BF16_EMULATED, label=f"states {case}",
                    against="oracle-bf16-products")
    # an empty sequence hands its initial state through, and its final-state errors back
    for b in np.flatnonzero(np.asarray(lengths) == 0):
        np.testing.assert_array_equal(gpu["h_n"][:, :, b], st["h0"][:, :, b])
        np.testing.assert_array_equal(gpu["dc0"][:, :, b], st["dc_n"][:, :, b])


@pytest.mark.parametrize("which", [("h0",), ("c0",), ("dh_n", "dc_n")], ids=["h0", "c0", "final-errors"])
def test_each_state_input_alone(which):
    """Each input on its own (the others NULL), so that a term wired to the wrong input shows."""
    w = synthetic.custom(2, 1, 16, 64, [9, 0, 4, 13, 13, 2, 7], seed=5, weight_range=0.3)
    st = _states(w, 11, which=which)
    compare_all(run_gpu(w, states=st), run_oracle(w, states=st), TOL_F32, label=f"state {which}")


def test_zero_states_equal_the_plain_entry_points():
    """lstm_fwd_state / lstm_bwd_state with no state give lstm_fwd / lstm_bwd bit for bit, and
    still the gradients of the (zero) initial state, which the loss depends on through R and
    the forget gate and peepholes."""
    w = synthetic.custom(2, 2, 16, 64, [9, 0, 4, 13, 13, 2, 7], seed=6, weight_range=0.3)
    a = run_gpu(w)
    none = {"h0": None, "c0": None, "dh_n": None, "dc_n": None}
    b = run_gpu(w, states=none)
    for k in ("y", "dx", "h_n", "c_n"):
        assert np.array_equal(a[k], b[k]), k
    for ga, gb in zip(a["grads"], b["grads"]):
        for k in ga:
            assert np.array_equal(ga[k], gb[k]), k
    compare_all(b, run_oracle(w, states=none), TOL_F32, label="zero states")


def test_padded_plan_refuses_states():
    from padding_free_variable_gb300 import _lib
    w = synthetic.custom(2, 1, 16, 64, [9, 4, 13], seed=8, weight_range=0.3)
    with pytest.raises(_lib.LSTMError) as e:
        run_gpu(w, padded=True, states=_states(w, 3))
    assert e.value.code == _lib.LSTM_ERR_UNSUPPORTED


def test_all_sequences_empty():
    w = synthetic.custom(2, 1, 16, 64, [0, 0, 0], seed=9, weight_range=0.3)
    st = _states(w, 4)
    gpu = run_gpu(w, states=st)
    np.testing.assert_array_equal(gpu["h_n"], st["h0"])
    np.testing.assert_array_equal(gpu["c_n"], st["c0"])
    np.testing.assert_array_equal(gpu["dh0"], st["dh_n"])
    np.testing.assert_array_equal(gpu["dc0"], st["dc_n"])
