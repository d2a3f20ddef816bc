"""The 2-D example-packing plan of the CUDA library, computed on the host (no GPU).

The library's placement must equal the packing oracle's exactly (Algorithm 1 of "No
Padding Please", App. B), and its wavefront schedule must be a valid one: every pixel
once per scan direction, predecessors one step earlier (Sec. IV-A: a skewed column
depends only on the previous one), successors the inverse of predecessors, and the
step count of each schedule as stated (canvas: height + width - 1 skewed columns;
diagonal: the longest example's h + w - 1).
"""
import numpy as np
import pytest

import oracle
from padding_free_variable_gb300 import ops


CASES = [
    ([3, 2, 3, 3, 2], [5, 4, 2, 3, 7], 0),
    ([1], [1], 0),
    ([4, 0, 2], [3, 5, 0], 0),
    ([2, 2, 2, 2], [1, 6, 3, 3], 5),
    ([5, 1, 5, 1], [2, 9, 2, 9], 3),
]


def _random_case(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 30))
    return list(rng.integers(0, 7, n)), list(rng.integers(0, 15, n)), int(rng.integers(0, 25))


ALL = CASES + [_random_case(s) for s in range(8)]


@pytest.mark.parametrize("case", ALL, ids=[f"case{i}" for i in range(len(ALL))])
def test_placement_matches_the_packing_oracle(case):
    hs, ws, rw = case
    ref = oracle.example_pack(hs, ws, rw)
    got = ops.md_compute_host(hs, ws, rw, 1, 0)
    assert list(got["y0"]) == ref["y0"] and list(got["x0"]) == ref["x0"]
    assert (got["height"], got["width"], got["rows"]) == (ref["height"], ref["width"], len(ref["rows"]))


@pytest.mark.parametrize("schedule", [0, 1], ids=["canvas", "diagonal"])
@pytest.mark.parametrize("case", ALL, ids=[f"case{i}" for i in range(len(ALL))])
def test_schedule_is_a_valid_wavefront(case, schedule):
    hs, ws, rw = case
    nd = 4
    t = ops.md_compute_host(hs, ws, rw, nd, schedule)
    hs_, ws_ = np.asarray(hs), np.asarray(ws)
    N = int((hs_ * ws_).sum())
    live = (hs_ > 0) & (ws_ > 0)
    ref = oracle.example_pack(hs, ws, rw)
    if N == 0:
        assert t["steps"] == 0
        return
    if schedule == 0:
        assert t["steps"] == ref["height"] + ref["width"] - 1
    else:
        assert t["steps"] == int((hs_ + ws_ - 1)[live].max())
    so = t["step_off"]
    assert so.shape == (nd, t["steps"] + 1)
    step_of = np.empty(nd * N, dtype=np.int64)
    for d in range(nd):
        assert so[d, 0] == d * N and so[d, -1] == (d + 1) * N
        assert (np.diff(so[d]) >= 0).all()
        for k in range(t["steps"]):
            step_of[so[d, k]:so[d, k + 1]] = k
    pix_off = np.concatenate([[0], np.cumsum(hs_ * ws_)])
    for d in range(nd):
        cells = np.arange(d * N, (d + 1) * N)
        assert sorted(t["src"][cells]) == list(range(N))          # every pixel once per direction
    fx = np.array([d & 1 for d in range(nd)])
    fy = np.array([(d >> 1) & 1 for d in range(nd)])
    ex = np.searchsorted(pix_off, t["src"], side="right") - 1
    for p in range(nd * N):
        d = p // N
        e = ex[p]
        h, w = int(hs_[e]), int(ws_[e])
        q = t["src"][p] - pix_off[e]
        y, x = divmod(int(q), w)
        ys = h - 1 - y if fy[d] else y
        xs = w - 1 - x if fx[d] else x
        if schedule == 1:
            assert step_of[p] == ys + xs
        else:
            yo = ref["height"] - ref["y0"][e] - h if fy[d] else ref["y0"][e]
            xo = ref["width"] - ref["x0"][e] - w if fx[d] else ref["x0"][e]
            assert step_of[p] == yo + xo + ys + xs          # the skewed canvas column
        for pred, succ, has in ((t["pred1"], t["succ1"], ys > 0), (t["pred2"], t["succ2"], xs > 0)):
            q1 = pred[p]
            if not has:
                assert q1 == -1
            else:
                assert q1 >= 0 and q1 // N == d and ex[q1] == e and step_of[q1] == step_of[p] - 1
                assert succ[q1] == p
    # within a step, cells follow the packing order of their examples
    order = {e: i for i, e in enumerate(i for r in ref["rows"] for i in r)}
    for d in range(nd):
        for k in range(t["steps"]):
            es = [order[int(ex[p])] for p in range(so[d, k], so[d, k + 1])]
            assert es == sorted(es)


def test_plan_arguments_are_checked():
    from padding_free_variable_gb300 import _lib
    with pytest.raises(_lib.LSTMError):
        ops.md_compute_host([2], [2], 0, 5, 0)           # at most four directions
    with pytest.raises(_lib.LSTMError):
        ops.md_compute_host([2], [-1], 0, 1, 0)
    with pytest.raises(_lib.LSTMError):
        ops.md_compute_host([2], [2], 0, 1, 2)           # schedules 0 and 1
