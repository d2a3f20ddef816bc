"""Pins of the 2-D MDLSTM oracle and of the 2-D packing oracle to facts outside them.

"No Padding Please: Efficient Neural Handwriting Recognition" prints no worked MDLSTM
example and no equations, so the layer oracle is pinned by:
  * a closed form: with zero input and recurrent weights and no input/forget
    peepholes, every cell has the same gates and c(y, x) is i z times a sum over the
    monotone lattice paths into (y, x), f1 per vertical and f2 per horizontal step;
    the output gate's peepholes read the predecessors' states (Sec. III's variant);
  * reduction to the 1-D LSTM oracle (itself pinned against torch.nn.LSTM, finite
    differences and closed forms): a one-row image is a 1-D LSTM along x with
    predecessor-2 weights, a one-column image one along y with predecessor-1
    weights (output-gate peepholes zero, where the 1-D cell reads c_t);
  * a symmetry: transposing the image and swapping the roles of the two
    predecessors (U1 <-> U2, f1 <-> f2, each peephole pair) transposes the output;
  * central finite differences of L = <y, G> for every parameter and the input,
    in all four scan directions.
The packing oracle (Algorithm 1, App. B) is pinned by a hand-worked placement and by
the properties the page asks of a packing (same-height rows, separator pixels, the
greedy fill).
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import mdlstm


def sig(v):
    return 1.0 / (1.0 + np.exp(-v))


def rand_layer(rng, nd, D, H, r=0.4):
    return {"W": rng.uniform(-r, r, (nd, 5 * H, D)), "U1": rng.uniform(-r, r, (nd, 5 * H, H)),
            "U2": rng.uniform(-r, r, (nd, 5 * H, H)), "b": rng.uniform(-r, r, (nd, 5 * H)),
            "peep": rng.uniform(-r, r, (nd, 6, H))}


def test_lattice_path_closed_form():
    """W = U1 = U2 = 0, p_i = p_f = 0: i, f1, f2, z are constants and
    c(y, x) = i z sum_{a<=y, b<=x} C(a+b, a) f1^a f2^b; o reads the predecessors' states."""
    H, D, h, w = 2, 3, 3, 4
    b = np.array([0.3, -0.2, 0.5, 0.1, -0.4, 0.2, 0.7, -0.6, 0.25, -0.15])   # i, f1, f2, z, o blocks
    peep = np.zeros((6, H))
    peep[4] = [0.8, -0.5]     # p_o1
    peep[5] = [-0.3, 0.6]     # p_o2
    layer = {"W": np.zeros((1, 5 * H, D)), "U1": np.zeros((1, 5 * H, H)), "U2": np.zeros((1, 5 * H, H)),
             "b": b[None], "peep": peep[None]}
    x = np.random.default_rng(0).standard_normal((h * w, D))
    y = oracle.md_layer([h], [w], x, layer)["y"].reshape(h, w, H)
    ig, f1, f2, zg = sig(b[0:2]), sig(b[2:4]), sig(b[4:6]), np.tanh(b[6:8])
    c = np.zeros((h, w, H))
    for yy in range(h):
        for xx in range(w):
            c[yy, xx] = ig * zg * sum(math.comb(a + bb, a) * f1 ** a * f2 ** bb
                                      for a in range(yy + 1) for bb in range(xx + 1))
    for yy in range(h):
        for xx in range(w):
            s1 = c[yy - 1, xx] if yy > 0 else 0.0
            s2 = c[yy, xx - 1] if xx > 0 else 0.0
            og = sig(b[8:10] + peep[4] * s1 + peep[5] * s2)
            np.testing.assert_allclose(y[yy, xx], og * np.tanh(c[yy, xx]), rtol=1e-13, atol=1e-15)


def _to_1d(layer, d, which):
    """The 1-D LSTM parameters that a one-row (which = 2) or one-column (which = 1) image sees."""
    H = layer["U1"].shape[2]
    i, f1, f2, z, o = (slice(k * H, (k + 1) * H) for k in range(5))
    f = f2 if which == 2 else f1
    U = layer["U2"] if which == 2 else layer["U1"]
    p = layer["peep"][d]
    rows = lambda A: np.concatenate([A[i], A[f], A[z], A[o]])
    return {"W": rows(layer["W"][d]), "R": rows(U[d]), "b": rows(layer["b"][d]),
            "peep": np.stack([p[1] if which == 2 else p[0], p[3] if which == 2 else p[2], np.zeros(H)])}


@pytest.mark.parametrize("which", [1, 2], ids=["one-column", "one-row"])
def test_single_line_images_reduce_to_the_1d_lstm(which):
    rng = np.random.default_rng(11 + which)
    H, D, L = 3, 4, 7
    layer = rand_layer(rng, 4, D, H)
    layer["peep"][:, 4:6] = 0.0            # the 1-D cell's output peephole reads c_t; 2-D reads S
    x = rng.standard_normal((L, D))
    h, w = (L, 1) if which == 1 else (1, L)
    y2 = oracle.md_layer([h], [w], x, layer)["y"]
    # direction d scans forward along the line when its flip bit for that axis is clear
    for d in range(4):
        flip = (d >> 1) & 1 if which == 1 else d & 1
        l1 = _to_1d(layer, d, which)
        if flip:
            one = {k: np.stack([np.zeros_like(v), v]) for k, v in l1.items()}
            y1 = oracle.lstm_stack([L], x, [one], 2, H)["y"][:, H:]
        else:
            one = {k: v[None] for k, v in l1.items()}
            y1 = oracle.lstm_stack([L], x, [one], 1, H)["y"]
        np.testing.assert_allclose(y2[:, d * H:(d + 1) * H], y1, rtol=1e-12, atol=1e-14)


def test_transposition_swaps_the_predecessors():
    rng = np.random.default_rng(5)
    H, D, h, w = 2, 3, 3, 5
    layer = rand_layer(rng, 4, D, H)
    x = rng.standard_normal((h, w, D))
    y = oracle.md_layer([h], [w], x.reshape(-1, D), layer)["y"].reshape(h, w, 4, H)
    # the transposed image's direction dt (x- and y-flips exchanged) takes direction d's
    # parameters with the two predecessors' roles swapped
    tr = [((d & 1) << 1) | ((d >> 1) & 1) for d in range(4)]
    Hs, F2 = slice(H, 2 * H), slice(2 * H, 3 * H)
    sw = {k: np.zeros_like(v) for k, v in layer.items()}
    for d in range(4):
        W, U1, U2, b = (layer[k][d].copy() for k in ("W", "U1", "U2", "b"))
        for a in (W, U1, U2, b):
            a[Hs], a[F2] = a[F2].copy(), a[Hs].copy()                  # f1 <-> f2 blocks
        sw["W"][tr[d]], sw["U1"][tr[d]], sw["U2"][tr[d]], sw["b"][tr[d]] = W, U2, U1, b
        sw["peep"][tr[d]] = layer["peep"][d][[1, 0, 3, 2, 5, 4]]
    yt = oracle.md_layer([w], [h], x.transpose(1, 0, 2).reshape(-1, D), sw)["y"].reshape(w, h, 4, H)
    for d in range(4):
        np.testing.assert_allclose(yt[:, :, tr[d]].transpose(1, 0, 2), y[:, :, d], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("d", range(4))
def test_finite_differences(d):
    rng = np.random.default_rng(20 + d)
    H, D = 2, 2
    hs, ws = [2, 3], [3, 2]
    N = 12
    layer = rand_layer(rng, 1, D, H)
    full = rand_layer(rng, 4, D, H)
    for k in full:
        full[k][d] = layer[k][0]
        for e in range(4):
            if e != d:
                full[k][e] = 0.0
    x = rng.standard_normal((N, D))
    G = np.zeros((N, 4 * H))
    G[:, d * H:(d + 1) * H] = rng.standard_normal((N, H))
    out = oracle.md_layer(hs, ws, x, full, G)

    def loss(lay, xx):
        return float((oracle.md_layer(hs, ws, xx, lay)["y"] * G).sum())

    eps = 1e-6
    for k in ("W", "U1", "U2", "b", "peep"):
        it = np.nditer(full[k][d], flags=["multi_index"])
        for _ in it:
            idx = (d,) + it.multi_index
            lp = {kk: v.copy() for kk, v in full.items()}
            lm = {kk: v.copy() for kk, v in full.items()}
            lp[k][idx] += eps
            lm[k][idx] -= eps
            num = (loss(lp, x) - loss(lm, x)) / (2 * eps)
            assert abs(num - out["grads"][k][idx]) <= 1e-6 * max(1.0, abs(num)), (k, idx, num, out["grads"][k][idx])
    for i in range(N):
        for j in range(D):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += eps
            xm[i, j] -= eps
            num = (loss(full, xp) - loss(full, xm)) / (2 * eps)
            assert abs(num - out["dx"][i, j]) <= 1e-6 * max(1.0, abs(num))


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "md_packing_example.txt")


def _read_golden():
    rec = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            rec[k.strip()] = [int(t) for t in v.split()]
    return rec


def test_packing_matches_hand_worked_example():
    g = _read_golden()
    p = oracle.example_pack(g["heights"], g["widths"], g["row_width"][0])
    assert p["y0"] == g["y0"] and p["x0"] == g["x0"]
    assert [p["height"], p["width"]] == g["canvas"]
    assert [len(r) for r in p["rows"]] == g["row_sizes"]


@pytest.mark.parametrize("seed", range(6))
def test_packing_properties(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    hs = rng.integers(0, 6, n)
    ws = rng.integers(0, 12, n)
    rw = int(rng.integers(0, 20))
    p = oracle.example_pack(hs, ws, rw)
    live = [i for i in range(n) if hs[i] > 0 and ws[i] > 0]
    assert sorted(i for r in p["rows"] for i in r) == live
    W = rw if rw > 0 else max([ws[i] for i in live], default=0)
    owner = -np.ones((p["height"], p["width"]), dtype=int)
    for i in live:
        blk = owner[p["y0"][i]:p["y0"][i] + hs[i], p["x0"][i]:p["x0"][i] + ws[i]]
        assert (blk == -1).all()
        blk[:] = i
    # no two examples touch: every 4-neighbour of an example pixel is the same example or empty
    for yy in range(p["height"]):
        for xx in range(p["width"]):
            if owner[yy, xx] < 0:
                continue
            for dy, dx in ((1, 0), (0, 1)):
                y2, x2 = yy + dy, xx + dx
                if y2 < p["height"] and x2 < p["width"] and owner[y2, x2] >= 0:
                    assert owner[y2, x2] == owner[yy, xx]
    for r in p["rows"]:
        assert len({int(hs[i]) for i in r}) == 1                     # one height a row
        used = sum(int(ws[i]) for i in r) + len(r) - 1
        assert used <= W or len(r) == 1
    # greedy: when a row closed with examples of its height still to place, none of them fit
    placed = set()
    for k, r in enumerate(p["rows"]):
        placed.update(r)
        used = sum(int(ws[i]) for i in r) + len(r) - 1
        rest = [i for i in live if i not in placed and hs[i] == hs[r[0]]]
        if rest:
            assert all(used + 1 + ws[i] > W for i in rest)
