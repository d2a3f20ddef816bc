"""Pins of the fp64 CPU oracle to facts outside itself.

The pages print no worked LSTM example, so the oracle is pinned by:
  * closed forms of special cases (zero weights; one-step sequences);
  * a fixed point solved by a library root finder (peepholes on i and f);
  * torch.nn.LSTM, a library routine, for the peephole-free case (forward,
    final states and every gradient through autograd);
  * central finite differences of the loss for every parameter and input;
  * invariants: packed == padded-and-masked, permutation of sequences,
    direction symmetry, zero input weights give zero input gradient;
  * hand-counted zero-padding statistics.
Each targets a plausible slip: a wrong gate order, a transposed W or R, a
peephole reading c_t instead of c_{t-1} (or the reverse), a dropped carry
term, a wrong sign, an off-by-one in the reverse direction.
"""
import math

import numpy as np
import pytest

import oracle
from padding_free_variable_gb300 import synthetic


def sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def zero_layer(ndir, D, H):
    return {"W": np.zeros((ndir, 4 * H, D)), "R": np.zeros((ndir, 4 * H, H)),
            "b": np.zeros((ndir, 4 * H)), "peep": np.zeros((ndir, 3, H))}


def rand_layer(rng, ndir, D, H, a=0.5, peep=True):
    lay = {"W": rng.uniform(-a, a, (ndir, 4 * H, D)), "R": rng.uniform(-a, a, (ndir, 4 * H, H)),
           "b": rng.uniform(-a, a, (ndir, 4 * H)), "peep": rng.uniform(-a, a, (ndir, 3, H))}
    if not peep:
        lay["peep"][:] = 0.0
    return lay


def concat_offsets(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(int)


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("ndir", [1, 2])
def test_zero_weights_closed_form(ndir):
    """W = R = 0, p = 0: gates are sigmoid(b), c_t = i z (1 - f^t) / (1 - f)."""
    H, D = 5, 3
    lay = zero_layer(ndir, D, H)
    rng = np.random.default_rng(7)
    lay["b"][:] = rng.uniform(-2, 2, (ndir, 4 * H))
    lengths = np.array([6, 1, 3])
    x = rng.standard_normal((lengths.sum(), D))
    out = oracle.lstm_stack(lengths, x, [lay], ndir, H)
    st = concat_offsets(lengths)
    for d in range(ndir):
        b = lay["b"][d]
        i, f, z, o = sig(b[:H]), sig(b[H:2 * H]), np.tanh(b[2 * H:3 * H]), sig(b[3 * H:])
        for s, L in enumerate(lengths):
            for t in range(L):
                k = t + 1 if d == 0 else L - t       # steps taken when position t is emitted
                c = i * z * (1 - f ** k) / (1 - f)
                h = o * np.tanh(c)
                np.testing.assert_allclose(out["y"][st[s] + t, d * H:(d + 1) * H], h, rtol=1e-13, atol=1e-15)
            kk = L
            c = i * z * (1 - f ** kk) / (1 - f)
            np.testing.assert_allclose(out["c_n"][0, d, s], c, rtol=1e-13, atol=1e-15)


def test_half_gates_closed_form():
    """b_i = b_f = 0 (gates exactly 1/2): c_t = tanh(b_z) (1 - 0.5^t)."""
    H, D = 4, 2
    lay = zero_layer(1, D, H)
    bz = np.array([1.0, -0.5, 2.0, 0.25])
    lay["b"][0, 2 * H:3 * H] = bz
    lengths = np.array([8])
    out = oracle.lstm_stack(lengths, np.ones((8, D)), [lay], 1, H)
    for t in range(8):
        c = np.tanh(bz) * (1 - 0.5 ** (t + 1))
        np.testing.assert_allclose(out["y"][t], 0.5 * np.tanh(c), rtol=1e-14)


@pytest.mark.parametrize("ndir", [1, 2])
def test_length_one_closed_form_with_peepholes(ndir):
    """One frame from the zero state: c = sig(a_i) tanh(a_z) (i/f peepholes see c_0 = 0),
    h = sig(a_o + p_o c) tanh(c) (the output peephole sees the new state)."""
    rng = np.random.default_rng(11)
    H, D = 6, 4
    lay = rand_layer(rng, ndir, D, H, a=1.0)
    x = rng.standard_normal((1, D))
    out = oracle.lstm_stack(np.array([1]), x, [lay], ndir, H)
    for d in range(ndir):
        a = lay["W"][d] @ x[0] + lay["b"][d]
        c = sig(a[:H]) * np.tanh(a[2 * H:3 * H])
        h = sig(a[3 * H:] + lay["peep"][d, 2] * c) * np.tanh(c)
        np.testing.assert_allclose(out["y"][0, d * H:(d + 1) * H], h, rtol=1e-13)
        np.testing.assert_allclose(out["c_n"][0, d, 0], c, rtol=1e-13)


def test_fixed_point_with_peepholes():
    """W = R = 0, constant input: the cell state converges to the root of
    c = sig(b_f + p_f c) c + sig(b_i + p_i c) tanh(b_z), found by brentq;
    then h = sig(b_o + p_o c) tanh(c)."""
    brentq = pytest.importorskip("scipy.optimize").brentq
    H = 3
    lay = zero_layer(1, 2, H)
    b = lay["b"][0]
    b[:H] = [0.3, -0.7, 1.1]           # i
    b[H:2 * H] = [-1.0, -0.2, -2.0]    # f
    b[2 * H:3 * H] = [0.8, -1.5, 0.4]  # z
    b[3 * H:] = [0.1, 0.9, -0.6]       # o
    p = lay["peep"][0]
    p[0] = [0.4, -0.3, 0.2]            # p_i
    p[1] = [-0.5, 0.6, 0.25]           # p_f
    p[2] = [0.7, -0.8, 0.35]           # p_o
    L = 400
    out = oracle.lstm_stack(np.array([L]), np.zeros((L, 2)), [lay], 1, H)
    for u in range(H):
        g = lambda c: sig(b[H + u] + p[1, u] * c) * c + sig(b[u] + p[0, u] * c) * np.tanh(b[2 * H + u]) - c
        cstar = brentq(g, -10, 10, xtol=1e-15)
        hstar = sig(b[3 * H + u] + p[2, u] * cstar) * np.tanh(cstar)
        assert abs(out["c_n"][0, 0, 0, u] - cstar) < 1e-12
        assert abs(out["y"][L - 1, u] - hstar) < 1e-12


def test_fixed_point_distinguishes_peephole_sides():
    """Swapping p_i and p_f moves the fixed point: the pin above sees which is which."""
    brentq = pytest.importorskip("scipy.optimize").brentq
    bi, bf, bz, pi, pf = 0.3, -1.0, 0.8, 0.9, -0.9
    g1 = lambda c: sig(bf + pf * c) * c + sig(bi + pi * c) * np.tanh(bz) - c
    g2 = lambda c: sig(bf + pi * c) * c + sig(bi + pf * c) * np.tanh(bz) - c
    assert abs(brentq(g1, -10, 10) - brentq(g2, -10, 10)) > 1e-3


# --------------------------------------------------------------------------- torch.nn.LSTM

def torch_reference(lengths, x, layers, ndir, H, G):
    torch = pytest.importorskip("torch")
    from torch.nn.utils.rnn import pack_sequence, pad_packed_sequence
    D0 = x.shape[1]
    nl = len(layers)
    mod = torch.nn.LSTM(D0, H, num_layers=nl, bidirectional=(ndir == 2)).double()
    with torch.no_grad():
        for l, lay in enumerate(layers):
            for d in range(ndir):
                sfx = f"_l{l}" + ("_reverse" if d else "")
                getattr(mod, "weight_ih" + sfx).copy_(torch.from_numpy(lay["W"][d]))
                getattr(mod, "weight_hh" + sfx).copy_(torch.from_numpy(lay["R"][d]))
                getattr(mod, "bias_ih" + sfx).copy_(torch.from_numpy(lay["b"][d]))
                getattr(mod, "bias_hh" + sfx).zero_()
    st = concat_offsets(lengths)
    seqs = [torch.tensor(x[st[i]:st[i + 1]], dtype=torch.float64, requires_grad=True)
            for i in range(len(lengths))]
    packed = pack_sequence(seqs, enforce_sorted=False)
    y, (h_n, c_n) = mod(packed)
    ypad, _ = pad_packed_sequence(y, batch_first=True)
    ycat = torch.cat([ypad[i, :lengths[i]] for i in range(len(lengths))])
    loss = (ycat * torch.from_numpy(G)).sum()
    loss.backward()
    res = {"y": ycat.detach().numpy(),
           "h_n": h_n.detach().numpy().reshape(nl, ndir, len(lengths), H),
           "c_n": c_n.detach().numpy().reshape(nl, ndir, len(lengths), H),
           "dx": torch.cat([s.grad for s in seqs]).numpy(), "grads": []}
    for l in range(nl):
        g = {"W": [], "R": [], "b": []}
        for d in range(ndir):
            sfx = f"_l{l}" + ("_reverse" if d else "")
            g["W"].append(getattr(mod, "weight_ih" + sfx).grad.numpy())
            g["R"].append(getattr(mod, "weight_hh" + sfx).grad.numpy())
            g["b"].append(getattr(mod, "bias_ih" + sfx).grad.numpy())
        res["grads"].append({k: np.stack(v) for k, v in g.items()})
    return res


@pytest.mark.parametrize("ndir,nl", [(1, 1), (2, 1), (2, 2), (1, 3)])
def test_matches_torch_lstm_without_peepholes(ndir, nl):
    rng = np.random.default_rng(100 + 10 * ndir + nl)
    H, D0 = 5, 3
    lengths = np.array([4, 7, 1, 3, 7])
    layers = [rand_layer(rng, ndir, D0 if l == 0 else ndir * H, H, peep=False) for l in range(nl)]
    x = rng.standard_normal((lengths.sum(), D0))
    G = rng.standard_normal((lengths.sum(), ndir * H))
    ref = torch_reference(lengths, x, layers, ndir, H, G)
    out = oracle.lstm_stack(lengths, x, layers, ndir, H, G=G)
    for k in ("y", "h_n", "c_n", "dx"):
        np.testing.assert_allclose(out[k], ref[k], rtol=1e-11, atol=1e-13, err_msg=k)
    for l in range(nl):
        for k in ("W", "R", "b"):
            np.testing.assert_allclose(out["grads"][l][k], ref["grads"][l][k], rtol=1e-11, atol=1e-13,
                                       err_msg=f"layer {l} d{k}")


# --------------------------------------------------------------------------- finite differences

def loss_of(lengths, x, layers, ndir, H, G):
    y = oracle.lstm_stack(lengths, x, layers, ndir, H)["y"]
    return float((y * G).sum())


@pytest.mark.parametrize("ndir,nl", [(1, 1), (2, 1), (2, 2)])
def test_gradients_match_central_differences(ndir, nl):
    rng = np.random.default_rng(200 + 10 * ndir + nl)
    H, D0 = 4, 3
    lengths = np.array([1, 2, 5])
    layers = [rand_layer(rng, ndir, D0 if l == 0 else ndir * H, H, a=0.6) for l in range(nl)]
    x = rng.standard_normal((lengths.sum(), D0))
    G = rng.standard_normal((lengths.sum(), ndir * H))
    out = oracle.lstm_stack(lengths, x, layers, ndir, H, G=G)
    eps = 1e-6

    def check(arr, grad, name):
        flat = arr.reshape(-1)
        gflat = grad.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            lp = loss_of(lengths, x, layers, ndir, H, G)
            flat[i] = keep - eps
            lm = loss_of(lengths, x, layers, ndir, H, G)
            flat[i] = keep
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - gflat[i]) <= 1e-7 * max(1.0, abs(fd)), (name, i, fd, gflat[i])

    check(x, out["dx"], "x")
    for l in range(nl):
        for k in ("W", "R", "b", "peep"):
            check(layers[l][k], out["grads"][l][k], f"layer{l}.{k}")


def test_zero_input_weights_give_zero_input_gradient():
    rng = np.random.default_rng(5)
    lay = rand_layer(rng, 2, 3, 4)
    lay["W"][:] = 0.0
    lengths = np.array([3, 2])
    G = rng.standard_normal((5, 8))
    out = oracle.lstm_stack(lengths, rng.standard_normal((5, 3)), [lay], 2, 4, G=G)
    assert np.all(out["dx"] == 0.0)
    assert np.any(out["grads"][0]["W"] != 0.0)


# --------------------------------------------------------------------------- invariants

def to_padded(lengths, x):
    T, B = int(max(lengths)), len(lengths)
    st = concat_offsets(lengths)
    pad = np.zeros((T, B, x.shape[1]))
    mask = np.zeros((T, B), np.uint8)
    for b, L in enumerate(lengths):
        pad[:L, b] = x[st[b]:st[b + 1]]
        mask[:L, b] = 1
    return pad, mask


@pytest.mark.parametrize("ndir", [1, 2])
def test_padded_masked_equals_per_sequence(ndir):
    """Invariant: a masked, zero-padded batch gives the per-sequence results."""
    rng = np.random.default_rng(300 + ndir)
    H, D = 5, 4
    lengths = np.array([6, 0, 2, 9, 1, 6])
    lay = rand_layer(rng, ndir, D, H)
    N = lengths.sum()
    x = rng.standard_normal((N, D))
    G = rng.standard_normal((N, ndir * H))
    ref = oracle.lstm_stack(lengths, x, [lay], ndir, H, G=G)
    xp, mask = to_padded(lengths, x)
    Gp, _ = to_padded(lengths, G)
    Gp[mask == 0] = rng.standard_normal(((mask == 0).sum(), ndir * H))   # must be ignored
    out = oracle.lstm_padded_layer(xp, mask, lay, ndir, H, dy_pad=Gp)
    st = concat_offsets(lengths)
    for b, L in enumerate(lengths):
        np.testing.assert_allclose(out["y"][:L, b], ref["y"][st[b]:st[b + 1]], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out["dx"][:L, b], ref["dx"][st[b]:st[b + 1]], rtol=1e-12, atol=1e-14)
        assert np.all(out["y"][L:, b] == 0.0)
    np.testing.assert_allclose(out["h_n"], ref["h_n"][0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out["c_n"], ref["c_n"][0], rtol=1e-12, atol=1e-14)
    for k in ("W", "R", "b", "peep"):
        np.testing.assert_allclose(out["grads"][k], ref["grads"][0][k], rtol=1e-11, atol=1e-13, err_msg=k)


def test_permuting_sequences_permutes_results():
    rng = np.random.default_rng(41)
    H, D = 4, 3
    lengths = np.array([3, 5, 1, 4])
    lay = rand_layer(rng, 2, D, H)
    st = concat_offsets(lengths)
    x = rng.standard_normal((lengths.sum(), D))
    G = rng.standard_normal((lengths.sum(), 2 * H))
    ref = oracle.lstm_stack(lengths, x, [lay], 2, H, G=G)
    perm = np.array([2, 0, 3, 1])
    xs = np.concatenate([x[st[i]:st[i + 1]] for i in perm])
    Gs = np.concatenate([G[st[i]:st[i + 1]] for i in perm])
    out = oracle.lstm_stack(lengths[perm], xs, [lay], 2, H, G=Gs)
    yref = np.concatenate([ref["y"][st[i]:st[i + 1]] for i in perm])
    dxref = np.concatenate([ref["dx"][st[i]:st[i + 1]] for i in perm])
    np.testing.assert_allclose(out["y"], yref, rtol=1e-14)
    np.testing.assert_allclose(out["dx"], dxref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out["h_n"], ref["h_n"][:, :, perm], rtol=1e-14)
    for k in ("W", "R", "b", "peep"):
        np.testing.assert_allclose(out["grads"][0][k], ref["grads"][0][k], rtol=1e-12, atol=1e-14)


def test_backward_direction_is_forward_on_reversed_sequences():
    """With equal parameters in both directions, the reverse direction on x equals the
    forward direction on each sequence reversed, read back in reverse."""
    rng = np.random.default_rng(17)
    H, D = 4, 3
    one = rand_layer(rng, 1, D, H)
    both = {k: np.concatenate([v, v]) for k, v in one.items()}
    lengths = np.array([5, 2, 7])
    st = concat_offsets(lengths)
    x = rng.standard_normal((lengths.sum(), D))
    G = rng.standard_normal((lengths.sum(), H))
    bi = oracle.lstm_stack(lengths, x, [both], 2, H, G=np.concatenate([np.zeros_like(G), G], 1))
    xr = np.concatenate([x[st[i]:st[i + 1]][::-1] for i in range(3)])
    Gr = np.concatenate([G[st[i]:st[i + 1]][::-1] for i in range(3)])
    uni = oracle.lstm_stack(lengths, xr, [one], 1, H, G=Gr)
    for i in range(3):
        np.testing.assert_allclose(bi["y"][st[i]:st[i + 1], H:], uni["y"][st[i]:st[i + 1]][::-1], rtol=1e-13)
        np.testing.assert_allclose(bi["dx"][st[i]:st[i + 1]], uni["dx"][st[i]:st[i + 1]][::-1],
                                   rtol=1e-12, atol=1e-14)
    for k in ("W", "R", "b", "peep"):
        np.testing.assert_allclose(bi["grads"][0][k][1], uni["grads"][0][k][0], rtol=1e-12, atol=1e-14)
        assert np.all(bi["grads"][0][k][0] == 0.0)      # zero upstream error into the forward half


def test_threads_do_not_change_results():
    w = synthetic.custom(2, 2, 6, 5, [9, 3, 0, 7, 7, 1], seed=3)
    a = oracle.lstm_stack(w.lengths, w.x, w.layers, 2, 5, G=w.G, nthreads=1)
    b = oracle.lstm_stack(w.lengths, w.x, w.layers, 2, 5, G=w.G, nthreads=4)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["dx"], b["dx"])
    for l in range(2):
        for k in ("W", "R", "b", "peep"):
            np.testing.assert_allclose(a["grads"][l][k], b["grads"][l][k], rtol=1e-13, atol=1e-15)


def test_empty_sequences_have_zero_final_state():
    w = synthetic.custom(2, 1, 3, 4, [0, 3, 0], seed=9)
    out = oracle.lstm_stack(w.lengths, w.x, w.layers, 2, 4, G=w.G)
    assert np.all(out["h_n"][:, :, [0, 2]] == 0.0)
    assert np.all(out["c_n"][:, :, [0, 2]] == 0.0)
    assert np.any(out["h_n"][:, :, 1] != 0.0)


# --------------------------------------------------------------------------- padding statistics

def test_zero_padding_rate_hand_counted():
    # one batch [3, 5, 2]: pads 2 + 0 + 3 = 5 frames over 10 real ones
    assert oracle.zero_padding_rate([[3, 5, 2]]) == pytest.approx(0.5)
    assert oracle.waste_fraction([[3, 5, 2]]) == pytest.approx(5 / 15)
    # two batches [4, 4] and [1, 3]: pads 0 + 2 over 12
    assert oracle.zero_padding_rate([[4, 4], [1, 3]]) == pytest.approx(2 / 12)
    # sorted, equal lengths: nothing padded
    assert oracle.zero_padding_rate([[7, 7, 7]]) == 0.0


def test_bucket_batches_cover_each_sequence_once():
    lengths = np.array([100, 199, 200, 555, 1000, 901, 899])
    buckets = oracle.bucket_batches(lengths, 100, 100)
    got = sorted(int(i) for b in buckets for i in b)
    assert got == list(range(len(lengths)))
    for b in buckets:
        lens = lengths[b]
        assert lens.max() - lens.min() <= 100
    # [100,200) holds 100 and 199; the top bucket [900, 1000] holds 901 and 1000
    assert [list(b) for b in buckets][0] == [0, 1]
    assert list(buckets[-1]) == [4, 5]


def test_bf16_rounding_of_generator_is_representable():
    w = synthetic.workload(3, batch=2)
    for arr in (w.x, w.layers[0]["W"], w.layers[0]["R"]):
        bits = np.ascontiguousarray(arr, np.float32).view(np.uint32)
        assert np.all((bits & 0xFFFF) == 0)
    # ties go to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert synthetic.round_bf16(np.array([1 + 2 ** -8], np.float32))[0] == 1.0
    assert synthetic.round_bf16(np.array([1 + 3 * 2 ** -8], np.float32))[0] == 1 + 2 ** -6
    assert math.isclose(float(synthetic.round_bf16(np.array([0.1], np.float32))[0]), 0.10009765625)


# --------------------------------------------------------------------------- bf16-product rounding

def _nearest_bf16_by_definition(v: float) -> float:
    """The bfloat16 nearest to fp32(v), ties to the neighbour with an even last mantissa bit,
    found by comparing distances to the two bf16 neighbours that bracket it (exact in fp64)."""
    f = np.float32(v)
    if not np.isfinite(f):
        return float(f)
    bits = int(np.array([f], np.float32).view(np.uint32)[0])
    lo_bits = bits & 0xFFFF0000                     # bf16 neighbour toward zero (same sign)
    hi_bits = lo_bits + 0x10000                     # next bf16 away from zero
    lo = float(np.array([lo_bits], np.uint32).view(np.float32)[0])
    hi = float(np.array([hi_bits & 0xFFFFFFFF], np.uint32).view(np.float32)[0])
    dlo, dhi = abs(float(f) - lo), abs(hi - float(f))
    if dlo < dhi:
        return lo
    if dhi < dlo:
        return hi
    return lo if ((lo_bits >> 16) & 1) == 0 else hi


def test_oracle_bf16_rounding_nearest_ties_to_even():
    """The oracle's bf16-product mode rounds like the kernels' cvt.rn.bf16: fp32 first, then the
    nearest bf16 with ties to even; Inf and NaN pass through."""
    one = 1.0
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (even: 1); 1 + 3*2^-8 halfway
    # between 1 + 2^-7 and 1 + 2^-6 (even: 1 + 2^-6); the same below zero
    assert oracle.round_bf16(one + 2.0 ** -8) == one
    assert oracle.round_bf16(one + 3 * 2.0 ** -8) == one + 2.0 ** -6
    assert oracle.round_bf16(-(one + 2.0 ** -8)) == -one
    assert oracle.round_bf16(one + 2.0 ** -8 + 2.0 ** -20) == one + 2.0 ** -7    # just past the tie
    assert oracle.round_bf16(0.0) == 0.0 and math.copysign(1.0, oracle.round_bf16(-0.0)) == -1.0
    assert oracle.round_bf16(float("inf")) == float("inf")
    assert oracle.round_bf16(float("-inf")) == float("-inf")
    assert math.isnan(oracle.round_bf16(float("nan")))
    rng = np.random.default_rng(2024)
    vals = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                           rng.uniform(-1, 1, 2000)])
    for v in vals:
        r = oracle.round_bf16(float(v))
        assert r == _nearest_bf16_by_definition(float(v)), v
        assert r == float(synthetic.round_bf16(np.array([v]))[0]), v


# --------------------------------------------------------------------------- initial states

def _state_inputs(rng, nl, ndir, B, H, scale=0.5):
    return [rng.uniform(-scale, scale, (nl, ndir, B, H)) for _ in range(4)]     # h0, c0, dh_n, dc_n


@pytest.mark.parametrize("ndir,nl", [(1, 1), (2, 1), (2, 2)])
def test_initial_states_match_torch_lstm(ndir, nl):
    """torch.nn.LSTM given (h0, c0), no peepholes, the loss reading y, h_n and c_n: outputs,
    final states and the gradients of x, every weight, h0 and c0 through autograd."""
    torch = pytest.importorskip("torch")
    from torch.nn.utils.rnn import pack_sequence, pad_packed_sequence
    rng = np.random.default_rng(300 + 10 * ndir + nl)
    H, D0 = 5, 3
    lengths = np.array([4, 7, 1, 3, 7])
    B = len(lengths)
    layers = [rand_layer(rng, ndir, D0 if l == 0 else ndir * H, H, peep=False) for l in range(nl)]
    x = rng.standard_normal((lengths.sum(), D0))
    G = rng.standard_normal((lengths.sum(), ndir * H))
    h0, c0, Gh, Gc = _state_inputs(rng, nl, ndir, B, H)
    out = oracle.lstm_stack(lengths, x, layers, ndir, H, G=G, h0=h0, c0=c0, dh_n=Gh, dc_n=Gc)

    mod = torch.nn.LSTM(D0, H, num_layers=nl, bidirectional=(ndir == 2)).double()
    with torch.no_grad():
        for l, lay in enumerate(layers):
            for d in range(ndir):
                sfx = f"_l{l}" + ("_reverse" if d else "")
                getattr(mod, "weight_ih" + sfx).copy_(torch.from_numpy(lay["W"][d]))
                getattr(mod, "weight_hh" + sfx).copy_(torch.from_numpy(lay["R"][d]))
                getattr(mod, "bias_ih" + sfx).copy_(torch.from_numpy(lay["b"][d]))
                getattr(mod, "bias_hh" + sfx).zero_()
    st = concat_offsets(lengths)
    seqs = [torch.tensor(x[st[i]:st[i + 1]], dtype=torch.float64, requires_grad=True) for i in range(B)]
    th0 = torch.tensor(h0.reshape(nl * ndir, B, H), requires_grad=True)
    tc0 = torch.tensor(c0.reshape(nl * ndir, B, H), requires_grad=True)
    y, (h_n, c_n) = mod(pack_sequence(seqs, enforce_sorted=False), (th0, tc0))
    ypad, _ = pad_packed_sequence(y, batch_first=True)
    ycat = torch.cat([ypad[i, :lengths[i]] for i in range(B)])
    loss = (ycat * torch.from_numpy(G)).sum() + (h_n * torch.from_numpy(Gh.reshape(nl * ndir, B, H))).sum() \
        + (c_n * torch.from_numpy(Gc.reshape(nl * ndir, B, H))).sum()
    loss.backward()
    tol = dict(rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(out["y"], ycat.detach().numpy(), **tol)
    np.testing.assert_allclose(out["h_n"], h_n.detach().numpy().reshape(nl, ndir, B, H), **tol)
    np.testing.assert_allclose(out["c_n"], c_n.detach().numpy().reshape(nl, ndir, B, H), **tol)
    np.testing.assert_allclose(out["dx"], torch.cat([s.grad for s in seqs]).numpy(), **tol)
    np.testing.assert_allclose(out["dh0"], th0.grad.numpy().reshape(nl, ndir, B, H), **tol)
    np.testing.assert_allclose(out["dc0"], tc0.grad.numpy().reshape(nl, ndir, B, H), **tol)
    for l in range(nl):
        for k, tk in (("W", "weight_ih"), ("R", "weight_hh"), ("b", "bias_ih")):
            ref = np.stack([getattr(mod, f"{tk}_l{l}" + ("_reverse" if d else "")).grad.numpy()
                            for d in range(ndir)])
            np.testing.assert_allclose(out["grads"][l][k], ref, err_msg=f"layer {l} d{k}", **tol)


@pytest.mark.parametrize("ndir,nl", [(1, 1), (2, 2)])
def test_initial_state_gradients_match_central_differences(ndir, nl):
    """With peepholes (which read c0 at the first step): dh0, dc0 and every parameter
    gradient against central differences of L = <y, G> + <h_n, Gh> + <c_n, Gc>."""
    rng = np.random.default_rng(400 + 10 * ndir + nl)
    H, D0 = 4, 3
    lengths = np.array([1, 2, 5, 0])
    B = len(lengths)
    layers = [rand_layer(rng, ndir, D0 if l == 0 else ndir * H, H, a=0.6) for l in range(nl)]
    x = rng.standard_normal((lengths.sum(), D0))
    G = rng.standard_normal((lengths.sum(), ndir * H))
    h0, c0, Gh, Gc = _state_inputs(rng, nl, ndir, B, H, scale=0.8)
    out = oracle.lstm_stack(lengths, x, layers, ndir, H, G=G, h0=h0, c0=c0, dh_n=Gh, dc_n=Gc)

    def loss():
        r = oracle.lstm_stack(lengths, x, layers, ndir, H, h0=h0, c0=c0)
        return float((r["y"] * G).sum() + (r["h_n"] * Gh).sum() + (r["c_n"] * Gc).sum())

    eps = 1e-6

    def check(arr, grad, name):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            lp = loss()
            flat[i] = keep - eps
            lm = loss()
            flat[i] = keep
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - gflat[i]) <= 1e-7 * max(1.0, abs(fd)), (name, i, fd, gflat[i])

    check(h0, out["dh0"], "h0")
    check(c0, out["dc0"], "c0")
    check(x, out["dx"], "x")
    for l in range(nl):
        for k in ("W", "R", "b", "peep"):
            check(layers[l][k], out["grads"][l][k], f"layer{l}.{k}")
    # an empty sequence consumes nothing: its final state is its initial state
    np.testing.assert_array_equal(out["h_n"][:, :, 3], h0[:, :, 3])
    np.testing.assert_array_equal(out["dc0"][:, :, 3], Gc[:, :, 3])


def test_passing_the_final_state_on_equals_one_longer_sequence():
    """RETURNN paper, Sec. 3.2 (one RNN's final state as another's initial state): running
    frames [0, L1) and then [L1, L) from the first part's final state gives the outputs and
    final state of running all L frames at once (forward direction)."""
    rng = np.random.default_rng(17)
    H, D = 6, 4
    lay = rand_layer(rng, 1, D, H)
    x = rng.standard_normal((11, D))
    whole = oracle.lstm_stack(np.array([11]), x, [lay], 1, H)
    a = oracle.lstm_stack(np.array([4]), x[:4], [lay], 1, H)
    b = oracle.lstm_stack(np.array([7]), x[4:], [lay], 1, H, h0=a["h_n"], c0=a["c_n"])
    np.testing.assert_allclose(np.concatenate([a["y"], b["y"]]), whole["y"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(b["h_n"], whole["h_n"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(b["c_n"], whole["c_n"], rtol=1e-14, atol=1e-15)
