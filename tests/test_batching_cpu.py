"""Host-side batch formation and segment lists (no GPU): the frame-budget batch former
("On batching variable size inputs...", Sec. 2, dynamic batch size) and RETURNN-style
chunking into segments (RETURNN paper, Sec. 4), through the C ABI's host-only calls,
against hand-counted cases and brute-force restatements."""
import numpy as np
import pytest

from padding_free_variable_gb300 import _lib, ops


def _greedy(lengths, budget, padded):
    """The dynamic batch size written out plainly: walk the sequences in order and open a new
    batch whenever adding the next one would exceed the budget."""
    out, cur = [], []
    b = 0
    for L in lengths:
        trial = cur + [L]
        size = len(trial) * max(trial) if padded else sum(trial)
        if cur and size > budget:
            b += 1
            cur = [L]
        else:
            cur = trial
        out.append(b)
    return out


def test_form_batches_hand_counted():
    # packed budget 10: [3, 4] (7), [5, 2] (7; +6 would be 13), [6, 4] (10), [11] (alone over budget), [1]
    lengths = [3, 4, 5, 2, 6, 4, 11, 1]
    assert list(ops.form_batches(lengths, 10)) == [0, 0, 1, 1, 2, 2, 3, 4]
    # padded budget 10: [3] (+4 -> 2x4 = 8 ok), [3, 4] then 5 -> 3x5 = 15: new; [5] + 2 -> 2x5 = 10 ok;
    # [5, 2] + 6 -> 3x6: new; [6] + 4 -> 2x6 = 12: new; [4] + 11: new; [11]; [11] + 1 -> 22: new
    assert list(ops.form_batches(lengths, 10, padded_budget=True)) == [0, 0, 1, 1, 2, 3, 4, 5]


@pytest.mark.parametrize("padded", [False, True])
def test_form_batches_matches_greedy_and_budget(padded):
    rng = np.random.default_rng(42 + padded)
    lengths = rng.integers(0, 60, 300)
    budget = 200
    got = ops.form_batches(lengths, budget, padded_budget=padded)
    assert list(got) == _greedy(list(lengths), budget, padded)
    # batches are contiguous runs; each fits the budget unless it holds one sequence; no batch could
    # have taken the next batch's first sequence
    assert np.all(np.diff(got) >= 0) and np.all(np.diff(got) <= 1)
    for b in range(got.max() + 1):
        L = lengths[got == b]
        size = len(L) * L.max() if padded else L.sum()
        assert size <= budget or len(L) == 1
        nxt = np.flatnonzero(got == b + 1)
        if nxt.size:
            L2 = np.append(L, lengths[nxt[0]])
            assert (len(L2) * L2.max() if padded else L2.sum()) > budget


def test_form_batches_rejects_bad_arguments():
    lib = _lib.load()
    import ctypes
    lens = np.array([3, -1], np.int32)
    out = np.zeros(2, np.int32)
    nb = ctypes.c_int32()
    P = ctypes.POINTER(ctypes.c_int32)
    assert lib.lstm_form_batches(lens.ctypes.data_as(P), 2, 10, 0, out.ctypes.data_as(P),
                                 ctypes.byref(nb)) == _lib.LSTM_ERR_INVALID_ARG
    assert lib.lstm_form_batches(lens.ctypes.data_as(P), 1, 0, 0, out.ctypes.data_as(P),
                                 ctypes.byref(nb)) == _lib.LSTM_ERR_INVALID_ARG
    assert lib.lstm_form_batches(None, 0, 10, 0, None, ctypes.byref(nb)) == _lib.LSTM_OK and nb.value == 0


def test_segments_hand_counted():
    # L = 10, chunk 4, step 4: [0,4) [4,8) [8,10); L = 0: one empty segment; L = 4: one segment
    seq, start, length = ops.segments_host([10, 0, 4], 4, 4)
    assert list(seq) == [0, 0, 0, 1, 2]
    assert list(start) == [0, 4, 8, 0, 0]
    assert list(length) == [4, 4, 2, 0, 4]
    # overlapping: L = 10, chunk 6, step 4: [0,6) [4,10) and stop (the end is reached)
    seq, start, length = ops.segments_host([10], 6, 4)
    assert list(start) == [0, 4] and list(length) == [6, 6]


@pytest.mark.parametrize("chunk,step", [(5, 5), (7, 3), (1, 1), (50, 50)])
def test_segments_cover_every_frame(chunk, step):
    rng = np.random.default_rng(chunk * 10 + step)
    lengths = rng.integers(0, 40, 25)
    seq, start, length = ops.segments_host(lengths, chunk, step)
    for b, L in enumerate(lengths):
        mine = np.flatnonzero(seq == b)
        assert mine.size >= 1
        assert np.all(start[mine] == step * np.arange(mine.size))
        assert np.all(length[mine] == np.minimum(chunk, L - start[mine]).clip(min=0))
        covered = np.zeros(L, bool)
        for u in mine:
            covered[start[u]:start[u] + length[u]] = True
        assert covered.all()
        assert start[mine[-1]] + length[mine[-1]] == L     # the last reaches the end
        assert mine.size == 1 or start[mine[-2]] + length[mine[-2]] < L   # and no earlier one does


def test_segments_reject_bad_arguments():
    with pytest.raises(_lib.LSTMError):
        ops.segments_host([5], 4, 5)          # step > chunk
    with pytest.raises(_lib.LSTMError):
        ops.segments_host([5], 0, 0)
