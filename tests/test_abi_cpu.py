"""CPU-only checks of the C ABI: it builds, loads without a GPU, exports every
declared symbol, rejects bad arguments before touching the device, and its
host-side packing tables match a brute-force construction."""
import ctypes
import os
import re

import numpy as np
import pytest

from padding_free_variable_gb300 import _lib, build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return _lib.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "lstm_packed.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lstm_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(_lib.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.lstm_status_string(code)
    assert b"unknown" in lib.lstm_status_string(99)


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def test_rejects_bad_arguments_without_a_device(lib):
    h = ctypes.c_void_p()
    assert lib.lstm_plan_create(_ip(np.array([3, -1], np.int32)), 2, ctypes.byref(h)) == _lib.LSTM_ERR_INVALID_ARG
    assert lib.lstm_plan_create(_ip(np.array([3], np.int32)), 0, ctypes.byref(h)) == _lib.LSTM_ERR_INVALID_ARG
    assert lib.lstm_plan_create(None, 2, ctypes.byref(h)) == _lib.LSTM_ERR_INVALID_ARG
    shape = _lib.LayerShape(40, 256, 2, 0)
    assert lib.lstm_fwd(None, ctypes.byref(shape), None, None, None, None, None, None, None, None) == \
        _lib.LSTM_ERR_INVALID_ARG
    assert lib.lstm_workspace_bytes(None, ctypes.byref(shape)) == 0
    assert lib.lstm_plan_destroy(None) == _lib.LSTM_OK
    assert lib.lstm_status_poll(None, None) == _lib.LSTM_ERR_INVALID_ARG


def host_tables(lib, lengths, padded=False):
    lengths = np.asarray(lengths, np.int32)
    T, rows = ctypes.c_int32(), ctypes.c_int64()
    assert lib.lstm_plan_dims(_ip(lengths), len(lengths), int(padded), ctypes.byref(T), ctypes.byref(rows)) == 0
    T, rows, B = T.value, rows.value, len(lengths)
    out = {k: np.full(n, -7, np.int32) for k, n in
           (("bs", T), ("off", T + 1), ("perm", B), ("len", B), ("row_src", rows), ("prev_fwd", rows),
            ("prev_rev", rows))}
    assert lib.lstm_plan_compute_host(_ip(lengths), B, int(padded), *[_ip(out[k]) for k in
                                      ("bs", "off", "perm", "len", "row_src", "prev_fwd", "prev_rev")]) == 0
    return T, rows, out


def brute_force(lengths):
    """Packed layout written out the long way: step t holds, in order, every
    sequence longer than t, longest first, ties in caller order."""
    B = len(lengths)
    order = sorted(range(B), key=lambda b: (-lengths[b], b))
    start = np.concatenate([[0], np.cumsum(lengths)])
    rows = []
    for t in range(max(lengths) if B else 0):
        for j, b in enumerate(order):
            if lengths[b] > t:
                rows.append((t, j, b, start[b] + t))
    return order, rows


@pytest.mark.parametrize("lengths", [[3, 1, 4, 0, 2], [5], [0, 0, 2], [7, 7, 7, 1], [2, 9, 2, 9, 5, 1]])
def test_host_tables_match_brute_force(lib, lengths):
    T, rows, tab = host_tables(lib, lengths)
    order, brute = brute_force(lengths)
    assert T == max(lengths) and rows == sum(lengths)
    assert list(tab["perm"]) == order
    assert list(tab["len"]) == [lengths[b] for b in order]
    where = {}
    for r, (t, j, b, src) in enumerate(brute):
        assert tab["row_src"][r] == src
        assert tab["off"][t] + j == r
        where[(t, j)] = r
    for t in range(T):
        assert tab["bs"][t] == sum(1 for L in lengths if L > t)
    for (t, j), r in where.items():
        assert tab["prev_fwd"][r] == where.get((t - 1, j), -1)
        assert tab["prev_rev"][r] == where.get((t + 1, j), -1)


def test_hand_worked_fixture(lib):
    """tests/golden/pack_plan_example.txt: a layout worked out by hand."""
    path = os.path.join(ROOT, "tests", "golden", "pack_plan_example.txt")
    fields = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=")
            fields[k.strip()] = [int(x) for x in v.split()]
    T, rows, tab = host_tables(lib, fields["lengths"])
    for k in ("bs", "off", "perm", "row_src", "prev_fwd", "prev_rev"):
        assert list(tab[k]) == fields[k], k


def test_padded_tables(lib):
    lengths = [2, 0, 3]
    T, rows, tab = host_tables(lib, lengths, padded=True)
    assert T == 3 and rows == 9
    assert list(tab["bs"]) == [3, 3, 3]
    assert list(tab["perm"]) == [0, 1, 2]
    # rows (t, b) = t*3 + b; source frames 0,1 | none | 2,3,4
    assert list(tab["row_src"]) == [0, -1, 2, 1, -1, 3, -1, -1, 4]
    assert list(tab["prev_fwd"]) == [-1, -1, -1, 0, 1, 2, 3, 4, 5]
    assert list(tab["prev_rev"]) == [3, 4, 5, 6, 7, 8, -1, -1, -1]


def test_tie_break_is_stable(lib):
    _, _, tab = host_tables(lib, [4, 6, 4, 6, 4])
    assert list(tab["perm"]) == [1, 3, 0, 2, 4]
