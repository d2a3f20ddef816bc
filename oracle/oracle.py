"""ctypes binding of ``lstm_oracle.c`` (test infrastructure only).

Every array crosses as float64.  For the bf16 workloads the caller passes the
bf16-rounded x, W and R values (the generator already rounds them), so the
oracle computes the exact fp64 result of the same rounded operands.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lstm_oracle.c")
_SRCS = (_SRC, os.path.join(_HERE, "mdlstm_oracle.c"))
_LIB = os.path.join(_HERE, "liblstm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, OpenMP over sequences, no fast-math)."""
    if force or not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-o", tmp, *_SRCS, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_lstm_stack.restype = ctypes.c_int
            lib.oracle_lstm_stack.argtypes = [
                ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, dp, ctypes.POINTER(dp), dp, dp, dp, dp, dp, ctypes.POINTER(dp),
                ctypes.c_int]
            lib.oracle_lstm_stack_state.restype = ctypes.c_int
            lib.oracle_lstm_stack_state.argtypes = [
                ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, dp, ctypes.POINTER(dp), dp, dp, dp, dp, dp, dp, dp, dp, dp,
                ctypes.POINTER(dp), dp, dp, ctypes.c_int]
            lib.oracle_lstm_padded_layer.restype = ctypes.c_int
            lib.oracle_lstm_padded_layer.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp,
                ctypes.POINTER(ctypes.c_ubyte), dp, dp, dp, dp, dp, dp, dp]
            lib.oracle_set_bf16_products.restype = None
            lib.oracle_set_bf16_products.argtypes = [ctypes.c_int]
            lib.oracle_round_bf16.restype = ctypes.c_double
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_layer_param_count.restype = ctypes.c_long
            lib.oracle_layer_param_count.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
            ip = ctypes.POINTER(ctypes.c_int)
            lib.oracle_md_param_count.restype = ctypes.c_long
            lib.oracle_md_param_count.argtypes = [ctypes.c_int, ctypes.c_int]
            lib.oracle_md_layer.restype = ctypes.c_int
            lib.oracle_md_layer.argtypes = [ctypes.c_int, ip, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            dp, dp, dp, dp, dp, dp]
            lib.oracle_md_forward.restype = None
            lib.oracle_md_forward.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, dp, dp, dp, dp, dp]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def pack_layer_params(layer: dict) -> np.ndarray:
    """Flat fp64 block W, R, b, peep (the layout ``lstm_oracle.c`` reads)."""
    return np.concatenate([_f64(layer[k]).ravel() for k in ("W", "R", "b", "peep")])


def unpack_layer_grads(flat: np.ndarray, ndir: int, D: int, H: int) -> dict:
    out, o = {}, 0
    for k, shape in (("W", (ndir, 4 * H, D)), ("R", (ndir, 4 * H, H)), ("b", (ndir, 4 * H)),
                     ("peep", (ndir, 3, H))):
        n = int(np.prod(shape))
        out[k] = flat[o:o + n].reshape(shape)
        o += n
    assert o == flat.size
    return out


def lstm_stack(lengths, x, layers, num_directions: int, hidden_size: int, G=None,
               nthreads: int = 1, bf16_products: bool = False, h0=None, c0=None, dh_n=None,
               dc_n=None) -> dict:
    """Forward (and, if ``G`` is given, BPTT) of a layer stack, each sequence on its own.

    lengths[B]; x[N, D0] in caller order; layers: list of dicts W, R, b, peep;
    G[N, ndir*H] = dL/dy of the top layer.  Returns y, h_n, c_n [layers, ndir, B, H]
    and, with G, dx and grads (list of dicts).

    h0, c0 [layers, ndir, B, H]: initial states (None = zero); dh_n, dc_n: dL/d of
    the final states from outside the stack (None = zero).  With G, the result also
    holds dh0 and dc0 [layers, ndir, B, H].

    bf16_products=True is a diagnostic (not the parity reference): h and the
    gate errors are rounded to bf16 before each product.
    """
    lib = _load()
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    B = int(lengths.size)
    N = int(lengths.sum())
    nd, H = int(num_directions), int(hidden_size)
    x = _f64(x).reshape(N, -1)
    D0 = x.shape[1]
    nl = len(layers)
    params = [pack_layer_params(layer) for layer in layers]
    for i, p in enumerate(params):
        D = D0 if i == 0 else nd * H
        assert p.size == lib.oracle_layer_param_count(nd, D, H), "layer shape mismatch"
    dp = ctypes.POINTER(ctypes.c_double)
    parr = (dp * nl)(*[_ptr(p) for p in params])
    y = np.zeros((N, nd * H))
    h_n = np.zeros((nl, nd, B, H))
    c_n = np.zeros((nl, nd, B, H))
    out = {"y": y, "h_n": h_n, "c_n": c_n}
    dy = dx = None
    garr = None
    grads = None
    if G is not None:
        dy = _f64(G).reshape(N, nd * H)
        dx = np.zeros((N, D0))
        grads = [np.zeros_like(p) for p in params]
        garr = (dp * nl)(*[_ptr(g) for g in grads])
    st_shape = (nl, nd, B, H)
    states = [None if a is None else _f64(a).reshape(st_shape) for a in (h0, c0, dh_n, dc_n)]
    dh0 = np.zeros(st_shape) if G is not None else None
    dc0 = np.zeros(st_shape) if G is not None else None
    lib.oracle_set_bf16_products(1 if bf16_products else 0)
    rc = lib.oracle_lstm_stack_state(B, lengths.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), nl, nd, H, D0,
                                     _ptr(x), parr, _ptr(dy), *[_ptr(a) for a in states], _ptr(y), _ptr(h_n),
                                     _ptr(c_n), _ptr(dx), garr, _ptr(dh0), _ptr(dc0), int(nthreads))
    lib.oracle_set_bf16_products(0)
    if rc != 0:
        raise ValueError("oracle_lstm_stack rejected its arguments")
    if G is not None:
        out["dx"] = dx
        out["grads"] = [unpack_layer_grads(g, nd, D0 if i == 0 else nd * H, H)
                        for i, g in enumerate(grads)]
        out["dh0"] = dh0
        out["dc0"] = dc0
    return out


def round_bf16(v: float) -> float:
    """The bf16-product mode's rounding of one value (fp32, then nearest bf16, ties to even)."""
    return float(_load().oracle_round_bf16(float(v)))


def lstm_padded_layer(x_pad, mask, layer: dict, num_directions: int, hidden_size: int,
                      dy_pad=None) -> dict:
    """One layer over a right-padded time-major batch x_pad[T, B, D] with mask[T, B]."""
    lib = _load()
    x_pad = _f64(x_pad)
    T, B, D = x_pad.shape
    nd, H = int(num_directions), int(hidden_size)
    mask = np.ascontiguousarray(mask, dtype=np.uint8)
    assert mask.shape == (T, B)
    params = pack_layer_params(layer)
    assert params.size == lib.oracle_layer_param_count(nd, D, H)
    y = np.zeros((T, B, nd * H))
    h_n = np.zeros((nd, B, H))
    c_n = np.zeros((nd, B, H))
    out = {"y": y, "h_n": h_n, "c_n": c_n}
    dy = dx = grads = None
    if dy_pad is not None:
        dy = _f64(dy_pad).reshape(T, B, nd * H)
        dx = np.zeros((T, B, D))
        grads = np.zeros_like(params)
    rc = lib.oracle_lstm_padded_layer(T, B, D, H, nd, _ptr(x_pad),
                                      mask.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                      _ptr(params), _ptr(dy), _ptr(y), _ptr(h_n), _ptr(c_n),
                                      _ptr(dx), _ptr(grads))
    if rc != 0:
        raise ValueError("oracle_lstm_padded_layer rejected its arguments")
    if dy_pad is not None:
        out["dx"] = dx
        out["grads"] = unpack_layer_grads(grads, nd, D, H)
    return out
