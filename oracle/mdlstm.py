"""2-D MDLSTM layer and 2-D example-packing -- TEST INFRASTRUCTURE ONLY.

``md_layer`` marshals numpy arrays into ``mdlstm_oracle.c`` (fp64, each example
and scan direction on its own: "No Padding Please: Efficient Neural
Handwriting Recognition", Sec. III and App. A; the cell is stated in that
file's header).  ``example_pack`` restates the page's packing algorithm
(Sec. V-A and App. B, Algorithm 1) in plain Python; the CUDA library's plan
must place every example exactly where this places it.
"""
from __future__ import annotations

import ctypes

import numpy as np

from .oracle import _f64, _load, _ptr

GATES = ("i", "f1", "f2", "z", "o")
PEEPS = ("i1", "i2", "f1", "f2", "o1", "o2")


def md_param_count(D: int, H: int) -> int:
    return int(_load().oracle_md_param_count(D, H))


def pack_md_params(layer: dict) -> np.ndarray:
    """Flat fp64 blocks, one per direction: W[5H][D], U1[5H][H], U2[5H][H], b[5H], p[6][H]."""
    nd = layer["W"].shape[0]
    return np.concatenate([np.concatenate([_f64(layer[k][d]).ravel() for k in ("W", "U1", "U2", "b", "peep")])
                           for d in range(nd)])


def unpack_md_grads(flat: np.ndarray, ndir: int, D: int, H: int) -> dict:
    out = {k: [] for k in ("W", "U1", "U2", "b", "peep")}
    o = 0
    for _ in range(ndir):
        for k, shape in (("W", (5 * H, D)), ("U1", (5 * H, H)), ("U2", (5 * H, H)), ("b", (5 * H,)),
                         ("peep", (6, H))):
            n = int(np.prod(shape))
            out[k].append(flat[o:o + n].reshape(shape))
            o += n
    assert o == flat.size
    return {k: np.stack(v) for k, v in out.items()}


def md_layer(heights, widths, x, layer: dict, G=None) -> dict:
    """One MDLSTM layer over a list of examples, each example and direction on its own.

    heights[n], widths[n]; x[N, D] = the examples' pixels (row-major) back to back;
    layer: W[ndir,5H,D], U1/U2[ndir,5H,H], b[ndir,5H], peep[ndir,6,H].  Returns y[N, ndir*H]
    and, with G = dL/dy [N, ndir*H], dx[N, D] and grads (same keys as layer)."""
    lib = _load()
    hs = np.ascontiguousarray(heights, dtype=np.int32)
    ws = np.ascontiguousarray(widths, dtype=np.int32)
    n = int(hs.size)
    N = int((hs.astype(np.int64) * ws).sum())
    x = _f64(x).reshape(N, -1)
    D = x.shape[1]
    nd, H = layer["W"].shape[0], layer["U1"].shape[2]
    blk = pack_md_params(layer)
    assert blk.size == nd * md_param_count(D, H)
    y = np.zeros((N, nd * H))
    dy = dx = g = None
    if G is not None:
        dy = _f64(G).reshape(N, nd * H)
        dx = np.zeros((N, D))
        g = np.zeros_like(blk)
    ip = ctypes.POINTER(ctypes.c_int)
    rc = lib.oracle_md_layer(n, hs.ctypes.data_as(ip), ws.ctypes.data_as(ip), D, H, nd, _ptr(x), _ptr(blk),
                             _ptr(dy), _ptr(y), _ptr(dx), _ptr(g))
    if rc != 0:
        raise ValueError("oracle_md_layer rejected its arguments")
    out = {"y": y}
    if G is not None:
        out["dx"] = dx
        out["grads"] = unpack_md_grads(g, nd, D, H)
    return out


def example_pack(heights, widths, row_width: int = 0) -> dict:
    """Algorithm 1 of "No Padding Please" (App. B), one plain step at a time.

    1. Bucket the examples by height (buckets in descending height; empty examples
       are left out: they have no pixel to place).
    2. Fill rows bucket by bucket: repeatedly add the widest example of the bucket
       that still fits beside the row's examples and one separator pixel; ties go to
       the lower example index.  When none fits, the row is closed and a new one
       begins; an empty row takes the widest example even if it is wider than the
       row (the row then holds it alone).  The last row of a bucket is closed when
       the bucket runs out (a row holds one height).
    3. Tile: rows top to bottom with one separator row between consecutive rows,
       examples left to right with one separator column between neighbours.
    The row width defaults to the widest example.  Returns rows (lists of example
    indices), y0/x0 per example (-1 for empty ones), the canvas height and width
    (the widest row), and the canvas mask (1 = example pixel)."""
    hs = [int(v) for v in heights]
    ws = [int(v) for v in widths]
    n = len(hs)
    live = [i for i in range(n) if hs[i] > 0 and ws[i] > 0]
    W = int(row_width) if row_width > 0 else max([ws[i] for i in live], default=0)
    rows = []
    for hgt in sorted({hs[i] for i in live}, reverse=True):
        bucket = [i for i in live if hs[i] == hgt]
        row, used = [], 0
        while bucket:
            room = W - used - (1 if row else 0)
            fit = [i for i in bucket if ws[i] <= room]
            if not fit and not row:
                fit = list(bucket)
            if fit:
                best = max(fit, key=lambda i: (ws[i], -i))
                bucket.remove(best)
                used += ws[best] + (1 if row else 0)
                row.append(best)
            else:
                rows.append(row)
                row, used = [], 0
        if row:
            rows.append(row)
    y0 = [-1] * n
    x0 = [-1] * n
    R, Wc, top = 0, 0, 0
    for r, row in enumerate(rows):
        if r > 0:
            top += 1
        left = 0
        for k, i in enumerate(row):
            if k > 0:
                left += 1
            y0[i], x0[i] = top, left
            left += ws[i]
        Wc = max(Wc, left)
        top += hs[row[0]]
    R = top
    mask = np.zeros((R, Wc), dtype=np.uint8)
    for i in live:
        mask[y0[i]:y0[i] + hs[i], x0[i]:x0[i] + ws[i]] = 1
    return {"rows": rows, "y0": y0, "x0": x0, "height": R, "width": Wc, "mask": mask}
