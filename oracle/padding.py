"""Zero-padding statistics (test infrastructure only).

"On batching variable size inputs for training end-to-end speech enhancement
systems", Sec. 4: the zero-padding rate (ZPR) is the total number of padded
zeros relative to the original dataset length.  The page's formula was lost;
the plain reading, with l_i the length of sequence i and p_i the padding
added to it, is

    ZPR = sum_i p_i / sum_i l_i .

The waste fraction is the share of computed frames that are padding:
sum_i p_i / (sum_i p_i + sum_i l_i); for a single padded batch of B
sequences that is (B*T_max - N) / (B*T_max).
"""
from __future__ import annotations

import numpy as np


def _padding(batches):
    pad = 0
    real = 0
    for lens in batches:
        lens = np.asarray(lens, dtype=np.int64)
        if lens.size == 0:
            continue
        pad += int((lens.max() - lens).sum())
        real += int(lens.sum())
    return pad, real


def zero_padding_rate(batches) -> float:
    """ZPR over a list of batches, each padded to its own longest sequence."""
    pad, real = _padding(batches)
    return pad / real if real else 0.0


def waste_fraction(batches) -> float:
    """Padded share of all computed frames over a list of padded batches."""
    pad, real = _padding(batches)
    return pad / (pad + real) if (pad + real) else 0.0


def bucket_batches(lengths, width: int, lo: int):
    """Sorted buckets of the given width: [lo, lo+width), [lo+width, lo+2*width), ...

    Returns the lists of sequence indices per non-empty bucket, each in
    ascending index order.  The top bucket is closed at the maximum length.
    """
    lengths = np.asarray(lengths)
    top = int(lengths.max()) if lengths.size else lo
    nb = max(1, (top - lo) // width + (1 if (top - lo) % width else 0))
    out = []
    for k in range(nb):
        a, b = lo + k * width, lo + (k + 1) * width
        sel = (lengths >= a) & ((lengths < b) | ((k == nb - 1) & (lengths <= b)))
        idx = np.nonzero(sel)[0]
        if idx.size:
            out.append(idx)
    return out
