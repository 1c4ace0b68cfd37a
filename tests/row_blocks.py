"""Whole-tensor oracle checks, split into row blocks over the host's cores.

The oracle is single-threaded C reached through ctypes, and ctypes lets go of
the GIL for the length of a foreign call, so row blocks of one tensor run
side by side on a thread pool; the numpy comparisons that follow each block
release it too.  The blocks cover every row once, so a test that checks each
block against the oracle checks every element of the tensor.

Row-indexed parts of a chain stay correct under the split: the dropout
counter of element i is offset + i / 8, so a block starting at row r0 keys its
oracle call with offset + r0 * cols / 8 (the block start keeps r0 * cols a
multiple of 8), and the causal mask depends on the row modulo its period, so
mask blocks start at multiples of the period.
"""
import os
from concurrent.futures import ThreadPoolExecutor


def host_workers(limit=32):
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, limit))


def blocks(rows, block=None, align=1):
    """Consecutive [r0, r1) ranges covering 0 .. rows, each starting at a
    multiple of ``align``; by default about four blocks per worker."""
    if rows <= 0:
        return []
    if block is None:
        block = -(-rows // (4 * host_workers()))
    block = max(align, -(-block // align) * align)
    return [(r0, min(rows, r0 + block)) for r0 in range(0, rows, block)]


def map_row_blocks(rows, work, block=None, align=1):
    """work(r0, r1) for every block, on a thread pool; the results in row
    order.  The first exception raised by any block is raised here."""
    spans = blocks(rows, block, align)
    with ThreadPoolExecutor(host_workers()) as ex:
        futs = [ex.submit(work, r0, r1) for r0, r1 in spans]
        return [f.result() for f in futs]


def worst(stats):
    """Combine assert_close's (max abs error, max error / limit) pairs."""
    if not stats:
        return (0.0, 0.0)
    return (max(s[0] for s in stats), max(s[1] for s in stats))


def dropout_block_offset(offset, r0, cols):
    """The generator offset of an oracle call that starts at row r0."""
    start = r0 * cols
    assert start % 8 == 0, "dropout blocks must start at a multiple of 8 elements"
    return offset + start // 8

