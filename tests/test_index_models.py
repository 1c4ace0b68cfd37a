"""Host models of the index arithmetic of the kernels for rows off the 16-byte
grid (no GPU): the shifted one-CTA kernel (head, whole vectors, tail; the
per-column copies; the staged ring) and the shifted form of the cluster
kernel (each CTA's share of the whole vectors, head and tail on rank 0).  For
every dtype, every common offset within 16 bytes and a spread of lengths and
block sizes they check that every element of a row is read and written
exactly once, that every vector access lies inside its row and starts on a
16-byte boundary, that the copies and the bulk copies stay inside their
shared-memory areas, and that the grid rule keeps each CTA on one row offset.
The formulas are written here from the kernels' description, not shared with
them."""
import pytest

LENGTHS = [8, 9, 15, 31, 33, 257, 1031, 2051, 4099, 4100, 8195, 32767]
BLOCKS = [32, 96, 288, 1024]


def ceil_div(a, b):
    return -(-a // b)


def head(m0, row, cols, es):
    """Elements before the row's first 16-byte boundary."""
    off = (m0 + row * cols * es) % 16
    return ((16 - off) % 16) // es


@pytest.mark.parametrize("es,vec", [(4, 4), (4, 8), (2, 8)], ids=["f32", "f32x8", "bf16"])
def test_shifted_rows_cover_each_element_once(es, vec):
    for cols in LENGTHS:
        if cols < 2 * vec:
            continue
        cstride = (cols + 15) // 16 * 16
        for m0 in range(0, 16, es):
            for row in range(4):
                h = head(m0, row, cols, es)
                nb = (cols - h) // vec
                ne = cols - nb * vec
                assert nb >= 1 and h < 16 // es and ne < 2 * vec
                for threads in BLOCKS:
                    if ne > threads:
                        continue
                    vpt = ceil_div(nb, threads)
                    seen = [0] * cols
                    for tid in range(threads):
                        for k in range(vpt):
                            vi = tid + k * threads
                            vc = min(vi, nb - 1)                     # clamped re-read
                            start = h + vc * vec
                            assert 0 <= start and start + vec <= cols
                            assert (m0 + (row * cols + start) * es) % 16 == 0
                            # the per-column copy from column h on: slot reads
                            # inside the copy, 16-byte aligned in it
                            assert vc * vec + vec <= cols - h <= cstride
                            assert (vc * vec * es) % 16 == 0 and (cstride * es) % 16 == 0
                            if vi < nb:
                                for e in range(vec):
                                    seen[start + e] += 1
                        if tid < ne:
                            col = tid if tid < h else h + nb * vec + (tid - h)
                            seen[col] += 1
                    assert seen == [1] * cols, (cols, m0, row, threads)
                # the staged ring: one bulk copy of the row's whole vectors per
                # input, 16-byte aligned at both ends and inside a stage
                nbytes = nb * vec * es
                assert nbytes % 16 == 0 and nbytes <= cstride * es
                assert (m0 + (row * cols + h) * es) % 16 == 0


@pytest.mark.parametrize("es", [2, 4], ids=["bf16", "f32"])
def test_column_copies(es):
    """The 4-byte asynchronous copies of a per-column array from column h on
    (element by element for bf16 arrays whose column h is not 4-byte
    aligned): every element of the copy written once, reads inside the array,
    both addresses 4-byte aligned."""
    for cols in LENGTHS:
        for h in range(16 // es):
            if h >= cols:
                continue
            n = cols - h
            for array_off in ((0, 2) if es == 2 else (0,)):     # array start, bytes past 4
                src = array_off + h * es
                for threads in BLOCKS:
                    written = [0] * n
                    if es == 4 or src % 4 == 0:
                        per = 4 // es
                        for tid in range(threads):
                            for m in range(tid, n // per, threads):
                                assert (src + m * per * es) % 4 == 0 and (m * per * es) % 4 == 0
                                assert h + m * per + per <= cols
                                for e in range(per):
                                    written[m * per + e] += 1
                        if per == 2 and n % 2:
                            written[n - 1] += 1
                    else:
                        for tid in range(threads):
                            for j in range(tid, n, threads):
                                written[j] += 1
                    assert written == [1] * n


@pytest.mark.parametrize("es,vec", [(4, 4), (4, 8), (2, 8)], ids=["f32", "f32x8", "bf16"])
def test_shifted_cluster_rows(es, vec):
    """The cluster kernel's shifted form: slices sized for the most whole
    vectors a row has, each rank holding those of its slice that the row has,
    rank 0 the head and tail; every element once, vector accesses inside the
    row and aligned, each rank's bulk copy inside its stage."""
    for cols in [33, 1031, 4099, 32769, 50257, 65537]:
        if cols < 2 * vec:
            continue
        nvec = cols // vec
        for cs0 in (2, 4, 8, 16):
            cs = min(cs0, nvec)
            slice_v = ceil_div(nvec, cs)
            cs = ceil_div(nvec, slice_v)
            if cs < 2:
                continue
            threads = min(1024, ceil_div(slice_v, 4) // 32 * 32 + 32)
            vpt = ceil_div(slice_v, threads)
            for m0 in range(0, 16, es):
                for row in range(3):
                    h = head(m0, row, cols, es)
                    nb = (cols - h) // vec
                    ne = cols - nb * vec
                    assert ne <= threads
                    seen = [0] * cols
                    for rank in range(cs):
                        lo = rank * slice_v * vec
                        nv = max(0, min(nb - rank * slice_v, slice_v))
                        assert nv * vec * es <= slice_v * vec * es          # inside the stage
                        if nv:
                            assert (m0 + (row * cols + h + lo) * es) % 16 == 0
                        for tid in range(threads):
                            for k in range(vpt):
                                vi = tid + k * threads
                                if nv == 0:
                                    continue
                                start = h + lo + min(vi, nv - 1) * vec
                                assert 0 <= start and start + vec <= cols
                                if vi < nv:
                                    for e in range(vec):
                                        seen[start + e] += 1
                            if rank == 0 and tid < ne:
                                seen[tid if tid < h else h + nb * vec + (tid - h)] += 1
                    assert seen == [1] * cols, (cols, cs, m0, row)


@pytest.mark.parametrize("es", [2, 4], ids=["bf16", "f32"])
def test_grid_keeps_each_cta_on_one_offset(es):
    """A grid of G CTAs, G a multiple of the period of the rows' offsets
    within 16 bytes, gives each CTA rows of one head (so it copies its
    per-column values once); the period divides 8, and so any grid of whole
    SMs on 152 SMs."""
    for cols in LENGTHS + [4097, 8193]:
        step = (cols * es) % 16
        period = 1
        while (step * period) % 16:
            period *= 2
        assert period in (1, 2, 4, 8) and (152 % period) == 0
        for m0 in range(0, 16, es):
            grid = 3 * period
            for b in range(grid):
                heads = {head(m0, b + k * grid, cols, es) for k in range(6)}
                assert len(heads) == 1
