"""Host-side checks of index layouts the kernels rely on.

* The standalone filter's swizzled shared rows (16-byte group g stored at
  g ^ ((g >> 3) & 1)): for every window offset a lane group of eight reads
  eight distinct 16-byte bank groups (the property that makes the 16-warp
  form conflict-free), while the plain layout collides.
* The many-geometry kernel's units (rows of quads; narrow frames as P whole
  rows side by side, or as eight row lanes of a 32-quad slice where whole
  rows would idle more threads; eight rows each): over every unit of a job,
  every output pixel is formed exactly once, for widths from 1 to past one
  unit.
* The uint8 filter tables' 2x fast path: the kernel groups (8, 4, 2 pixels
  for 1, 3, 4 channels) tile the row.
"""
import numpy as np
import pytest

THREADS, ROWS = 256, 8


def swz(e):
    g = e >> 2
    return ((g ^ ((g >> 3) & 1)) << 2) | (e & 3)


@pytest.mark.parametrize("layout", ["swizzled", "plain"])
def test_filter_window_loads_bank_groups(layout):
    f = swz if layout == "swizzled" else (lambda e: e)
    conflicts = 0
    for kc in range(0, 72, 8):               # chunk offsets up to the widest filter
        for q in range(4):                   # the four 16-byte loads of a window
            for phase in range(4):           # eight lanes per phase of a 16-byte load
                groups = {(f(8 * t + kc + 4 * q) >> 2) % 8 for t in range(8 * phase, 8 * phase + 8)}
                conflicts += len(groups) != 8
    if layout == "swizzled":
        assert conflicts == 0
    else:
        assert conflicts > 0


def test_swizzle_is_a_permutation_within_the_row():
    for row_floats in (272, 328, 264 + 64):
        idx = [swz(e) for e in range(row_floats)]
        assert sorted(idx) == list(range(row_floats))


def unit_shape(out_w):
    # (quads per row lane, row lanes, column units), as the kernel picks them
    qpr = (out_w + 3) // 4
    if qpr >= THREADS:
        return THREADS, 1, (qpr + THREADS - 1) // THREADS
    P, n32 = THREADS // qpr, (qpr + 31) // 32
    if 8 > P * n32:
        return 32, THREADS // 32, n32
    return qpr, P, 1


def multi_cover(out_h, out_w):
    qw, P, col_units = unit_shape(out_w)
    rows_per_unit = ROWS * P
    units = ((out_h + rows_per_unit - 1) // rows_per_unit) * col_units
    seen = np.zeros((out_h, out_w), np.int64)
    for u in range(units):
        rb, cu = divmod(u, col_units)
        for t in range(THREADS):
            p = t // qw
            q = cu * qw + t - p * qw
            x0 = 4 * q
            if x0 >= out_w or p >= P:
                continue
            for k8 in range(ROWS):
                dy = rb * rows_per_unit + p + k8 * P
                if dy >= out_h:
                    break
                seen[dy, x0:min(x0 + 4, out_w)] += 1
    return seen


@pytest.mark.parametrize("out_w", [1, 3, 4, 5, 31, 56, 100, 224, 320, 350, 371, 516, 530, 640, 1020, 1023, 1024,
                                   1025, 2050])
@pytest.mark.parametrize("out_h", [1, 7, 8, 9, 65, 300])
def test_multi_units_cover_each_pixel_once(out_h, out_w):
    seen = multi_cover(out_h, out_w)
    assert (seen == 1).all()


@pytest.mark.parametrize("C, px", [(1, 8), (3, 4), (4, 2)])
def test_down2_groups_tile_the_row(C, px):
    for OW in (1, 7, 8, 9, 960, 1919, 1920):
        full = OW // px
        cols = [p for j in range(full) for p in range(j * px, j * px + px)] + list(range(full * px, OW))
        assert cols == list(range(OW))
        assert 2 * px * C in (16, 24)        # source bytes per row and group: one 16- or 24-byte load set


@pytest.mark.parametrize("out_w, shape", [(640, (32, 8, 5)), (530, (32, 8, 5)), (371, (32, 8, 3)),
                                          (300, (75, 3, 1)), (224, (56, 4, 1)), (320, (80, 3, 1)),
                                          (1030, (256, 1, 2))])
def test_multi_unit_shapes_of_the_workload_widths(out_w, shape):
    # 640-pixel rows (160 quads) go to 32-quad slices, which keep every
    # thread busy; 300/224/320-pixel rows stay whole rows side by side
    assert unit_shape(out_w) == shape
