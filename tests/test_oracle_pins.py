"""Pins for the CPU oracle: facts the pages print, closed forms and brute force.

None of these tests re-types the oracle's formulas.  The gather is checked
against an independent formulation (numpy strided views, zero padding and
slicing); the swizzle against the page's identity case, a typed chunk table,
per-mode chunk rules and brute-force bijection; the store against numpy slice
assignment and guard bytes; the tile enumeration against the positions the
CuTe-DSL page prints.
"""
import json
import os

import numpy as np
import pytest

import datagen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLDEN, "page_facts.json")))


# --------------------------------------------------------------------------
# independent helpers (numpy array semantics, no oracle code)
# --------------------------------------------------------------------------
def np_view(buf: np.ndarray, v: oracle.View) -> np.ndarray:
    """Element view of ``buf`` as an array shaped outermost-first + (esize,) bytes."""
    shape = tuple(int(d) for d in reversed(v.dims)) + (v.esize,)
    strides = tuple(int(s) for s in reversed(v.strides)) + (1,)
    return np.lib.stride_tricks.as_strided(buf, shape=shape, strides=strides, writeable=True)


def np_box(buf: np.ndarray, v: oracle.View, origin) -> np.ndarray:
    """The box at ``origin`` (innermost first) with zero bytes outside the tensor.

    Built by zero-padding every dimension by the box extent and slicing.
    """
    a = np_view(buf, v)
    c = [int(x) for x in reversed(origin)]
    b = [int(x) for x in reversed(v.box)]
    n = [int(x) for x in reversed(v.dims)]
    pads = [(max(0, -ci), max(0, ci + bi - ni)) for ci, bi, ni in zip(c, b, n)]
    p = np.pad(a, pads + [(0, 0)])
    sl = tuple(slice(ci + lo, ci + lo + bi) for ci, bi, (lo, _) in zip(c, b, pads))
    return p[sl]  # shape outermost-first box + (esize,)


def chunk_permutation(box_bytes: int, mode: str) -> np.ndarray:
    """dest_offset[src_offset] built from 16-byte chunk rules per 128-byte line.

    NONE keeps every chunk; 32B/64B/128B XOR the chunk number inside each
    128-byte line with the line number modulo 2/4/8 (the swizzle span divided
    by 16 bytes).  Written with integer division and modulo over lines and
    chunks, not with bit masks.
    """
    period_lines = {"none": 1, "32B": 2, "64B": 4, "128B": 8}[mode]
    span_chunks = period_lines  # chunks that can move: 2, 4 or 8 of the 8 per line
    dest = np.empty(box_bytes, dtype=np.int64)
    for o in range(box_bytes):
        line, within = divmod(o, 128)
        chunk, byte = divmod(within, 16)
        group, low = divmod(chunk, span_chunks)
        low = low ^ (line % period_lines)
        dest[o] = line * 128 + (group * span_chunks + low) * 16 + byte
    return dest


def swizzle_image(unswizzled: np.ndarray, mode: str) -> np.ndarray:
    dest = chunk_permutation(unswizzled.size, mode)
    out = np.empty_like(unswizzled)
    out[dest] = unswizzled
    return out


# --------------------------------------------------------------------------
# page facts
# --------------------------------------------------------------------------
def test_single_tile_is_16384_bytes():
    f = FACTS["single_tile_fp32"]
    v = oracle.View(4, (64, 64), (4, 256), (64, 64))
    assert oracle.box_bytes(v) == f["box_bytes"] == 16384
    assert oracle.box_bytes(oracle.View(*_c(datagen.C1))) == 16384


def test_cute_dsl_payload_and_smem_request():
    f = FACTS["cute_dsl_fp16_strips"]
    v = oracle.View(*_c(datagen.C2))
    assert oracle.box_bytes(v) == f["payload_bytes"] == 32768
    # the allocation is payload plus one 8-byte barrier; the expected
    # transaction count is the payload alone
    assert oracle.box_bytes(v) + f["barrier_bytes"] == f["smem_request_bytes"]


def test_cute_dsl_924_tiles_and_block1_iter2():
    f = FACTS["cute_dsl_fp16_strips"]
    v = oracle.View(*_c(datagen.C2))
    assert oracle.grid_count(v) == f["tile_loads"] == f["blocks"] * f["tiles_per_block"]
    coords = oracle.grid_coords(v)
    # block b owns row strip b and walks j = 0..6: tile index b*7 + j
    t = f["example_block"] * f["tiles_per_block"] + f["example_iteration"]
    x, y = coords[t]
    assert (y, x) == tuple(f["example_element_origin_row_col"])
    # load that tile from matrices whose elements hold their own row (resp.
    # column) index and read which rows and columns it actually covers
    rows, cols = 8448, 1792
    row_of = np.ascontiguousarray(np.broadcast_to(np.arange(rows, dtype=np.uint16)[:, None], (rows, cols)))
    col_of = np.ascontiguousarray(np.broadcast_to(np.arange(cols, dtype=np.uint16)[None, :], (rows, cols)))
    for val, (lo, hi) in ((row_of, f["example_rows"]), (col_of, f["example_cols"])):
        img = oracle.tile_load(v, val.view(np.uint8).ravel(), coords[t:t + 1])
        got = img.view(np.uint16).reshape(64, 256)
        assert got.min() == lo and got.max() == hi


def test_identity_swizzle_leaves_offsets_unchanged():
    f = FACTS["cute_dsl_identity_swizzle"]
    assert f["bits"] == 0
    for o in range(0, 1 << 16):
        assert oracle.swizzle(o, "none") == o


def test_swizzle128_matches_chunk_table():
    rows = [list(map(int, ln.split())) for ln in open(os.path.join(GOLDEN, "swizzle128_chunk_table.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 8
    for rep in range(3):  # pattern repeats every 1024 bytes
        for r in range(8):
            for c in range(8):
                for b in (0, 7, 15):
                    src = rep * 1024 + r * 128 + c * 16 + b
                    dst = rep * 1024 + r * 128 + rows[r][c] * 16 + b
                    assert oracle.swizzle(src, "128B") == dst


@pytest.mark.parametrize("mode", ["none", "32B", "64B", "128B"])
def test_swizzle_chunk_rules(mode):
    n = 4096
    dest = chunk_permutation(n, mode)
    got = np.array([oracle.swizzle(o, mode) for o in range(n)])
    np.testing.assert_array_equal(got, dest)


@pytest.mark.parametrize("mode", ["none", "32B", "64B", "128B"])
@pytest.mark.parametrize("box_bytes", [128, 1024, 4096, 8192, 16384, 32768])
def test_swizzle_is_bijection_on_box(mode, box_bytes):
    img = np.array([oracle.swizzle(o, mode) for o in range(box_bytes)])
    assert img.min() == 0 and img.max() == box_bytes - 1
    assert np.unique(img).size == box_bytes


def test_swizzle_keeps_16_byte_chunks_and_lines():
    for mode in ("32B", "64B", "128B"):
        for o in range(0, 8192, 3):
            s = oracle.swizzle(o, mode)
            assert s % 16 == o % 16          # bytes inside a chunk stay in order
            assert s // 128 == o // 128      # a chunk never leaves its 128-byte line


# --------------------------------------------------------------------------
# gather / store vs an independent numpy formulation
# --------------------------------------------------------------------------
def _c(w: datagen.Workload):
    return (w.esize, w.dims, w.strides, w.box, w.swizzle)


@pytest.mark.parametrize("esize", [1, 2, 4, 8])
def test_gather_brute_force_small_2d(esize):
    rows, cols = 5, 7
    v = oracle.View(esize, (cols, rows), (esize, cols * esize), (4, 4))
    buf = datagen.random_bytes(rows * cols * esize, 11 + esize)
    origins = np.array([(x, y) for y in range(-4, 9) for x in range(-4, 9)], dtype=np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        want = np_box(buf, v, o).reshape(-1)
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], want, err_msg=f"origin {o}")


@pytest.mark.parametrize("mode", ["32B", "64B", "128B"])
def test_gather_swizzled_small(mode):
    span = {"32B": 32, "64B": 64, "128B": 128}[mode]
    esize = 2
    inner = span // esize
    rows, cols = 37, inner * 3 - 5  # ragged in both directions
    v = oracle.View(esize, (cols, rows), (esize, cols * esize + 16), (inner, 16), mode)
    buf = datagen.random_bytes(v.span_bytes() + 64, 21)
    origins = np.array([(x, y) for y in (-15, -1, 0, 5, 21, 36) for x in (-inner, -8, 0, 8, cols - 8, cols)],
                       dtype=np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        want = swizzle_image(np_box(buf, v, o).reshape(-1), mode)
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], want, err_msg=f"origin {o}")


def test_gather_permuted_3d_view():
    # storage [6, 3, 8] fp32 contiguous, view = permute(1, 0, 2): shape [3, 6, 8]
    S = datagen.random_bytes(6 * 3 * 8 * 4, 31)
    v = oracle.View(4, (8, 6, 3), (4, 3 * 8 * 4, 8 * 4), (4, 4, 2), "none")
    arr = S.view(np.uint32).reshape(6, 3, 8).transpose(1, 0, 2)  # numpy's own permute
    g = datagen.rng(5)
    origins = np.stack([g.integers(-3, 8, 200), g.integers(-3, 6, 200), g.integers(-1, 3, 200)], 1).astype(np.int32)
    packed = oracle.tile_load(v, S, origins).view(np.uint32)
    for i, (x, y, z) in enumerate(origins):
        want = np.zeros((2, 4, 4), dtype=np.uint32)
        for kz in range(2):
            for ky in range(4):
                for kx in range(4):
                    zz, yy, xx = z + kz, y + ky, x + kx
                    if 0 <= zz < 3 and 0 <= yy < 6 and 0 <= xx < 8:
                        want[kz, ky, kx] = arr[zz, yy, xx]
        np.testing.assert_array_equal(packed[i * 32:(i + 1) * 32], want.ravel())


@pytest.mark.parametrize("rank", [1, 2, 3, 4, 5])
def test_gather_each_rank(rank):
    dims = (9, 4, 3, 2, 3)[:rank]
    box = (4, 3, 2, 2, 2)[:rank]
    esize = 2
    strides = [esize]
    for d in range(1, rank):
        strides.append(strides[-1] * dims[d - 1] + (16 if d == 1 else 0))
    v = oracle.View(esize, dims, tuple(strides), box)
    buf = datagen.random_bytes(v.span_bytes() + 32, 40 + rank)
    g = datagen.rng(rank)
    origins = np.stack([g.integers(-b + 1, n, 64) for n, b in zip(dims, box)], 1).astype(np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], np_box(buf, v, o).reshape(-1))


def test_store_matches_slice_assignment_and_keeps_guard_bytes():
    rows, cols, esize = 11, 13, 4
    pitch = cols * esize + 12  # 12 guard bytes after every row
    v = oracle.View(esize, (cols, rows), (esize, pitch), (8, 4))
    fill = 0xA5
    base = np.full(pitch * rows + 64, fill, dtype=np.uint8)
    origins = np.array([(x, y) for y in (-3, 0, 4, 8, 10) for x in (-7, 0, 5, 8, 12)], dtype=np.int32)
    packed = datagen.random_bytes(len(origins) * oracle.box_bytes(v), 51)
    oracle.tile_store(v, base, origins, packed)
    # independent: numpy slice assignment, in list order, clipped to the tensor
    want = np.full_like(base, fill)
    a = np_view(want, v)
    bb = oracle.box_bytes(v)
    for i, (x, y) in enumerate(origins):
        img = packed[i * bb:(i + 1) * bb].reshape(4, 8, esize)
        y0, y1 = max(y, 0), min(y + 4, rows)
        x0, x1 = max(x, 0), min(x + 8, cols)
        if y0 < y1 and x0 < x1:
            a[y0:y1, x0:x1] = img[y0 - y:y1 - y, x0 - x:x1 - x]
    np.testing.assert_array_equal(base, want)
    # guard bytes between rows and after the tensor never change
    for r in range(rows):
        assert (base[r * pitch + cols * esize:(r + 1) * pitch] == fill).all()
    assert (base[rows * pitch:] == fill).all()


@pytest.mark.parametrize("mode", ["none", "128B"])
def test_store_after_load_is_identity(mode):
    rows, cols, esize = 300, 200, 2
    box = (64, 32) if mode == "128B" else (40, 24)
    v = oracle.View(esize, (cols, rows), (esize, cols * esize), box, mode)
    src = datagen.random_bytes(rows * cols * esize, 61)
    coords = oracle.grid_coords(v)
    packed = oracle.tile_load(v, src, coords)
    dst = np.zeros_like(src)
    oracle.tile_store(v, dst, coords, packed)
    np.testing.assert_array_equal(dst, src)
    dst2 = np.full_like(src, 7)
    oracle.roundtrip(v, src, v, dst2, coords)
    np.testing.assert_array_equal(dst2, src)


def test_c3_edge_tiles_zero_counts():
    w = datagen.C3
    v = oracle.View(*_c(w))
    assert oracle.grid_count(v) == 79 * 47 == 3713
    coords = oracle.grid_coords(v)
    # nonzero storage so that every zero byte in an image is fill
    buf = (datagen.random_bytes(w.storage_bytes, 3) | np.uint8(1))
    bb = oracle.box_bytes(v)
    last_row = np.nonzero(coords[:, 1] == 78 * 128)[0]
    last_col = np.nonzero(coords[:, 0] == 46 * 64)[0]
    corner = np.intersect1d(last_row, last_col)
    assert len(last_row) == 47 and len(last_col) == 79 and len(corner) == 1
    packed = oracle.tile_load(v, buf, coords[[0, last_row[0], last_col[0], corner[0]]])
    zeros = [(packed[i * bb:(i + 1) * bb] == 0).sum() for i in range(4)]
    valid_rows, valid_cols = 10000 - 78 * 128, 3000 - 46 * 64
    assert (valid_rows, valid_cols) == (16, 56)
    assert zeros[0] == 0
    assert zeros[1] == (128 - valid_rows) * 64 * 2
    assert zeros[2] == 128 * (64 - valid_cols) * 2
    assert zeros[3] == (128 * 64 - valid_rows * valid_cols) * 2


def test_c4_random_origins_touch_tensor_and_span_every_offset():
    w = datagen.C4
    c = datagen.workload_coords(w)
    assert c.shape == (4096, 3)
    for d in range(3):
        assert (c[:, d] + w.box[d] - 1 >= 0).all() and (c[:, d] < w.dims[d]).all()
        assert c[:, d].min() == -(w.box[d] - 1) and c[:, d].max() == w.dims[d] - 1  # the whole range is drawn
    # every element offset along x: all four 4-byte phases of a 16-byte chunk occur
    phases = np.bincount(c[:, 0] % 4, minlength=4) / len(c)
    assert (np.abs(phases - 0.25) < 0.04).all()
    partial = ((c[:, 0] < 0) | (c[:, 0] + 32 > 1024) | (c[:, 1] < 0) | (c[:, 1] + 64 > 512)).mean()
    assert 0.15 < partial < 0.4


def test_day76_sixteen_tiles():
    f = FACTS["day76_matrix"]
    v = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    assert oracle.grid_count(v) == f["tiles"]
    coords = oracle.grid_coords(v)
    # coordinates are innermost first: tile (blockIdx.x, blockIdx.y) -> (64 bx, 64 by)
    assert [tuple(c) for c in coords[:5]] == [(0, 0), (64, 0), (128, 0), (192, 0), (0, 64)]


def test_swapped_coordinates_load_transposed_positions():
    # swapping x and y fetches the mirror tile: a whole tile of wrong values
    v = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    buf = datagen.random_bytes(256 * 256 * 4, 77)
    right = oracle.tile_load(v, buf, np.array([[64, 128]], dtype=np.int32))
    swapped = oracle.tile_load(v, buf, np.array([[128, 64]], dtype=np.int32))
    assert (right.view(np.uint32) != swapped.view(np.uint32)).mean() > 0.99
    a = buf.view(np.uint32).reshape(256, 256)
    np.testing.assert_array_equal(right.view(np.uint32).reshape(64, 64), a[128:192, 64:128])


# --------------------------------------------------------------------------
# fp32 update between load and store ("Day 76", +1.0f per element)
# --------------------------------------------------------------------------
def test_add_f32_closed_forms():
    x = np.array([0.0, 1.5, -2.0, 2.0**24, 3.0e38, -0.0, 1e-45], dtype=np.float32)
    got = oracle.add_f32(x.view(np.uint8), 1.0).view(np.float32)
    np.testing.assert_array_equal(got[:3], np.array([1.0, 2.5, -1.0], dtype=np.float32))
    assert got[3] == np.float32(2.0**24)        # 2^24 + 1 rounds to even: 2^24
    assert got[4] == np.float32(3.0e38)         # absorbed
    assert got[5] == 1.0 and got[6] == 1.0      # -0 + 1 and denormal + 1
    z = oracle.add_f32(np.array([-0.0], dtype=np.float32).view(np.uint8), 0.0).view(np.uint32)
    assert z[0] == 0                            # IEEE: -0 + +0 = +0


def test_add_f32_matches_numpy_float32():
    x = datagen.finite_f32_bytes(1 << 16, 8)
    for addend in (1.0, -3.25, 1e-40, 6.5e37):
        got = oracle.add_f32(x, addend).view(np.uint32)
        with np.errstate(over="ignore"):  # finite + 6.5e37 may round to inf, as IEEE says
            want = (x.view(np.float32) + np.float32(addend)).view(np.uint32)
        np.testing.assert_array_equal(got, want)


def test_roundtrip_add_f32_day76_matrix():
    f = FACTS["day76_matrix"]
    v = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    src = datagen.finite_f32_bytes(256 * 256, 76)
    dst = np.zeros_like(src)
    oracle.roundtrip_add_f32(v, src, v, dst, oracle.grid_coords(v), 1.0)
    assert oracle.grid_count(v) == f["tiles"]
    want = (src.view(np.float32) + np.float32(1.0)).view(np.uint8)
    np.testing.assert_array_equal(dst, want)


def test_roundtrip_add_f32_edges_get_addend_where_source_is_outside():
    # destination larger than the source: its extra elements read source zeros
    vs = oracle.View(4, (20, 10), (4, 80), (16, 4))
    vd = oracle.View(4, (32, 12), (4, 128), (16, 4))
    src = datagen.finite_f32_bytes(200, 9)
    dst = np.full(12 * 128, 0xCD, dtype=np.uint8)
    oracle.roundtrip_add_f32(vs, src, vd, dst, oracle.grid_coords(vd), 2.0)
    d = dst.view(np.float32).reshape(12, 32)
    s = src.view(np.float32).reshape(10, 20)
    np.testing.assert_array_equal(d[:10, :20], s + np.float32(2.0))
    assert (d[:12, 20:32] == 2.0).all() and (d[10:12, :20] == 2.0).all()


# --------------------------------------------------------------------------
# traversal steps (elementStrides): every e-th element along outer dimensions
# --------------------------------------------------------------------------
def np_box_stepped(buf, v, origin):
    """Box with traversal steps by numpy: zero-pad, then slice with a step."""
    a = np_view(buf, v)
    c = [int(x) for x in reversed(origin)]
    b = [int(x) for x in reversed(v.box)]
    e = [int(x) for x in reversed(v.estr)]
    n = [int(x) for x in reversed(v.dims)]
    pads = [(max(0, -ci), max(0, ci + bi - ni)) for ci, bi, ni in zip(c, b, n)]
    p = np.pad(a, pads + [(0, 0)])
    sl = tuple(slice(ci + lo, ci + lo + bi, ei) for ci, bi, ei, (lo, _) in zip(c, b, e, pads))
    return p[sl]


def test_box_bytes_with_traversal_steps():
    v = oracle.View(2, (64, 40, 9), (2, 128, 5120), (64, 8, 3), "none", (1, 2, 3))
    assert oracle.box_bytes(v) == 64 * 4 * 1 * 2
    v = oracle.View(4, (64, 40), (4, 256), (32, 7), "128B", (1, 3))
    assert oracle.box_bytes(v) == 32 * 3 * 4  # ceil(7 / 3) = 3 visits


@pytest.mark.parametrize("steps", [(1, 2), (1, 3), (1, 8)])
def test_gather_with_traversal_steps_brute_force(steps):
    rows, cols, esize = 23, 40, 2
    v = oracle.View(esize, (cols, rows), (esize, cols * esize + 16), (16, 9), "none", steps)
    buf = datagen.random_bytes(v.span_bytes() + 32, 91)
    origins = np.array([(x, y) for y in range(-9, 24, 4) for x in range(-16, 41, 8)], dtype=np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], np_box_stepped(buf, v, o).reshape(-1),
                                      err_msg=f"origin {o}")


def test_gather_3d_steps_and_swizzle():
    esize = 4
    dims, box, steps = (32, 11, 13), (32, 5, 6), (1, 2, 4)
    strides = (4, 128 + 16, (128 + 16) * 11)
    v = oracle.View(esize, dims, strides, box, "128B", steps)
    buf = datagen.random_bytes(v.span_bytes() + 16, 92)
    g = datagen.rng(3)
    origins = np.stack([g.integers(-1, 2, 50) * 32, g.integers(-4, 11, 50), g.integers(-5, 13, 50)], 1).astype(np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        want = swizzle_image(np_box_stepped(buf, v, o).reshape(-1), "128B")
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], want)


def test_gather_4d_steps_on_middle_dimensions_brute_force():
    # a step on every outer dimension, the two middle ones included; any x origin
    esize = 2
    dims, box, steps = (8, 7, 6, 5), (8, 5, 4, 3), (1, 2, 3, 2)
    strides = (2, 32, 32 * 7 + 16, (32 * 7 + 16) * 6)
    v = oracle.View(esize, dims, strides, box, "none", steps)
    assert oracle.box_bytes(v) == 8 * 3 * 2 * 2 * esize  # ceil(5/2), ceil(4/3), ceil(3/2) visits
    buf = datagen.random_bytes(v.span_bytes() + 16, 94)
    g = datagen.rng(4)
    origins = np.stack([g.integers(-7, 8, 60)] + [g.integers(-b, n, 60) for b, n in zip(box[1:], dims[1:])],
                       1).astype(np.int32)
    packed = oracle.tile_load(v, buf, origins)
    bb = oracle.box_bytes(v)
    for i, o in enumerate(origins):
        np.testing.assert_array_equal(packed[i * bb:(i + 1) * bb], np_box_stepped(buf, v, o).reshape(-1),
                                      err_msg=f"origin {o}")


def test_store_overlapping_boxes_later_box_wins():
    # boxes are applied in list order: where two boxes with different images
    # overlap, the one listed later leaves its bytes
    v = oracle.View(1, (32, 4), (1, 32), (16, 4))
    ones, twos = np.full(64, 0x11, np.uint8), np.full(64, 0x22, np.uint8)
    base = np.zeros(128, dtype=np.uint8)
    oracle.tile_store(v, base, np.array([[0, 0], [8, 0]], dtype=np.int32), np.concatenate([ones, twos]))
    rows = base.reshape(4, 32)
    assert (rows[:, :8] == 0x11).all() and (rows[:, 8:24] == 0x22).all() and (rows[:, 24:] == 0).all()
    base[:] = 0
    oracle.tile_store(v, base, np.array([[8, 0], [0, 0]], dtype=np.int32), np.concatenate([twos, ones]))
    assert (rows[:, :16] == 0x11).all() and (rows[:, 16:24] == 0x22).all() and (rows[:, 24:] == 0).all()


def test_store_with_steps_writes_only_visited_elements():
    rows, cols = 17, 32
    v = oracle.View(4, (cols, rows), (4, 128), (32, 8), "none", (1, 3))
    base = np.full(rows * 128, 0x11, dtype=np.uint8)
    origins = np.array([[0, 0], [0, 8], [0, 16]], dtype=np.int32)
    packed = datagen.random_bytes(3 * oracle.box_bytes(v), 93)
    oracle.tile_store(v, base, origins, packed)
    a = base.view(np.uint32).reshape(rows, cols)
    img = packed.view(np.uint32).reshape(3, 3, 32)  # ceil(8 / 3) = 3 rows per box
    for i, y0 in enumerate((0, 8, 16)):
        for k in range(3):
            y = y0 + 3 * k
            if y < rows:
                np.testing.assert_array_equal(a[y], img[i, k])
    untouched = [y for y in range(rows) if (y % 8) % 3 != 0 or (y % 8) > 6]
    assert (base.reshape(rows, 128)[untouched] == 0x11).all()


# --------------------------------------------------------------------------
# out-of-bounds mask (the bytes a NaN-filling load fills instead of reading)
# --------------------------------------------------------------------------
def np_inside_image(v: oracle.View, origin, mode: str) -> np.ndarray:
    """1 per image byte whose element is inside the tensor, by numpy: a buffer
    of ones seen through the view, zero-padded, sliced with the steps, then
    placed by the chunk rules."""
    ones = np.ones(v.span_bytes(), dtype=np.uint8)
    return swizzle_image(np_box_stepped(ones, v, origin).reshape(-1), mode)


@pytest.mark.parametrize("mode,steps", [("none", (1, 1)), ("128B", (1, 1)), ("64B", (1, 3)), ("32B", (1, 2))])
def test_oob_mask_brute_force(mode, steps):
    esize = 4
    inner = {"none": 12, "32B": 8, "64B": 16, "128B": 32}[mode]
    rows, cols = 19, inner * 2 + 4
    v = oracle.View(esize, (cols, rows), (esize, cols * esize + 16), (inner, 7), mode, steps)
    origins = np.array([(x, y) for y in range(-7, 20, 3) for x in range(-inner, cols + 1, 4)], dtype=np.int32)
    mask = oracle.tile_oob_mask(v, origins)
    bb = oracle.box_bytes(v)
    assert mask.size == len(origins) * bb and set(np.unique(mask)) <= {0, 1}
    for i, o in enumerate(origins):
        np.testing.assert_array_equal(mask[i * bb:(i + 1) * bb], 1 - np_inside_image(v, o, mode),
                                      err_msg=f"origin {o}")


def test_oob_mask_c3_edge_tiles_closed_form():
    w = datagen.C3
    v = oracle.View(*_c(w))
    coords = oracle.grid_coords(v)
    pick = [0, int(np.nonzero(coords[:, 1] == 78 * 128)[0][0]), int(np.nonzero(coords[:, 0] == 46 * 64)[0][0]),
            len(coords) - 1]
    mask = oracle.tile_oob_mask(v, coords[pick]).reshape(4, -1)
    valid_rows, valid_cols = 16, 56
    assert mask[0].sum() == 0
    assert mask[1].sum() == (128 - valid_rows) * 64 * 2
    assert mask[2].sum() == 128 * (64 - valid_cols) * 2
    assert mask[3].sum() == (128 * 64 - valid_rows * valid_cols) * 2


def test_oob_mask_marks_whole_elements_and_a_box_outside_is_all_fill():
    v = oracle.View(8, (6, 5), (8, 48), (4, 4), "none")
    mask = oracle.tile_oob_mask(v, np.array([[4, 3], [-4, 0], [0, 5]], dtype=np.int32)).reshape(3, 4, 4, 8)
    assert ((mask.min(axis=3) == mask.max(axis=3))).all()  # all 8 bytes of an element agree
    assert mask[1].all() and mask[2].all()  # entirely left of / below the tensor
    np.testing.assert_array_equal(mask[0, :, :, 0], [[0, 0, 1, 1], [0, 0, 1, 1], [1, 1, 1, 1], [1, 1, 1, 1]])


def test_roundtrip_between_different_views_matches_numpy():
    # source 13 x 9 f16 (row pitch 32 B), destination 11 x 7 f16 (row pitch 48 B); boxes 8 x 4
    # in list order: later boxes overwrite earlier ones where they overlap
    vs = oracle.View(2, (13, 9), (2, 32), (8, 4))
    vd = oracle.View(2, (11, 7), (2, 48), (8, 4))
    src = datagen.random_bytes(9 * 32, 61)
    dst = np.full(7 * 48, 0xA5, dtype=np.uint8)
    origins = np.array([(x, y) for y in (-2, 0, 3, 5, 8) for x in (-8, -4, 0, 4, 8, 12)], dtype=np.int32)
    want = dst.copy()
    a_dst = np_view(want, vd)  # [7, 11, 2] bytes, writable view into `want`
    for o in origins:
        img = np_box(src, vs, o)  # [4, 8, 2], zero outside the source
        x0, y0 = int(o[0]), int(o[1])
        for ky in range(4):
            for kx in range(8):
                y, x = y0 + ky, x0 + kx
                if 0 <= y < 7 and 0 <= x < 11:
                    a_dst[y, x] = img[ky, kx]
    oracle.roundtrip(vs, src, vd, dst, origins)
    np.testing.assert_array_equal(dst, want)


def test_swizzled_view_whose_image_would_overflow_is_refused():
    # The swizzle keeps chunks inside their 128-byte line: a 128B-swizzled box
    # of 144 bytes (nine 16-byte rows) would move its last chunk past the box.
    with pytest.raises(ValueError):
        oracle.View(4, (8, 9, 7), (4, 32, 288), (4, 3, 3), "128B")
    with pytest.raises(ValueError):
        oracle.View(2, (8, 9), (2, 16), (8, 3), "64B")  # 48 bytes under a 64-byte period
    assert oracle.box_bytes(oracle.View(2, (8, 9), (2, 16), (8, 4), "64B")) == 64
    assert oracle.box_bytes(oracle.View(1, (48, 9), (1, 48), (48, 3), "none")) == 144
