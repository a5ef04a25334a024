"""Seeded random configurations, every operation, byte for byte against the oracle.

Each case draws a rank (1..5), an element size, extents, a box that the
encoder accepts (inner box bytes a multiple of 16, or exactly the swizzle
span), traversal steps, padded and sometimes permuted strides, random
origins (partly outside the tensor) and a random pipeline shape, then checks
the listed gather, the grid gather, the listed store and the listed round trip.
"""
import numpy as np
import pytest

import datagen
import oracle
from gpu_helpers import assert_bytes_equal, dev_bytes, dev_empty, host, torch_cuda

pytestmark = pytest.mark.gpu

DTYPES = ["u8", "f16", "bf16", "f32", "f64"]
SPANS = {"32B": 32, "64B": 64, "128B": 128}


def draw_case(seed):
    g = np.random.default_rng(seed)
    dtype = DTYPES[g.integers(len(DTYPES))]
    esize = datagen.ESIZE[dtype]
    rank = int(g.integers(1, 6))
    swizzle = "none" if rank == 1 else ["none", "32B", "64B", "128B"][g.integers(4)]
    if swizzle == "none":
        box0 = (16 // esize) * int(g.integers(1, 9))
    else:
        box0 = SPANS[swizzle] // esize
    box0 = min(box0, 256)
    dims = [int(g.integers(1, 3 * box0 + 8))]
    box = [box0]
    steps = [1]
    for d in range(1, rank):
        dims.append(int(g.integers(1, 14 if rank <= 3 else 6)))
        box.append(int(g.integers(1, 9 if rank <= 3 else 4)))
        steps.append(int([1, 1, 2, 3][g.integers(4)]))
    # nested strides with row padding, outer dimensions in a random order
    order = list(range(1, rank))
    g.shuffle(order)
    strides = [esize] + [0] * (rank - 1)
    step = ((dims[0] * esize + 16 * int(g.integers(0, 3)) + 15) // 16) * 16
    for d in order:
        strides[d] = step
        step *= dims[d]
    nbytes = max(step, 16)
    launch = {}
    if g.random() < 0.7:
        launch = dict(stages=int(g.integers(1, 7)), ctas=int(g.integers(1, 9)),
                      store_groups=int(g.integers(1, 4)), schedule=["strided", "contiguous"][g.integers(2)])
    n = int(g.integers(1, 90))
    if seed % 2:  # every other case also runs the stage bookkeeping check (no draw, so cases stay put)
        launch = dict(launch, checks=1)
    if seed % 3 == 1:  # the one-thread drain where it serves, freeing stages before the next store where it may
        launch = dict(launch, consumer="drain")
        if launch.get("stages", 0) > launch.get("store_groups", 0) > 0:
            launch["release"] = "before_store"
    return dict(dtype=dtype, esize=esize, dims=tuple(dims), strides=tuple(strides), box=tuple(box),
                swizzle=swizzle, steps=tuple(steps), nbytes=nbytes, launch=launch, n=n, seed=seed)


@pytest.fixture(scope="module")
def atb():
    torch_cuda()
    import async_bulk_tensor_gb300 as atb

    atb.init_device()
    atb.device_status()
    return atb


def draw_large_case(seed):
    """Larger shapes: rank 2-3, boxes up to 256 along outer dimensions (at most
    16 KiB per box), up to 2000 listed boxes, deeper rings, up to 39 CTAs, so
    that every CTA wraps its ring many times and several store groups are in
    flight."""
    g = np.random.default_rng(seed)
    dtype = DTYPES[g.integers(len(DTYPES))]
    esize = datagen.ESIZE[dtype]
    rank = int(g.integers(2, 4))
    swizzle = ["none", "32B", "64B", "128B"][g.integers(4)]
    box0 = (16 // esize) * int(g.integers(1, 17)) if swizzle == "none" else SPANS[swizzle] // esize
    box0 = min(box0, 256)
    budget = 16384 // (box0 * esize)
    box, dims, steps = [box0], [int(g.integers(box0 // 2 + 1, 6 * box0 + 9))], [1]
    for d in range(1, rank):
        b = int(g.integers(1, max(2, min(256, budget) + 1)))
        budget = max(1, budget // b)
        box.append(b)
        dims.append(int(g.integers(1, 5 * b + 3)))
        steps.append(int([1, 1, 1, 2, 4][g.integers(5)]))
    order = list(range(1, rank))
    g.shuffle(order)
    strides = [esize] + [0] * (rank - 1)
    step = ((dims[0] * esize + 16 * int(g.integers(0, 3)) + 15) // 16) * 16
    for d in order:
        strides[d] = step
        step *= dims[d]
    launch = dict(stages=int(g.integers(1, 9)), ctas=int(g.integers(1, 40)), store_groups=int(g.integers(1, 5)),
                  schedule=["strided", "contiguous"][g.integers(2)], checks=int(g.integers(2)))
    if g.random() < 0.3:
        launch = {}
    if seed % 3 == 2:  # as for the small cases (no draw)
        launch = dict(launch, consumer="drain")
        if launch.get("stages", 0) > launch.get("store_groups", 0) > 0:
            launch["release"] = "before_store"
    return dict(dtype=dtype, esize=esize, dims=tuple(dims), strides=tuple(strides), box=tuple(box),
                swizzle=swizzle, steps=tuple(steps), nbytes=max(step, 16), launch=launch,
                n=int(g.integers(1, 2000)), seed=seed)


@pytest.mark.parametrize("seed", range(400))
def test_random_configuration(atb, seed):
    _check_case(atb, draw_case(10_000 + seed))


@pytest.mark.parametrize("seed", range(40))
def test_random_large_configuration(atb, seed):
    _check_case(atb, draw_large_case(20_000 + seed), grid_round_trip=True)


def _check_case(atb, c, grid_round_trip=False):
    v = oracle.View(c["esize"], c["dims"], c["strides"], c["box"], c["swizzle"], c["steps"])
    src_h = datagen.random_bytes(c["nbytes"], c["seed"])
    coords_h = datagen.random_box_origins(c["dims"], c["box"], c["esize"], c["n"], c["seed"] + 1)
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled(c["dtype"], src, c["dims"], c["strides"], c["box"], c["swizzle"],
                          elem_strides=c["steps"])
    bb = atb.box_bytes(ms)
    assert bb == oracle.box_bytes(v)
    n = c["n"]
    what = f"case {c}"

    guard = 4096  # bytes past every destination must keep their fill
    packed = dev_empty(n * bb + guard, fill=0xEE)
    atb.tile_load(ms, coords, n, packed, **c["launch"])
    want_packed = oracle.tile_load(v, src_h, coords_h)
    assert atb.device_status().code == 0
    got = host(packed)
    assert_bytes_equal(got, want_packed, "listed gather " + what, image_bytes=bb)
    assert (got[n * bb:] == 0xEE).all(), "listed gather wrote past its buffer " + what

    grid_h = oracle.grid_coords(v)
    packed_g = dev_empty(len(grid_h) * bb + guard, fill=0xEE)
    atb.tile_load(ms, None, 0, packed_g, **c["launch"])
    assert atb.device_status().code == 0
    got_g = host(packed_g)
    assert_bytes_equal(got_g, oracle.tile_load(v, src_h, grid_h), "grid gather " + what, image_bytes=bb)
    assert (got_g[len(grid_h) * bb:] == 0xEE).all(), "grid gather wrote past its buffer " + what

    out = dev_empty(c["nbytes"] + guard, fill=0x5A)
    md = atb.encode_tiled(c["dtype"], out, c["dims"], c["strides"], c["box"], c["swizzle"],
                          elem_strides=c["steps"])
    atb.tile_store(md, coords, n, packed, **c["launch"])
    assert atb.device_status().code == 0
    want = np.full(c["nbytes"] + guard, 0x5A, dtype=np.uint8)
    oracle.tile_store(v, want, coords_h, want_packed)
    assert_bytes_equal(host(out), want, "listed store " + what)

    out2 = dev_empty(c["nbytes"] + guard, fill=0x33)
    md2 = atb.encode_tiled(c["dtype"], out2, c["dims"], c["strides"], c["box"], c["swizzle"],
                           elem_strides=c["steps"])
    atb.tile_roundtrip(ms, md2, coords, n, **c["launch"])
    assert atb.device_status().code == 0
    want2 = np.full(c["nbytes"] + guard, 0x33, dtype=np.uint8)
    oracle.roundtrip(v, src_h, v, want2, coords_h)
    assert_bytes_equal(host(out2), want2, "listed round trip " + what)

    if grid_round_trip:
        out3 = dev_empty(c["nbytes"] + guard, fill=0x77)
        md3 = atb.encode_tiled(c["dtype"], out3, c["dims"], c["strides"], c["box"], c["swizzle"],
                               elem_strides=c["steps"])
        atb.tile_roundtrip(ms, md3, None, 0, **c["launch"])
        assert atb.device_status().code == 0
        want3 = np.full(c["nbytes"] + guard, 0x77, dtype=np.uint8)
        oracle.roundtrip(v, src_h, v, want3, grid_h)
        assert_bytes_equal(host(out3), want3, "grid round trip " + what)


def test_draws_cover_the_space():
    cases = [draw_case(10_000 + s) for s in range(40)]
    assert {c["dtype"] for c in cases} == set(DTYPES)
    assert {len(c["dims"]) for c in cases} == {1, 2, 3, 4, 5}
    assert {c["swizzle"] for c in cases} == {"none", "32B", "64B", "128B"}
    assert any(max(c["steps"]) > 1 for c in cases)


def test_large_draws_fit_and_vary():
    cases = [draw_large_case(20_000 + s) for s in range(40)]
    for c in cases:
        bb = c["esize"]
        for b, e in zip(c["box"], c["steps"]):
            bb *= -(-b // e)
        assert bb <= 16384 and all(1 <= b <= 256 for b in c["box"])
    assert {c["swizzle"] for c in cases} == {"none", "32B", "64B", "128B"}
    assert max(c["n"] for c in cases) > 1000 and any(c["launch"].get("checks") for c in cases)
