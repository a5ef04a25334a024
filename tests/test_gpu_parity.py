"""GPU parity: every output of the CUDA path compared byte for byte with the
CPU oracle on the same seeded inputs, through the C ABI (Python binding).

Covers the five workloads (single 64x64 fp32 tile; 8448x1792 fp16 in 132 x 7
boxes of 64x256; ragged 10000x3000 bf16 with 128-byte swizzle and edge boxes;
a permuted 3-D fp32 view with 4096 random, partly out-of-bounds boxes; the
512 MiB fp16 round trip in the launch configuration the benchmark times),
small multi-tile cases with ragged tails over every rank, element size and
swizzle mode, and the edge cases (no boxes, one box, maximum box extents,
origins off the 16-byte grid, boxes entirely outside the tensor).
"""
import numpy as np
import pytest

import datagen
import oracle
from gpu_helpers import assert_bytes_equal, dev_bytes, dev_empty, encode, host, oracle_view, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def atb():
    torch_cuda()
    import async_bulk_tensor_gb300 as atb

    atb.init_device()
    atb.device_status()
    return atb


def device_ok(atb):
    rep = atb.device_status()
    assert rep.code == 0, rep.as_dict()


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
def test_c1_single_tile_round_trip(atb):
    w = datagen.C1
    src_h = datagen.storage(w)
    src, dst = dev_bytes(src_h), dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, src), encode(atb, w, dst)
    assert atb.box_bytes(ms) == 16384 and atb.grid_tiles(ms) == 1
    atb.tile_roundtrip(ms, md, stages=1, ctas=1)
    device_ok(atb)
    v = oracle_view(w)
    want = np.zeros_like(src_h)
    oracle.roundtrip(v, src_h, v, want, oracle.grid_coords(v))
    assert_bytes_equal(host(dst), want, "c1", view=v)


def test_day76_sixteen_tiles_one_block_each(atb):
    # 256x256 fp32, sixteen 64x64 tiles, one CTA per tile
    v = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    src_h = datagen.random_bytes(256 * 1024, 76)
    src, dst = dev_bytes(src_h), dev_empty(256 * 1024, fill=0)
    ms = atb.encode_tiled("f32", src, v.dims, v.strides, v.box)
    md = atb.encode_tiled("f32", dst, v.dims, v.strides, v.box)
    atb.tile_roundtrip(ms, md, ctas=16, stages=1)
    device_ok(atb)
    assert_bytes_equal(host(dst), src_h, "day76", view=v)


def test_c2_132_blocks_by_7_column_tiles(atb):
    w = datagen.C2
    src_h = datagen.storage(w)
    src, dst = dev_bytes(src_h), dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, src), encode(atb, w, dst)
    assert atb.grid_tiles(ms) == 924 and atb.box_bytes(ms) == 32768
    atb.tile_roundtrip(ms, md, ctas=w.ctas, schedule=w.schedule, stages=2)
    device_ok(atb)
    v = oracle_view(w)
    want = np.zeros_like(src_h)
    oracle.roundtrip(v, src_h, v, want, oracle.grid_coords(v))
    assert_bytes_equal(host(dst), want, "c2", view=v)


def test_c3_ragged_bf16_gather_with_swizzle(atb):
    w = datagen.C3
    src_h = datagen.storage(w)
    src = dev_bytes(src_h)
    ms = encode(atb, w, src)
    n = atb.grid_tiles(ms)
    assert n == 3713
    bb = atb.box_bytes(ms)
    packed = dev_empty(n * bb, fill=0xEE)
    atb.tile_load(ms, None, 0, packed)
    device_ok(atb)
    v = oracle_view(w)
    want = oracle.tile_load(v, src_h, oracle.grid_coords(v))
    assert_bytes_equal(host(packed), want, "c3", image_bytes=bb)


def test_c4_permuted_view_random_gather_then_store(atb):
    w = datagen.C4
    src_h = datagen.storage(w)
    coords_h = datagen.workload_coords(w)
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = encode(atb, w, src)
    bb = atb.box_bytes(ms)
    assert bb == 8192
    n = coords_h.shape[0]
    packed = dev_empty(n * bb, fill=0xEE)
    atb.tile_load(ms, coords, n, packed)
    device_ok(atb)
    v = oracle_view(w)
    want_packed = oracle.tile_load(v, src_h, coords_h)
    assert_bytes_equal(host(packed), want_packed, "c4 gather", image_bytes=bb)
    packed_pf = dev_empty(n * bb, fill=0xEE)
    atb.tile_load(ms, coords, n, packed_pf, prefetch_boxes=8)
    device_ok(atb)
    assert_bytes_equal(host(packed_pf), want_packed, "c4 gather with L2 prefetch", image_bytes=bb)

    fresh = dev_empty(w.storage_bytes, fill=0xFF)
    md = encode(atb, w, fresh)
    atb.tile_store(md, coords, n, packed)
    device_ok(atb)
    want = np.full(w.storage_bytes, 0xFF, dtype=np.uint8)
    oracle.tile_store(v, want, coords_h, want_packed)
    assert_bytes_equal(host(fresh), want, "c4 store")


@pytest.fixture(scope="module")
def c5_input():
    return datagen.storage(datagen.C5A)


@pytest.fixture(scope="module")
def c5_device(c5_input, atb):
    return dev_bytes(c5_input)


@pytest.mark.parametrize("w", [datagen.C5A, datagen.C5B], ids=["box64x256", "box128x64_sw128"])
def test_c5_full_round_trip_default_launch(atb, w, c5_input, c5_device):
    dst = dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, c5_device), encode(atb, w, dst)
    atb.tile_roundtrip(ms, md)  # the library defaults, which the benchmark times
    device_ok(atb)
    v = oracle_view(w)
    want = np.zeros_like(c5_input)
    oracle.roundtrip(v, c5_input, v, want, oracle.grid_coords(v))
    assert_bytes_equal(host(dst), want, w.name, view=v)


@pytest.mark.parametrize("consumer", ["drain", "warp", "drain_after_store", "drain_before_store"])
@pytest.mark.parametrize("w", [datagen.C5A, datagen.C5B], ids=["box64x256", "box128x64_sw128"])
def test_c5_full_round_trip_each_consumer(atb, w, consumer, c5_input, c5_device):
    dst = dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, c5_device), encode(atb, w, dst)
    kw = dict(consumer=consumer) if "_" not in consumer else \
        dict(consumer="drain", release=consumer.split("_", 1)[1], stages=5, store_groups=2, ctas_per_sm=1)
    atb.tile_roundtrip(ms, md, **kw)
    device_ok(atb)
    assert_bytes_equal(host(dst), c5_input, f"{w.name} {consumer}", view=oracle_view(w))


def test_library_default_launch_shapes(atb):
    # What the library resolves for tile-grid round trips of a 32 MiB fp16
    # tensor (1024 x 16384), per box size, and that each launch moves every byte.
    dims, strides = (16384, 1024), (2, 32768)
    src_h = datagen.random_bytes(dims[0] * dims[1] * 2, 77)
    src = dev_bytes(src_h)

    def run(box, swizzle, **kw):
        dst = dev_empty(src_h.size, fill=0)
        ms = atb.encode_tiled("f16", src, dims, strides, box, swizzle)
        md = atb.encode_tiled("f16", dst, dims, strides, box, swizzle)
        atb.tile_roundtrip(ms, md, **kw)
        shape = atb.last_launch()
        device_ok(atb)
        assert_bytes_equal(host(dst), src_h, f"box {box} {kw}")
        return shape

    import torch

    sm = torch.cuda.get_device_properties(0).multi_processor_count
    # 16 KiB stages: the drain's own ring, 64 KiB of stages for loads + 48 KiB of store groups
    s16 = run((64, 128), "128B")
    assert (s16["consumer"], s16["release"], s16["stages"], s16["store_groups"], s16["ctas_per_sm"]) == \
        ("drain", "before_store", 7, 3, 1), s16
    assert s16["ctas"] == sm and s16["boxes"] == 2048
    # 8 KiB: 8 + 6 stages
    s8 = run((64, 64), "128B")
    assert (s8["consumer"], s8["release"], s8["stages"], s8["store_groups"]) == ("drain", "before_store", 14, 6), s8
    # 32 KiB: the drain on the common default ring, freeing after the store; 1,024 boxes are a short
    # launch (under four ring-fulls per CTA at one CTA per SM), spread over two CTAs per SM
    s32 = run((256, 64), "none")
    assert (s32["consumer"], s32["release"], s32["stages"], s32["store_groups"], s32["ctas_per_sm"]) == \
        ("drain", "after_store", 3, 2, 2), s32
    # 4 KiB: the drain's ring at two CTAs per SM, 8 + 4 stages
    s4 = run((64, 32), "128B")
    assert (s4["consumer"], s4["release"], s4["stages"], s4["store_groups"], s4["ctas_per_sm"]) == \
        ("drain", "before_store", 12, 4, 2), s4
    # 2 KiB, or an explicit ring shape below 32 KiB: the warp consumer
    assert run((64, 16), "128B")["consumer"] == "warp"
    assert run((64, 128), "128B", stages=3)["consumer"] == "warp"
    # an explicit order on an explicit ring
    sb = run((64, 128), "128B", consumer="drain", release="before_store", stages=4, store_groups=3, ctas_per_sm=2)
    assert (sb["release"], sb["stages"], sb["store_groups"], sb["ctas_per_sm"]) == ("before_store", 4, 3, 2), sb
    sa = run((64, 128), "128B", consumer="drain", release="after_store")
    assert (sa["release"], sa["stages"], sa["store_groups"]) == ("after_store", 7, 3), sa
    sw = run((64, 128), "128B", consumer="warp", release="before_store", stages=4, store_groups=2)
    assert (sw["consumer"], sw["release"], sw["stages"], sw["store_groups"]) == ("warp", "before_store", 4, 2), sw
    # freeing before the next store needs a stage beyond the store groups
    dst = dev_empty(src_h.size, fill=0)
    ms = atb.encode_tiled("f16", src, dims, strides, (64, 128), "128B")
    md = atb.encode_tiled("f16", dst, dims, strides, (64, 128), "128B")
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(ms, md, consumer="drain", release="before_store", stages=3, store_groups=3)
    assert e.value.code == atb.ATB_ERR_ARG and "store_groups" in str(e.value)
    assert atb.last_launch()["boxes"] == 0
    # coordinate lists run the kernel with several consumer warps
    coords = dev_bytes(np.array([[0, 0], [64, 128]], dtype=np.int32).reshape(-1).view(np.uint8))
    packed = dev_empty(2 * 16384, fill=0)
    atb.tile_load(ms, coords, 2, packed)
    sl = atb.last_launch()
    assert (sl["consumer"], sl["release"], sl["stages"], sl["store_groups"], sl["ctas_per_sm"], sl["boxes"]) == \
        ("warps", "before_store", 5, 3, 2, 2), sl
    device_ok(atb)
    # the fp32 update over the tile grid takes the several-warp kernel's own ring (16 KiB boxes of fp32)
    fv = oracle.View(4, (8192, 512), (4, 32768), (32, 128), "128B")
    f_h = datagen.finite_f32_bytes(8192 * 512, 78)
    fsrc, fdst = dev_bytes(f_h), dev_empty(f_h.size, fill=0)
    mfs = atb.encode_tiled("f32", fsrc, fv.dims, fv.strides, fv.box, "128B")
    mfd = atb.encode_tiled("f32", fdst, fv.dims, fv.strides, fv.box, "128B")
    atb.tile_roundtrip_add_f32(mfs, mfd, 1.0)
    sf = atb.last_launch()
    assert (sf["consumer"], sf["release"], sf["stages"], sf["store_groups"], sf["ctas_per_sm"]) == \
        ("warps", "before_store", 5, 3, 2), sf
    device_ok(atb)
    want = np.zeros_like(f_h)
    oracle.roundtrip_add_f32(fv, f_h, fv, want, oracle.grid_coords(fv), 1.0)
    assert_bytes_equal(host(fdst), want, "fp32 update on the several-warp ring", view=fv)


@pytest.mark.parametrize("w", [datagen.C5A, datagen.C5B], ids=["box64x256", "box128x64_sw128"])
def test_c5_ring_check_full_size(atb, w, c5_input, c5_device):
    # the stage bookkeeping check over every box of the 512 MiB round trip, in
    # the default launch shape and in a deep ring with four groups in flight
    for launch in (dict(checks=atb.CHECK_RING), dict(checks=atb.CHECK_RING, stages=6, store_groups=4)):
        dst = dev_empty(w.storage_bytes, fill=0)
        ms, md = encode(atb, w, c5_device), encode(atb, w, dst)
        atb.tile_roundtrip(ms, md, **launch)
        device_ok(atb)
        assert_bytes_equal(host(dst), c5_input, f"{w.name} {launch}", view=oracle_view(w))


@pytest.mark.parametrize("stages", [2, 4, 6, 8])
@pytest.mark.parametrize("w", [datagen.C5A, datagen.C5B], ids=["box64x256", "box128x64_sw128"])
def test_c5_stage_sweep(atb, w, stages, c5_input, c5_device):
    dst = dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, c5_device), encode(atb, w, dst)
    if stages * atb.box_bytes(ms) > 227 * 1024:
        # 8 stages of 32 KiB do not fit in one block's shared memory
        with pytest.raises(atb.AtbError) as e:
            atb.tile_roundtrip(ms, md, stages=stages)
        assert e.value.code == atb.ATB_ERR_SMEM_BUDGET
        return
    atb.tile_roundtrip(ms, md, stages=stages)
    device_ok(atb)
    # the oracle's full-grid round trip reproduces its input (pinned on the
    # CPU by the store-after-load identity), so the input is the expectation
    assert_bytes_equal(host(dst), c5_input, f"{w.name} stages={stages}", view=oracle_view(w))


# --------------------------------------------------------------------------
# small multi-tile cases: every rank, element size and swizzle mode
# --------------------------------------------------------------------------
def _strides(esize, dims, pitch_pad=16, order=None):
    """Byte strides for dims (innermost first); outer dimensions nested in
    ``order`` (default: increasing), innermost run padded by pitch_pad bytes."""
    rank = len(dims)
    order = list(range(1, rank)) if order is None else order
    strides = [esize] + [0] * (rank - 1)
    step = ((dims[0] * esize + pitch_pad + 15) // 16) * 16
    for d in order:
        strides[d] = step
        step *= dims[d]
    return tuple(strides), step


SMALL = [
    # name, dtype, dims, box, swizzle, outer order
    ("r1_u8", "u8", (1000,), (48,), "none", None),
    ("r2_f16", "f16", (300, 77), (64, 16), "none", None),
    ("r2_bf16_sw128", "bf16", (200, 150), (64, 32), "128B", None),
    ("r2_f32_sw64", "f32", (100, 45), (16, 8), "64B", None),
    ("r2_u8_sw32", "u8", (333, 41), (32, 8), "32B", None),
    ("r2_f64", "f64", (50, 33), (8, 8), "none", None),
    ("r3_f32_sw64_permuted", "f32", (64, 20, 7), (16, 8, 3), "64B", [2, 1]),
    ("r4_f16_sw64", "f16", (40, 9, 5, 4), (32, 4, 2, 3), "64B", None),
    ("r5_u8_sw32", "u8", (70, 6, 5, 4, 3), (32, 3, 2, 2, 2), "32B", [3, 1, 4, 2]),
    ("r2_f16_box256", "f16", (700, 300), (256, 256), "none", None),
]


def _small_case(name, dtype, dims, box, swizzle, order, seed):
    esize = datagen.ESIZE[dtype]
    strides, nbytes = _strides(esize, dims, order=order)
    v = oracle.View(esize, dims, strides, box, swizzle)
    src_h = datagen.random_bytes(nbytes, seed)
    g = datagen.rng(seed + 1)
    rand = datagen.random_box_origins(dims, box, esize, 97, seed + 2)
    # plus boxes wholly outside the tensor on both sides and one far away
    extra = []
    for d in range(len(dims)):
        q = max(1, 16 // esize)
        lo = [0] * len(dims)
        lo[d] = -((box[d] + q - 1) // q) * q if d == 0 else -box[d]
        hi = [0] * len(dims)
        hi[d] = ((dims[d] + q - 1) // q) * q if d == 0 else dims[d]
        extra += [lo, hi]
    coords = np.concatenate([rand, np.array(extra, dtype=np.int32)])
    g.shuffle(coords)
    return v, src_h, nbytes, coords


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("launch", [dict(stages=1, ctas=1), dict(stages=3, ctas=5, store_groups=2),
                                    dict(stages=2, ctas=3, schedule="contiguous"), dict(),
                                    dict(prefetch_boxes=3, l2_hints=3, poll_suspend_ns=20000),
                                    dict(checks=1), dict(checks=1, stages=2, ctas=3, store_groups=2),
                                    dict(consumer="drain"), dict(consumer="warp", stages=2, store_groups=1),
                                    dict(consumer="drain", release="before_store", stages=2, store_groups=1),
                                    dict(consumer="drain", release="before_store", stages=4, store_groups=2, ctas=3),
                                    dict(consumer="drain", release="before_store", stages=5, store_groups=3, ctas=2,
                                         checks=1, l2_hints=3),
                                    dict(consumer="drain", release="after_store"),
                                    dict(consumer="warp", release="before_store", stages=3, store_groups=2, ctas=4)],
                         ids=["s1c1", "s3c5g2", "s2c3contig", "default", "prefetch3_hints", "ring_check",
                              "ring_check_s2c3g2", "drain", "warp_s2g1", "before_s2g1", "before_s4g2c3",
                              "before_s5g3c2_check_hints", "drain_after", "warp_before_s3g2c4"])
def test_small_cases_all_ops(atb, case, launch):
    name, dtype, dims, box, swizzle, order = case
    v, src_h, nbytes, coords_h = _small_case(name, dtype, dims, box, swizzle, order, 1000 + len(name))
    if box == (256, 256) and launch.get("stages", 4) > 1:
        launch = dict(launch, stages=1)  # one 128 KiB stage
        launch.pop("release", None)  # one stage leaves nothing to free before the next store
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled(dtype, src, dims, v.strides, box, swizzle)
    bb = atb.box_bytes(ms)
    n = coords_h.shape[0]

    # gather, listed origins (guard bytes after the packed images must survive)
    guard = 4096
    packed = dev_empty(n * bb + guard, fill=0xEE)
    atb.tile_load(ms, coords, n, packed, **launch)
    device_ok(atb)
    want_packed = oracle.tile_load(v, src_h, coords_h)
    got = host(packed)
    assert_bytes_equal(got, want_packed, f"{name} load", image_bytes=bb)
    assert (got[n * bb:] == 0xEE).all(), f"{name} load wrote past the packed buffer"
    packed = packed[: n * bb]

    # gather, tile grid
    grid_h = oracle.grid_coords(v)
    packed_g = dev_empty(len(grid_h) * bb + guard, fill=0xEE)
    atb.tile_load(ms, None, 0, packed_g, **launch)
    device_ok(atb)
    got_g = host(packed_g)
    assert_bytes_equal(got_g, oracle.tile_load(v, src_h, grid_h), f"{name} grid load", image_bytes=bb)
    assert (got_g[len(grid_h) * bb:] == 0xEE).all(), f"{name} grid load wrote past the packed buffer"

    # scatter of random images: over the tile grid, whose boxes are disjoint, so
    # the result does not depend on the order the boxes are written in (listed
    # origins may overlap; they are stored below with images of one load, which
    # carry identical bytes wherever boxes overlap)
    images_h = datagen.random_bytes(len(grid_h) * bb, 7)
    images = dev_bytes(images_h)
    out = dev_empty(nbytes + guard, fill=0x5A)  # bytes past the tensor must stay 0x5A
    md = atb.encode_tiled(dtype, out, dims, v.strides, box, swizzle)
    atb.tile_store(md, None, 0, images, **launch)
    device_ok(atb)
    want = np.full(nbytes + guard, 0x5A, dtype=np.uint8)
    oracle.tile_store(v, want, grid_h, images_h)
    assert_bytes_equal(host(out), want, f"{name} grid store")

    # listed origins, overlapping boxes carry identical bytes (images of a load)
    out2 = dev_empty(nbytes + guard, fill=0x5A)
    md2 = atb.encode_tiled(dtype, out2, dims, v.strides, box, swizzle)
    atb.tile_store(md2, coords, n, packed, **launch)
    device_ok(atb)
    want2 = np.full(nbytes + guard, 0x5A, dtype=np.uint8)
    oracle.tile_store(v, want2, coords_h, want_packed)
    assert_bytes_equal(host(out2), want2, f"{name} listed store")

    # round trip with listed origins into a prefilled tensor
    out3 = dev_empty(nbytes + guard, fill=0x33)
    md3 = atb.encode_tiled(dtype, out3, dims, v.strides, box, swizzle)
    atb.tile_roundtrip(ms, md3, coords, n, **launch)
    device_ok(atb)
    want3 = np.full(nbytes + guard, 0x33, dtype=np.uint8)
    oracle.roundtrip(v, src_h, v, want3, coords_h)
    assert_bytes_equal(host(out3), want3, f"{name} roundtrip")


# --------------------------------------------------------------------------
# edge cases and device-side errors
# --------------------------------------------------------------------------
def test_zero_boxes_launch_nothing(atb):
    src = dev_empty(4096, fill=1)
    packed = dev_empty(1024, fill=0xEE)
    ms = atb.encode_tiled("f32", src, (32, 32), (4, 128), (32, 8))
    coords = dev_empty(16)
    atb.tile_load(ms, coords, 0, packed)
    atb.tile_store(ms, coords, 0, packed)
    atb.tile_roundtrip(ms, ms, coords, 0)
    device_ok(atb)
    assert (host(packed) == 0xEE).all()


# boxes whose x origin is off the 16-byte grid (the engine may not start a copy
# there; the consumer threads move them): every phase of a 16-byte chunk, at
# and across the start and the end of whole and ragged rows, and wholly outside
OFF_GRID = [
    # name, dtype, dims, box, swizzle, outer order
    ("r1_u8", "u8", (1000,), (64,), "none", None),
    ("r2_u8_ragged", "u8", (1001, 9), (48, 4), "none", None),
    ("r2_f16_sw128", "f16", (300, 40), (64, 8), "128B", None),
    ("r2_bf16_ragged_sw64", "bf16", (301, 33), (32, 5), "64B", None),
    ("r2_f32_sw32", "f32", (130, 20), (8, 6), "32B", None),
    ("r2_f32_box256", "f32", (600, 7), (256, 3), "none", None),
    ("r2_f64_ragged", "f64", (51, 12), (8, 3), "none", None),
    ("r3_f32_sw128_permuted", "f32", (70, 9, 6), (32, 4, 2), "128B", [2, 1]),
    ("r4_f16_sw32", "f16", (45, 7, 5, 3), (16, 3, 2, 2), "32B", None),
]


def _off_grid_origins(dims, box, esize, seed):
    q = 16 // esize
    d0, b0 = dims[0], box[0]
    xs = sorted(set(range(-b0 - q, -b0 + 2 * q)) | set(range(-2 * q, 2 * q + 1)) |
                set(range(d0 - b0 - q, d0 - b0 + q + 1)) | set(range(d0 - 2 * q, d0 + q + 1)))
    g = datagen.rng(seed)
    c = np.empty((len(xs), len(dims)), dtype=np.int32)
    c[:, 0] = xs
    for d in range(1, len(dims)):
        c[:, d] = g.integers(-(box[d] - 1), dims[d], size=len(xs))
    c = np.concatenate([c, datagen.random_box_origins(dims, box, esize, 60, seed + 1)])
    g.shuffle(c)
    return c


@pytest.mark.parametrize("case", OFF_GRID, ids=[c[0] for c in OFF_GRID])
@pytest.mark.parametrize("launch", [dict(), dict(stages=1, ctas=1), dict(checks=1, stages=2, ctas=3)],
                         ids=["default", "s1c1", "ring_check_s2c3"])
def test_off_grid_origins_all_ops(atb, case, launch):
    name, dtype, dims, box, swizzle, order = case
    esize = datagen.ESIZE[dtype]
    strides, nbytes = _strides(esize, dims, order=order)
    v = oracle.View(esize, dims, strides, box, swizzle)
    src_h = datagen.random_bytes(nbytes, 4100 + len(name))
    coords_h = _off_grid_origins(dims, box, esize, 4200 + len(name))
    assert ((coords_h[:, 0].astype(np.int64) * esize) % 16 != 0).mean() > 0.3
    src, coords = dev_bytes(src_h), dev_bytes(coords_h.view(np.uint8))
    n = len(coords_h)
    ms = atb.encode_tiled(dtype, src, dims, strides, box, swizzle)
    bb = atb.box_bytes(ms)
    guard = 4096

    packed = dev_empty(n * bb + guard, fill=0xEE)
    atb.tile_load(ms, coords, n, packed, **launch)
    device_ok(atb)
    want_packed = oracle.tile_load(v, src_h, coords_h)
    got = host(packed)
    assert_bytes_equal(got, want_packed, f"{name} gather", image_bytes=bb)
    assert (got[n * bb:] == 0xEE).all(), f"{name} gather wrote past the packed buffer"

    out = dev_empty(nbytes + guard, fill=0x5A)
    md = atb.encode_tiled(dtype, out, dims, strides, box, swizzle)
    atb.tile_store(md, coords, n, packed[: n * bb], **launch)
    device_ok(atb)
    want = np.full(nbytes + guard, 0x5A, dtype=np.uint8)
    oracle.tile_store(v, want, coords_h, want_packed)
    assert_bytes_equal(host(out), want, f"{name} store")

    out2 = dev_empty(nbytes + guard, fill=0x33)
    md2 = atb.encode_tiled(dtype, out2, dims, strides, box, swizzle)
    atb.tile_roundtrip(ms, md2, coords, n, **launch)
    device_ok(atb)
    want2 = np.full(nbytes + guard, 0x33, dtype=np.uint8)
    oracle.roundtrip(v, src_h, v, want2, coords_h)
    assert_bytes_equal(host(out2), want2, f"{name} round trip")

    if dtype == "f32":
        fin_h = datagen.finite_f32_bytes(nbytes // 4, 4300 + len(name))
        fin = dev_bytes(fin_h)
        mf = atb.encode_tiled(dtype, fin, dims, strides, box, swizzle)
        out3 = dev_empty(nbytes + guard, fill=0x44)
        md3 = atb.encode_tiled(dtype, out3, dims, strides, box, swizzle)
        atb.tile_roundtrip_add_f32(mf, md3, 1.0, coords, n, **launch)
        device_ok(atb)
        want3 = np.full(nbytes + guard, 0x44, dtype=np.uint8)
        oracle.roundtrip_add_f32(v, fin_h, v, want3, coords_h, 1.0)
        assert_bytes_equal(host(out3), want3, f"{name} fp32 update")


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32", "f64"])
def test_off_grid_nan_fill_matches_the_engine_fill(atb, dtype):
    # Whether the engine or the consumer threads filled an element outside the
    # tensor, its bytes are the same NaN (0x7FF7 in every 16-bit half).
    esize = datagen.ESIZE[dtype]
    q = 16 // esize
    dims, box = (120 + 1, 9), (32 // esize * 2, 4)
    strides, nbytes = _strides(esize, dims)
    v = oracle.View(esize, dims, strides, box, "none")
    src_h = datagen.random_bytes(nbytes, 4400)
    xs = list(range(-box[0] - q, q + 1)) + list(range(dims[0] - box[0] - q, dims[0] + q))
    coords_h = np.array([[x, y] for x in xs for y in (-3, 2, 7)], dtype=np.int32)
    src, coords = dev_bytes(src_h), dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled(dtype, src, dims, strides, box, oob_fill="nan")
    bb = atb.box_bytes(ms)
    packed = dev_empty(len(coords_h) * bb, fill=0)
    atb.tile_load(ms, coords, len(coords_h), packed)
    device_ok(atb)
    got = host(packed)
    _check_nan_fill(got, v, src_h, coords_h, dtype, f"{dtype} off-grid NaN fill")
    mask = oracle.tile_oob_mask(v, coords_h).reshape(len(coords_h), bb)
    imgs = got.reshape(len(coords_h), bb)
    on_grid = (coords_h[:, 0] * esize) % 16 == 0
    for which, rows in (("engine", on_grid), ("threads", ~on_grid)):
        filled = imgs[rows][mask[rows] == 1].reshape(-1, 2)
        assert filled.size and (filled == np.array([0xF7, 0x7F], dtype=np.uint8)).all(), which


def test_origin_beyond_range_is_reported_and_never_issued(atb):
    # origins beyond +-2^30 are refused per box before any copy is issued; the
    # other boxes of the call still move
    v = oracle.View(2, (128, 64), (2, 256), (64, 16))
    src_h = datagen.random_bytes(64 * 256, 91)
    src = dev_bytes(src_h)
    far = (1 << 30) + 16
    coords_h = np.array([[0, 0], [0, far], [64, 16], [-far, 0], [64, 48]], dtype=np.int32)
    coords = dev_bytes(coords_h.view(np.uint8))
    good = [0, 2, 4]
    ms = atb.encode_tiled("f16", src, v.dims, v.strides, v.box)
    bb = atb.box_bytes(ms)

    packed = dev_empty(5 * bb, fill=0xEE)
    atb.tile_load(ms, coords, 5, packed, stages=2, ctas=1)
    rep = atb.device_status()
    assert rep.code == atb.ATB_ERR_COORD_RANGE and rep.tile == 1 and rep.errors == 2, rep.as_dict()
    got = host(packed).reshape(5, bb)
    want = oracle.tile_load(v, src_h, coords_h[good]).reshape(3, bb)
    for i, j in enumerate(good):
        assert_bytes_equal(got[j], want[i], f"box {j}")
    assert (got[[1, 3]] == 0xEE).all()  # refused boxes left untouched

    for op in ("store", "roundtrip"):
        out = dev_empty(64 * 256, fill=0x5A)
        md = atb.encode_tiled("f16", out, v.dims, v.strides, v.box)
        if op == "store":
            atb.tile_store(md, coords, 5, packed)
        else:
            atb.tile_roundtrip(ms, md, coords, 5)
        rep = atb.device_status()
        assert rep.code == atb.ATB_ERR_COORD_RANGE and rep.errors == 2, (op, rep.as_dict())
        want_t = np.full(64 * 256, 0x5A, dtype=np.uint8)
        oracle.tile_store(v, want_t, coords_h[good], oracle.tile_load(v, src_h, coords_h[good]))
        assert_bytes_equal(host(out), want_t, f"{op} with refused origins")
    device_ok(atb)


def test_bounded_wait_times_out_and_gpu_stays_usable(atb):
    import time

    t0 = time.time()
    atb.selftest_wait_timeout(50_000_000)  # 50 ms; nothing ever completes the barrier
    rep = atb.device_status()
    elapsed = time.time() - t0
    assert rep.code == atb.ATB_ERR_TIMEOUT and rep.where == 5, rep.as_dict()
    assert elapsed < 10
    test_c1_single_tile_round_trip(atb)


def test_host_side_errors(atb):
    a = dev_empty(1 << 16)
    b = dev_empty(1 << 16)
    ms = atb.encode_tiled("f16", a, (256, 64), (2, 512), (64, 16))
    md = atb.encode_tiled("f16", b, (256, 64), (2, 512), (32, 16))
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(ms, md)
    assert e.value.code == atb.ATB_ERR_ARG
    with pytest.raises(atb.AtbError) as e:
        atb.tile_load(ms, None, 0, a.data_ptr() + 8)
    assert e.value.code == atb.ATB_ERR_SMEM_ALIGN
    with pytest.raises(atb.AtbError) as e:
        atb.tile_load(ms, None, 0, b, stages=17)
    assert e.value.code == atb.ATB_ERR_ARG
    c = dev_empty(1 << 17)
    big = atb.encode_tiled("f16", c, (256, 256), (2, 512), (256, 256))
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(big, big, stages=2)
    assert e.value.code == atb.ATB_ERR_SMEM_BUDGET
    # the binding refuses buffers a call would overrun, and host memory, before the library runs
    with pytest.raises(atb.AtbError) as e:
        atb.encode_tiled("f16", a, (256, 256), (2, 512), (256, 256))
    assert e.value.code == atb.ATB_ERR_ARG and "tensor base" in str(e.value)
    with pytest.raises(atb.AtbError) as e:
        atb.tile_load(ms, None, 0, b[: atb.grid_tiles(ms) * atb.box_bytes(ms) - 1].clone())
    assert e.value.code == atb.ATB_ERR_ARG and "packed buffer" in str(e.value)
    with pytest.raises(atb.AtbError) as e:
        atb.tile_load(ms, None, 0, b.cpu())
    assert e.value.code == atb.ATB_ERR_ARG and "host memory" in str(e.value)
    device_ok(atb)


def test_non_default_stream(atb):
    torch = torch_cuda()
    w = datagen.C2
    src_h = datagen.storage(w, seed=222)
    src, dst = dev_bytes(src_h), dev_empty(w.storage_bytes, fill=0)
    ms, md = encode(atb, w, src), encode(atb, w, dst)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        atb.tile_roundtrip(ms, md, stream=s)
    s.synchronize()
    device_ok(atb)
    assert_bytes_equal(host(dst), src_h, "stream roundtrip")


@pytest.mark.parametrize("kind", ["cpasync", "ldst_v4", "memcpy"])
def test_ablation_copies(atb, kind):
    nbytes = (64 << 20) + 48
    src_h = datagen.random_bytes(nbytes, 99)
    src, dst = dev_bytes(src_h), dev_empty(nbytes, fill=0)
    {"cpasync": atb.copy_cpasync, "ldst_v4": atb.copy_ldst_v4, "memcpy": atb.copy_memcpy}[kind](src, dst, nbytes)
    device_ok(atb)
    assert_bytes_equal(host(dst), src_h, kind)


# --------------------------------------------------------------------------
# fp32 update in shared memory between load and store (generic-proxy writes,
# fence.proxy.async, tensor store)
# --------------------------------------------------------------------------
def test_add_f32_day76_sixteen_tiles(atb):
    v = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    src_h = datagen.finite_f32_bytes(256 * 256, 760)
    src, dst = dev_bytes(src_h), dev_empty(256 * 1024, fill=0)
    ms = atb.encode_tiled("f32", src, v.dims, v.strides, v.box)
    md = atb.encode_tiled("f32", dst, v.dims, v.strides, v.box)
    atb.tile_roundtrip_add_f32(ms, md, 1.0, ctas=16, stages=1)
    device_ok(atb)
    want = np.zeros_like(src_h)
    oracle.roundtrip_add_f32(v, src_h, v, want, oracle.grid_coords(v), 1.0)
    assert_bytes_equal(host(dst), want, "day76 +1.0f", view=v)


@pytest.mark.parametrize("swizzle,box", [("none", (64, 16)), ("128B", (32, 16)), ("64B", (16, 8)),
                                         ("none", (64, 128)), ("128B", (32, 160))])  # 32 KiB; 20 KiB boxes
@pytest.mark.parametrize("launch", [dict(), dict(stages=1, ctas=1), dict(stages=4, ctas=7, store_groups=3),
                                    dict(checks=1, stages=3, ctas=5)],
                         ids=["default", "s1c1", "s4c7g3", "ring_check"])
def test_add_f32_ragged_lists_and_grid(atb, swizzle, box, launch):
    rows, cols = 300, 200
    strides = (4, 816)  # padded rows
    v = oracle.View(4, (cols, rows), strides, box, swizzle)
    src_h = datagen.finite_f32_bytes(816 * rows // 4, 761)
    coords_h = datagen.random_box_origins((cols, rows), box, 4, 257, 762)
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled("f32", src, (cols, rows), strides, box, swizzle)
    for name, cl, nl in (("grid", None, 0), ("list", coords, len(coords_h))):
        out = dev_empty(816 * rows, fill=0x7B)
        md = atb.encode_tiled("f32", out, (cols, rows), strides, box, swizzle)
        atb.tile_roundtrip_add_f32(ms, md, -0.75, cl, nl, **launch)
        device_ok(atb)
        want = np.full(816 * rows, 0x7B, dtype=np.uint8)
        oracle.roundtrip_add_f32(v, src_h, v, want, oracle.grid_coords(v) if cl is None else coords_h, -0.75)
        assert_bytes_equal(host(out), want, f"add_f32 {swizzle} {name}")


def test_add_f32_full_size(atb):
    # 16384 x 8192 fp32 (512 MiB), box 32x128 with 128B swizzle, library defaults
    rows, cols = 8192, 16384
    v = oracle.View(4, (cols, rows), (4, cols * 4), (32, 128), "128B")
    src_h = datagen.finite_f32_bytes(rows * cols, 763)
    src, dst = dev_bytes(src_h), dev_empty(rows * cols * 4, fill=0)
    ms = atb.encode_tiled("f32", src, v.dims, v.strides, v.box, "128B")
    md = atb.encode_tiled("f32", dst, v.dims, v.strides, v.box, "128B")
    atb.tile_roundtrip_add_f32(ms, md, 1.0)
    device_ok(atb)
    want = np.zeros_like(src_h)
    oracle.roundtrip_add_f32(v, src_h, v, want, oracle.grid_coords(v), 1.0)
    assert_bytes_equal(host(dst), want, "add_f32 512 MiB", view=v)


def test_add_f32_rejects_other_types(atb):
    a = dev_empty(1 << 16)
    m16 = atb.encode_tiled("f16", a, (256, 64), (2, 512), (64, 16))
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip_add_f32(m16, m16, 1.0)
    assert e.value.code == atb.ATB_ERR_DTYPE


# --------------------------------------------------------------------------
# host-resident round trip: slab-wise H2D copy, boxes, D2H copy on three streams
# --------------------------------------------------------------------------
HOST_CASES = [
    # name, dtype, dims, strides, box, swizzle, slabs
    ("padded_f16_5slabs", "f16", (1000, 777), (2, 2016), (64, 32), "none", 5),
    ("nested_3d_f32_sw128", "f32", (64, 30, 17), (4, 272, 8160), (32, 8, 4), "128B", 4),
    ("permuted_3d_one_slab", "f32", (64, 30, 17), (4, 4352, 256), (32, 8, 2), "128B", 3),
    ("rank1_u8", "u8", (5000,), (1,), (64,), "none", 7),
]


@pytest.mark.parametrize("case", HOST_CASES, ids=[c[0] for c in HOST_CASES])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_round_trip(atb, case, pinned):
    torch = torch_cuda()
    name, dtype, dims, strides, box, swizzle, slabs = case
    esize = datagen.ESIZE[dtype]
    v = oracle.View(esize, dims, strides, box, swizzle)
    nbytes = ((v.span_bytes() + 15) // 16) * 16
    src_h = datagen.random_bytes(nbytes, 800 + slabs)
    dst_h = np.full(nbytes, 0x5A, dtype=np.uint8)
    if pinned:
        src_host = torch.from_numpy(src_h).pin_memory()
        dst_host = torch.from_numpy(dst_h).pin_memory()
    else:
        src_host, dst_host = src_h.copy(), dst_h.copy()
    d_src, d_dst = dev_empty(nbytes, fill=0), dev_empty(nbytes, fill=0x5A)
    ms = atb.encode_tiled(dtype, d_src, dims, strides, box, swizzle)
    md = atb.encode_tiled(dtype, d_dst, dims, strides, box, swizzle)
    s = torch.cuda.Stream()
    atb.tile_roundtrip_host(ms, md, src_host, dst_host, slabs, stream=s)
    s.synchronize()
    device_ok(atb)
    got = dst_host.numpy() if pinned else dst_host
    want = dst_h.copy()
    oracle.roundtrip(v, src_h, v, want, oracle.grid_coords(v))
    assert_bytes_equal(got, want, f"host round trip {name}")


def test_host_round_trip_full_size(atb, c5_input):
    torch = torch_cuda()
    w = datagen.C5B
    src_pin = torch.from_numpy(c5_input).pin_memory()
    dst_pin = torch.zeros(w.storage_bytes, dtype=torch.uint8).pin_memory()
    d_src, d_dst = dev_empty(w.storage_bytes), dev_empty(w.storage_bytes)
    ms, md = encode(atb, w, d_src), encode(atb, w, d_dst)
    atb.tile_roundtrip_host(ms, md, src_pin, dst_pin)
    torch.cuda.synchronize()
    device_ok(atb)
    # the oracle's full-grid round trip reproduces its input (pinned on the CPU)
    assert_bytes_equal(dst_pin.numpy(), c5_input, "host round trip 512 MiB", view=oracle_view(w))


# --------------------------------------------------------------------------
# traversal steps (elementStrides): every e-th element along outer dimensions
# --------------------------------------------------------------------------
STEP_CASES = [
    # name, dtype, dims, box, swizzle, steps
    ("f16_2d_step2", "f16", (300, 90), (64, 16), "none", (1, 2)),
    ("f32_2d_step3_sw128", "f32", (200, 77), (32, 10), "128B", (1, 3)),
    ("u8_3d_steps_sw64", "u8", (256, 20, 15), (64, 6, 4), "64B", (1, 2, 4)),
    ("bf16_4d_step8", "bf16", (64, 5, 33, 3), (32, 2, 16, 2), "64B", (1, 1, 8, 2)),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_traversal_steps_all_ops(atb, case):
    name, dtype, dims, box, swizzle, steps = case
    esize = datagen.ESIZE[dtype]
    strides, nbytes = _strides(esize, dims)
    v = oracle.View(esize, dims, strides, box, swizzle, steps)
    src_h = datagen.random_bytes(nbytes, 900 + len(name))
    coords_h = datagen.random_box_origins(dims, box, esize, 61, 901)
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled(dtype, src, dims, strides, box, swizzle, elem_strides=steps)
    bb = atb.box_bytes(ms)
    assert bb == oracle.box_bytes(v)
    n = len(coords_h)
    guard = 4096  # bytes past the packed images and past the tensor must survive
    packed = dev_empty(n * bb + guard, fill=0xEE)
    atb.tile_load(ms, coords, n, packed)
    device_ok(atb)
    want_packed = oracle.tile_load(v, src_h, coords_h)
    got = host(packed)
    assert_bytes_equal(got, want_packed, f"{name} load", image_bytes=bb)
    assert (got[n * bb:] == 0xEE).all(), f"{name} load wrote past the packed buffer"

    grid_h = oracle.grid_coords(v)
    images_h = datagen.random_bytes(len(grid_h) * bb, 902)
    out = dev_empty(nbytes + guard, fill=0x5A)
    md = atb.encode_tiled(dtype, out, dims, strides, box, swizzle, elem_strides=steps)
    atb.tile_store(md, None, 0, dev_bytes(images_h))
    device_ok(atb)
    want = np.full(nbytes + guard, 0x5A, dtype=np.uint8)
    oracle.tile_store(v, want, grid_h, images_h)
    assert_bytes_equal(host(out), want, f"{name} grid store")

    out2 = dev_empty(nbytes + guard, fill=0x33)
    md2 = atb.encode_tiled(dtype, out2, dims, strides, box, swizzle, elem_strides=steps)
    atb.tile_roundtrip(ms, md2, coords, n)
    device_ok(atb)
    want2 = np.full(nbytes + guard, 0x33, dtype=np.uint8)
    oracle.roundtrip(v, src_h, v, want2, coords_h)
    assert_bytes_equal(host(out2), want2, f"{name} listed round trip")


def test_tensor_larger_than_4gib(atb):
    # fp16 36864 x 65536 (4.5 GiB): 64-bit offsets end to end; every byte by the
    # round-trip property (the oracle's full-grid round trip is the identity, pinned
    # on the CPU), 48 sampled boxes by the oracle itself
    torch = torch_cuda()
    rows, cols = 36864, 65536
    nbytes = rows * cols * 2
    v = oracle.View(2, (cols, rows), (2, cols * 2), (64, 128), "128B")
    src_h = datagen.random_bytes(nbytes, 4096)
    src, dst = dev_bytes(src_h), dev_empty(nbytes, fill=0)
    ms = atb.encode_tiled("f16", src, v.dims, v.strides, v.box, "128B")
    md = atb.encode_tiled("f16", dst, v.dims, v.strides, v.box, "128B")
    atb.tile_roundtrip(ms, md)
    device_ok(atb)
    assert torch.equal(src, dst)
    dst_h = host(dst)
    g = datagen.rng(4097)
    sample = np.stack([g.integers(0, cols // 64, 48) * 64, g.integers(0, rows // 128, 48) * 128], 1).astype(np.int32)
    sample[-1] = (cols - 64, rows - 128)  # the box with the largest offsets
    assert_bytes_equal(oracle.tile_load(v, dst_h, sample), oracle.tile_load(v, src_h, sample), "4.5 GiB sampled",
                       image_bytes=oracle.box_bytes(v))



def test_two_million_small_boxes(atb):
    # many boxes in one call: 2^21 listed 16-byte boxes (list indices past 2^20)
    n = 1 << 21
    dims = (4096, 1024)
    v = oracle.View(1, dims, (1, 4096), (16, 1))
    src_h = datagen.random_bytes(4096 * 1024, 777)
    g = datagen.rng(778)
    coords_h = np.stack([g.integers(-1, 257, n) * 16, g.integers(-1, 1025, n)], 1).astype(np.int32)
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled("u8", src, dims, v.strides, v.box)
    packed = dev_empty(n * 16, fill=0xEE)
    atb.tile_load(ms, coords, n, packed)
    device_ok(atb)
    assert_bytes_equal(host(packed), oracle.tile_load(v, src_h, coords_h), "2M boxes", image_bytes=16)


def test_sixteen_stages_and_single_cta(atb):
    w = datagen.C2
    src_h = datagen.storage(w, seed=16)
    src, dst = dev_bytes(src_h), dev_empty(w.storage_bytes, fill=0)
    m16 = atb.encode_tiled("f16", src, (1792, 8448), (2, 3584), (64, 32))  # 4 KiB boxes
    d16 = atb.encode_tiled("f16", dst, (1792, 8448), (2, 3584), (64, 32))
    atb.tile_roundtrip(m16, d16, stages=16, ctas=1, store_groups=8)
    device_ok(atb)
    assert_bytes_equal(host(dst), src_h, "16 stages, one CTA")


# --------------------------------------------------------------------------
# CUDA graphs: the calls capture into a graph and replay exactly
# --------------------------------------------------------------------------
def test_cuda_graph_capture_and_replay(atb):
    torch = torch_cuda()
    w = datagen.C3
    v = oracle_view(w)
    src_h = datagen.storage(w)
    src = dev_bytes(src_h)
    ms = encode(atb, w, src)
    n = atb.grid_tiles(ms)
    bb = atb.box_bytes(ms)
    packed = dev_empty(n * bb, fill=0)
    out = dev_empty(w.storage_bytes, fill=0)
    md = encode(atb, w, out)
    atb.init_device()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first calls outside the capture (per-kernel set-up)
        atb.tile_load(ms, None, 0, packed)
        atb.tile_store(md, None, 0, packed)
        atb.tile_roundtrip(ms, md)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        atb.tile_load(ms, None, 0, packed)   # grid gather into packed images
        atb.tile_store(md, None, 0, packed)  # and back into the second tensor
        atb.tile_roundtrip(ms, md)           # then a direct round trip over it
    # the fp32 update, captured on its own: 256x256 fp32, sixteen 64x64 tiles, +1.0f
    v32 = oracle.View(4, (256, 256), (4, 1024), (64, 64))
    a32, b32 = dev_empty(256 * 1024), dev_empty(256 * 1024, fill=0)
    m_a = atb.encode_tiled("f32", a32, v32.dims, v32.strides, v32.box)
    m_b = atb.encode_tiled("f32", b32, v32.dims, v32.strides, v32.box)
    with torch.cuda.stream(s):
        atb.tile_roundtrip_add_f32(m_a, m_b, 1.0)
    s.synchronize()
    g32 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g32, stream=s):
        atb.tile_roundtrip_add_f32(m_a, m_b, 1.0)
    h32 = datagen.finite_f32_bytes(256 * 256, 33)
    a32.copy_(torch.from_numpy(h32))
    torch.cuda.synchronize()
    g32.replay()
    torch.cuda.synchronize()
    want32 = np.zeros_like(h32)
    oracle.roundtrip_add_f32(v32, h32, v32, want32, oracle.grid_coords(v32), 1.0)
    assert_bytes_equal(host(b32), want32, "graph fp32 update")

    for seed in (31, 32):
        new_h = datagen.storage(w, seed=seed)
        src.copy_(torch.from_numpy(new_h))
        out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        device_ok(atb)
        assert_bytes_equal(host(packed), oracle.tile_load(v, new_h, oracle.grid_coords(v)), f"graph gather {seed}",
                           image_bytes=bb)
        want = np.zeros_like(new_h)
        oracle.roundtrip(v, new_h, v, want, oracle.grid_coords(v))
        assert_bytes_equal(host(out), want, f"graph round trip {seed}")


# --------------------------------------------------------------------------
# NaN out-of-bounds fill: in-bounds bytes exact, every filled element a NaN
# --------------------------------------------------------------------------
def _is_nan_bits(img: np.ndarray, dtype: str) -> np.ndarray:
    """Per element of the images: is it a NaN of ``dtype`` (by its bit fields)."""
    if dtype in ("f16", "bf16"):
        x = img.view(np.uint16)
        exp, man = (0x7C00, 0x03FF) if dtype == "f16" else (0x7F80, 0x007F)
    elif dtype == "f32":
        x, exp, man = img.view(np.uint32), 0x7F800000, 0x007FFFFF
    else:
        x, exp, man = img.view(np.uint64), 0x7FF0000000000000, 0x000FFFFFFFFFFFFF
    return ((x & x.dtype.type(exp)) == exp) & ((x & x.dtype.type(man)) != 0)


def _check_nan_fill(got: np.ndarray, v: oracle.View, src_h, coords_h, dtype, what):
    want = oracle.tile_load(v, src_h, coords_h)  # zero fill: right wherever the mask is 0
    mask = oracle.tile_oob_mask(v, coords_h)
    got = got[: want.size]
    inside = mask == 0
    bad = np.flatnonzero(got[inside] != want[inside])
    assert bad.size == 0, f"{what}: {bad.size} in-bounds bytes differ"
    elem_out = mask.reshape(-1, v.esize)[:, 0] == 1
    assert elem_out.any(), f"{what}: the case has no out-of-bounds element"
    nan = _is_nan_bits(got, dtype)
    assert nan[elem_out].all(), f"{what}: {int((~nan[elem_out]).sum())} filled elements are not NaN"


NAN_CASES = [c for c in SMALL if c[1] in ("f16", "bf16", "f32", "f64")]


@pytest.mark.parametrize("case", NAN_CASES, ids=[c[0] for c in NAN_CASES])
def test_nan_fill_gather_and_round_trip(atb, case):
    name, dtype, dims, box, swizzle, order = case
    v, src_h, nbytes, coords_h = _small_case(name, dtype, dims, box, swizzle, order, 3000 + len(name))
    launch = dict(stages=1) if box == (256, 256) else {}
    src = dev_bytes(src_h)
    coords = dev_bytes(coords_h.view(np.uint8))
    ms = atb.encode_tiled(dtype, src, dims, v.strides, box, swizzle, oob_fill="nan")
    bb = atb.box_bytes(ms)
    n = coords_h.shape[0]

    packed = dev_empty(n * bb, fill=0)
    atb.tile_load(ms, coords, n, packed, **launch)
    device_ok(atb)
    _check_nan_fill(host(packed), v, src_h, coords_h, dtype, f"{name} listed gather")

    grid_h = oracle.grid_coords(v)
    packed_g = dev_empty(len(grid_h) * bb, fill=0)
    atb.tile_load(ms, None, 0, packed_g, **launch)
    device_ok(atb)
    if (oracle.tile_oob_mask(v, grid_h) == 1).any():
        _check_nan_fill(host(packed_g), v, src_h, grid_h, dtype, f"{name} grid gather")
    else:
        assert_bytes_equal(host(packed_g), oracle.tile_load(v, src_h, grid_h), f"{name} grid gather")

    # a store never writes outside the tensor, so the fill cannot reach the output
    out = dev_empty(nbytes, fill=0x33)
    md = atb.encode_tiled(dtype, out, dims, v.strides, box, swizzle, oob_fill="nan")
    atb.tile_roundtrip(ms, md, coords, n, **launch)
    device_ok(atb)
    want = np.full(nbytes, 0x33, dtype=np.uint8)
    oracle.roundtrip(v, src_h, v, want, coords_h)
    assert_bytes_equal(host(out), want, f"{name} round trip")


def test_nan_fill_workload3_edges_and_steps(atb):
    # ragged 10000 x 3000 bf16, 128-byte swizzle: NaN exactly where the edge boxes overhang
    w = datagen.C3
    v = oracle_view(w)
    src_h = datagen.storage(w)
    src = dev_bytes(src_h)
    ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle, oob_fill="nan")
    grid_h = oracle.grid_coords(v)
    packed = dev_empty(len(grid_h) * atb.box_bytes(ms), fill=0)
    atb.tile_load(ms, None, 0, packed)
    device_ok(atb)
    _check_nan_fill(host(packed), v, src_h, grid_h, "bf16", "workload 3 grid gather")

    # traversal steps with the NaN fill: f32, step 3 along rows
    dims, box, steps = (200, 77), (32, 10), (1, 3)
    strides, nbytes = _strides(4, dims)
    vs = oracle.View(4, dims, strides, box, "128B", steps)
    s_h = datagen.random_bytes(nbytes, 3100)
    c_h = datagen.random_box_origins(dims, box, 4, 80, 3101)
    s_d = dev_bytes(s_h)  # keep the source alive while the map is in use
    m = atb.encode_tiled("f32", s_d, dims, strides, box, "128B", elem_strides=steps, oob_fill="nan")
    p = dev_empty(len(c_h) * atb.box_bytes(m), fill=0)
    atb.tile_load(m, dev_bytes(c_h.view(np.uint8)), len(c_h), p)
    device_ok(atb)
    _check_nan_fill(host(p), vs, s_h, c_h, "f32", "stepped gather")


def test_nan_fill_fp32_update_matches_zero_fill(atb):
    # the +1.0f update sees NaN + 1 in the overhang, which the clipped store drops
    dims, box = (300, 70), (32, 16)
    strides, nbytes = _strides(4, dims)
    v = oracle.View(4, dims, strides, box, "128B")
    src_h = datagen.finite_f32_bytes(nbytes // 4, 3200)
    coords_h = datagen.random_box_origins(dims, box, 4, 120, 3201)
    src = dev_bytes(src_h)  # keep the source alive while the map is in use
    ms = atb.encode_tiled("f32", src, dims, strides, box, "128B", oob_fill="nan")
    out = dev_empty(nbytes, fill=0x44)
    md = atb.encode_tiled("f32", out, dims, strides, box, "128B", oob_fill="nan")
    atb.tile_roundtrip_add_f32(ms, md, 1.0, dev_bytes(coords_h.view(np.uint8)), len(coords_h))
    device_ok(atb)
    want = np.full(nbytes, 0x44, dtype=np.uint8)
    oracle.roundtrip_add_f32(v, src_h, v, want, coords_h, 1.0)
    assert_bytes_equal(host(out), want, "fp32 update with NaN fill")


# --------------------------------------------------------------------------
# ordering: dependent calls back to back, and independent calls on several streams
# --------------------------------------------------------------------------
def _c4_finite():
    """Workload 4's permuted fp32 view over finite values (the fp32 update is
    compared bit for bit, which NaN payloads would not allow)."""
    w = datagen.C4
    return w, oracle_view(w), datagen.finite_f32_bytes(w.storage_bytes // 4, 4400)


def test_dependent_calls_back_to_back_without_host_sync(atb):
    # each call reads what the previous one wrote; the kernels overlap their
    # set-up with the previous grid (programmatic dependent launch) and must
    # still see its writes
    torch = torch_cuda()
    w, v, src_h = _c4_finite()
    coords_h = datagen.workload_coords(w)
    n = len(coords_h)
    src, coords = dev_bytes(src_h), dev_bytes(coords_h.view(np.uint8))
    packed = dev_empty(n * 8192, fill=0)
    fresh = dev_empty(w.storage_bytes, fill=0x3F)  # 0x3F3F3F3F is a finite fp32
    out2 = dev_empty(w.storage_bytes, fill=0)
    out3 = dev_empty(w.storage_bytes, fill=0)
    packed2 = dev_empty(n * 8192, fill=0)
    m_src, m_fresh, m_out2, m_out3 = (encode(atb, w, t) for t in (src, fresh, out2, out3))
    torch.cuda.synchronize()
    atb.tile_load(m_src, coords, n, packed)                    # 1 gather
    atb.tile_store(m_fresh, coords, n, packed)                 # 2 reads 1
    atb.tile_roundtrip(m_fresh, m_out2)                        # 3 reads 2 (whole grid)
    atb.tile_roundtrip_add_f32(m_out2, m_out3, 1.0)            # 4 reads 3
    atb.tile_load(m_out3, coords, n, packed2, stages=2)        # 5 reads 4
    device_ok(atb)

    want_packed = oracle.tile_load(v, src_h, coords_h)
    want_fresh = np.full(w.storage_bytes, 0x3F, dtype=np.uint8)
    oracle.tile_store(v, want_fresh, coords_h, want_packed)
    grid = oracle.grid_coords(v)
    want2 = np.zeros(w.storage_bytes, dtype=np.uint8)
    oracle.roundtrip(v, want_fresh, v, want2, grid)
    want3 = np.zeros(w.storage_bytes, dtype=np.uint8)
    oracle.roundtrip_add_f32(v, want2, v, want3, grid, 1.0)
    assert_bytes_equal(host(fresh), want_fresh, "step 2 store")
    assert_bytes_equal(host(out3), want3, "step 4 fp32 update")
    assert_bytes_equal(host(packed2), oracle.tile_load(v, want3, coords_h), "step 5 gather", image_bytes=8192)


def test_independent_calls_on_four_streams(atb):
    torch = torch_cuda()
    w2, w3 = datagen.C2, datagen.C3
    s2_h, s3_h = datagen.storage(w2, seed=4501), datagen.storage(w3, seed=4502)
    w4, v4, s4_h = _c4_finite()
    c4_h = datagen.workload_coords(w4)
    src2, dst2 = dev_bytes(s2_h), dev_empty(w2.storage_bytes, fill=0)
    src3 = dev_bytes(s3_h)
    packed3 = dev_empty(3713 * 16384, fill=0)
    src4, c4 = dev_bytes(s4_h), dev_bytes(c4_h.view(np.uint8))
    packed4 = dev_empty(len(c4_h) * 8192, fill=0)
    out4 = dev_empty(w4.storage_bytes, fill=0x3F)
    upd = dev_empty(w4.storage_bytes, fill=0)
    maps = dict(s2=encode(atb, w2, src2), d2=encode(atb, w2, dst2), s3=encode(atb, w3, src3),
                s4=encode(atb, w4, src4), o4=encode(atb, w4, out4), u=encode(atb, w4, upd))
    streams = [torch.cuda.Stream() for _ in range(4)]
    torch.cuda.synchronize()
    atb.tile_roundtrip(maps["s2"], maps["d2"], stream=streams[0])
    atb.tile_load(maps["s3"], None, 0, packed3, stream=streams[1])
    atb.tile_load(maps["s4"], c4, len(c4_h), packed4, stream=streams[2])
    atb.tile_store(maps["o4"], c4, len(c4_h), packed4, stream=streams[2])
    atb.tile_roundtrip_add_f32(maps["s4"], maps["u"], -2.5, stream=streams[3])
    torch.cuda.synchronize()
    device_ok(atb)

    assert_bytes_equal(host(dst2), s2_h, "stream 1 round trip")
    v3 = oracle_view(w3)
    assert_bytes_equal(host(packed3), oracle.tile_load(v3, s3_h, oracle.grid_coords(v3)), "stream 2 gather",
                       image_bytes=16384)
    want_p4 = oracle.tile_load(v4, s4_h, c4_h)
    want_o4 = np.full(w4.storage_bytes, 0x3F, dtype=np.uint8)
    oracle.tile_store(v4, want_o4, c4_h, want_p4)
    assert_bytes_equal(host(out4), want_o4, "stream 3 gather then store")
    want_u = np.zeros(w4.storage_bytes, dtype=np.uint8)
    oracle.roundtrip_add_f32(v4, s4_h, v4, want_u, oracle.grid_coords(v4), -2.5)
    assert_bytes_equal(host(upd), want_u, "stream 4 fp32 update")


# --------------------------------------------------------------------------
# round trips between different views: the maps share box, element size and
# swizzle, while extents, strides and dimension order differ
# --------------------------------------------------------------------------
VIEW_PAIRS = [
    # name, dtype, src dims, dst dims, box, swizzle, src outer order, dst outer order
    ("f16_into_smaller", "f16", (300, 77), (200, 50), (64, 16), "none", None, None),
    ("bf16_into_larger_sw128", "bf16", (130, 40), (260, 90), (64, 8), "128B", None, None),
    ("f32_3d_permuted_dst", "f32", (64, 20, 7), (40, 9, 11), (16, 8, 3), "64B", None, [2, 1]),
    ("u8_ragged_rows", "u8", (333, 41), (201, 29), (32, 8), "32B", None, None),
]


@pytest.mark.parametrize("case", VIEW_PAIRS, ids=[c[0] for c in VIEW_PAIRS])
@pytest.mark.parametrize("listed", [False, True], ids=["grid", "listed"])
def test_round_trip_between_different_views(atb, case, listed):
    name, dtype, sdims, ddims, box, swizzle, sorder, dorder = case
    esize = datagen.ESIZE[dtype]
    sstr, sbytes = _strides(esize, sdims, order=sorder)
    dstr, dbytes = _strides(esize, ddims, pitch_pad=48, order=dorder)
    vs = oracle.View(esize, sdims, sstr, box, swizzle)
    vd = oracle.View(esize, ddims, dstr, box, swizzle)
    src_h = datagen.random_bytes(sbytes, 5000 + len(name))
    src = dev_bytes(src_h)
    guard = 4096
    out = dev_empty(dbytes + guard, fill=0x6C)
    ms = atb.encode_tiled(dtype, src, sdims, sstr, box, swizzle)
    md = atb.encode_tiled(dtype, out, ddims, dstr, box, swizzle)
    if listed:
        coords_h = datagen.random_box_origins(sdims, box, esize, 150, 5100 + len(name))
        coords = dev_bytes(coords_h.view(np.uint8))
        atb.tile_roundtrip(ms, md, coords, len(coords_h))
    else:
        coords_h = oracle.grid_coords(vs)
        atb.tile_roundtrip(ms, md)
    device_ok(atb)
    want = np.full(dbytes + guard, 0x6C, dtype=np.uint8)
    oracle.roundtrip(vs, src_h, vd, want, coords_h)
    assert_bytes_equal(host(out), want, f"{name} {'listed' if listed else 'grid'} round trip")

    # the same move as two calls: gather from one view, store the images into the other
    out2 = dev_empty(dbytes + guard, fill=0x6C)
    md2 = atb.encode_tiled(dtype, out2, ddims, dstr, box, swizzle)
    bb = atb.box_bytes(ms)
    packed = dev_empty(len(coords_h) * bb, fill=0)
    c_dev = dev_bytes(np.ascontiguousarray(coords_h, dtype=np.int32).view(np.uint8))
    atb.tile_load(ms, c_dev, len(coords_h), packed)
    atb.tile_store(md2, c_dev, len(coords_h), packed)
    device_ok(atb)
    assert_bytes_equal(host(out2), want, f"{name} gather then store")
