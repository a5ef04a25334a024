"""C ABI checks that need no GPU: the library loads, exports every function
include/atb.h declares, agrees with the binding on struct layouts, and the
encoder rejects each broken rule with its own status before the driver is
asked ("Day 76: The Tensor Memory Accelerator (TMA)", "Pitfalls": the driver
alone answers every broken rule with one invalid-value code)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "atb.h")


@pytest.fixture(scope="module")
def atb():
    import async_bulk_tensor_gb300 as atb

    return atb


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(atb_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("atb_encode_tiled", "atb_tile_load", "atb_tile_store", "atb_tile_roundtrip",
                     "atb_device_status", "atb_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(atb):
    out = subprocess.run(["nm", "-D", "--defined-only", atb.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT\s+(atb_\w+)", out.stdout))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(atb.lib, n)


def test_struct_layouts(atb):
    assert atb.lib.atb_tensor_map_size() == ctypes.sizeof(atb.TensorMap)
    assert ctypes.sizeof(atb.Launch) == 48
    assert ctypes.sizeof(atb.DeviceReport) == 32
    assert ctypes.sizeof(atb.LaunchShape) == 48


def test_last_launch_is_empty_after_a_refused_call(atb):
    m = atb.TensorMap()  # never encoded: refused before any launch
    with pytest.raises(atb.AtbError):
        atb.tile_roundtrip(m, m)
    shape = atb.last_launch()
    assert shape["consumer"] is None and shape["boxes"] == 0 and shape["ctas"] == 0


def test_status_strings(atb):
    for i, name in enumerate(atb.STATUS):
        assert atb.status_string(i) == name


def _expect(atb, code, **kw):
    args = dict(dtype="f16", base=0x10000, dims=(1024, 64), strides_bytes=(2, 2048), box=(64, 16))
    args.update(kw)
    with pytest.raises(atb.AtbError) as e:
        atb.encode_tiled(**args)
    assert e.value.code == code, str(e.value)
    return str(e.value)


def test_encoder_rules_each_have_their_own_status(atb):
    _expect(atb, atb.ATB_ERR_RANK, dims=(2,) * 6, strides_bytes=(2,) + (16,) * 5, box=(8,) * 6)
    _expect(atb, atb.ATB_ERR_RANK, dims=(), strides_bytes=(), box=())
    _expect(atb, atb.ATB_ERR_DTYPE, dtype=42)
    _expect(atb, atb.ATB_ERR_ARG, base=0)
    assert "0x10008" in _expect(atb, atb.ATB_ERR_BASE_ALIGN, base=0x10008)
    _expect(atb, atb.ATB_ERR_DIM_RANGE, dims=(1024, 0))
    _expect(atb, atb.ATB_ERR_DIM_RANGE, dims=((1 << 32) + 1, 4))
    msg = _expect(atb, atb.ATB_ERR_STRIDE_ALIGN, strides_bytes=(2, 2040))
    assert "strides_bytes[1]" in msg and "2040" in msg
    _expect(atb, atb.ATB_ERR_STRIDE_RANGE, strides_bytes=(2, 1 << 40))
    msg = _expect(atb, atb.ATB_ERR_BOX_DIM, box=(64, 257))
    assert "box[1]" in msg
    _expect(atb, atb.ATB_ERR_BOX_DIM, box=(0, 16))
    _expect(atb, atb.ATB_ERR_INNER_BYTES, box=(12, 16))  # 24 bytes
    _expect(atb, atb.ATB_ERR_SWIZZLE, swizzle=9)
    _expect(atb, atb.ATB_ERR_SWIZZLE_SPAN, box=(32, 16), swizzle="128B")  # 64 bytes != 128
    _expect(atb, atb.ATB_ERR_SWIZZLE_SPAN, box=(64, 16), swizzle="32B")
    _expect(atb, atb.ATB_ERR_ARG, elem_strides=(2, 1))  # no step along the contiguous dimension
    _expect(atb, atb.ATB_ERR_ARG, elem_strides=(1, 9))  # steps are 1..8
    _expect(atb, atb.ATB_ERR_ARG, elem_strides=(1, 0))
    _expect(atb, atb.ATB_ERR_ARG, oob_fill=7)
    for integer in ("u8", "u16", "u32", "i32", "u64", "i64"):  # the NaN fill is for floating-point types
        msg = _expect(atb, atb.ATB_ERR_DTYPE, dtype=integer, box=(64, 16), oob_fill="nan")
        assert "NaN" in msg


def test_valid_map_reaches_the_driver(atb):
    # With no GPU driver the entry point is unavailable; on a GPU the map encodes.
    try:
        m = atb.encode_tiled("f16", 0x10000, (1024, 64), (2, 2048), (64, 16))
        atb.encode_tiled("bf16", 0x10000, (1024, 64), (2, 2048), (64, 16), oob_fill="nan")
    except atb.AtbError as e:
        assert e.code == atb.ATB_ERR_DRIVER
    else:
        assert atb.box_bytes(m) == 64 * 16 * 2


def test_null_maps_are_rejected_without_a_device(atb):
    m = atb.TensorMap()  # never encoded
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(m, m)
    assert e.value.code == atb.ATB_ERR_ARG
    assert atb.box_bytes(m) == 0 and atb.grid_tiles(m) == 0



def test_unknown_launch_options_are_rejected_before_any_device_work(atb):
    # a map record that passes the library's validity check (magic and rank);
    # the launch must refuse the unknown bit before asking for a device
    m = atb.TensorMap()
    m.magic, m.rank, m.esize, m.dtype = 0x31425441, 2, 2, atb.DTYPES["f16"]
    m.base, m.box_bytes = 0x10000, 2048
    for d, (n, b) in enumerate(((1024, 64), (64, 16))):
        m.dims[d], m.box[d], m.elem_strides[d] = n, b, 1
    m.strides[0], m.strides[1] = 2, 2048
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(m, m, checks=2)
    assert e.value.code == atb.ATB_ERR_ARG and "check bits" in str(e.value)
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(m, m, consumer=3)
    assert e.value.code == atb.ATB_ERR_ARG and "consumer" in str(e.value)
    with pytest.raises(atb.AtbError) as e:
        atb.tile_roundtrip(m, m, release=3)
    assert e.value.code == atb.ATB_ERR_ARG and "release" in str(e.value)


class _FakeDeviceTensor:
    """Just enough of a CUDA tensor for the binding's buffer checks (no GPU)."""

    is_cuda = True

    def __init__(self, nbytes, offset=0):
        self._n, self._off = nbytes, offset

    def untyped_storage(self):
        n = self._n

        class _S:
            def nbytes(self):
                return n

        return _S()

    def storage_offset(self):
        return self._off

    def element_size(self):
        return 1

    def data_ptr(self):
        return 0x10000 + self._off


def test_binding_refuses_host_and_short_buffers_before_the_library(atb):
    import numpy as np
    import torch

    m = atb.TensorMap()
    m.magic, m.rank, m.esize, m.dtype = 0x31425441, 2, 2, atb.DTYPES["f16"]
    m.base, m.box_bytes = 0x10000, 2048
    for d, (n, b) in enumerate(((1024, 64), (64, 16))):
        m.dims[d], m.box[d], m.elem_strides[d] = n, b, 1
    m.strides[0], m.strides[1] = 2, 2048
    assert atb.span_bytes(m) == 63 * 2048 + 1024 * 2
    cases = [
        (lambda: atb.tile_load(m, None, 0, torch.empty(1 << 20, dtype=torch.uint8)), "host memory"),
        (lambda: atb.tile_load(m, None, 0, np.empty(1 << 20, dtype=np.uint8)), "host memory"),
        (lambda: atb.tile_load(m, None, 0, _FakeDeviceTensor(64 * 2048 - 1)), "touches 131072"),  # 64 boxes
        (lambda: atb.tile_store(m, _FakeDeviceTensor(8 * 2 * 4 - 4), 8, _FakeDeviceTensor(1 << 20)), "coordinate"),
        (lambda: atb.tile_store(m, _FakeDeviceTensor(64), 8, _FakeDeviceTensor(8 * 2048 - 16, 16)), "packed"),
        (lambda: atb.tile_roundtrip(m, m, torch.zeros(16, dtype=torch.int32), 8), "host memory"),
        (lambda: atb.tile_roundtrip_host(m, m, np.empty(atb.span_bytes(m) - 1, np.uint8),
                                         np.empty(atb.span_bytes(m), np.uint8)), "host source"),
        (lambda: atb.tile_roundtrip_host(m, m, np.empty(atb.span_bytes(m), np.uint8),
                                         _FakeDeviceTensor(1 << 20)), "device memory"),
        (lambda: atb.encode_tiled("f16", torch.empty(4096, dtype=torch.uint8), (1024, 64), (2, 2048), (64, 16)),
         "host memory"),
        (lambda: atb.encode_tiled("f16", _FakeDeviceTensor(atb.span_bytes(m) - 2), (1024, 64), (2, 2048), (64, 16)),
         "tensor base"),
        (lambda: atb.copy_memcpy(_FakeDeviceTensor(100), _FakeDeviceTensor(99), 100), "destination"),
    ]
    for call, text in cases:
        with pytest.raises(atb.AtbError) as e:
            call()
        assert e.value.code == atb.ATB_ERR_ARG and text in str(e.value), str(e.value)
