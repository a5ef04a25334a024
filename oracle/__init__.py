"""Plain CPU oracle for tiled tensor movement -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the
``async_bulk_tensor_gb300`` package and its CUDA library) never does, and the
two share no code.  The arithmetic lives in ``oracle.c`` (plain C, one byte at
a time, each function citing the page section it follows); this module only
compiles it with gcc and marshals numpy buffers through ctypes.

Every function here is pinned by tests in ``tests/test_oracle_pins.py``
against facts the pages print and against properties fixed by mathematics
(see that file); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

MAX_RANK = 5
SWIZZLE_BITS = {"none": 0, "32B": 1, "64B": 2, "128B": 3}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no GPU involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC]
        )
        os.replace(tmp, _LIB)
    return _LIB


class _View(ctypes.Structure):
    _fields_ = [
        ("rank", ctypes.c_int32),
        ("esize", ctypes.c_int32),
        ("swizzle_bits", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("dims", ctypes.c_uint64 * MAX_RANK),
        ("strides", ctypes.c_uint64 * MAX_RANK),
        ("box", ctypes.c_uint32 * MAX_RANK),
        ("estr", ctypes.c_uint32 * MAX_RANK),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the mutation tests run the pins against a deliberately
        # broken build of this same source; it is never set otherwise.
        lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        P = ctypes.POINTER(_View)
        u8p = ctypes.c_void_p
        lib.oracle_swizzle.argtypes = [ctypes.c_uint64, ctypes.c_int32]
        lib.oracle_swizzle.restype = ctypes.c_uint64
        lib.oracle_box_bytes.argtypes = [P]
        lib.oracle_box_bytes.restype = ctypes.c_uint64
        lib.oracle_grid_count.argtypes = [P]
        lib.oracle_grid_count.restype = ctypes.c_uint64
        lib.oracle_grid_coords.argtypes = [P, u8p]
        lib.oracle_grid_coords.restype = None
        lib.oracle_tile_load.argtypes = [P, u8p, u8p, ctypes.c_uint64, u8p]
        lib.oracle_tile_load.restype = None
        lib.oracle_tile_oob_mask.argtypes = [P, u8p, ctypes.c_uint64, u8p]
        lib.oracle_tile_oob_mask.restype = None
        lib.oracle_tile_store.argtypes = [P, u8p, u8p, ctypes.c_uint64, u8p]
        lib.oracle_tile_store.restype = None
        lib.oracle_roundtrip.argtypes = [P, u8p, P, u8p, u8p, ctypes.c_uint64]
        lib.oracle_roundtrip.restype = ctypes.c_int32
        lib.oracle_add_f32.argtypes = [u8p, ctypes.c_uint64, ctypes.c_float]
        lib.oracle_add_f32.restype = None
        lib.oracle_roundtrip_add_f32.argtypes = [P, u8p, P, u8p, u8p, ctypes.c_uint64, ctypes.c_float]
        lib.oracle_roundtrip_add_f32.restype = ctypes.c_int32
        _lib = lib
    return _lib


@dataclass
class View:
    """A strided tensor seen through a box, innermost dimension first.

    ``strides`` are byte strides for every dimension; ``strides[0]`` must
    equal ``esize`` (the innermost dimension is contiguous).
    """

    esize: int
    dims: tuple
    strides: tuple
    box: tuple
    swizzle: str = "none"
    estr: tuple | None = None  # traversal steps per dimension (None = all 1)
    rank: int = field(init=False)

    def __post_init__(self):
        self.rank = len(self.dims)
        assert 1 <= self.rank <= MAX_RANK
        assert len(self.strides) == self.rank and len(self.box) == self.rank
        assert self.strides[0] == self.esize
        assert self.estr is None or (len(self.estr) == self.rank and self.estr[0] == 1)
        # The swizzle keeps every 16-byte chunk inside its 128-byte line; an
        # image whose last line holds a number of chunks the XOR does not map
        # onto itself would send chunks past the end of the box.  Such a view
        # has no image of box_bytes bytes, and is refused before any C call.
        bits = SWIZZLE_BITS[self.swizzle]
        visited = self.esize
        for d in range(self.rank):
            e = self.estr[d] if self.estr is not None else 1
            visited *= (int(self.box[d]) + e - 1) // e
        if bits and visited % (16 << bits) != 0:
            raise ValueError(f"a {self.swizzle} swizzle needs box bytes that are a multiple of {16 << bits}, "
                             f"not {visited}")

    def _c(self) -> _View:
        v = _View()
        v.rank = self.rank
        v.esize = self.esize
        v.swizzle_bits = SWIZZLE_BITS[self.swizzle]
        for d in range(self.rank):
            v.dims[d] = int(self.dims[d])
            v.strides[d] = int(self.strides[d])
            v.box[d] = int(self.box[d])
            v.estr[d] = int(self.estr[d]) if self.estr is not None else 1
        return v

    def span_bytes(self) -> int:
        """Bytes from the base to one past the last element of the tensor."""
        return sum((int(n) - 1) * int(s) for n, s in zip(self.dims, self.strides)) + self.esize


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def swizzle(offset: int, mode: str) -> int:
    return int(_load().oracle_swizzle(offset, SWIZZLE_BITS[mode]))


def box_bytes(v: View) -> int:
    return int(_load().oracle_box_bytes(ctypes.byref(v._c())))


def grid_count(v: View) -> int:
    return int(_load().oracle_grid_count(ctypes.byref(v._c())))


def grid_coords(v: View) -> np.ndarray:
    n = grid_count(v)
    out = np.zeros((n, v.rank), dtype=np.int32)
    _load().oracle_grid_coords(ctypes.byref(v._c()), _ptr(out))
    return out


def _check_base(v: View, base: np.ndarray):
    assert base.dtype == np.uint8 and base.ndim == 1
    assert base.nbytes >= v.span_bytes(), "buffer smaller than the view"


def _coords(coords: np.ndarray, v: View) -> np.ndarray:
    c = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, v.rank)
    return c


def tile_load(v: View, base: np.ndarray, coords: np.ndarray) -> np.ndarray:
    """Packed box images (uint8, n * box_bytes) gathered from ``base``."""
    _check_base(v, base)
    c = _coords(coords, v)
    out = np.empty(c.shape[0] * box_bytes(v), dtype=np.uint8)
    if c.shape[0]:
        _load().oracle_tile_load(ctypes.byref(v._c()), _ptr(base), _ptr(c), c.shape[0], _ptr(out))
    return out


def tile_oob_mask(v: View, coords: np.ndarray) -> np.ndarray:
    """Per byte of the packed images of ``tile_load``: 1 where the element lies
    outside the tensor (the bytes a load fills), else 0."""
    c = _coords(coords, v)
    out = np.empty(c.shape[0] * box_bytes(v), dtype=np.uint8)
    if c.shape[0]:
        _load().oracle_tile_oob_mask(ctypes.byref(v._c()), _ptr(c), c.shape[0], _ptr(out))
    return out


def tile_store(v: View, base: np.ndarray, coords: np.ndarray, packed: np.ndarray) -> None:
    """Scatter packed images into ``base`` in place (in-bounds elements only)."""
    _check_base(v, base)
    c = _coords(coords, v)
    assert packed.dtype == np.uint8 and packed.nbytes >= c.shape[0] * box_bytes(v)
    if c.shape[0]:
        _load().oracle_tile_store(ctypes.byref(v._c()), _ptr(base), _ptr(c), c.shape[0], _ptr(np.ascontiguousarray(packed)))


def roundtrip(src: View, src_base: np.ndarray, dst: View, dst_base: np.ndarray, coords: np.ndarray) -> None:
    """``store(dst, coords, load(src, coords))`` applied to ``dst_base`` in place."""
    _check_base(src, src_base)
    _check_base(dst, dst_base)
    c = _coords(coords, src)
    rc = _load().oracle_roundtrip(ctypes.byref(src._c()), _ptr(src_base), ctypes.byref(dst._c()),
                                  _ptr(dst_base), _ptr(c), c.shape[0])
    if rc != 0:
        raise ValueError("oracle roundtrip: box shape, element size or swizzle differ, or out of memory")


def add_f32(packed: np.ndarray, addend: float) -> np.ndarray:
    """Copy of ``packed`` with ``addend`` added to every fp32 element."""
    out = np.array(packed, dtype=np.uint8, copy=True)
    _load().oracle_add_f32(_ptr(out), out.nbytes, float(addend))
    return out


def roundtrip_add_f32(src: View, src_base: np.ndarray, dst: View, dst_base: np.ndarray, coords: np.ndarray,
                      addend: float) -> None:
    """``store(dst, coords, load(src, coords) + addend)`` applied to ``dst_base`` in place."""
    _check_base(src, src_base)
    _check_base(dst, dst_base)
    c = _coords(coords, src)
    rc = _load().oracle_roundtrip_add_f32(ctypes.byref(src._c()), _ptr(src_base), ctypes.byref(dst._c()),
                                          _ptr(dst_base), _ptr(c), c.shape[0], float(addend))
    if rc != 0:
        raise ValueError("oracle fp32 round trip: views differ, element size is not 4, or out of memory")
