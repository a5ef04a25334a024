"""Python binding of libatb: tiled tensor movement through the TMA on sm_103a.

Argument marshalling only.  Every step of the data path runs in the CUDA
kernels of ``libatb.so`` (built in-tree by ``_build.build()``); this module
converts Python values to the C ABI declared in ``include/atb.h`` and raises
``AtbError`` on any non-OK status.  It never falls back to another
implementation: importing it without the built library raises ImportError.

Pointers may be given as ints or as any object with ``data_ptr()`` (a torch
tensor); streams as ints (``cudaStream_t`` handles) or objects with a
``cuda_stream`` attribute; ``None`` means torch's current stream when torch is
loaded, else the legacy default stream.
"""
from __future__ import annotations

import ctypes
import os
import sys

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libatb.so")

MAX_RANK = 5

STATUS = [
    "ATB_OK", "ATB_ERR_RANK", "ATB_ERR_BOX_DIM", "ATB_ERR_STRIDE_ALIGN", "ATB_ERR_BASE_ALIGN",
    "ATB_ERR_SMEM_ALIGN", "ATB_ERR_SWIZZLE", "ATB_ERR_SWIZZLE_SPAN", "ATB_ERR_INNER_BYTES", "ATB_ERR_DTYPE",
    "ATB_ERR_DRIVER", "ATB_ERR_UNSUPPORTED_DEVICE", "ATB_ERR_SMEM_BUDGET", "ATB_ERR_ARG", "ATB_ERR_TIMEOUT",
    "ATB_ERR_CUDA", "ATB_ERR_COORD_ALIGN", "ATB_ERR_COORD_RANGE", "ATB_ERR_STRIDE_RANGE", "ATB_ERR_DIM_RANGE",
    "ATB_ERR_RING_CHECK",
]
for _i, _n in enumerate(STATUS):
    globals()[_n] = _i

DTYPES = {"u8": 0, "u16": 1, "u32": 2, "i32": 3, "u64": 4, "i64": 5, "f16": 6, "f32": 7, "f64": 8, "bf16": 9}
SWIZZLES = {"none": 0, "32B": 1, "64B": 2, "128B": 3}
L2_PROMOTIONS = {"none": 0, "64B": 1, "128B": 2, "256B": 3}
OOB_FILLS = {"zero": 0, "nan": 1}
SCHEDULES = {"strided": 0, "contiguous": 1}
CHECK_RING = 1  # atb_launch.checks: stage bookkeeping check


class AtbError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        self.name = STATUS[code] if 0 <= code < len(STATUS) else f"status {code}"
        super().__init__(f"{where}: {self.name}" + (f": {detail}" if detail else ""))


class TensorMap(ctypes.Structure):
    """Mirror of ``atb_tensor_map`` (checked against ``atb_tensor_map_size()``)."""

    _fields_ = [
        ("map", ctypes.c_ubyte * 128),
        ("map_wide", ctypes.c_ubyte * 128),
        ("base", ctypes.c_uint64),
        ("dims", ctypes.c_uint64 * MAX_RANK),
        ("strides", ctypes.c_uint64 * MAX_RANK),
        ("box", ctypes.c_uint32 * MAX_RANK),
        ("elem_strides", ctypes.c_uint32 * MAX_RANK),
        ("rank", ctypes.c_uint32),
        ("esize", ctypes.c_uint32),
        ("dtype", ctypes.c_uint32),
        ("swizzle", ctypes.c_uint32),
        ("l2_promotion", ctypes.c_uint32),
        ("oob_fill", ctypes.c_uint32),
        ("box_bytes", ctypes.c_uint32),
        ("wide_box0", ctypes.c_uint32),
        ("magic", ctypes.c_uint32),
    ]


class Launch(ctypes.Structure):
    """Mirror of ``atb_launch``; zero fields take the library defaults."""

    _fields_ = [
        ("stages", ctypes.c_uint32),
        ("ctas", ctypes.c_uint32),
        ("ctas_per_sm", ctypes.c_uint32),
        ("schedule", ctypes.c_uint32),
        ("store_groups", ctypes.c_uint32),
        ("l2_hints", ctypes.c_uint32),
        ("no_pdl", ctypes.c_uint32),
        ("poll_suspend_ns", ctypes.c_uint32),
        ("prefetch_boxes", ctypes.c_uint32),
        ("checks", ctypes.c_uint32),
        ("consumer", ctypes.c_uint32),
        ("release", ctypes.c_uint32),
    ]


class DeviceReport(ctypes.Structure):
    _fields_ = [
        ("code", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("tile", ctypes.c_int32),
        ("where", ctypes.c_int32),
        ("errors", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32 * 3),
    ]

    def as_dict(self):
        return {"code": self.code, "name": STATUS[self.code] if 0 <= self.code < len(STATUS) else "?",
                "block": self.block, "tile": self.tile, "where": self.where, "errors": self.errors}


class LaunchShape(ctypes.Structure):
    """Mirror of ``atb_launch_shape``."""

    _fields_ = [(name, ctypes.c_uint32) for name in ("consumer", "release", "stages", "store_groups",
                                                     "ctas_per_sm", "ctas", "threads", "smem_bytes", "boxes")]
    _fields_ += [("reserved", ctypes.c_uint32 * 3)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libatb.so is not built ({LIB_PATH} missing); run async_bulk_tensor_gb300._build.build() "
            "or __graft_entry__.build() first -- there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    S, P, U32, U64, SZ = ctypes.c_int, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
    MapP, LaunchP = ctypes.POINTER(TensorMap), ctypes.POINTER(Launch)
    sig = {
        "atb_version": (ctypes.c_int, []),
        "atb_tensor_map_size": (SZ, []),
        "atb_status_string": (ctypes.c_char_p, [S]),
        "atb_last_error": (ctypes.c_char_p, []),
        "atb_encode_tiled": (S, [MapP, S, U32, P, P, P, P, P, S, S, S]),
        "atb_box_bytes": (SZ, [MapP]),
        "atb_grid_tiles": (U64, [MapP]),
        "atb_pipeline_smem_bytes": (S, [MapP, U32, ctypes.POINTER(SZ)]),
        "atb_tile_load": (S, [MapP, P, U64, P, LaunchP, P]),
        "atb_tile_store": (S, [MapP, P, U64, P, LaunchP, P]),
        "atb_tile_roundtrip": (S, [MapP, MapP, P, U64, LaunchP, P]),
        "atb_init_device": (S, []),
        "atb_device_status": (S, [P, ctypes.POINTER(DeviceReport)]),
        "atb_status_block_allocated": (ctypes.c_int, []),
        "atb_last_launch": (S, [ctypes.POINTER(LaunchShape)]),
        "atb_set_wait_timeout_ns": (None, [U64]),
        "atb_selftest_wait_timeout": (S, [U64, P]),
        "atb_tile_roundtrip_noalloc": (S, [MapP, MapP, P, U64, LaunchP, P, ctypes.POINTER(DeviceReport)]),
        "atb_tile_roundtrip_add_f32": (S, [MapP, MapP, P, U64, ctypes.c_float, LaunchP, P]),
        "atb_tile_roundtrip_host": (S, [MapP, MapP, P, P, U32, LaunchP, P]),
        "atb_copy_cpasync": (S, [P, P, SZ, LaunchP, P]),
        "atb_copy_ldst_v4": (S, [P, P, SZ, LaunchP, P]),
        "atb_copy_memcpy": (S, [P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if lib.atb_tensor_map_size() != ctypes.sizeof(TensorMap):
        raise ImportError("atb_tensor_map layout mismatch between libatb.so and the binding")
    return lib


lib = _load()


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError(f"expected a pointer (int) or an object with data_ptr(), got {type(x).__name__}")


ESIZE = {"u8": 1, "u16": 2, "u32": 4, "i32": 4, "u64": 8, "i64": 8, "f16": 2, "f32": 4, "f64": 8, "bf16": 2}


def _bytes_from(x) -> int | None:
    """Bytes a torch tensor can reach from its data pointer to the end of its
    storage, or a numpy array's size; None for a raw pointer."""
    if hasattr(x, "untyped_storage"):
        return int(x.untyped_storage().nbytes()) - int(x.storage_offset()) * int(x.element_size())
    if hasattr(x, "nbytes") and hasattr(x, "ctypes"):
        return int(x.nbytes)
    return None


def _device_ptr(x, need: int, what: str) -> int | None:
    """Device address of ``x`` for a call that touches ``need`` bytes from it.

    A torch tensor must live on a CUDA device and reach at least ``need`` bytes
    from its data pointer; anything else raises AtbError(ATB_ERR_ARG) before the
    library is called, so that a host buffer or a short one never reaches a
    kernel.  Raw integer addresses are passed through unchecked, as in C.
    """
    if x is None or isinstance(x, int):
        return x
    if getattr(x, "is_cuda", None) is False or (hasattr(x, "ctypes") and hasattr(x, "dtype")):
        raise AtbError(ATB_ERR_ARG, what, f"{what} is in host memory; this call needs device memory")  # noqa: F821
    have = _bytes_from(x)
    if have is not None and have < need:
        raise AtbError(ATB_ERR_ARG, what, f"{what} reaches {have} bytes; the call touches {need}")  # noqa: F821
    return _ptr(x)


def _host_ptr(x, need: int, what: str) -> int:
    """Host address of ``x`` (a CPU tensor, a numpy array or an int) for a call
    that touches ``need`` bytes from it; a device tensor or a short buffer
    raises AtbError(ATB_ERR_ARG)."""
    if isinstance(x, int):
        return x
    if getattr(x, "is_cuda", False):
        raise AtbError(ATB_ERR_ARG, what, f"{what} is device memory; this call needs host memory")  # noqa: F821
    have = _bytes_from(x)
    if have is not None and have < need:
        raise AtbError(ATB_ERR_ARG, what, f"{what} reaches {have} bytes; the call touches {need}")  # noqa: F821
    return x.ctypes.data if hasattr(x, "ctypes") and hasattr(x, "dtype") else _ptr(x)


def span_bytes(m: "TensorMap") -> int:
    """Bytes from a map's base to one past its last element."""
    span = int(m.esize)
    for d in range(int(m.rank)):
        span += (int(m.dims[d]) - 1) * (int(m.esize) if d == 0 else int(m.strides[d]))
    return span


def _boxes(m: "TensorMap", coords, n: int) -> int:
    return int(n) if coords is not None else grid_tiles(m)


def _coords_ptr(m: "TensorMap", coords, n: int) -> int | None:
    return _device_ptr(coords, int(n) * int(m.rank) * 4, "coordinate list")


def _stream(s) -> int | None:
    if s is None:
        torch = sys.modules.get("torch")
        if torch is not None and torch.cuda.is_available() and torch.cuda.is_initialized():
            return int(torch.cuda.current_stream().cuda_stream) or None
        return None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream) or None


def _check(code: int, where: str):
    if code != ATB_OK:  # noqa: F821 (defined from STATUS above)
        raise AtbError(code, where, lib.atb_last_error().decode(errors="replace"))


HINT_LOAD_EVICT_FIRST, HINT_STORE_EVICT_FIRST, HINT_STORE_EVICT_LAST = 1, 2, 4


CONSUMERS = {"auto": 0, "drain": 1, "warp": 2}
RELEASES = {"auto": 0, "after_store": 1, "before_store": 2}


def _launch(stages=0, ctas=0, ctas_per_sm=0, schedule="strided", store_groups=0, l2_hints=0, pdl=True,
            poll_suspend_ns=0, prefetch_boxes=0, checks=0, consumer="auto", release="auto") -> Launch:
    """The ``atb_launch`` record of every call's keyword options; 0 / "auto" leave a field to the library.

    stages, ctas, ctas_per_sm, store_groups: the ring's shape (giving any of stages, ctas_per_sm or
    store_groups turns the consumers' own rings off); schedule: "strided" or "contiguous"; l2_hints:
    ATB_HINT_* bits; pdl: programmatic dependent launch; poll_suspend_ns, prefetch_boxes, checks
    (CHECK_RING); consumer: "auto", "drain" or "warp" (tile-grid launches); release: "auto",
    "after_store" or "before_store" (when the consumer frees a stage).
    ``last_launch()`` reports what a call resolved.
    """
    return Launch(stages, ctas, ctas_per_sm, SCHEDULES[schedule] if isinstance(schedule, str) else schedule,
                  store_groups, l2_hints, 0 if pdl else 1, poll_suspend_ns, prefetch_boxes, checks,
                  CONSUMERS[consumer] if isinstance(consumer, str) else consumer,
                  RELEASES[release] if isinstance(release, str) else release)


def version() -> int:
    return lib.atb_version()


def status_string(code: int) -> str:
    return lib.atb_status_string(code).decode()


def encode_tiled(dtype: str, base, dims, strides_bytes, box, swizzle="none", l2_promotion="none",
                 elem_strides=None, oob_fill="zero") -> TensorMap:
    """Encode a tiled tensor map (``atb_encode_tiled``); sequences are innermost first.

    ``strides_bytes`` lists a byte stride per dimension; entry 0 is ignored.
    ``oob_fill`` is "zero" or "nan" (floating-point types only).
    """
    rank = len(dims)
    if not isinstance(base, int) and base is not None and isinstance(dtype, str) and dtype in ESIZE \
            and strides_bytes is not None and len(strides_bytes) == rank and rank >= 1:
        need = ESIZE[dtype] + sum((int(dims[d]) - 1) * (ESIZE[dtype] if d == 0 else int(strides_bytes[d]))
                                  for d in range(rank))
        _device_ptr(base, need, "tensor base")
    m = TensorMap()
    a_dims = (ctypes.c_uint64 * max(rank, 1))(*[int(d) for d in dims])
    a_str = (ctypes.c_uint64 * max(rank, 1))(*[int(s) for s in strides_bytes]) if strides_bytes is not None else None
    a_box = (ctypes.c_uint32 * max(len(box), 1))(*[int(b) for b in box])
    a_es = (ctypes.c_uint32 * rank)(*elem_strides) if elem_strides is not None else None
    code = lib.atb_encode_tiled(ctypes.byref(m), DTYPES[dtype] if isinstance(dtype, str) else dtype, rank,
                                _ptr(base), a_dims, a_str, a_box, a_es,
                                SWIZZLES[swizzle] if isinstance(swizzle, str) else swizzle,
                                L2_PROMOTIONS[l2_promotion] if isinstance(l2_promotion, str) else l2_promotion,
                                OOB_FILLS[oob_fill] if isinstance(oob_fill, str) else oob_fill)
    _check(code, "atb_encode_tiled")
    return m


def box_bytes(m: TensorMap) -> int:
    return int(lib.atb_box_bytes(ctypes.byref(m)))


def grid_tiles(m: TensorMap) -> int:
    return int(lib.atb_grid_tiles(ctypes.byref(m)))


def pipeline_smem_bytes(m: TensorMap, stages: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib.atb_pipeline_smem_bytes(ctypes.byref(m), stages, ctypes.byref(out)), "atb_pipeline_smem_bytes")
    return int(out.value)


def tile_load(src: TensorMap, coords, n: int, packed, stream=None, **launch):
    """``atb_tile_load``: gather boxes into packed images; ``coords=None`` = tile grid."""
    c = _coords_ptr(src, coords, n)
    p = _device_ptr(packed, _boxes(src, coords, n) * box_bytes(src), "packed buffer")
    _check(lib.atb_tile_load(ctypes.byref(src), c, int(n), p, ctypes.byref(_launch(**launch)), _stream(stream)),
           "atb_tile_load")


def tile_store(dst: TensorMap, coords, n: int, packed, stream=None, **launch):
    """``atb_tile_store``: scatter packed images into the tensor; ``coords=None`` = tile grid."""
    c = _coords_ptr(dst, coords, n)
    p = _device_ptr(packed, _boxes(dst, coords, n) * box_bytes(dst), "packed buffer")
    _check(lib.atb_tile_store(ctypes.byref(dst), c, int(n), p, ctypes.byref(_launch(**launch)), _stream(stream)),
           "atb_tile_store")


def tile_roundtrip(src: TensorMap, dst: TensorMap, coords=None, n: int = 0, stream=None, **launch):
    """``atb_tile_roundtrip``: store(dst, coords, load(src, coords)); ``coords=None`` = tile grid."""
    _check(lib.atb_tile_roundtrip(ctypes.byref(src), ctypes.byref(dst), _coords_ptr(src, coords, n), int(n),
                                  ctypes.byref(_launch(**launch)), _stream(stream)), "atb_tile_roundtrip")


def tile_roundtrip_host(src: TensorMap, dst: TensorMap, h_src, h_dst, slabs: int = 0, stream=None, **launch):
    """``atb_tile_roundtrip_host``: host source -> device -> boxes -> device -> host destination.

    ``h_src``/``h_dst`` are host pointers (ints, or CPU tensors / numpy arrays
    via ``data_ptr()``/``ctypes.data``), laid out as the device maps describe.
    """
    hs = _host_ptr(h_src, span_bytes(src), "host source")
    hd = _host_ptr(h_dst, span_bytes(dst), "host destination")
    _check(lib.atb_tile_roundtrip_host(ctypes.byref(src), ctypes.byref(dst), hs, hd, int(slabs),
                                       ctypes.byref(_launch(**launch)), _stream(stream)), "atb_tile_roundtrip_host")


def tile_roundtrip_add_f32(src: TensorMap, dst: TensorMap, addend: float, coords=None, n: int = 0, stream=None,
                           **launch):
    """``atb_tile_roundtrip_add_f32``: store(dst, coords, load(src, coords) + addend) in fp32."""
    _check(lib.atb_tile_roundtrip_add_f32(ctypes.byref(src), ctypes.byref(dst), _coords_ptr(src, coords, n), int(n),
                                          float(addend), ctypes.byref(_launch(**launch)), _stream(stream)),
           "atb_tile_roundtrip_add_f32")


def tile_roundtrip_noalloc(src: TensorMap, dst: TensorMap, coords=None, n: int = 0, stream=None,
                           report: bool = True, **launch) -> DeviceReport | None:
    """``atb_tile_roundtrip_noalloc``: the round trip without any device allocation.

    With ``report=True`` the call waits for the stream and returns the kernel's
    error record (a non-OK record is returned, not raised); with ``report=False``
    it returns None right after the launch.
    """
    rep = DeviceReport() if report else None
    code = lib.atb_tile_roundtrip_noalloc(ctypes.byref(src), ctypes.byref(dst), _coords_ptr(src, coords, n), int(n),
                                          ctypes.byref(_launch(**launch)), _stream(stream),
                                          ctypes.byref(rep) if rep is not None else None)
    if rep is None or code != rep.code:
        _check(code, "atb_tile_roundtrip_noalloc")
    return rep


def init_device():
    _check(lib.atb_init_device(), "atb_init_device")


def last_launch() -> dict:
    """``atb_last_launch``: the shape of this thread's most recent pipeline launch
    (all zero when it launched nothing)."""
    out = LaunchShape()
    _check(lib.atb_last_launch(ctypes.byref(out)), "atb_last_launch")
    d = {name: getattr(out, name) for name, _ in LaunchShape._fields_ if name != "reserved"}
    d["consumer"] = {0: None, 1: "drain", 2: "warp", 3: "warps"}.get(d["consumer"], d["consumer"])
    d["release"] = {0: None, 1: "after_store", 2: "before_store"}.get(d["release"], d["release"])
    return d


def status_block_allocated() -> int:
    """``atb_status_block_allocated``: 1 if this process's library has allocated
    the current device's status block, 0 if not, -1 if no device is readable."""
    return int(lib.atb_status_block_allocated())


def device_status(stream=None) -> DeviceReport:
    """Synchronise, read and reset the device status block; returns the report (no raise)."""
    rep = DeviceReport()
    code = lib.atb_device_status(_stream(stream), ctypes.byref(rep))
    if code == ATB_ERR_CUDA or code == ATB_ERR_UNSUPPORTED_DEVICE:  # noqa: F821
        _check(code, "atb_device_status")
    return rep


def check_device(stream=None):
    """Raise AtbError if a kernel recorded an error since the last check."""
    rep = device_status(stream)
    if rep.code != 0:
        raise AtbError(rep.code, "device", str(rep.as_dict()))


def set_wait_timeout_ns(ns: int):
    lib.atb_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(timeout_ns: int, stream=None):
    _check(lib.atb_selftest_wait_timeout(int(timeout_ns), _stream(stream)), "atb_selftest_wait_timeout")


def copy_cpasync(src, dst, nbytes: int, stream=None, **launch):
    _check(lib.atb_copy_cpasync(_device_ptr(src, int(nbytes), "source"), _device_ptr(dst, int(nbytes), "destination"),
                                int(nbytes), ctypes.byref(_launch(**launch)),
                                _stream(stream)), "atb_copy_cpasync")


def copy_ldst_v4(src, dst, nbytes: int, stream=None, **launch):
    _check(lib.atb_copy_ldst_v4(_device_ptr(src, int(nbytes), "source"), _device_ptr(dst, int(nbytes), "destination"),
                                int(nbytes), ctypes.byref(_launch(**launch)),
                                _stream(stream)), "atb_copy_ldst_v4")


def copy_memcpy(src, dst, nbytes: int, stream=None):
    _check(lib.atb_copy_memcpy(_device_ptr(src, int(nbytes), "source"), _device_ptr(dst, int(nbytes), "destination"),
                               int(nbytes), _stream(stream)), "atb_copy_memcpy")
