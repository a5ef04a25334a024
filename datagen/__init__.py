"""Seeded synthetic inputs and workload recipes for tiled tensor movement.

This module is shared by the tests, the smoke check and the benchmark, and by
both sides of every parity check: it makes input bytes and coordinate lists,
nothing else.  It holds none of the method's arithmetic (no box gather, no
swizzle, no tile enumeration); those live separately in the oracle and in the
CUDA library.

Recipes follow the workloads the pages describe:
  * a single 64x64 fp32 tile (16384 bytes) round trip -- "Day 76: The Tensor
    Memory Accelerator (TMA)", "The address arithmetic moves into a
    descriptor" and "An exact round trip";
  * an fp16 row-major matrix cut into 64x256 boxes, 132 row strips x 7 column
    tiles = 924 boxes -- "Understanding TMA loads in CuTe DSL", "The work
    assigned to each block"; the matrix extents (8448 x 1792) are the plainest
    reading of that decomposition;
  * ragged bf16 and permuted 3-D fp32 tensors with 128-byte swizzle and
    out-of-bounds boxes, and a 512 MiB fp16 bandwidth case, which exercise the
    descriptor rules and zero fill described in "GPU TMA tensor memory
    accelerator", "The architecture: every piece explained".
All values are seeded (numpy PCG64, or torch's CPU generator for the normal draws);
nothing is read from disk.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

ESIZE = {"u8": 1, "f16": 2, "bf16": 2, "f32": 4, "f64": 8}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # element type name (sizes in ESIZE)
    storage_bytes: int         # bytes of the backing allocation
    dims: tuple                # innermost first
    strides: tuple             # byte strides, innermost first (strides[0] == element size)
    box: tuple                 # innermost first
    swizzle: str               # none / 32B / 64B / 128B
    values: str                # bits / uniform_bf16 / normal_f16
    seed: int
    op: str                    # roundtrip / load / load_store
    coords: str = "grid"       # grid / random
    n_random: int = 0
    ctas: int = 0              # 0 = library default
    schedule: str = "strided"  # strided / contiguous
    description: str = ""
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def esize(self) -> int:
        return ESIZE[self.dtype]

    @property
    def rank(self) -> int:
        return len(self.dims)


def _row_major_2d(rows: int, cols: int, esize: int, row_stride_bytes: int | None = None):
    rs = row_stride_bytes if row_stride_bytes is not None else cols * esize
    return (cols, rows), (esize, rs), rs * rows


def _c1():
    dims, strides, nbytes = _row_major_2d(64, 64, 4)
    return Workload("c1_tile64x64_f32", "f32", nbytes, dims, strides, (64, 64), "none", "bits", 1,
                    "roundtrip", description="fp32 64x64 row-major, box 64x64, no swizzle, single-tile round trip")


def _c2():
    dims, strides, nbytes = _row_major_2d(8448, 1792, 2)
    return Workload("c2_f16_8448x1792_box64x256", "f16", nbytes, dims, strides, (256, 64), "none", "bits", 2,
                    "roundtrip", ctas=132, schedule="contiguous",
                    description="fp16 8448x1792, box 64x256, 132 blocks x 7 column tiles, round trip")


def _c3():
    dims, strides, nbytes = _row_major_2d(10000, 3000, 2, 6000)
    return Workload("c3_bf16_10000x3000_box128x64_sw128", "bf16", nbytes, dims, strides, (64, 128), "128B",
                    "uniform_bf16", 3, "load",
                    description="bf16 10000x3000 (row stride 6000 B), box 128x64, 128B swizzle, full grid "
                                "with edge tiles gathered into the packed swizzled buffer")


def _c4():
    # Storage S is a contiguous fp32 [512, 32, 1024] array; the view is
    # S.permute(1, 0, 2), shape [32, 512, 1024], element strides (1024, 32768, 1).
    # Innermost first: dims (1024, 512, 32), byte strides (4, 131072, 4096).
    return Workload("c4_f32_permuted_32x512x1024_gather", "f32", 512 * 32 * 1024 * 4, (1024, 512, 32),
                    (4, 131072, 4096), (32, 64, 1), "128B", "bits", 4, "load_store", coords="random",
                    n_random=4096,
                    description="fp32 [32,512,1024] view with permuted strides, box 1x64x32, 128B swizzle, "
                                "4096 random boxes gathered to packed then stored to a fresh tensor")


def _c5(box: str):
    dims, strides, nbytes = _row_major_2d(16384, 16384, 2)
    if box == "64x256":
        return Workload("c5_f16_16384x16384_box64x256", "f16", nbytes, dims, strides, (256, 64), "none",
                        "normal_f16", 5, "roundtrip",
                        description="fp16 16384x16384 (512 MiB) full round trip, box 64x256, no swizzle")
    return Workload("c5_f16_16384x16384_box128x64_sw128", "f16", nbytes, dims, strides, (64, 128), "128B",
                    "normal_f16", 5, "roundtrip",
                    description="fp16 16384x16384 (512 MiB) full round trip, box 128x64, 128B swizzle")


WORKLOADS = {w.name: w for w in (_c1(), _c2(), _c3(), _c4(), _c5("64x256"), _c5("128x64"))}
C1, C2, C3, C4 = (WORKLOADS[k] for k in list(WORKLOADS)[:4])
C5A = WORKLOADS["c5_f16_16384x16384_box64x256"]
C5B = WORKLOADS["c5_f16_16384x16384_box128x64_sw128"]


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def random_bytes(nbytes: int, seed: int) -> np.ndarray:
    """Uniform random byte patterns (every bit pattern possible, NaNs included).

    Raw 64-bit PCG64 outputs, viewed as little-endian bytes.
    """
    words = rng(seed).bit_generator.random_raw((nbytes + 7) // 8)
    return words.view(np.uint8)[:nbytes].copy()


def uniform_bf16_bytes(n_elems: int, seed: int) -> np.ndarray:
    """uniform[-1, 1) drawn in fp32, rounded to bf16 (nearest even) by torch on the CPU."""
    import torch

    x = rng(seed).random(n_elems, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)
    b = torch.from_numpy(x).to(torch.bfloat16)
    return b.view(torch.uint8).numpy().copy()


def normal_f16_bytes(n_elems: int, seed: int) -> np.ndarray:
    """normal(0, 1) drawn in fp32 by torch's seeded CPU generator, rounded to fp16."""
    import torch

    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n_elems, generator=g, dtype=torch.float32).to(torch.float16)
    return x.view(torch.uint8).numpy()


def finite_f32_bytes(n_elems: int, seed: int) -> np.ndarray:
    """Random fp32 bit patterns with every Inf/NaN pattern made finite
    (exponent 0xFF -> 0x7F); zeros of both signs and denormals are kept."""
    bits = random_bytes(4 * n_elems, seed).view(np.uint32).copy()
    inf_nan = (bits & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
    bits[inf_nan] &= np.uint32(0xBFFFFFFF)
    return bits.view(np.uint8)


def storage(w: Workload, seed: int | None = None) -> np.ndarray:
    """The workload's backing bytes (uint8, ``w.storage_bytes`` long)."""
    s = w.seed if seed is None else seed
    if w.values == "bits":
        return random_bytes(w.storage_bytes, s)
    if w.values == "uniform_bf16":
        return uniform_bf16_bytes(w.storage_bytes // 2, s)
    if w.values == "normal_f16":
        return normal_f16_bytes(w.storage_bytes // 2, s)
    raise ValueError(w.values)


def random_box_origins(dims, box, esize: int, n: int, seed: int, align_bytes: int = 0) -> np.ndarray:
    """``n`` box origins (int32, innermost first), each box touching the tensor.

    Along every dimension the origin is uniform in [-(box-1), dims-1], so about
    a quarter of the boxes hang over an edge.  With ``align_bytes`` > 0 the
    innermost origin is drawn on that grid instead (x * esize a multiple of
    ``align_bytes``); by default every element offset is possible.
    """
    g = rng(seed)
    out = np.empty((n, len(dims)), dtype=np.int32)
    if align_bytes:
        q = max(1, align_bytes // esize)
        lo0 = -((box[0] - 1) // q) * q
        hi0 = ((dims[0] - 1) // q) * q
        out[:, 0] = g.integers(lo0 // q, hi0 // q + 1, size=n) * q
    else:
        out[:, 0] = g.integers(-(box[0] - 1), dims[0], size=n)
    for d in range(1, len(dims)):
        out[:, d] = g.integers(-(box[d] - 1), dims[d], size=n)
    return out


def workload_coords(w: Workload, seed: int | None = None) -> np.ndarray | None:
    """Coordinate list for random-box workloads; None means the full tile grid."""
    if w.coords == "grid":
        return None
    s = (w.seed if seed is None else seed) + 1000
    return random_box_origins(w.dims, w.box, w.esize, w.n_random, s)
