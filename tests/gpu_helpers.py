"""Helpers shared by the GPU parity tests: device buffers, map encoding from a
workload recipe, and byte comparison that reports the first mismatch the way
"Day 76: The Tensor Memory Accelerator (TMA)" asks for (index, and the element
coordinates, so that a whole wrong tile reads as bad coordinates and scattered
bytes as a race)."""
from __future__ import annotations

import numpy as np

import datagen
import oracle


def torch_cuda():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def dev_bytes(host: np.ndarray):
    torch = torch_cuda()
    t = torch.from_numpy(np.ascontiguousarray(host)).to("cuda")
    assert t.data_ptr() % 256 == 0
    return t


def dev_empty(nbytes: int, fill: int | None = None):
    torch = torch_cuda()
    t = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


def host(t) -> np.ndarray:
    return t.cpu().numpy()


def oracle_view(w: datagen.Workload) -> oracle.View:
    return oracle.View(w.esize, w.dims, w.strides, w.box, w.swizzle)


def encode(atb, w: datagen.Workload, base, l2_promotion="none"):
    return atb.encode_tiled(w.dtype, base, w.dims, w.strides, w.box, w.swizzle, l2_promotion)


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str, view: oracle.View | None = None,
                       image_bytes: int | None = None):
    got = np.asarray(got).reshape(-1)
    want = np.asarray(want).reshape(-1)
    assert got.size >= want.size, f"{what}: {got.size} bytes, expected {want.size}"
    got = got[: want.size]
    if np.array_equal(got, want):
        return
    bad = np.flatnonzero(got != want)
    i = int(bad[0])
    msg = f"{what}: {bad.size} of {want.size} bytes differ; first at byte {i} (got {got[i]}, want {want[i]})"
    if image_bytes:
        msg += f"; packed image {i // image_bytes}, offset {i % image_bytes}"
        msg += f"; images with errors: {np.unique(bad // image_bytes)[:10].tolist()}"
    elif view is not None and view.rank == 2:
        row, col = i // view.strides[1], (i % view.strides[1]) // view.esize
        msg += f"; element row {row}, col {col} (box row {row % view.box[1]}, box col {col % view.box[0]})"
    raise AssertionError(msg)
