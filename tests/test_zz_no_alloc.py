"""The allocation-free round trip (atb_tile_roundtrip_noalloc) against the
regular one (atb_tile_roundtrip).

The regular call lets the library obtain a small status block with cudaMalloc
the first time it runs on a GPU.  Callers that may not allocate device memory
-- work captured into a CUDA graph in global capture mode, servers that hand
all GPU memory to their own pool at start-up, latency-critical threads -- use
the allocation-free call, which keeps that record in a static device array
instead.  These tests check, through the C ABI, that it moves exactly the same
bytes, on two calls in a row, and that each call starts from a clean record.

This file is collected last on purpose: the no-allocation call must work
both in a fresh process (its first call performs the one-time address lookup)
and after every other test has run.  The fresh-process case runs in a child
interpreter whose first library call on the GPU is the allocation-free round
trip; it checks the bytes against the oracle and that the library's status
block was never allocated, and that a second call leaves the device's free
memory unchanged.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import datagen
from gpu_helpers import assert_bytes_equal, dev_bytes, dev_empty, encode, host, torch_cuda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def atb():
    torch_cuda()
    import async_bulk_tensor_gb300 as atb

    return atb


def test_no_alloc_round_trip_matches_regular_call_twice(atb):
    w = datagen.C2
    for call, seed in enumerate((501, 502)):
        src_h = datagen.storage(w, seed=seed)
        src = dev_bytes(src_h)
        out_noalloc = dev_empty(w.storage_bytes, fill=0x11)
        out_regular = dev_empty(w.storage_bytes, fill=0x11)
        ms = encode(atb, w, src)
        rep = atb.tile_roundtrip_noalloc(ms, encode(atb, w, out_noalloc), ctas=w.ctas, schedule=w.schedule)
        assert rep.code == 0 and rep.errors == 0, (call, rep.as_dict())
        atb.tile_roundtrip(ms, encode(atb, w, out_regular), ctas=w.ctas, schedule=w.schedule)
        atb.check_device()
        got = host(out_noalloc)
        assert_bytes_equal(got, host(out_regular), f"call {call}: no-alloc vs regular")
        assert_bytes_equal(got, src_h, f"call {call}: no-alloc vs input")


def test_no_alloc_record_starts_clean_each_call(atb):
    # a listed round trip with one origin beyond +-2^30 records an error; the
    # next call must not see it again
    rows, cols = 64, 128
    src_h = datagen.random_bytes(rows * cols * 2, 503)
    src = dev_bytes(src_h)
    dims, strides, box = (cols, rows), (2, cols * 2), (64, 16)
    ms = atb.encode_tiled("f16", src, dims, strides, box)
    bad = dev_bytes(np.array([[0, 0], [0, (1 << 30) + 16]], dtype=np.int32).view(np.uint8))
    good = dev_bytes(np.array([[0, 0], [64, 16]], dtype=np.int32).view(np.uint8))
    out1 = dev_empty(rows * cols * 2, fill=0)
    rep1 = atb.tile_roundtrip_noalloc(ms, atb.encode_tiled("f16", out1, dims, strides, box), bad, 2, stages=1)
    assert rep1.code == atb.ATB_ERR_COORD_RANGE and rep1.errors == 1 and rep1.tile == 1, rep1.as_dict()
    out2 = dev_empty(rows * cols * 2, fill=0)
    rep2 = atb.tile_roundtrip_noalloc(ms, atb.encode_tiled("f16", out2, dims, strides, box), good, 2, stages=1)
    assert rep2.code == 0 and rep2.errors == 0, rep2.as_dict()
    want = np.zeros(rows * cols * 2, dtype=np.uint8)
    a, b = want.reshape(rows, cols * 2), src_h.reshape(rows, cols * 2)
    a[0:16, 0:128], a[16:32, 128:256] = b[0:16, 0:128], b[16:32, 128:256]
    assert_bytes_equal(host(out2), want, "listed no-alloc round trip")


def test_no_alloc_without_report_returns_after_launch(atb):
    torch = torch_cuda()
    w = datagen.C1
    src_h = datagen.storage(w, seed=504)
    src, dst = dev_bytes(src_h), dev_empty(w.storage_bytes, fill=0)
    assert atb.tile_roundtrip_noalloc(encode(atb, w, src), encode(atb, w, dst), report=False, stages=1) is None
    torch.cuda.synchronize()
    assert_bytes_equal(host(dst), src_h, "no-alloc without report")


FRESH_PROCESS = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import async_bulk_tensor_gb300 as atb
import datagen
import oracle

torch.cuda.set_device(0)
w = datagen.C2
src_h = datagen.storage(w, seed=505)
src = torch.from_numpy(src_h).cuda()
outs = [torch.full((w.storage_bytes,), 0x11, dtype=torch.uint8, device="cuda") for _ in range(2)]
ms = atb.encode_tiled(w.dtype, src, w.dims, w.strides, w.box, w.swizzle)
mds = [atb.encode_tiled(w.dtype, o, w.dims, w.strides, w.box, w.swizzle) for o in outs]
torch.cuda.synchronize()
assert atb.status_block_allocated() == 0, "status block allocated before any launch"
v = oracle.View(w.esize, w.dims, w.strides, w.box, w.swizzle)
want = np.full(w.storage_bytes, 0x11, dtype=np.uint8)
oracle.roundtrip(v, src_h, v, want, oracle.grid_coords(v))
# the library's first call on the GPU is the allocation-free round trip
rep = atb.tile_roundtrip_noalloc(ms, mds[0], ctas=w.ctas, schedule=w.schedule)
assert rep.code == 0 and rep.errors == 0, rep.as_dict()
assert atb.status_block_allocated() == 0, "the first call allocated the status block"
assert np.array_equal(outs[0].cpu().numpy(), want), "first call differs from the oracle"
torch.cuda.synchronize()
free_before = torch.cuda.mem_get_info()[0]
rep = atb.tile_roundtrip_noalloc(ms, mds[1], ctas=w.ctas, schedule=w.schedule)
assert rep.code == 0 and rep.errors == 0, rep.as_dict()
torch.cuda.synchronize()
free_after = torch.cuda.mem_get_info()[0]
assert free_after == free_before, f"free device memory changed by {free_before - free_after} bytes"
assert atb.status_block_allocated() == 0, "the second call allocated the status block"
assert np.array_equal(outs[1].cpu().numpy(), want), "second call differs from the oracle"
print("fresh process ok")
"""


def test_no_alloc_first_call_in_a_fresh_process_allocates_nothing():
    torch_cuda()
    r = subprocess.run([sys.executable, "-c", FRESH_PROCESS, ROOT], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0 and "fresh process ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
