"""Calls from several host threads at once: each thread has its own stream and
buffers and runs round trips, listed gathers and host round trips.  The
library's lazily initialised state (device table, status block, kernel
attributes, transfer streams) is created under locks; the ctypes calls release
the GIL, so the calls really overlap."""
import threading

import numpy as np
import pytest

import datagen
import oracle
from gpu_helpers import encode, oracle_view, torch_cuda

pytestmark = pytest.mark.gpu


def test_calls_from_four_host_threads():
    torch = torch_cuda()
    import async_bulk_tensor_gb300 as atb

    w = datagen.C2
    v = oracle_view(w)
    inputs = [datagen.storage(w, seed=7000 + i) for i in range(4)]
    coords_h = datagen.random_box_origins(w.dims, w.box, w.esize, 64, 7100)
    want_packed = [oracle.tile_load(v, h, coords_h) for h in inputs]
    errors = []
    start = threading.Barrier(4)

    def work(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                src = torch.from_numpy(inputs[i]).to("cuda")
                dst = torch.zeros(w.storage_bytes, dtype=torch.uint8, device="cuda")
                coords = torch.from_numpy(coords_h.view(np.uint8)).to("cuda")
                packed = torch.zeros(64 * 32768, dtype=torch.uint8, device="cuda")
            src_pin = torch.from_numpy(inputs[i]).pin_memory()
            out_pin = torch.zeros(w.storage_bytes, dtype=torch.uint8).pin_memory()
            s.synchronize()
            start.wait()
            for _ in range(5):
                ms, md = encode(atb, w, src), encode(atb, w, dst)
                atb.tile_roundtrip(ms, md, stream=s)
                atb.tile_load(ms, coords, 64, packed, stream=s)
                atb.tile_roundtrip_host(ms, md, src_pin, out_pin, 4, stream=s)
                s.synchronize()
                if not torch.equal(dst.cpu(), src.cpu()):
                    errors.append(f"thread {i}: round trip differs")
                if not np.array_equal(packed.cpu().numpy(), want_packed[i]):
                    errors.append(f"thread {i}: gather differs")
                if not torch.equal(out_pin, src_pin):
                    errors.append(f"thread {i}: host round trip differs")
                dst.zero_()
                out_pin.zero_()
                s.synchronize()
        except Exception as e:  # reported below, in the test's own thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors[:5]
    torch.cuda.synchronize()
    rep = atb.device_status()
    assert rep.code == 0, rep.as_dict()
