"""The README's Python example runs as written and moves the right bytes."""
import os
import re

import numpy as np
import pytest

import datagen  # noqa: F401  (tests directory on the path)
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def readme_example() -> str:
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    return blocks[0]


def test_readme_has_one_python_example():
    code = readme_example()
    assert "encode_tiled" in code and "tile_load" in code and "tile_store" in code


@pytest.mark.gpu
def test_readme_example_runs_and_matches_the_oracle():
    ns = {}
    exec(compile(readme_example(), "README.md", "exec"), ns)
    torch, atb = ns["torch"], ns["atb"]
    torch.cuda.synchronize()
    x, y = ns["x"], ns["y"]
    assert torch.equal(x, y)  # the full-grid round trip, then stores of boxes carrying x's own bytes
    v = oracle.View(2, (16384, 16384), (2, 32768), (64, 128), "128B")
    src_h = x.view(torch.uint8).reshape(-1).cpu().numpy()
    coords_h = ns["coords"].cpu().numpy()
    want = oracle.tile_load(v, src_h, coords_h)
    got = ns["packed"].cpu().numpy()
    np.testing.assert_array_equal(got, want)
    assert atb.device_status().code == 0
