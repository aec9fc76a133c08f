"""Seeded fuzz parity: random shapes, dtypes, strides, base offsets, aliasing
and forced paths through softmax_fwd, every result against the oracle.  The
cases are drawn from a fixed seed, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import DeviceCase, compare

pytestmark = pytest.mark.gpu

PATHS = [0, 0, 0, B.PATH_WARP, B.PATH_CTA, B.PATH_CLUSTER, B.PATH_STREAM, B.PATH_STREAM, B.PATH_PACKED,
         B.PATH_GRID]


def draw_cases(n: int, seed: int = 20261202):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        dtype = ["f32", "f16", "bf16"][rng.integers(3)]
        # widths log-uniform over 1 .. 200000, rows so that the case stays small
        cols = int(np.exp(rng.uniform(0, np.log(200000))))
        rows = int(max(1, min(rng.integers(1, 600), 3_000_000 // max(cols, 1))))
        pad = int(rng.choice([0, 0, 1, 3, 8, 13]))
        off = int(rng.integers(0, 8))
        inplace = bool(rng.integers(4) == 0)
        path = int(PATHS[rng.integers(len(PATHS))])
        cases.append((i, dtype, rows, cols, cols + pad, off, inplace, path))
    return cases


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    yield
    B.set_force_path(0)


@pytest.mark.parametrize("case", draw_cases(160), ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}s{c[4]}o{c[5]}"
                         f"{'i' if c[6] else ''}p{c[7]}")
def test_fuzz(case):
    _, dtype, rows, cols, stride, off, inplace, path = case
    x = W.make_random(rows, cols, dtype, seed=rows * 7919 + cols, row_stride=stride, sigma=2.5)
    dc = DeviceCase(x, dtype, in_off=off, out_off=off, inplace=inplace)
    st = dc.run(cols, path=path)
    if path and st == B.ERR_UNSUPPORTED:
        # a forced path that cannot take this shape (cluster: 16-bit rows
        # only; packed: dense narrow rows; warp / block: short rows; grid:
        # out != in and three vectors or more)
        pytest.skip(f"path {path} refuses this shape")
    assert st == B.OK, B.status_string(st)
    assert B.check_device_error() == B.OK
    compare(dc.result(cols), x, dtype, cols)
    if path:
        assert B.last_path() == path
