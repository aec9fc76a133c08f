"""softmax_fwd_noalloc: the entry point for callers that cannot allocate
device memory (an allocator owned by a host framework, real-time loops,
processes that must not grow their device footprint).  It runs the split
path with its scratch in a fixed array inside the library.  These tests go
through the C ABI and check two calls in a row -- the second one finding the
first one's states still in that array -- element by element against the
double-precision oracle (the parity harness's comparison: same NaN pattern,
absolute tolerance per dtype, fp32 row sums) and against softmax_fwd's output
on the same input within the same tolerance; and that requests larger than
the array are refused before any launch, while a request exactly at the limit
is exact on random rows.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import os
import re

import numpy as np
import pytest
import torch

from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import TOL, compare, decode

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mbrs_softmax.h")
MAX_STATES = int(re.search(r"#define SOFTMAX_NOALLOC_MAX_STATES (\d+)", open(HEADER).read()).group(1))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    torch.cuda.init()
    B.set_force_path(0)


def _device(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int32 if dtype == "f32" else np.int16)).cuda()


def _bits(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)


def _noalloc(d_in_ptr, d_out_ptr, rows, cols, stride, dtype):
    st = B.softmax_fwd_noalloc_ptr(d_in_ptr, d_out_ptr, rows, cols, stride, B.DTYPE_CODES[dtype],
                                   torch.cuda.current_stream().cuda_stream)
    assert st == B.OK, B.status_string(st)
    torch.cuda.synchronize()
    assert B.check_device_error() == B.OK


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("rows,cols", [(3, 70001), (64, 1000), (257, 4103), (1024, 2048)])
def test_two_calls_in_a_row_match_the_oracle(dtype, rows, cols):
    stream = torch.cuda.current_stream().cuda_stream
    code = B.DTYPE_CODES[dtype]
    # two different inputs: the second call runs over the first call's states
    xs = [W.make_random(rows, cols, dtype, seed=s, sigma=3.0) for s in (11, 12)]
    for x in xs:
        d_in = _device(x, dtype)
        ref = torch.empty_like(d_in)
        got = torch.empty_like(d_in)
        _noalloc(d_in.data_ptr(), got.data_ptr(), rows, cols, cols, dtype)
        compare(_bits(got, dtype), x, dtype, cols)
        assert B.softmax_fwd_ptr(d_in.data_ptr(), ref.data_ptr(), rows, cols, cols, code, stream) == B.OK
        torch.cuda.synchronize()
        y_ref, y = decode(_bits(ref, dtype), dtype), decode(_bits(got, dtype), dtype)
        assert np.abs(y - y_ref).max() <= TOL[dtype]


def test_in_place_and_misaligned():
    rows, cols = 33, 5003
    x = W.make_random(rows, cols, "f16", seed=5, sigma=2.0)
    buf = torch.zeros(rows * cols + 3, dtype=torch.int16, device="cuda")
    buf[1:1 + x.size] = _device(x.reshape(-1), "f16")
    ptr = buf.data_ptr() + 2  # one element in: rows are not 16-byte aligned
    _noalloc(ptr, ptr, rows, cols, cols, "f16")
    got = _bits(buf[1:1 + rows * cols], "f16").reshape(rows, cols)
    compare(got, x, "f16", cols)
    assert (_bits(buf[:1], "f16") == 0).all() and (_bits(buf[1 + rows * cols:], "f16") == 0).all()


def test_requests_beyond_the_array_are_refused():
    stream = torch.cuda.current_stream().cuda_stream
    rows = MAX_STATES + 1
    d = torch.zeros(rows * 4, dtype=torch.float32, device="cuda")
    o = torch.full_like(d, 7.0)
    st = B.softmax_fwd_noalloc_ptr(d.data_ptr(), o.data_ptr(), rows, 4, 4, 0, stream)
    assert st == B.ERR_SCRATCH_LIMIT
    assert "scratch" in B.status_string(st)
    torch.cuda.synchronize()
    assert (o == 7.0).all()  # nothing was launched


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_at_the_limit_on_random_rows(dtype):
    # exactly MAX_STATES rows: one state per row fills the whole array, twice
    # in a row on different inputs
    for seed in (21, 22):
        x = W.make_random(MAX_STATES, 37, dtype, seed=seed, sigma=3.0)
        d_in = _device(x, dtype)
        d_out = torch.empty_like(d_in)
        _noalloc(d_in.data_ptr(), d_out.data_ptr(), MAX_STATES, 37, 37, dtype)
        compare(_bits(d_out, dtype), x, dtype, 37)
