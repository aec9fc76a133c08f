"""softmax_fwd_host: host buffers through the library's chunked copy / softmax /
copy pipeline, against the oracle -- one chunk and many, in place, padded
strides, page-locked and pageable memory, and the stream ordering -- and the
zero-copy mode, in which the kernels work on the host buffers in place."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import TOL, decode

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()


def host_tensor(x: np.ndarray, dtype: str, pinned: bool) -> torch.Tensor:
    bits = torch.from_numpy(np.ascontiguousarray(W.bits_view(x, dtype)).view(np.int32 if dtype == "f32" else np.int16))
    t = bits.view(TORCH[dtype])
    return t.pin_memory() if pinned else t.clone()


def check(y: torch.Tensor, x: np.ndarray, dtype: str, cols: int):
    bits = y.view(torch.int32 if dtype == "f32" else torch.int16).numpy()
    got = decode(bits[:, :cols].view(np.uint32 if dtype == "f32" else np.uint16), dtype)
    ref = oracle.softmax(x, dtype, cols=cols, threads=8)
    assert np.abs(got - ref).max() <= TOL[dtype]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(1, 7), (37, 1000), (4096, 2048), (300, 40000)])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffers(dtype, rows, cols, pinned):
    x = W.make_random(rows, cols, dtype, seed=rows + cols, sigma=2.0)
    h = host_tensor(x, dtype, pinned)
    y = B.softmax_fwd_host(h)
    check(y, x, dtype, cols)


@pytest.mark.parametrize("dtype", DTYPES)
def test_many_chunks_in_place_and_strided(dtype):
    rows, cols, stride = 999, 1001, 1013
    x = W.make_random(rows, cols, dtype, seed=11, row_stride=stride, sigma=2.0)
    h = host_tensor(x, dtype, True)[:, :cols]          # a padded view: row stride 1013
    ws = torch.empty(3 * 40 * stride * 4, dtype=torch.uint8, device="cuda")  # ~40-row chunks: 25 of them
    B.softmax_fwd_host(h, out=h, workspace=ws)          # in place
    check(h, x, dtype, cols)


@pytest.mark.parametrize("dtype", DTYPES)
def test_padding_between_rows_is_not_touched(dtype):
    rows, cols, stride = 500, 300, 307
    x = W.make_random(rows, cols, dtype, seed=12, row_stride=stride)
    full = host_tensor(x, dtype, True)                  # (rows, stride), padding holds the NaN sentinel
    out_full = host_tensor(np.zeros_like(x), dtype, True)
    ws = torch.empty(3 * 64 * stride * 4, dtype=torch.uint8, device="cuda")
    B.softmax_fwd_host(full[:, :cols], out=out_full[:, :cols], workspace=ws)
    check(out_full, x, dtype, cols)
    pad = out_full.view(torch.int32 if dtype == "f32" else torch.int16).numpy()[:, cols:]
    assert (pad == 0).all()


def test_ordered_on_the_callers_stream():
    # a kernel queued on the stream before the call must finish before the
    # copies read the host input, and the copies must land before work queued
    # after the call: fill the input on the device, copy it to host memory on
    # the stream, run the host call on the same stream, read the result there
    s = torch.cuda.Stream()
    rows, cols = 2048, 2048
    g = torch.Generator(device="cuda").manual_seed(3)
    with torch.cuda.stream(s):
        d = torch.randn(rows, cols, generator=g, device="cuda")
        h = torch.empty(rows, cols, pin_memory=True)
        h.copy_(d, non_blocking=True)
        out = torch.empty(rows, cols, pin_memory=True)
        ws = torch.empty(B.host_workspace_bytes(rows, cols, cols, "f32"), dtype=torch.uint8, device="cuda")
        st = B.lib().softmax_fwd_host(h.data_ptr(), out.data_ptr(), rows, cols, cols, 0, ws.data_ptr(),
                                      ws.numel(), s.cuda_stream)
        assert st == B.OK
    s.synchronize()
    ref = torch.softmax(d.double(), dim=1).cpu()
    assert (out.double() - ref).abs().max().item() <= TOL["f32"]


def test_workspace_too_small_is_refused():
    h = torch.zeros(4, 100, pin_memory=True)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    assert B.lib().softmax_fwd_host(h.data_ptr(), h.data_ptr(), 4, 100, 100, 0, ws.data_ptr(), 256, 0) == B.ERR_ARG


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(1, 7), (37, 1000), (4096, 2048), (300, 40000), (512, 131072)])
def test_zero_copy_on_page_locked_memory(dtype, rows, cols):
    if rows * cols > 20_000_000:
        rows = 128
    x = W.make_random(rows, cols, dtype, seed=rows * 3 + cols, sigma=2.0)
    h = host_tensor(x, dtype, True)
    y = B.softmax_fwd_host(h, zero_copy=True)
    check(y, x, dtype, cols)


@pytest.mark.parametrize("dtype", DTYPES)
def test_zero_copy_in_place_strided(dtype):
    rows, cols, stride = 700, 3001, 3009
    x = W.make_random(rows, cols, dtype, seed=13, row_stride=stride, sigma=2.0)
    full = host_tensor(x, dtype, True)
    view = full[:, :cols]
    B.softmax_fwd_host(view, out=view, zero_copy=True)
    check(full, x, dtype, cols)
    pad = full.view(torch.int32 if dtype == "f32" else torch.int16).numpy()[:, cols:]
    want = W.bits_view(np.ascontiguousarray(x), dtype)[:, cols:].view(np.int32 if dtype == "f32" else np.int16)
    assert (pad == want).all()  # the padding columns are never written


def test_zero_copy_on_pageable_memory_runs_or_is_refused():
    # pageable memory: run in place where the device reaches it through the
    # host's page tables (a coherent CPU-GPU link), refused before any launch
    # elsewhere -- either way never a fault
    rows, cols = 300, 5000
    x = W.make_random(rows, cols, "f32", seed=14, sigma=2.0)
    a_in = np.ascontiguousarray(x)
    a_out = np.full_like(a_in, 7.0)
    st = B.lib().softmax_fwd_host(a_in.ctypes.data, a_out.ctypes.data, rows, cols, cols, 0, None, 0,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    if st == B.ERR_ARG:
        assert (a_out == 7.0).all()
    else:
        assert st == B.OK
        ref = oracle.softmax(x, "f32", cols=cols, threads=8)
        assert np.abs(a_out.astype(np.float64) - ref).max() <= TOL["f32"]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("pinned", [True, False])
def test_zero_copy_few_very_long_rows(dtype, pinned):
    # rows * 16 < SMs and 1 MiB rows: the grid path, whose chunk states and
    # block counter live in the host output rows (atomics on host memory where
    # the device performs them natively, else the streaming cluster); pageable
    # memory runs where the device reaches it, else it is refused
    rows, cols = 2, 700_001
    x = W.make_random(rows, cols, dtype, seed=16, sigma=2.0)
    h = host_tensor(x, dtype, pinned)
    out = torch.full_like(h, 3.0)
    st = B.lib().softmax_fwd_host(h.data_ptr(), out.data_ptr(), rows, cols, cols, B.DTYPE_CODES[dtype], None, 0,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    if st == B.ERR_ARG and not pinned:
        assert (out == 3.0).all()
        return
    assert st == B.OK
    assert B.last_path() in (B.PATH_GRID, B.PATH_STREAM)
    assert B.check_device_error() == B.OK
    check(out, x, dtype, cols)


def test_zero_copy_needs_both_ranges_reachable():
    # a device buffer for in and a pinned one for out is fine; a NULL
    # workspace with a non-zero size is an error, as before
    rows, cols = 64, 1000
    x = W.make_random(rows, cols, "f32", seed=15)
    d = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = torch.empty(rows, cols, pin_memory=True)
    st = B.lib().softmax_fwd_host(d.data_ptr(), out.data_ptr(), rows, cols, cols, 0, None, 0,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == B.OK
    torch.cuda.synchronize()
    check(out, x, "f32", cols)
    assert B.lib().softmax_fwd_host(d.data_ptr(), out.data_ptr(), rows, cols, cols, 0, None, 64, None) == B.ERR_NULL
