"""GPU parity of softmax_fwd_masked (scaled, causally masked rows) against the
oracle's masked softmax: every path it runs (lane groups, blocks, the
streaming cluster), offsets that keep nothing / part / everything, grouped
rows, misaligned rows, in place, and masked inputs that hold NaN (they must
never be read)."""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import TOL, DeviceCase, decode

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    yield
    B.set_force_path(0)


def kept(r, cols, off, period):
    q = r % period if period > 0 else r
    return max(0, min(cols, q + off + 1))


def run_masked(x, dtype, scale, off, period=0, *, path=0, threads=0, vpt=0, group=0, in_off=0, out_off=0,
               inplace=False, poison=False):
    rows, cols = x.shape
    xin = x.copy()
    if poison:  # masked inputs hold NaN: reading any of them would show
        nan = W.quantise(np.asarray([np.nan]), dtype)[0]
        for r in range(rows):
            xin[r, kept(r, cols, off, period):] = nan
    case = DeviceCase(xin, dtype, in_off=in_off, out_off=out_off, inplace=inplace)
    B.set_force_path(path, threads, vpt, group)
    try:
        st = B.softmax_fwd_masked_ptr(case.in_ptr, case.out_ptr, rows, cols, cols, W.DTYPES.index(dtype), scale,
                                      off, period, torch.cuda.current_stream().cuda_stream)
    finally:
        B.set_force_path(0)
    assert st == B.OK, B.status_string(st)
    assert B.check_device_error() == B.OK
    y = decode(case.result(cols), dtype)
    ref = oracle.softmax_masked(x, dtype, scale, off, period, threads=8)
    nan_ref = np.isnan(ref)
    assert (np.isnan(y) == nan_ref).all(), "NaN pattern differs from the oracle"
    fin = ~nan_ref
    err = float(np.abs(y[fin] - ref[fin]).max()) if fin.any() else 0.0
    assert err <= TOL[dtype], f"max abs err {err:.3e} > {TOL[dtype]:.0e} ({dtype})"
    assert (y[fin & (ref == 0)] == 0).all(), "a masked output is not exactly 0"
    return B.last_path()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [1, 7, 33, 100, 1000, 2048, 3001, 20011, 70001])
def test_causal_square_blocks(dtype, cols):
    # the attention shape: rows grouped into sequences of `period` queries
    rows = 96 if cols <= 3001 else 24
    period = min(rows, cols)
    run_masked(W.make_random(rows, cols, dtype, seed=cols, sigma=2.0), dtype, 0.125, cols - period, period)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("off", [-200, -3, 0, 5, 10 ** 12])
def test_offsets(dtype, off):
    x = W.make_random(150, 600, dtype, seed=7, sigma=1.5)
    run_masked(x, dtype, 1.0, off)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("path,cols", [(B.PATH_WARP, 300), (B.PATH_WARP, 1000), (B.PATH_CTA, 1000),
                                       (B.PATH_CTA, 9000), (B.PATH_STREAM, 1000), (B.PATH_STREAM, 40000),
                                       (B.PATH_CLUSTER, 5000)])
def test_forced_paths(dtype, path, cols):
    x = W.make_random(64, cols, dtype, seed=path * 10 + cols, sigma=2.0)
    got = run_masked(x, dtype, 0.7, cols // 2 - 32, 0, path=path)
    want = path if path in (B.PATH_WARP, B.PATH_CTA, B.PATH_STREAM) else B.PATH_STREAM
    assert got == want


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("threads,vpt,group", [(256, 4, 1), (256, 2, 3), (512, 4, 16), (1024, 4, 5)])
def test_stream_shapes(dtype, threads, vpt, group):
    x = W.make_random(20, 50001, dtype, seed=threads + group, sigma=2.0)
    assert run_masked(x, dtype, 0.3, 25000, 0, path=B.PATH_STREAM, threads=threads, vpt=vpt,
                      group=group) == B.PATH_STREAM


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols,path", [(100, 0), (1000, B.PATH_WARP), (3001, 0), (3001, B.PATH_STREAM),
                                       (40000, 0)])
def test_masked_inputs_are_never_read(dtype, cols, path):
    x = W.make_random(48, cols, dtype, seed=cols + 1)
    run_masked(x, dtype, 0.5, cols // 3, 0, path=path, poison=True)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [100, 3001, 40000])
@pytest.mark.parametrize("in_off", [1, 3])
def test_misaligned_and_in_place(dtype, cols, in_off):
    x = W.make_random(40, cols, dtype, seed=cols * in_off)
    run_masked(x, dtype, 2.0, 7, 16, in_off=in_off, out_off=in_off)
    run_masked(x, dtype, 2.0, 7, 16, in_off=in_off, inplace=True)


def test_the_fp16_causal_workload_at_full_size():
    # the fp16 8192 x 4096 workload whose mask is in its data (x = -inf for
    # c > r mod 4096), stride 4104: the masked call reads only the kept half
    # and must give the plain softmax of the same rows
    w = W.CONFIGS["c4"]
    x = W.make_input(w)
    case = DeviceCase(x, w.dtype)
    st = B.softmax_fwd_masked_ptr(case.in_ptr, case.out_ptr, w.rows, w.cols, w.stride, 1, 1.0, 0,
                                  w.causal_period, torch.cuda.current_stream().cuda_stream)
    assert st == B.OK and B.check_device_error() == B.OK
    y = decode(case.result(w.cols), w.dtype)
    rows = list(range(0, w.rows, 97)) + [4095, 4096, w.rows - 1]
    ref = oracle.softmax(x, w.dtype, cols=w.cols, rows=rows, threads=8)
    err = float(np.abs(y[rows] - ref).max())
    assert err <= TOL["f16"]
    print(w.name + "_masked", {"max_abs_err": err, "rows_checked": len(rows)})


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("off,period,threads", [(0, 0, 64), (0, 150, 256), (-3, 100, 0), (5000, 0, 1024),
                                                (-10000, 0, 32), (7, 64, 128)])
def test_masked_copy_moves_the_masked_pattern(dtype, off, period, threads):
    # the diagnostic softmax_masked_copy: kept entries bit for bit, the rest
    # zero bits, padding and guards untouched (rows of whole 16-byte vectors)
    rows, cols, stride = 300, 1024, 1032
    x = W.make_random(rows, cols, dtype, seed=31 + threads, row_stride=stride, sigma=2.0)
    case = DeviceCase(x, dtype)
    st = B.masked_copy_ptr(case.in_ptr, case.out_ptr, rows, cols, stride, W.DTYPES.index(dtype), off, period,
                           threads, torch.cuda.current_stream().cuda_stream)
    assert st == B.OK, B.status_string(st)
    y = case.result(cols)
    xb = W.bits_view(np.ascontiguousarray(x), dtype)[:, :cols]
    keep = np.array([kept(r, cols, off, period) for r in range(rows)])
    live = np.arange(cols)[None, :] < keep[:, None]
    assert (y[live] == xb[live]).all() and (y[~live] == 0).all()


def test_rejects_bad_scale_and_period():
    d = torch.zeros(64, device="cuda")
    p = d.data_ptr()
    for scale in (0.0, -1.0, float("inf"), float("nan")):
        assert B.softmax_fwd_masked_ptr(p, p, 4, 8, 8, 0, scale, 0, 0) == B.ERR_ARG
    assert B.softmax_fwd_masked_ptr(p, p, 4, 8, 8, 0, 1.0, 0, -1) == B.ERR_ARG


@pytest.mark.parametrize("tdtype,name", [(torch.float32, "f32"), (torch.float16, "f16"), (torch.bfloat16, "bf16")])
def test_torch_binding_matches_torch_on_a_masked_score_matrix(tdtype, name):
    # an attention-score matrix: 2 sequences of 300 queries over 300 keys
    g = torch.Generator(device="cpu").manual_seed(5)
    x = (torch.randn(600, 300, generator=g) * 4).to(tdtype).cuda()
    y = B.softmax_fwd_masked(x, scale=0.125, causal_offset=0, rows_per_seq=300)
    q = torch.arange(600).remainder(300)[:, None]
    s = (x.double() * 0.125).masked_fill(torch.arange(300)[None, :].cuda() > q.cuda(), float("-inf"))
    assert (y.double() - torch.softmax(s, dim=1)).abs().max().item() <= TOL[name]
