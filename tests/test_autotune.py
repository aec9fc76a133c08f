"""Shape-keyed autotune: the candidate set (host only), every candidate shape
against the oracle, and the tuner's cache and its use by softmax_fwd."""
import numpy as np
import pytest
import torch

from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import DeviceCase, compare, run_and_compare

A_IN, A_OUT = 1 << 24, 1 << 40   # aligned addresses for host-only plans


# -- host only ------------------------------------------------------------------------------

def _paths(cands):
    return {c[0] for c in cands}


def test_candidates_start_with_the_automatic_choice():
    for cols in (5, 1000, 3001, 40000, 300000):
        c = B.tune_candidates(A_IN, A_OUT, 64, cols, cols, "f32")
        assert c[0] == (0, 0, 0, 0) and len(c) == len(set(c))


def test_candidates_follow_the_row_length():
    narrow = B.tune_candidates(A_IN, A_OUT, 64, 1000, 1000, "f32")
    assert _paths(narrow) == {0, B.PATH_WARP, B.PATH_CTA}
    dense = B.tune_candidates(A_IN, A_OUT, 64, 39, 39, "f32")
    assert B.PATH_PACKED in _paths(dense)
    assert B.PATH_PACKED not in _paths(B.tune_candidates(A_IN, A_OUT, 64, 39, 40, "f32"))  # padded
    medium = B.tune_candidates(A_IN, A_OUT, 64, 16384, 16384, "f32")      # 4096 vectors
    assert {B.PATH_CTA, B.PATH_STREAM} <= _paths(medium)
    assert B.PATH_WARP not in _paths(medium)
    assert B.PATH_CLUSTER not in _paths(medium)                          # fp32 slices would spill
    assert B.PATH_CLUSTER in _paths(B.tune_candidates(A_IN, A_OUT, 64, 16384, 16384, "f16"))
    long_ = B.tune_candidates(A_IN, A_OUT, 64, 1 << 20, 1 << 20, "f32")
    assert _paths(long_) == {0, B.PATH_STREAM, B.PATH_GRID}              # nothing else holds the row
    in_place = B.tune_candidates(A_IN, A_IN, 64, 1 << 20, 1 << 20, "f32")
    assert _paths(in_place) == {0, B.PATH_STREAM}                        # the grid path keeps states in out
    bf16 = B.tune_candidates(A_IN, A_OUT, 512, 131072, 131072, "bf16")
    assert (B.PATH_CLUSTER, 256, 8, 0) in bf16                           # register-held slices


@pytest.mark.parametrize("rows,cols,stride,dt,in_off", [(64, 1000, 1000, "f32", 0), (4096, 2048, 2048, "f16", 0),
                                                        (7, 3001, 3001, "bf16", 2), (300, 40000, 40000, "f32", 0),
                                                        (512, 131072, 131072, "bf16", 0), (9, 70001, 70001, "f32", 4)])
def test_every_candidate_can_be_planned(rows, cols, stride, dt, in_off):
    es = W.ELEM_BYTES[dt]
    for shape in B.tune_candidates(A_IN + in_off * es, A_OUT + in_off * es, rows, cols, stride, dt):
        B.set_force_path(*shape)
        try:
            p = B.plan(A_IN + in_off * es, A_OUT + in_off * es, rows, cols, stride, dt, num_sms=152)
        finally:
            B.set_force_path(0)
        if shape[0]:
            assert p["path"] == shape[0]


def test_bad_arguments_and_empty_cache():
    assert B.lib().softmax_tune_candidates(A_IN, A_OUT, 4, 0, 4, 0, 0, None, 0) == -B.ERR_SHAPE
    assert B.lib().softmax_tune_candidates(A_IN, A_OUT, 4, 8, 8, 0, 0, None, -1) == -B.ERR_ARG
    B.autotune_clear()
    assert B.autotune_size() == 0


# -- on the GPU -------------------------------------------------------------------------------

CASES = [(64, 1000, "f32", 0), (300, 2048, "f16", 0), (7, 3001, "bf16", 1), (40, 40000, "f32", 0),
         (24, 70001, "f16", 3), (20, 131072, "bf16", 0), (3000, 39, "f32", 0), (700, 13, "bf16", 1)]


@pytest.fixture()
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    B.autotune_clear()
    yield
    B.autotune_clear()
    B.set_force_path(0)


@pytest.mark.gpu
@pytest.mark.parametrize("rows,cols,dt,in_off", CASES)
def test_every_candidate_shape_matches_the_oracle(cuda_lib, rows, cols, dt, in_off):
    x = W.make_random(rows, cols, dt, seed=rows + cols, sigma=2.0)
    case = DeviceCase(x, dt, in_off=in_off, out_off=in_off)
    shapes = B.tune_candidates(case.in_ptr, case.out_ptr, rows, cols, cols, dt)
    assert len(shapes) > 1
    for shape in shapes:
        res = run_and_compare(x, dt, in_off=in_off, out_off=in_off, path=shape[0], threads=shape[1],
                              vpt=shape[2], group=shape[3])
        if shape[0]:
            assert res["path"] == shape[0]


@pytest.mark.gpu
@pytest.mark.parametrize("rows,cols,dt,in_off", CASES)
def test_autotune_keeps_a_shape_no_slower_than_automatic(cuda_lib, rows, cols, dt, in_off):
    x = W.make_random(rows, cols, dt, seed=3 * rows + cols, sigma=2.0)
    case = DeviceCase(x, dt, in_off=in_off, out_off=in_off)
    code = W.DTYPES.index(dt)
    stream = torch.cuda.current_stream().cuda_stream
    r = B.autotune_ptr(case.in_ptr, case.out_ptr, rows, cols, cols, code, stream, iters=10)
    assert r["candidates"] >= 2 and r["best_us"] <= r["auto_us"]
    assert B.autotune_size() == 1
    # the tuner's own output is a correct softmax
    compare(case.result(cols), x, dt, cols)
    # later calls with the same key take the kept shape and stay exact
    kept = r["plan"]
    p = B.plan(case.in_ptr, case.out_ptr, rows, cols, cols, dt)
    assert (p["path"], p["threads"], p["vpt"], p["group"]) == (kept["path"], kept["threads"], kept["vpt"],
                                                               kept["group"])
    res = run_and_compare(x, dt, in_off=in_off, out_off=in_off)
    assert res["path"] == kept["path"]
    # another key (rows in another power-of-two bucket) is not affected
    off = in_off * W.ELEM_BYTES[dt]
    other = B.plan(A_IN + off, A_OUT + off, rows * 4 + 1, cols, cols, dt)
    B.autotune_clear()
    assert other == B.plan(A_IN + off, A_OUT + off, rows * 4 + 1, cols, cols, dt)


@pytest.mark.gpu
def test_autotune_refuses_in_place(cuda_lib):
    d = torch.zeros(64 * 1000, device="cuda")
    st = B.lib().softmax_autotune(d.data_ptr(), d.data_ptr(), 64, 1000, 1000, 0, 0, 5, None)
    assert st == B.ERR_ARG and B.autotune_size() == 0


@pytest.mark.gpu
@pytest.mark.parametrize("rows", [2, 3])
def test_a_tuned_shape_never_breaks_other_calls_of_its_key(cuda_lib, rows):
    # tuning runs out of place; a few very long rows may keep the grid path,
    # which cannot run in place: in-place calls with the same sizes and
    # phases keep the automatic choice, and a tuned shape that another row
    # count of the same power-of-two bucket cannot take gives way to it
    cols, dt = 400_003, "f32"
    x = W.make_random(rows, cols, dt, seed=rows, sigma=2.0)
    case = DeviceCase(x, dt)
    stream = torch.cuda.current_stream().cuda_stream
    r = B.autotune_ptr(case.in_ptr, case.out_ptr, rows, cols, cols, 0, stream, iters=5)
    assert B.autotune_size() == 1 and r["best_us"] <= r["auto_us"]
    res = run_and_compare(x, dt, inplace=True)
    assert res["path"] == B.PATH_STREAM
    res = run_and_compare(x, dt)
    assert res["path"] == r["plan"]["path"]
    # the planner agrees (host side, same key, in place)
    assert B.plan(case.in_ptr, case.in_ptr, rows, cols, cols, dt)["path"] == B.PATH_STREAM
