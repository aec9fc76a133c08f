"""The C-ABI library on the host, without a GPU: it loads, exports every
function the header declares, rejects bad arguments before touching CUDA,
and plans launches that cover every row."""
import ctypes
import os
import re

import numpy as np
import pytest

from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_mod.build()
    B.set_force_path(0)
    yield
    B.set_force_path(0)


def declared_functions():
    names = []
    for f in sorted(os.listdir(HEADER_DIR)):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(softmax_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert "softmax_fwd" in names and len(names) >= 8
    lib = ctypes.CDLL(B._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(names) <= set(B.SIGNATURES), "binding lacks a signature for a declared function"


def test_status_strings():
    for s in range(11):
        assert B.status_string(s) and B.status_string(s) != "unknown status"
    assert B.status_string(99) == "unknown status"
    assert B.abi_version() == 20200


@pytest.mark.parametrize("args,expect", [
    ((0, 0, 5, 3, 3, 0), B.ERR_NULL),
    ((0, 0, 0, 3, 3, 0), B.OK),               # rows == 0: nothing to do, nothing launched
    ((0, 0, -1, 3, 3, 0), B.ERR_SHAPE),
    ((0, 0, 5, 0, 3, 0), B.ERR_SHAPE),
    ((0, 0, 5, 3, 2, 0), B.ERR_STRIDE),
    ((0, 0, 5, 3, 3, 7), B.ERR_DTYPE),
    ((0, 0, 5, 3, 3, -1), B.ERR_DTYPE),
    ((4096, 4096 + 40, 5, 3, 3, 0), B.ERR_OVERLAP),
    ((4096, 4096 + 64, 5, 3, 3, 0), B.OK),    # out starts past in's 60-byte extent: planner only
    ((4098, 8192, 5, 3, 3, 0), B.ERR_ALIGN),
    ((4097, 8192, 5, 3, 3, 1), B.ERR_ALIGN),
    ((4096, 8192, 2**62, 3, 2**62, 0), B.ERR_SHAPE),
])
def test_argument_checks(args, expect):
    i, o, rows, cols, stride, dt = args
    if expect == B.OK and rows > 0:
        # a valid call would launch: check the host planner instead of calling
        assert B.plan(i, o, rows, cols, stride, dt, num_sms=152)["path"] > 0
    else:
        assert B.softmax_fwd_ptr(i, o, rows, cols, stride, dt, 0) == expect


def test_in_place_is_allowed():
    assert B.plan(1 << 20, 1 << 20, 7, 100, 100, "f32", num_sms=152)["path"] == B.PATH_WARP


CASES = [(64, 1000, 1000, "f32"), (4096, 2048, 2048, "f16"), (4096, 4096, 4096, "f32"),
         (8192, 4096, 4104, "f16"), (512, 131072, 131072, "bf16"), (1, 1 << 24, 1 << 24, "f32"),
         (1562500, 32, 32, "f32"), (1282051, 39, 39, "f32"), (3050, 16391, 16391, "f32"),
         (3, 5, 5, "bf16"), (2, 524288, 524288, "bf16"), (100, 600000, 600000, "f16")]


@pytest.mark.parametrize("rows,cols,stride,dt", CASES)
@pytest.mark.parametrize("in_off", [0, 4, 12])
def test_plans_cover_every_row(rows, cols, stride, dt, in_off):
    es = 4 if dt == "f32" else 2
    V = 16 // es
    p = B.plan((1 << 24) + in_off, (1 << 40) + in_off, rows, cols, stride, dt, num_sms=152)
    uniform = (stride * es) % 16 == 0
    head = (in_off // es) % V if uniform else V - 1
    nv = -(-(head + cols) // V)
    path = p["path"]
    assert p["vec_store"] == 1
    if path == B.PATH_WARP:
        assert (cols <= 1024 or p["whole_vectors"] or es == 2) and p["group"] * p["vpt"] >= nv
        assert p["grid"] * p["threads"] // p["group"] >= min(rows, p["grid"] * p["threads"] // p["group"])
    elif path == B.PATH_CTA:
        assert p["threads"] * p["vpt"] >= nv and p["grid"] == rows
    elif path == B.PATH_CLUSTER:
        assert es == 2 and p["vpt"] == 8 and p["threads"] in (256, 512)
        assert 1 <= p["group"] <= 16 and -(-nv // p["group"]) <= p["threads"] * p["vpt"]
        assert p["grid"] == rows * p["group"] and p["smem_bytes"] <= 227 * 1024
    elif path == B.PATH_PACKED:  # dense narrow rows, one thread each, 128 rows per staged span
        assert stride == cols and cols <= 48 and p["threads"] == 128 and p["grid"] == -(-rows // 128)
        assert p["smem_bytes"] >= 128 * cols * 4
    elif path == B.PATH_GRID:  # a few rows of 1 MiB or more, spread over the grid (out != in)
        assert rows * 16 < 152 and cols * es >= 1 << 20
        assert p["group"] == max(1, min(2 * 152 // rows, nv // max(3, nv // max(1, 2 * 152 // rows))))
        assert p["threads"] == 512 and p["grid"] == min(rows * p["group"], 152 * 4)
    else:  # any slice length; enough blocks to fill the GPU (or 16 per row)
        assert path == B.PATH_STREAM
        assert 1 <= p["group"] <= 16 and p["grid"] == rows * p["group"]
        assert rows * p["group"] >= min(152, rows * 16)
    assert p["scratch_bytes"] == 0  # nothing allocated
    assert p["launches"] == (2 if path == B.PATH_GRID else 1)
    mult = 3 if path in (B.PATH_STREAM, B.PATH_GRID) else 2
    assert p["hbm_bytes"] == mult * rows * cols * es


@pytest.mark.parametrize("in_off,out_off,cols,stride,dt,whole", [
    (0, 0, 2048, 2048, "f16", 1),      # aligned rows of whole vectors
    (0, 0, 1000, 1000, "f32", 1),      # 4000-byte rows: whole vectors
    (0, 0, 1001, 1001, "f32", 0),      # the width leaves a partial last vector
    (0, 0, 1000, 1001, "f32", 0),      # the stride moves later rows off 16 bytes
    (4, 4, 1000, 1000, "f32", 0),      # in and out start inside a vector
    (0, 8, 1000, 1000, "f32", 0),      # out not aligned
    (0, 0, 8, 8, "bf16", 1),
    (0, 0, 7, 8, "bf16", 0),
])
def test_plan_reports_whole_vector_rows(in_off, out_off, cols, stride, dt, whole):
    p = B.plan((1 << 24) + in_off, (1 << 40) + out_off, 64, cols, stride, dt, num_sms=152)
    assert p["whole_vectors"] == whole


def test_dispatch_follows_width_rule():
    plan = lambda r, c, dt="f32": B.plan(1 << 24, 1 << 40, r, c, c, dt, num_sms=152)["path"]
    assert plan(64, 1000) == B.PATH_WARP          # cols <= 1024: a warp per row
    assert plan(1000, 39) == B.PATH_PACKED        # narrow dense rows off the 16-byte grid: staged
    assert plan(1000, 40) == B.PATH_WARP          # ... but 40 fp32 are whole vectors
    assert plan(1000, 71) == B.PATH_WARP          # ... and 71 is too wide for a thread per row
    assert B.plan(1 << 24, 1 << 40, 1000, 39, 41, "f32", num_sms=152)["path"] == B.PATH_WARP  # padded
    assert plan(64, 1024) == B.PATH_WARP
    assert plan(64, 1025) == B.PATH_CTA           # misaligned medium rows: a block per row
    assert plan(4096, 16391) == B.PATH_CTA
    assert plan(4096, 2048, "f16") == B.PATH_WARP  # whole vectors, 256 per row: still a warp
    assert plan(4096, 1100) == B.PATH_WARP         # 275 whole vectors
    assert B.plan(1 << 24, 1 << 40, 4096, 2047, 2047, "bf16", num_sms=152)["path"] == B.PATH_WARP  # 16-bit edges
    assert B.plan(1 << 24, 1 << 40, 8192, 2055, 2055, "f16", num_sms=152)["path"] == B.PATH_WARP
    assert plan(4096, 2047) == B.PATH_CTA            # ragged fp32 rows past 1024: a block per row
    assert B.plan(1 << 24, 1 << 40, 8192, 2305, 2305, "f16", num_sms=152)["path"] == B.PATH_CTA  # > 288 vectors
    assert plan(4096, 16384) == B.PATH_CTA           # 512 x 8 keeps two 64 KB rows per SM
    assert plan(512, 131072, "bf16") == B.PATH_CLUSTER   # long 16-bit rows: a cluster, registers
    assert plan(512, 65536) == B.PATH_STREAM             # long fp32 rows: a cluster streaming them twice
    assert plan(512, 65537) == B.PATH_STREAM             # ... aligned or not
    assert plan(512, 131079, "bf16") == B.PATH_CLUSTER   # long misaligned rows, enough of them
    assert plan(4, 131072, "bf16") == B.PATH_STREAM      # too few rows to fill the GPU: 16 blocks each
    assert plan(64, 1 << 22) == B.PATH_STREAM            # too long to hold on chip: stream it twice
    assert plan(9, 1 << 22) == B.PATH_GRID               # 9 rows of 16 MiB: chunks over the whole grid
    assert B.plan(1 << 24, 1 << 24, 9, 1 << 22, 1 << 22, "f32", num_sms=152)["path"] == B.PATH_STREAM  # in place
    assert plan(9, 1 << 18) == B.PATH_GRID               # 1 MiB rows
    assert plan(9, (1 << 18) - 1) == B.PATH_STREAM       # ... but not shorter ones


def test_few_long_rows_take_one_tile_per_block():
    # rows * 16 < SMs: the stream blocks grow (up to 1024 threads) until each
    # holds about one 4-vector tile of its slice
    p = B.plan(1 << 24, 1 << 40, 9, 262144, 262144, "bf16", num_sms=152)
    assert (p["path"], p["group"], p["threads"]) == (B.PATH_STREAM, 16, 512)
    p = B.plan(1 << 24, 1 << 24, 3, 1_000_000, 1_000_000, "f32", num_sms=152)   # in place
    assert (p["path"], p["group"], p["threads"]) == (B.PATH_STREAM, 16, 1024)
    p = B.plan(1 << 24, 1 << 40, 1, 40000, 40000, "f32", num_sms=152)
    assert (p["path"], p["group"], p["threads"]) == (B.PATH_STREAM, 10, 256)


def test_few_very_long_rows_spread_over_the_grid():
    # out != in and rows of 1 MiB or more: about two 512-thread blocks per SM
    # over all rows, each row in equal chunks, the states kept in the output row
    p = B.plan(1 << 24, 1 << 40, 3, 1_000_000, 1_000_000, "f32", num_sms=152)
    assert (p["path"], p["threads"], p["vpt"], p["launches"]) == (B.PATH_GRID, 512, 4, 2)
    assert p["group"] == 101 and p["grid"] == 303 and p["scratch_bytes"] == 0
    p = B.plan(1 << 24, 1 << 40, 1, 4_000_000, 4_000_000, "f32", num_sms=152)
    assert p["path"] == B.PATH_GRID and p["group"] == 304 and p["grid"] == 304
    p = B.plan(1 << 24, 1 << 40, 1, 1 << 26, 1 << 26, "bf16", num_sms=152)
    assert p["path"] == B.PATH_GRID and p["group"] == 304 and p["grid"] == 304
    try:
        B.set_force_path(B.PATH_GRID, group=7)   # forced: any chunk count, chunks of 3 vectors or more
        p = B.plan(1 << 24, 1 << 40, 5, 100, 100, "f32", num_sms=152)
        assert (p["path"], p["group"], p["grid"]) == (B.PATH_GRID, 7, 35)
        p = B.plan(1 << 24, 1 << 40, 5, 9, 9, "f32", num_sms=152)         # 3 vectors: one chunk
        assert (p["path"], p["group"]) == (B.PATH_GRID, 1)
        for cols in (1, 8):                        # fewer than 3 vectors: no room for the states
            with pytest.raises(B.SoftmaxError) as e:
                B.plan(1 << 24, 1 << 40, 5, cols, cols, "f32", num_sms=152)
            assert e.value.status == B.ERR_UNSUPPORTED
        B.set_force_path(B.PATH_GRID, group=300)   # at most 2048 threads per SM
        p = B.plan(1 << 24, 1 << 40, 5, 100000, 100000, "f32", num_sms=152)
        assert (p["group"], p["grid"]) == (300, 152 * 4)
        B.set_force_path(B.PATH_GRID, 1024, 4, 300)
        p = B.plan(1 << 24, 1 << 40, 5, 100000, 100000, "f32", num_sms=152)
        assert (p["threads"], p["vpt"], p["group"], p["grid"]) == (1024, 4, 300, 152 * 2)
        for shape in ((128, 4), (256, 2), (512, 8)):   # not instantiated
            B.set_force_path(B.PATH_GRID, *shape)
            with pytest.raises(B.SoftmaxError):
                B.plan(1 << 24, 1 << 40, 5, 100000, 100000, "f32", num_sms=152)
        B.set_force_path(B.PATH_GRID, group=1 << 20)   # chunks of 3 vectors: the state region still fits
        p = B.plan(1 << 24, 1 << 40, 5, 100000, 100000, "f32", num_sms=152)
        assert p["group"] == 25000 // 3 and 8 * p["group"] + 8 <= 400000
        with pytest.raises(B.SoftmaxError) as e:   # the states need an output row apart from the input
            B.plan(1 << 24, 1 << 24, 5, 100, 100, "f32", num_sms=152)
        assert e.value.status == B.ERR_UNSUPPORTED
    finally:
        B.set_force_path(0)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_no_automatic_plan_takes_scratch(dt):
    # softmax_fwd allocates nothing: every automatic plan, over rows from 1 to
    # 2^21 and widths from 1 to 2^24, has scratch_bytes == 0 and one kernel
    # (two for the grid-wide path, whose states live in the output)
    for rows in (1, 2, 3, 5, 9, 10, 64, 1000, 1 << 21):
        for cols in (1, 39, 1000, 2055, 20000, 40961, 131072, 1_000_000, 1 << 24):
            if rows * cols > 1 << 34:
                continue
            for off in (0, 4):
                p = B.plan((1 << 24) + off, (1 << 46) + off, rows, cols, cols, dt, num_sms=152)
                assert p["scratch_bytes"] == 0 and p["path"] != B.PATH_SPLIT
                assert p["launches"] == (2 if p["path"] == B.PATH_GRID else 1)


def test_forced_paths_and_rejections():
    try:
        for retired in (B.PATH_SPLIT, 5):  # the split path is softmax_fwd_noalloc's; 5 is unused
            with pytest.raises(B.SoftmaxError) as e:
                B.set_force_path(retired)
            assert e.value.status == B.ERR_ARG
        B.set_force_path(B.PATH_WARP)
        with pytest.raises(B.SoftmaxError) as e:
            B.plan(1 << 24, 1 << 40, 64, 5000, 5000, "f32", num_sms=152)
        assert e.value.status == B.ERR_UNSUPPORTED
        B.set_force_path(B.PATH_CLUSTER)
        with pytest.raises(B.SoftmaxError):   # fp32 rows would spill in a register-held cluster
            B.plan(1 << 24, 1 << 40, 64, 50000, 50000, "f32", num_sms=152)
        assert B.plan(1 << 24, 1 << 40, 64, 50000, 50000, "bf16", num_sms=152)["path"] == B.PATH_CLUSTER
        B.set_force_path(B.PATH_CLUSTER, 256, 2, 2)   # only 8 vectors per thread exist
        with pytest.raises(B.SoftmaxError):
            B.plan(1 << 24, 1 << 40, 64, 5000, 5000, "bf16", num_sms=152)
        with pytest.raises(B.SoftmaxError):
            B.set_force_path(9)
    finally:
        B.set_force_path(0)


def test_masked_argument_checks_need_no_gpu():
    p = 1 << 24
    q = 1 << 40
    for scale in (0.0, -2.0, float("inf"), float("nan")):
        assert B.softmax_fwd_masked_ptr(p, q, 4, 8, 8, 0, scale, 0, 0) == B.ERR_ARG
    assert B.softmax_fwd_masked_ptr(p, q, 4, 8, 8, 0, 1.0, 0, -1) == B.ERR_ARG
    assert B.softmax_fwd_masked_ptr(p, q, 0, 8, 8, 0, 1.0, 0, 0) == B.OK      # no rows: nothing to do
    assert B.softmax_fwd_masked_ptr(p, q, 4, 8, 7, 0, 1.0, 0, 0) == B.ERR_STRIDE
    assert B.softmax_fwd_masked_ptr(p, p + 4, 4, 8, 8, 0, 1.0, 0, 0) == B.ERR_OVERLAP


def test_masked_copy_argument_checks_need_no_gpu():
    p, q = 1 << 24, 1 << 40
    assert B.masked_copy_ptr(p, q, 4, 8, 8, 0, 0, -1) == B.ERR_ARG             # rows_per_seq < 0
    for threads in (16, 48, 2048):
        assert B.masked_copy_ptr(p, q, 4, 8, 8, 0, 0, 0, threads) == B.ERR_ARG
    assert B.masked_copy_ptr(p, q, 4, 6, 8, 0, 0, 0) == B.ERR_UNSUPPORTED      # 24-byte rows
    assert B.masked_copy_ptr(p, q, 4, 8, 9, 0, 0, 0) == B.ERR_UNSUPPORTED      # 36-byte stride
    assert B.masked_copy_ptr(p + 4, q + 4, 4, 8, 8, 0, 0, 0) == B.ERR_UNSUPPORTED
    assert B.masked_copy_ptr(p, q, 0, 8, 8, 0, 0, 0) == B.OK                   # no rows: nothing to do
    assert B.masked_copy_ptr(p, p + 4, 4, 8, 8, 0, 0, 0) == B.ERR_OVERLAP


def test_host_workspace_sizes():
    # three slots of whole rows, about chunk_bytes each, never more than the matrix
    assert B.host_workspace_bytes(0, 10, 10, "f32") == 0
    small = B.host_workspace_bytes(5, 10, 10, "f32")
    assert small == 3 * 256                                  # 5 rows of 40 B: one 200-byte slot, 256-aligned
    big = B.host_workspace_bytes(4096, 2048, 2048, "f16", 1 << 20)
    assert big == 3 * (256 * 2048 * 2)                       # 256 rows of 4 KiB per 1 MiB chunk
    assert B.host_workspace_bytes(4096, 2048, 2048, "f16") == 3 * (1024 * 4096)  # a quarter: 4 MiB
    assert B.host_workspace_bytes(4096, 4096, 4096, "f32") == 3 * (8 << 20)      # capped at 8 MiB
    assert B.host_workspace_bytes(100, 100, 100, "f32") == 3 * 40192              # small: the whole matrix
    with pytest.raises(B.SoftmaxError):
        B.host_workspace_bytes(4, 10, 9, "f32")              # stride < cols


def test_host_call_argument_checks_need_no_gpu():
    h = 1 << 24
    assert B.lib().softmax_fwd_host(h, h + (1 << 20), 4, 8, 8, 0, None, 1 << 20, None) == B.ERR_NULL
    assert B.lib().softmax_fwd_host(h, h + 4, 4, 8, 8, 0, 1 << 30, 1 << 20, None) == B.ERR_OVERLAP
    assert B.lib().softmax_fwd_host(h, h + (1 << 20), 4, 8, 8, 0, (1 << 30) + 4, 1 << 20, None) == B.ERR_ARG
    assert B.lib().softmax_fwd_host(h, h + (1 << 20), 4, 8, 8, 0, 1 << 30, 16, None) == B.ERR_ARG  # too small


def _check_plan_covers(p, rows, cols, stride, dt, in_off, out_off):
    es = 4 if dt == "f32" else 2
    V = 16 // es
    uniform = (stride * es) % 16 == 0
    head = (in_off // es) % V if uniform else V - 1
    nv = -(-(head + cols) // V)
    path = p["path"]
    if path == B.PATH_WARP:
        assert p["group"] * p["vpt"] >= nv and p["threads"] % p["group"] == 0 and 32 <= p["threads"] <= 256
        assert p["grid"] * (p["threads"] // p["group"]) >= min(rows, p["grid"] * (p["threads"] // p["group"]))
    elif path == B.PATH_CTA:
        assert p["threads"] * p["vpt"] >= nv and p["grid"] == min(rows, 2 ** 31 - 1)
    elif path == B.PATH_CLUSTER:
        assert 1 <= p["group"] <= 16 and -(-nv // p["group"]) <= p["threads"] * p["vpt"]
        assert p["grid"] == rows * p["group"]
    elif path == B.PATH_PACKED:
        assert stride == cols and p["group"] == 1 and p["smem_bytes"] <= 48 * 1024
        assert p["grid"] * 128 * p["vpt"] >= rows
    elif path == B.PATH_GRID:
        assert p["group"] >= 1 and nv // p["group"] >= 3 and 1 <= p["grid"] <= rows * p["group"]
    else:
        assert path == B.PATH_STREAM
        assert 1 <= p["group"] <= 16 and p["grid"] == rows * p["group"]
    assert p["scratch_bytes"] == 0


def test_planner_fuzz_covers_every_row():
    # random shapes, strides and base offsets: the automatic plan always exists
    # and always covers the row (host only: an SM count is given)
    rng = np.random.default_rng(7)
    for _ in range(3000):
        dt = ["f32", "f16", "bf16"][rng.integers(3)]
        es = 4 if dt == "f32" else 2
        cols = int(np.exp(rng.uniform(0, np.log(3_000_000))))
        stride = cols + int(rng.choice([0, 0, 0, 1, 5, 8, 64]))
        rows = int(np.exp(rng.uniform(0, np.log(2_000_000))))
        off = int(rng.integers(0, 16 // es)) * es
        out_off = off if rng.integers(3) else int(rng.integers(0, 16 // es)) * es
        p = B.plan((1 << 30) + off, (1 << 46) + out_off, rows, cols, stride, dt,
                   num_sms=int(rng.choice([1, 16, 152])))
        _check_plan_covers(p, rows, cols, stride, dt, off, out_off)
        assert p["vec_store"] == (off == out_off)


# softmax_attention_fwd: every argument error is reported before any CUDA call
_A = 1 << 32  # well-separated fake device addresses, 16-byte aligned
_MB = 1 << 24


@pytest.mark.parametrize("args,expect", [
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, -1, 1, 128, 128, 1, 1, 0.1), B.ERR_SHAPE),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 0, 1, 1, 0.1), B.ERR_SHAPE),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 64, 1, 1, 0.1), B.ERR_UNSUPPORTED),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 0, 1, 0.1), B.ERR_UNSUPPORTED),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 7, 1, 0.1), B.ERR_DTYPE),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 2, 0.1), B.ERR_ARG),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, 0.0), B.ERR_ARG),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, float("inf")), B.ERR_ARG),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, float("nan")), B.ERR_ARG),
    ((0, 0, 0, 0, 0, 1, 128, 128, 1, 1, 0.1), B.OK),          # no work: nothing launched
    ((0, 0, 0, 0, 3, 2, 0, 128, 2, 0, 0.1), B.OK),
    ((0, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_NULL),
    ((_A, _A + _MB, _A + 2 * _MB, 0, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_NULL),
    ((_A + 8, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_ALIGN),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB + 2, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_ALIGN),
    ((_A, _A + _MB, _A + 2 * _MB, _A + _MB + 16, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_OVERLAP),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 2 * _MB - 16, 1, 1, 128, 128, 1, 1, 0.1), B.ERR_OVERLAP),
    ((_A, _A + _MB, _A + 2 * _MB, _A, 1, 1, 128, 128, 2, 0, 0.1), B.ERR_OVERLAP),
    ((_A, _A, _A, _A + 3 * _MB, 1, 1, 128, 128, 1, 1, 0.1), None),   # q, k, v may share memory
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1, 1, 1 << 31, 128, 1, 1, 0.1), B.ERR_SHAPE),
    ((_A, _A + _MB, _A + 2 * _MB, _A + 3 * _MB, 1 << 20, 1 << 10, 1024, 128, 1, 1, 0.1), B.ERR_SHAPE),
])
def test_attention_argument_checks(args, expect):
    if expect is None:
        # valid arguments would launch: only check that none of the argument
        # errors is raised (without a device the launch itself fails)
        st = B.lib().softmax_attention_fwd(*args, None)
        assert st not in (B.ERR_SHAPE, B.ERR_NULL, B.ERR_ALIGN, B.ERR_OVERLAP, B.ERR_ARG, B.ERR_DTYPE,
                          B.ERR_UNSUPPORTED)
        return
    assert B.lib().softmax_attention_fwd(*args, None) == expect


def test_attention_plan_on_the_host():
    # the pages' shape on 152 SMs: 4 x 32 heads x 16 items each, one block per SM,
    # head groups whose K and V (2 MiB per head at N = 4096) fit 48 MiB
    p = B.attention_plan(4, 32, 4096, num_sms=152)
    assert p["items"] == 4 * 32 * 16 and p["grid"] == 152 and p["head_group"] == 24
    assert p["threads"] == 320 and p["tmem_columns"] == 512 and p["smem_bytes"] <= 227 * 1024
    assert p["flops"] == 4.0 * 4 * 32 * 4096 ** 2 * 128 / 2
    assert B.attention_plan(4, 32, 16384, num_sms=152)["head_group"] == 6
    assert B.attention_plan(4, 32, 16384, causal=False, num_sms=152)["flops"] == 4.0 * 4 * 32 * 16384 ** 2 * 128
    # fewer items than SMs: one block per item; tiny contexts: every head in one group
    small = B.attention_plan(1, 3, 100, num_sms=152)
    assert small["items"] == 3 and small["grid"] == 3 and small["head_group"] == 3
    assert B.attention_plan(0, 3, 100, num_sms=152)["items"] == 0
    for args, status in [((1, 1, 128, 64), B.ERR_UNSUPPORTED), ((1, -1, 128, 128), B.ERR_SHAPE),
                         ((1, 1, 1 << 31, 128), B.ERR_SHAPE)]:
        with pytest.raises(B.SoftmaxError) as e:
            B.attention_plan(*args, num_sms=152)
        assert e.value.status == status
    with pytest.raises(B.SoftmaxError):
        B.attention_plan(1, 1, 128, dtype="f32", num_sms=152)
