"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle, element by element, on seeded inputs.

Covers every path (automatic and forced), ragged row counts, widths around
every vector / warp / block / cluster boundary, misaligned base pointers and
strides, padding that must stay untouched, in-place calls, the special values
(-inf masks, NaN, +inf, spikes), the workloads of the pages at full size, and
the bounded-wait error path.
"""
import numpy as np
import pytest
import torch

from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import DeviceCase, compare, decode, run_and_compare

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    torch.cuda.init()
    yield
    B.set_force_path(0)
    B.set_wait_test(0, False)


def rnd(rows, cols, dtype, seed, stride=0, sigma=2.0):
    return W.make_random(rows, cols, dtype, seed, row_stride=stride, sigma=sigma)


def skip_fp32_cluster(path, dtype):
    """The register-held cluster path takes 16-bit rows only (fp32 slices
    would spill); a forced fp32 call is refused, as its own test checks."""
    if path == B.PATH_CLUSTER and dtype == "f32":
        pytest.skip("the cluster path takes 16-bit rows only")


# -- automatic dispatch across widths -----------------------------------------------

WIDTHS = [1, 2, 3, 5, 7, 8, 9, 16, 31, 33, 63, 100, 255, 257, 1000, 1023, 1024, 1025, 2047, 2048, 2055,
          4096, 4103, 8192, 8199, 16391, 32768, 32775, 65536, 131079]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", WIDTHS)
def test_auto_widths(dtype, cols):
    rows = 5 if cols > 10000 else 7
    res = run_and_compare(rnd(rows, cols, dtype, seed=cols), dtype)
    assert res["path"] in (B.PATH_WARP, B.PATH_CTA, B.PATH_CLUSTER, B.PATH_STREAM, B.PATH_PACKED, B.PATH_GRID)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows", [1, 2, 3, 31, 33, 257, 1000])
@pytest.mark.parametrize("cols", [40, 700, 3000])
def test_ragged_row_counts(dtype, rows, cols):
    run_and_compare(rnd(rows, cols, dtype, seed=rows * 7 + cols), dtype)


def test_zero_rows_is_a_no_op():
    assert B.softmax_fwd_ptr(0, 0, 0, 5, 5, 0) == B.OK


# -- every path forced onto the widths it can take ---------------------------------------

FORCED = {
    B.PATH_WARP: [1, 2, 3, 7, 9, 17, 31, 33, 100, 255, 256, 257, 1000, 1024],
    B.PATH_CTA: [1, 9, 100, 1025, 2047, 4096, 4103, 8199, 16384],
    B.PATH_CLUSTER: [1, 100, 2048, 9000, 16391, 65536, 131079, 262151],
    B.PATH_STREAM: [1, 100, 4103, 65536, 262147],
    B.PATH_PACKED: [1, 7, 39, 90],
    B.PATH_GRID: [17, 100, 4103, 65536, 262147],
}


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("path,cols", [(p, c) for p, cs in FORCED.items() for c in cs])
def test_forced_path(dtype, path, cols):
    skip_fp32_cluster(path, dtype)
    res = run_and_compare(rnd(3, cols, dtype, seed=100 + cols), dtype, path=path)
    assert res["path"] == path


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [1, 2, 3, 5, 8, 16])
def test_cluster_sizes(dtype, group):
    # 2001 columns fit one 256 x 8-vector block, so every cluster size can
    # take the row (most slots of most slices empty)
    res = run_and_compare(rnd(4, 2001, dtype, seed=group), dtype, path=B.PATH_CLUSTER, threads=256, vpt=8,
                          group=group)
    assert res["path"] == B.PATH_CLUSTER


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("threads", [256, 512])
@pytest.mark.parametrize("group", [1, 2, 3, 8, 16])
def test_cluster_register_slices(dtype, threads, group):
    # 8 vectors per thread: the cluster path's variant that holds its slice in
    # registers instead of staging it in shared memory
    cols = min(8 * threads * 8 * group - 13, 140001)
    res = run_and_compare(rnd(5, cols, dtype, seed=group + threads), dtype, path=B.PATH_CLUSTER, threads=threads,
                          vpt=8, group=group)
    assert res["path"] == B.PATH_CLUSTER


def test_cluster_register_slices_refuse_fp32():
    case = DeviceCase(rnd(2, 4000, "f32", 1), "f32")
    assert case.run(4000, path=B.PATH_CLUSTER, threads=256, vpt=8, group=2) == B.ERR_UNSUPPORTED
    assert case.run(4000, path=B.PATH_CLUSTER) == B.ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("threads,vpt", [(64, 8), (128, 2), (512, 4), (1024, 2), (256, 3), (1024, 5)])
def test_cta_shapes(dtype, threads, vpt):
    cols = {"f32": 4 * threads * vpt - 5, "f16": 8 * threads * vpt - 9, "bf16": 8 * threads * vpt - 9}[dtype]
    res = run_and_compare(rnd(3, cols, dtype, seed=threads + vpt), dtype, path=B.PATH_CTA, threads=threads, vpt=vpt)
    assert res["path"] == B.PATH_CTA


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("group", [1, 2, 3, 5, 8, 16])
@pytest.mark.parametrize("threads,vpt", [(256, 2), (512, 4), (1024, 4)])
def test_stream_cluster_sizes_and_tiles(dtype, group, threads, vpt):
    # 70001 columns over `group` blocks: slices of one to many tiles, a partial
    # last tile, ragged edges on misaligned rows
    res = run_and_compare(rnd(3, 70001, dtype, seed=group * 13 + vpt), dtype, in_off=1, path=B.PATH_STREAM,
                          threads=threads, vpt=vpt, group=group)
    assert res["path"] == B.PATH_STREAM


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols", [(40, 65536), (200, 24576), (12, 400000), (1, 4_000_000), (3, 1_000_000)])
def test_stream_whole_rows(dtype, rows, cols):
    # aligned rows of whole vectors (the edge-free instantiations), automatic
    # cluster size
    res = run_and_compare(rnd(rows, cols, dtype, seed=rows + cols), dtype, path=B.PATH_STREAM)
    assert res["path"] == B.PATH_STREAM


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("group", [1, 2, 3, 7, 64, 1000, 5000])
@pytest.mark.parametrize("in_off,out_off", [(1, 1), (3, 0)])
def test_grid_chunk_counts(dtype, group, in_off, out_off):
    # 70001 columns in `group` chunks (down to 3 vectors each), misaligned
    # rows, out at in's 16-byte phase or not: every chunk's state passes
    # through the state region at the start of the output row
    res = run_and_compare(rnd(3, 70001, dtype, seed=group + in_off), dtype, in_off=in_off, out_off=out_off,
                          path=B.PATH_GRID, group=group)
    assert res["path"] == B.PATH_GRID


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("threads,vpt", [(256, 4), (256, 8), (512, 4), (1024, 4)])
@pytest.mark.parametrize("group", [1, 5, 40, 700])
def test_grid_block_shapes(dtype, threads, vpt, group):
    # every block shape, chunks of one to many tiles, the state region over
    # one chunk or several (700 chunks of 3-25 vectors)
    res = run_and_compare(rnd(4, 70001, dtype, seed=threads + vpt + group), dtype, in_off=3, out_off=3,
                          path=B.PATH_GRID, threads=threads, vpt=vpt, group=group)
    assert res["path"] == B.PATH_GRID


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("rows,cols,in_off,out_off", [(1, 4_000_000, 0, 0), (3, 1_000_000, 0, 0),
                                                      (9, 524288, 0, 0), (2, 3_000_001, 3, 1), (5, 777_777, 2, 2)])
def test_grid_rows(dtype, rows, cols, in_off, out_off):
    # a few rows of 1 MiB or more with out != in: the automatic choice
    x = rnd(rows, cols, dtype, seed=rows * 31 + cols)
    res = run_and_compare(x, dtype, in_off=in_off, out_off=out_off)
    es = 4 if dtype == "f32" else 2
    assert res["path"] == (B.PATH_GRID if cols * es >= 1 << 20 else B.PATH_STREAM)
    # in place the same rows stream through a cluster instead
    res = run_and_compare(x, dtype, inplace=True, in_off=in_off)
    assert res["path"] == B.PATH_STREAM


def test_grid_refuses_in_place_and_writes_nothing():
    x = rnd(3, 70001, "f32", seed=5)
    c = DeviceCase(x, "f32", inplace=True)
    before = c.result(70001).copy()
    assert c.run(70001, path=B.PATH_GRID) == B.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert np.array_equal(c.result(70001).view(np.uint32), before.view(np.uint32))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols", [1, 3, 8, 9, 33, 39, 71, 90])
@pytest.mark.parametrize("off", [0, 1, 3])
@pytest.mark.parametrize("rows,k", [(1, 1), (5, 1), (700, 2), (1537, 1)])
def test_packed_spans(dtype, cols, off, rows, k):
    # dense rows staged through shared memory: spans that end inside a vector,
    # a last partial span, the matrix starting `off` elements into a vector
    if k > 1 and 128 * k * cols * 4 > 48 * 1024:
        k = 1  # the span would not fit its 48 KB
    res = run_and_compare(rnd(rows, cols, dtype, seed=cols * 31 + rows + off), dtype, in_off=off, out_off=off,
                          path=B.PATH_PACKED, vpt=k)
    assert res["path"] == B.PATH_PACKED


@pytest.mark.parametrize("dtype", DTYPES)
def test_packed_refuses_what_it_cannot_stage(dtype):
    x = rnd(40, 39, dtype, 3, stride=41)                         # padded stride
    assert DeviceCase(x, dtype).run(39, path=B.PATH_PACKED) == B.ERR_UNSUPPORTED
    y = rnd(40, 300, dtype, 3)                                   # a 128-row span over 48 KB
    assert DeviceCase(y, dtype).run(300, path=B.PATH_PACKED) == B.ERR_UNSUPPORTED
    z = rnd(40, 39, dtype, 3)                                    # out in another 16-byte phase
    assert DeviceCase(z, dtype, in_off=1, out_off=2).run(39, path=B.PATH_PACKED) == B.ERR_UNSUPPORTED


def test_forced_shape_that_cannot_cover_the_row_is_rejected():
    case = DeviceCase(rnd(2, 5000, "f32", 1), "f32")
    assert case.run(5000, path=B.PATH_WARP) == B.ERR_UNSUPPORTED
    assert case.run(5000, path=B.PATH_CLUSTER, threads=256, vpt=2, group=2) == B.ERR_UNSUPPORTED


# -- alignment, strides, aliasing ------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("in_off,out_off", [(1, 1), (2, 2), (3, 3), (1, 0), (0, 3), (5, 2)])
@pytest.mark.parametrize("cols", [7, 100, 1000, 3001, 20011])
def test_misaligned_pointers(dtype, in_off, out_off, cols):
    run_and_compare(rnd(4, cols, dtype, seed=cols + in_off), dtype, in_off=in_off, out_off=out_off)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cols,extra", [(31, 1), (100, 3), (1000, 8), (2048, 5), (4096, 8), (20000, 7)])
def test_padded_strides(dtype, cols, extra):
    x = rnd(9, cols, dtype, seed=cols, stride=cols + extra)
    run_and_compare(x, dtype, cols)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("path", [0, B.PATH_WARP, B.PATH_CTA, B.PATH_CLUSTER, B.PATH_STREAM, B.PATH_PACKED])
def test_in_place(dtype, path):
    skip_fp32_cluster(path, dtype)
    cols = 1000 if path in (0, B.PATH_WARP) else 6007
    off = 1
    if path == B.PATH_PACKED:
        cols = 39
    run_and_compare(rnd(300, cols, dtype, seed=path), dtype, inplace=True, in_off=off, path=path)


def test_partial_overlap_is_rejected():
    d = torch.zeros(1000, device="cuda")
    p = d.data_ptr()
    assert B.softmax_fwd_ptr(p, p + 16, 10, 10, 10, 0) == B.ERR_OVERLAP


# -- special values ------------------------------------------------------------------

def special_rows(dtype, cols):
    """Rows 0..6: fully masked, one-hot, a NaN, a +inf, constant, a +100 spike, half masked."""
    x = W.make_random(8, cols, dtype, seed=77, sigma=1.0)

    def put(row, idx, v):
        x[row, idx] = W.quantise(np.asarray([v], dtype=np.float64), dtype)[0]

    put(0, slice(None), -np.inf)
    put(1, slice(None), -np.inf)
    put(1, cols // 2, 1.5)
    put(2, cols - 1, np.nan)
    put(3, 0, np.inf)
    put(4, slice(None), 0.375)
    put(5, cols // 3, float(decode(x[5], dtype).max()) + 100.0)
    put(6, slice(0, None, 2), -np.inf)
    return x


def _result_bits(x, dtype, path):
    c = DeviceCase(x, dtype)
    assert c.run(x.shape[1], path=path) == B.OK
    return c.result(x.shape[1])


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("path,cols", [(B.PATH_WARP, 33), (B.PATH_WARP, 1000), (B.PATH_CTA, 3000),
                                       (B.PATH_CLUSTER, 20000), (B.PATH_CLUSTER, 65536), (B.PATH_STREAM, 20000),
                                       (B.PATH_STREAM, 65536), (B.PATH_GRID, 20000), (B.PATH_GRID, 65536)])
def test_special_values(dtype, path, cols):
    skip_fp32_cluster(path, dtype)
    x = special_rows(dtype, cols)
    run_and_compare(x, dtype, path=path)
    y = decode(_result_bits(x, dtype, path), dtype)
    assert np.isnan(y[0]).all() and np.isnan(y[2]).all() and np.isnan(y[3]).all()
    assert y[1, cols // 2] == 1.0 and (np.delete(y[1], cols // 2) == 0).all()
    assert np.isfinite(y[5]).all() and abs(y[5, cols // 3] - 1.0) < 1e-3
    assert (y[6, ::2] == 0).all()


def test_constant_rows_are_exactly_one_over_n():
    for cols in (1, 2, 4, 1024, 4096, 131072):
        x = np.full((2, cols), 0.5, dtype=np.float32)
        c = DeviceCase(x, "f32")
        assert c.run(cols) == B.OK
        y = decode(c.result(cols), "f32")
        assert np.abs(y - 1.0 / cols).max() <= 1e-6 * (1.0 / cols) + 1e-12


# -- the pages' workloads at full size ----------------------------------------------------

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_config_full_size(name):
    w = W.CONFIGS[name]
    x = W.make_input(w)
    res = run_and_compare(x, w.dtype, w.cols)
    if name == "c3":  # the spike rows: the spiked entry carries almost all the mass
        rows, cols = W.spike_plan(w)
        c = DeviceCase(x, "f32")
        assert c.run(w.cols) == B.OK
        y = decode(c.result(w.cols), "f32")
        assert np.isfinite(y[rows]).all()
        assert (np.abs(y[rows, cols] - 1.0) < 1e-6).all()
    print(name, res)


@pytest.mark.parametrize("name", sorted(W.EXTRA_SHAPES))
def test_extra_shape_full_size(name):
    # the shapes the benchmark times beside the pages' workloads (ragged
    # 16-bit rows, a few very long rows), every element against the oracle
    w = W.EXTRA_SHAPES[name]
    x = W.make_input(w)
    res = run_and_compare(x, w.dtype, w.cols)
    print(w.name, B.PATH_NAMES[res["path"]], res)


@pytest.mark.parametrize("cols", W.SWEEP_WIDTHS)
def test_sweep_width_full_size(cols):
    w = W.sweep_workload(cols)
    x = W.make_input(w)
    rng = np.random.default_rng(cols)
    sample = np.unique(np.concatenate([[0, 1, 2, w.rows - 1], rng.integers(0, w.rows, 61)]))
    res = run_and_compare(x, "f32", rows=sample)
    print(w.name, res)


def test_offsets_beyond_int32():
    # 65539 rows x 32768 fp16: element offsets pass 2^31; tile 64 seeded rows
    rows, cols = 65539, 32768
    block = W.make_random(64, cols, "f16", seed=31, sigma=3.0)
    d_in = torch.from_numpy(block.view(np.int16)).cuda().repeat((rows + 63) // 64, 1)[:rows].contiguous()
    d_out = torch.empty_like(d_in)
    st = B.softmax_fwd_ptr(d_in.data_ptr(), d_out.data_ptr(), rows, cols, cols, 1,
                           torch.cuda.current_stream().cuda_stream)
    assert st == B.OK
    torch.cuda.synchronize()
    check = [0, 63, 64, 65535, 65536, 65538]
    got = d_out[check].cpu().numpy().view(np.uint16)
    compare(got, np.ascontiguousarray(block[[r % 64 for r in check]]), "f16", cols)
    del d_in, d_out
    torch.cuda.empty_cache()


# -- the bounded wait and the device error word ------------------------------------------

@pytest.mark.parametrize("path,threads,vpt,group", [(B.PATH_CLUSTER, 256, 8, 0), (B.PATH_CLUSTER, 512, 8, 1),
                                                    (B.PATH_STREAM, 256, 4, 1), (B.PATH_STREAM, 512, 4, 4)])
def test_wait_timeout_is_reported_and_recoverable(path, threads, vpt, group):
    # the cluster kernels' state exchange: with the hook no block sends its
    # state, so every block's bounded wait runs out
    x = rnd(4, 20000, "bf16", seed=5)
    c = DeviceCase(x, "bf16")
    B.set_wait_test(1_000_000, starve=True)  # 1 ms, and no state is ever sent
    try:
        assert c.run(20000, path=path, threads=threads, vpt=vpt, group=group) == B.OK
        assert B.check_device_error() == B.ERR_TIMEOUT
    finally:
        B.set_wait_test(0, False)
    assert B.check_device_error() == B.OK
    # outputs were skipped, the context is still usable and the next call is exact
    run_and_compare(x, "bf16", path=path, threads=threads, vpt=vpt, group=group)


# -- the tensor-level binding --------------------------------------------------------------

@pytest.mark.parametrize("tdtype,name", [(torch.float32, "f32"), (torch.float16, "f16"), (torch.bfloat16, "bf16")])
def test_torch_binding(tdtype, name):
    g = torch.Generator(device="cpu").manual_seed(3)
    x = (torch.randn(37, 3001, generator=g) * 3).to(tdtype).cuda()
    y = B.softmax_fwd(x)
    ref = torch.softmax(x.double(), dim=1)
    assert (y.double() - ref).abs().max().item() <= {"f32": 1e-6, "f16": 1e-3, "bf16": 4e-3}[name]
    out = torch.empty_like(x)
    assert B.softmax_fwd(x, out) is out
    assert torch.equal(out, y)
    z = x.clone()
    B.softmax_fwd(z, z)
    assert torch.equal(z, y)
    big = torch.randn(8, 4000, device="cuda").to(tdtype)
    view = big[:, 100:3100]  # a strided, differently aligned view: row stride 4000
    tol = {"f32": 1e-6, "f16": 1e-3, "bf16": 4e-3}[name]
    vref = torch.softmax(view.double(), dim=1)
    assert (B.softmax_fwd(view).double() - vref).abs().max().item() <= tol
    assert (B.softmax_fwd(view.contiguous()).double() - vref).abs().max().item() <= tol
    with pytest.raises(ValueError):
        B.softmax_fwd(x.t())


# -- launch overlap (programmatic dependent launch) ----------------------------------------

def _bits_tensor(x: np.ndarray, dtype: str) -> torch.Tensor:
    a = W.bits_view(np.ascontiguousarray(x), dtype)
    return torch.from_numpy(a.view(np.int32) if dtype == "f32" else a.view(np.int16)).cuda()


OVERLAP_CASES = [(B.PATH_WARP, 700), (B.PATH_CTA, 3000), (B.PATH_CLUSTER, 20011), (B.PATH_STREAM, 20011),
                 (0, 65536)]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("path,cols", OVERLAP_CASES)
def test_launch_overlap_orders_against_neighbours(dtype, path, cols):
    """Calls issued back to back on one stream, with the overlap on: before
    each call a torch kernel rewrites the shared input buffer (the call must
    read the new data, not the old) and right after it the next rewrite
    follows (it must not land before the call has read).  Each output is
    checked against the oracle, and a chain of in-place calls matches the
    same chain run in plain stream order bit for bit."""
    skip_fp32_cluster(path, dtype)
    rows, k = 48, 5
    xs = [rnd(rows, cols, dtype, 900 + i) for i in range(k)]
    srcs = [_bits_tensor(x, dtype) for x in xs]
    buf = torch.empty_like(srcs[0])
    outs = [torch.empty_like(buf) for _ in range(k)]
    code = W.DTYPES.index(dtype)
    stream = torch.cuda.current_stream().cuda_stream
    B.set_force_path(path)
    try:
        B.set_launch_overlap(True)
        for i in range(k):
            buf.copy_(srcs[i])
            assert B.softmax_fwd_ptr(buf.data_ptr(), outs[i].data_ptr(), rows, cols, cols, code, stream) == B.OK
        chains = {}
        for overlap in (True, False):
            B.set_launch_overlap(overlap)
            z = srcs[0].clone()
            for _ in range(4):
                assert B.softmax_fwd_ptr(z.data_ptr(), z.data_ptr(), rows, cols, cols, code, stream) == B.OK
            chains[overlap] = z
        torch.cuda.synchronize()
        assert B.check_device_error() == B.OK
    finally:
        B.set_launch_overlap(True)
        B.set_force_path(0)
    for i in range(k):
        compare(outs[i].cpu().numpy().view(W.storage_dtype(dtype)), xs[i], dtype, cols)
    assert torch.equal(chains[True], chains[False])


@pytest.mark.parametrize("dtype", DTYPES)
def test_grid_launches_order_against_neighbours(dtype):
    """The grid path's three launches, back to back with the overlap on: each
    call's input is rewritten right before it and right after it, and a chain
    of calls ping-pongs between two buffers (the path does not run in place),
    matching the same chain in plain stream order bit for bit."""
    rows, cols, k = 3, 300_007, 4
    xs = [rnd(rows, cols, dtype, 950 + i) for i in range(k)]
    srcs = [_bits_tensor(x, dtype) for x in xs]
    buf = torch.empty_like(srcs[0])
    outs = [torch.empty_like(buf) for _ in range(k)]
    code = W.DTYPES.index(dtype)
    stream = torch.cuda.current_stream().cuda_stream
    B.set_force_path(B.PATH_GRID)
    try:
        B.set_launch_overlap(True)
        for i in range(k):
            buf.copy_(srcs[i])
            assert B.softmax_fwd_ptr(buf.data_ptr(), outs[i].data_ptr(), rows, cols, cols, code, stream) == B.OK
        chains = {}
        for overlap in (True, False):
            B.set_launch_overlap(overlap)
            z = [srcs[0].clone(), torch.empty_like(srcs[0])]
            for j in range(4):
                a, b = z[j % 2], z[1 - j % 2]
                assert B.softmax_fwd_ptr(a.data_ptr(), b.data_ptr(), rows, cols, cols, code, stream) == B.OK
            chains[overlap] = z[0]
        torch.cuda.synchronize()
        assert B.check_device_error() == B.OK
    finally:
        B.set_launch_overlap(True)
        B.set_force_path(0)
    for i in range(k):
        compare(outs[i].cpu().numpy().view(W.storage_dtype(dtype)), xs[i], dtype, cols)
    assert torch.equal(chains[True], chains[False])
