"""Fused attention forward (softmax_attention_fwd) against the oracle's
one-head attention in double precision, on the same quantised inputs.

Tolerance, per output element o (derived from the kernel's arithmetic): with
u the unit roundoff of the 16-bit type (2^-11 fp16, 2^-8 bf16),
  * P is rounded to the type before the second product while the normaliser
    sums the unrounded fp32 values: |sum_j p_j e_j v_j| / l <= u max|v|;
  * O is rounded once: u |o|;
  * fp32 work: the scores' fp32 sums over 128 products perturb each exponent
    by at most 128 * 2^-24 * scale * sum_c |q_c k_c| (counted twice: numerator
    and normaliser), the PV sums over n kept keys add n * 2^-24 max|v|, and
    ex2.approx adds about 2^-22 relative twice (taken as 2^-21).
so |o_gpu - o| <= (u + 2 * score_err + n 2^-24 + 2^-21) max|v| + u |o|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import build as build_mod
from memory_bound_row_softmax_gb300 import workloads as W

from gpu_harness import decode

pytestmark = pytest.mark.gpu

U = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}
CODE = {"f16": 1, "bf16": 2}
D = 128
GUARD_ELEMS = 256  # guard elements on each side of O (512 bytes)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_mod.build()
    yield
    assert B.check_device_error() == B.OK


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(TORCH[dtype])


def from_dev(t: torch.Tensor, dtype: str) -> np.ndarray:
    return decode(t.view(torch.int16).cpu().numpy().view(np.uint16), dtype)


def run(q, k, v, dtype, causal, scale=None, guard=True):
    """softmax_attention_fwd on storage arrays [b, h, n, d]; returns O (float64)
    and checks that the guard regions around O were not written."""
    b, h, n, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype)
    total = b * h * n * d
    buf = torch.full((total + 2 * GUARD_ELEMS,), 0x7D0B, dtype=torch.int16, device="cuda")
    out_ptr = buf.data_ptr() + GUARD_ELEMS * 2
    st = B.attention_fwd_ptr(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), out_ptr, b, h, n, d, CODE[dtype], causal,
                             scale, torch.cuda.current_stream().cuda_stream)
    assert st == B.OK, B.status_string(st)
    torch.cuda.synchronize()
    assert B.check_device_error() == B.OK
    raw = buf.cpu().numpy()
    if guard:
        assert (raw[:GUARD_ELEMS] == 0x7D0B).all() and (raw[GUARD_ELEMS + total:] == 0x7D0B).all()
    return decode(raw[GUARD_ELEMS:GUARD_ELEMS + total].view(np.uint16), dtype).reshape(b, h, n, d)


def row_tolerance(q, k, v, dtype, scale, causal, rows=None):
    """Per-row bound of the module docstring for one head: q, k, v decoded to
    float64 (n, d); returns an (n_rows, 1) array."""
    n = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    qa, ka = np.abs(q[rows]), np.abs(k)
    score_err = 128 * 2.0 ** -24 * scale * (qa @ ka.T)           # (rows, n)
    keep = np.arange(n)[None, :] <= rows[:, None] if causal else np.ones((len(rows), n), bool)
    n_kept = keep.sum(axis=1)
    se = np.where(keep, score_err, 0).max(axis=1)
    vmax = np.array([np.abs(v[:c]).max() if causal else np.abs(v).max() for c in n_kept])
    return ((U[dtype] + 2 * se + n_kept * 2.0 ** -24 + 2.0 ** -21) * vmax)[:, None]


def check_head(o_gpu, q, k, v, dtype, scale, causal, rows=None):
    """One head against the oracle (all rows, or the listed query rows)."""
    qd, kd, vd = (decode(a, dtype) for a in (q, k, v))
    if rows is None:
        ref = oracle.attention_fwd(q, k, v, dtype, scale, causal=causal)
        got = o_gpu
    else:
        ref = np.concatenate([oracle.attention_fwd(q[i:i + 1], k, v, dtype, scale, causal=causal, causal_offset=i)
                              for i in rows])
        got = o_gpu[rows]
    tol = row_tolerance(qd, kd, vd, dtype, scale, causal, rows) + U[dtype] * np.abs(ref)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{len(bad)} elements off; first {bad[0]}: got {got[tuple(bad[0])]}, " \
                          f"ref {ref[tuple(bad[0])]}, tol {tol[bad[0][0], 0]}"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("b,h,n", [(1, 1, 128), (1, 1, 1), (1, 2, 200), (2, 1, 384), (1, 1, 1000), (1, 1, 129)])
def test_parity_small(dtype, causal, b, h, n):
    w = W.AttentionWorkload("t", b, h, n, D, dtype, seed=100 + n, causal=causal)
    q, k, v = W.make_qkv(w)
    scale = 1.0 / math.sqrt(D)
    o = run(q, k, v, dtype, causal, scale)
    for bi in range(b):
        for hi in range(h):
            check_head(o[bi, hi], q[bi, hi], k[bi, hi], v[bi, hi], dtype, scale, causal)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("scale", [0.02, 0.5])
def test_parity_scales(dtype, scale):
    # a small scale flattens the weights over all keys; a large one makes them
    # peaked (exercises the moving shift and the O rescale)
    w = W.AttentionWorkload("t", 1, 2, 640, D, dtype, seed=7, causal=True)
    q, k, v = W.make_qkv(w)
    o = run(q, k, v, dtype, True, scale)
    for hi in range(2):
        check_head(o[0, hi], q[0, hi], k[0, hi], v[0, hi], dtype, scale, True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_rising_scores_rescale(dtype):
    # keys whose scores rise along the sequence: the running max moves by more
    # than the 2^8 slack from one key tile to the next, so O is rescaled often
    n = 768
    w = W.AttentionWorkload("t", 1, 1, n, D, dtype, seed=9, causal=True)
    q, k, v = W.make_qkv(w)
    qd = np.ones((1, 1, n, D))
    kd = np.repeat(np.linspace(-1.0, 1.0, n)[:, None], D, axis=1)[None, None]
    q, k = W.quantise(qd, dtype), W.quantise(kd, dtype)
    o = run(q, k, v, dtype, True, 0.5)
    check_head(o[0, 0], q[0, 0], k[0, 0], v[0, 0], dtype, 0.5, True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("causal", [True, False])
def test_ones_value_gives_ones(dtype, causal):
    # V = 1 everywhere: every output is sum_j p~_j / sum_j p_j = 1 within u
    w = W.AttentionWorkload("t", 1, 3, 333, D, dtype, seed=11, causal=causal)
    q, k, _ = W.make_qkv(w)
    v = W.quantise(np.ones(q.shape), dtype)
    o = run(q, k, v, dtype, causal)
    # The kernel forms sum_j p~_j / l with |sum p~ / sum p - 1| <= u (P
    # rounding) and fp32 sums and ex2 adding far less than u / 2, then rounds
    # to the 16-bit grid.  Near 1 that grid is 1 - u, 1, 1 + 2u (spacing u
    # below 1, 2u above), so every value within u + u/2 below 1, and every
    # value up to the tie at 1 + u above it, lands on 1 - u or 1: the bound
    # is exactly u, and the fp32 terms of the general bound do not widen it.
    assert np.abs(o - 1.0).max() <= U[dtype]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_causal_first_query_is_first_value(dtype):
    # under the causal mask query 0 sees key 0 only: its weight is exactly 1
    w = W.AttentionWorkload("t", 2, 2, 300, D, dtype, seed=13, causal=True)
    q, k, v = W.make_qkv(w)
    o = run(q, k, v, dtype, True)
    assert (o[:, :, 0, :] == decode(v[:, :, 0, :], dtype)).all()


def test_equal_keys_average_the_values():
    # all keys equal: every kept key has the same weight, so query i gets the
    # mean of V[0..i] (causal) -- a closed form independent of the oracle
    n, dtype = 300, "f16"
    w = W.AttentionWorkload("t", 1, 1, n, D, dtype, seed=17, causal=True)
    q, _, v = W.make_qkv(w)
    k = W.quantise(np.full((1, 1, n, D), 0.25), dtype)
    o = run(q, k, v, dtype, True)
    vd = decode(v[0, 0], dtype)
    mean = np.cumsum(vd, axis=0) / np.arange(1, n + 1)[:, None]
    assert np.abs(o[0, 0] - mean).max() <= U[dtype] * (np.abs(vd).max() + np.abs(mean).max()) + 1e-5


def sampled_check(w, heads):
    """Inputs from a seeded device generator; sampled query rows (tile edges,
    first and last, a few random ones) of the listed (batch, head) pairs are
    checked against the oracle one by one."""
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    shape = (w.batch, w.heads, w.n_ctx, w.head_dim)
    q, k, v = (torch.randn(shape, generator=g, device="cuda").to(TORCH[w.dtype]) for _ in range(3))
    o = B.attention_fwd(q, k, v, causal=w.causal)
    torch.cuda.synchronize()
    assert B.check_device_error() == B.OK
    scale = 1.0 / math.sqrt(w.head_dim)
    rng = np.random.default_rng(5)
    rows = sorted({0, 1, 127, 128, 129, 255, 256, 1000, 2047, 2048, w.n_ctx - 129, w.n_ctx - 1,
                   *rng.integers(0, w.n_ctx, 6).tolist()})
    for bi, hi in heads:
        bits = [t[bi, hi].view(torch.int16).cpu().numpy().view(np.uint16) for t in (q, k, v)]
        got = from_dev(o[bi, hi], w.dtype)
        check_head(got, bits[0], bits[1], bits[2], w.dtype, scale, w.causal, rows=rows)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_bench_size_sampled_rows(dtype):
    # the benchmarked configuration (B4 H32 N4096, causal), fp16 and bf16
    from dataclasses import replace
    w = replace(W.ATTENTION_CONFIGS["a4k"], dtype=dtype)
    sampled_check(w, [(0, 0), (w.batch - 1, w.heads - 1), (1, 17), (2, 5)])


@pytest.mark.parametrize("causal", [True, False])
def test_long_context_partial_head_group(causal):
    # N = 16384: the block order takes heads in groups of 6, so 7 heads make a
    # full group and a group of one; every head is checked on sampled rows
    w = W.AttentionWorkload("long", 1, 7, 16384, D, "f16", seed=23, causal=causal)
    sampled_check(w, [(0, h) for h in range(7)])


def test_repeatable():
    # the same inputs twice give the same bits (no dependence on timing)
    w = W.AttentionWorkload("t", 2, 2, 500, D, "bf16", seed=19, causal=True)
    q, k, v = W.make_qkv(w)
    a = run(q, k, v, "bf16", True)
    b = run(q, k, v, "bf16", True)
    assert (a == b).all()


def test_bad_arguments_launch_nothing():
    q = torch.zeros(1, 1, 128, D, dtype=torch.float16, device="cuda")
    o = torch.zeros_like(q)
    p = q.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert B.attention_fwd_ptr(p, p, p, p, 1, 1, 128, D, 1, True, 0.1, s) == B.ERR_OVERLAP
    assert B.attention_fwd_ptr(p, p, p, o.data_ptr() + 2, 1, 1, 128, D, 1, True, 0.1, s) == B.ERR_ALIGN
    assert B.attention_fwd_ptr(p, p, p, o.data_ptr(), 1, 1, 128, 64, 1, True, 0.1, s) == B.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (o == 0).all()


def test_wait_timeout_is_reported_and_recoverable():
    # every block's first Q barrier left unarmed: its bounded wait (1 ms here)
    # runs out, the launch takes its abort path (drains its loads and MMAs,
    # frees tensor memory, resets its work counter) and reports a timeout;
    # the next 65 launches -- more than the 64 work-counter slots, so the
    # aborted launch's slot is used again -- are exact
    w = W.AttentionWorkload("t", 2, 3, 700, D, "f16", seed=29, causal=True)
    q, k, v = W.make_qkv(w)
    dq, dk, dv = to_dev(q, "f16"), to_dev(k, "f16"), to_dev(v, "f16")
    out = torch.empty_like(dq)
    s = torch.cuda.current_stream().cuda_stream
    args = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), out.data_ptr(), 2, 3, 700, D, CODE["f16"], True,
            1.0 / math.sqrt(D), s)
    B.set_wait_test(1_000_000)
    B.set_attention_wait_test(True)
    try:
        assert B.attention_fwd_ptr(*args) == B.OK
        assert B.check_device_error() == B.ERR_TIMEOUT
    finally:
        B.set_attention_wait_test(False)
        B.set_wait_test(0)
    for _ in range(65):
        assert B.attention_fwd_ptr(*args) == B.OK
    assert B.check_device_error() == B.OK
    got = from_dev(out, "f16")
    scale = 1.0 / math.sqrt(D)
    for bi in range(2):
        for hi in range(3):
            check_head(got[bi, hi], q[bi, hi], k[bi, hi], v[bi, hi], "f16", scale, True)


def test_plain_call_refuses_capture():
    # a captured plain call would keep its library counter slot on every
    # replay: it returns SOFTMAX_ERR_ARG without launching, and the capture
    # ends with nothing in it
    w = W.AttentionWorkload("t", 1, 2, 256, D, "f16", seed=31, causal=True)
    q, k, v = W.make_qkv(w)
    dq, dk, dv = to_dev(q, "f16"), to_dev(k, "f16"), to_dev(v, "f16")
    out = torch.zeros_like(dq)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = B.attention_fwd_ptr(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), out.data_ptr(), 1, 2, 256, D,
                                 CODE["f16"], True, 0.1, s.cuda_stream)
        out.add_(0)  # one captured kernel, so that the graph is not empty
    assert st == B.ERR_ARG
    g.replay()
    torch.cuda.synchronize()
    assert (out == 0).all()


def test_graph_replays_beside_direct_calls():
    # stream A replays a graph of counter-variant calls (the caller's own
    # counters) while stream B makes plain calls (the library's slots) at the
    # same time; every output equals the one a lone plain call gives, bit for
    # bit (each item's arithmetic does not depend on which block takes it)
    w1 = W.AttentionWorkload("t", 1, 4, 1000, D, "f16", seed=33, causal=True)
    w2 = W.AttentionWorkload("t", 2, 2, 700, D, "f16", seed=34, causal=False)
    scale = 1.0 / math.sqrt(D)
    ins = []
    for w in (w1, w2):
        q, k, v = W.make_qkv(w)
        ins.append((w, to_dev(q, "f16"), to_dev(k, "f16"), to_dev(v, "f16")))

    def call(w, dq, dk, dv, o, stream, counter=None):
        a = (dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), w.batch, w.heads, w.n_ctx, D, CODE["f16"],
             w.causal, scale)
        if counter is None:
            return B.attention_fwd_ptr(*a, stream)
        return B.attention_fwd_counter_ptr(*a, counter, stream)

    refs = []
    for w, dq, dk, dv in ins:
        o = torch.empty_like(dq)
        assert call(w, dq, dk, dv, o, torch.cuda.current_stream().cuda_stream) == B.OK
        refs.append(o)
    torch.cuda.synchronize()

    counter = torch.zeros(2, dtype=torch.int32, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    w, dq, dk, dv = ins[0]
    outs_a = [torch.empty_like(dq) for _ in range(3)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=sa):
        for o in outs_a:  # three calls in a row on one counter
            assert call(w, dq, dk, dv, o, sa.cuda_stream, counter.data_ptr()) == B.OK
    wb, qb, kb, vb = ins[1]
    outs_b = [torch.empty_like(qb) for _ in range(4)]
    for rep in range(3):
        for o in outs_a:
            o.zero_()
        for o in outs_b:
            o.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(sa):
            g.replay()
        for o in outs_b:
            assert call(wb, qb, kb, vb, o, sb.cuda_stream) == B.OK
        torch.cuda.synchronize()
        assert B.check_device_error() == B.OK
        for o in outs_a:
            assert torch.equal(o, refs[0]), f"graph replay {rep}"
        for o in outs_b:
            assert torch.equal(o, refs[1]), f"direct call beside replay {rep}"
    assert (counter == 0).all()  # left zero by every call


def test_counter_argument_checks():
    p = torch.zeros(4096, dtype=torch.int16, device="cuda")
    o = torch.zeros(1 * 1 * 128 * D, dtype=torch.int16, device="cuda")
    c = torch.zeros(4, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    a = (p.data_ptr(), p.data_ptr(), p.data_ptr(), o.data_ptr(), 1, 1, 128, D, 1, True, 0.1)
    assert B.attention_fwd_counter_ptr(*a, 0, s) == B.ERR_NULL
    assert B.attention_fwd_counter_ptr(*a, c.data_ptr() + 4, s) == B.ERR_ALIGN
    assert B.attention_fwd_counter_ptr(*a, o.data_ptr() + 64, s) == B.ERR_OVERLAP
    torch.cuda.synchronize()
    assert (o == 0).all() and (c == 0).all()
