"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

None of these re-types the oracle's own formula.  Each check is chosen so that
a plausible slip in the oracle (no max shift, a wrong sign, a dropped exp, the
wrong stride or axis, a bad fp16/bf16 decode, a wrong merge factor) fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from memory_bound_row_softmax_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32(rows):
    return np.asarray(rows, dtype=np.float32).reshape(len(rows), -1)


# -- storage decoding ------------------------------------------------------

def test_f16_decoder_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_bf16_decoder_matches_the_top_half_of_binary32():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.decode(bits, "bf16")
    ref = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


# -- closed forms ----------------------------------------------------------

def test_log_ramp_gives_linear_weights():
    # softmax(ln 1 .. ln 5) = (1..5)/15; the only error is fp32 rounding of ln k
    # (relative <= 2^-24 on values <= ln 5), i.e. below 2e-7 relative.
    x = f32([[math.log(k) for k in range(1, 6)]])
    y = oracle.softmax(x, "f32")[0]
    np.testing.assert_allclose(y, np.arange(1, 6) / 15.0, rtol=2e-7, atol=0)


@pytest.mark.parametrize("a,b", [(0.0, 0.0), (1.5, -2.25), (-7.0, 3.0), (1000.0, 1001.0), (-80.0, 80.0)])
def test_two_entries_are_a_logistic_pair(a, b):
    y = oracle.softmax(f32([[a, b]]), "f32")[0]
    sig = lambda t: 1.0 / (1.0 + math.exp(-t)) if t > -700 else 0.0
    assert abs(y[0] - sig(a - b)) < 1e-15
    assert abs(y[1] - sig(b - a)) < 1e-15


def test_hand_table_3x5():
    # e^k to 17 significant digits (tables of the exponential), k = 0..4.
    E = {0: 1.0, 1: 2.7182818284590452, 2: 7.3890560989306502, 3: 20.085536923187668,
         4: 54.598150033144239}
    rows = [[0, 1, 2, 3, 4], [4, 4, 0, 0, 1], [2, 0, 2, 0, 2]]
    y = oracle.softmax(f32(rows), "f32")
    for r, row in enumerate(rows):
        m = max(row)
        den = sum(E[m - k] ** -1 for k in row)  # e^(k-m) = 1 / e^(m-k)
        for c, k in enumerate(row):
            assert abs(y[r, c] - (E[m - k] ** -1) / den) < 1e-15, (r, c)


@pytest.mark.parametrize("n", [1, 2, 3, 1000, 131072])
def test_constant_row_is_exactly_one_over_n(n):
    y = oracle.softmax(np.full((1, n), 0.3125, dtype=np.float32), "f32")[0]
    assert (y == 1.0 / n).all()


# -- invariants --------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_rows_sum_to_one(dtype):
    x = W.make_random(17, 257, dtype, seed=11, sigma=3.0)
    y = oracle.softmax(x, dtype)
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-12
    assert (y >= 0).all()


@pytest.mark.parametrize("k", [-50.0, 3.75, 1000.0])
def test_shift_invariance(k):
    # x on a 1/16 grid and k exact, so x and x + k are both exact in fp32.
    rng = np.random.default_rng(5)
    x = (rng.integers(-160, 160, size=(6, 37)) / 16.0).astype(np.float32)
    xs = (x.astype(np.float64) + k).astype(np.float32)
    assert (xs.astype(np.float64) - k == x.astype(np.float64)).all()
    np.testing.assert_allclose(oracle.softmax(xs, "f32"), oracle.softmax(x, "f32"), rtol=0, atol=1e-12)


def test_spike_row_stays_finite():
    # the C3 construction: one entry 100 above the row max.  exp(x) without the
    # max shift overflows here (e^1100), the shifted form does not.
    x = W.make_random(1, 4096, "f32", seed=2).astype(np.float64)
    x = x + 1000.0
    x[0, 77] = x[0].max() + 100.0
    x = x.astype(np.float32)
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(x.astype(np.float64).max()))
    y = oracle.softmax(x, "f32")[0]
    assert np.isfinite(y).all()
    assert abs(y[77] - 1.0) < 4096 * math.exp(-90)
    assert np.delete(y, 77).max() < math.exp(-90)


def test_one_hot_when_all_but_one_masked():
    x = np.full((3, 9), -np.inf, dtype=np.float32)
    x[0, 0] = 5.0
    x[1, 8] = -3.0
    x[2, 4] = 0.0
    y = oracle.softmax(x, "f32")
    expect = np.zeros((3, 9))
    expect[0, 0] = expect[1, 8] = expect[2, 4] = 1.0
    assert (y == expect).all()


def test_causal_rows_match_their_unmasked_prefix():
    # row r of the C4 construction is the softmax of its first (r mod P)+1 entries
    w = W.CONFIGS["c4"]
    x = W.make_input(w.with_rows(6)).copy()
    x16 = x[:, : w.cols]
    y = oracle.softmax(x, "f16", cols=w.cols)
    for r in range(6):
        k = r % w.causal_period + 1
        pre = oracle.softmax(np.ascontiguousarray(x16[r : r + 1, :k]), "f16")[0]
        assert np.abs(y[r, :k] - pre).max() < 1e-15
        assert (y[r, k:] == 0.0).all()


def test_row_stride_skips_padding():
    # the padding holds NaN: reading it would poison the row
    w = W.CONFIGS["c4"]
    x = W.make_input(w.with_rows(4))
    assert np.isnan(x[:, w.cols :].view(np.float16)).all()
    y = oracle.softmax(x, "f16", cols=w.cols)
    assert np.isfinite(y).all()
    dense = np.ascontiguousarray(x[:, : w.cols])
    assert (oracle.softmax(dense, "f16") == y).all()


def test_softmax_is_over_rows_not_columns():
    x = f32([[0.0, 0.0, 0.0], [0.0, 1.0, 2.0]])
    y = oracle.softmax(x, "f32")
    assert (y[0] == 1.0 / 3.0).all()
    assert np.argmax(y[1]) == 2


# -- readings where the pages are silent ---------------------------------------

def test_fully_masked_row_is_nan():
    x = np.full((1, 5), -np.inf, dtype=np.float32)
    assert np.isnan(oracle.softmax(x, "f32")).all()


@pytest.mark.parametrize("bad", [np.nan, np.inf])
def test_nan_or_plus_inf_poisons_the_row(bad):
    x = f32([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0]])
    x[1, 1] = bad
    y = oracle.softmax(x, "f32")
    assert np.isfinite(y[0]).all()
    assert np.isnan(y[1]).all()


# -- the pages' worked examples ---------------------------------------------------

def _golden(name):
    lines = [ln.split() for ln in open(os.path.join(GOLDEN, name)) if ln.strip() and not ln.startswith("#")]
    return lines


def test_tree_example_from_page3():
    g = _golden("page3_tree_reduction.txt")
    vals = [float(v) for v in g[0][1:]]
    rounds = [[float(v) for v in ln[1:]] for ln in g[1:]]
    m, l, trace = oracle.tree_merge(vals, [1.0] * len(vals))
    assert trace == rounds
    assert m == 9.5
    # the normaliser of four single-element states is sum e^(v - 9.5)
    assert abs(l - sum(math.exp(v - 9.5) for v in vals)) < 1e-15


def test_mask_example_from_page3():
    # -inf padding up to the block contributes nothing (exp(-inf) = 0)
    g = dict((ln[0], ln[1:]) for ln in _golden("page3_mask.txt"))
    n, block = int(g["n_cols"][0]), int(g["block"][0])
    mask = np.array([int(v) for v in g["mask"]], dtype=bool)
    assert (mask == (np.arange(block) < n)).all()
    x = W.make_random(1, n, "f32", seed=3)
    padded = np.full((1, block), -np.inf, dtype=np.float32)
    padded[0, mask] = x[0]
    yp = oracle.softmax(padded, "f32")[0]
    assert (yp[~mask] == 0.0).all()
    assert np.abs(yp[mask] - oracle.softmax(x, "f32")[0]).max() < 1e-16


def test_partition_example_from_page3():
    # the strided partition covers each column once, and folding each
    # thread's columns then merging the threads gives the direct row state
    g = _golden("page3_partition.txt")
    n = int(g[0][1])
    t = int(g[1][1])
    parts = {int(ln[1]): [int(v) for v in ln[2:]] for ln in g[2:]}
    assert parts == {k: list(range(k, n, t)) for k in range(t)}
    assert sorted(c for p in parts.values() for c in p) == list(range(n))
    x = W.make_random(1, n, "f32", seed=9, sigma=4.0)
    ms, ls = [], []
    for k in range(t):
        m, l = -math.inf, 0.0
        for c in parts[k]:
            m, l = oracle.merge(m, l, *oracle.row_stats(x, "f32", 0, c, c + 1))
        ms.append(m)
        ls.append(l)
    m, l, _ = oracle.tree_merge(ms, ls)
    md, ld = oracle.row_stats(x, "f32", 0, 0, n)
    assert m == md
    assert abs(l - ld) < 1e-13


# -- the merge rule and the online form -----------------------------------------------

def test_online_chunks_match_direct_state():
    rng = np.random.default_rng(7)
    x = W.make_random(4, 3001, "bf16", seed=13, sigma=6.0)
    for r in range(4):
        cuts = np.sort(rng.choice(np.arange(1, 3001), size=rng.integers(1, 40), replace=False))
        bounds = np.concatenate([[0], cuts, [3001]])
        m_on, l_on = oracle.online_stats(x, "bf16", r, bounds)
        m_d, l_d = oracle.row_stats(x, "bf16", r, 0, 3001)
        assert m_on == m_d
        assert abs(l_on - l_d) <= 1e-13 * l_d


def test_merge_identity_and_symmetry():
    assert oracle.merge(-math.inf, 0.0, 2.0, 3.0) == (2.0, 3.0)
    assert oracle.merge(2.0, 3.0, -math.inf, 0.0) == (2.0, 3.0)
    a = oracle.merge(1.0, 2.0, 4.0, 0.5)
    b = oracle.merge(4.0, 0.5, 1.0, 2.0)
    assert a[0] == b[0] == 4.0 and abs(a[1] - b[1]) < 1e-15
    # merging with exactly the page's factor e^(m1 - m): 2 e^-3 + 0.5
    assert abs(a[1] - (2.0 * math.exp(-3.0) + 0.5)) < 1e-15


# -- an independent library ------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_agrees_with_torch_softmax_in_double(dtype):
    x = W.make_random(9, 777, dtype, seed=21, sigma=5.0)
    xd = oracle.decode(x, dtype) if dtype != "f32" else x.astype(np.float64)
    ref = torch.softmax(torch.from_numpy(xd), dim=1).numpy()
    assert np.abs(oracle.softmax(x, dtype) - ref).max() < 1e-14


def test_threaded_rows_equal_serial_rows():
    x = W.make_random(37, 129, "f16", seed=4)
    a = oracle.softmax(x, "f16")
    b = oracle.softmax(x, "f16", threads=4)
    c = oracle.softmax(x, "f16", rows=[5, 0, 36])
    assert (a == b).all()
    assert (c == a[[5, 0, 36]]).all()


# -- the scaled, causally masked variant ------------------------------------------------------

@pytest.mark.parametrize("off,period", [(0, 0), (3, 0), (-2, 0), (0, 4), (1, 3)])
def test_masked_constant_rows_are_one_over_kept(off, period):
    # every kept entry of a constant row is 1/n, n = query + off + 1 (clamped); the rest 0
    rows, cols = 9, 6
    y = oracle.softmax_masked(np.full((rows, cols), 0.7, np.float32), "f32", 1.5, off, period)
    for r in range(rows):
        q = r % period if period > 0 else r
        n = min(max(q + off + 1, 0), cols)
        if n == 0:
            assert np.isnan(y[r]).all()
        else:
            assert np.abs(y[r, :n] - 1.0 / n).max() < 1e-15 and (y[r, n:] == 0).all()


@pytest.mark.parametrize("a,b,scale", [(0.0, 1.0, 0.125), (2.0, -3.0, 3.0), (-1.5, 4.25, 1.0 / 3.0)])
def test_masked_pair_is_a_logistic_in_the_scaled_gap(a, b, scale):
    # row 1 keeps two columns: p0 = 1 / (1 + e^(scale (b - a))), a closed form
    x = f32([[a, b, 9.0], [a, b, 9.0]])
    y = oracle.softmax_masked(x, "f32", scale, 0)
    p0 = 1.0 / (1.0 + math.exp(scale * (float(np.float32(b)) - float(np.float32(a)))))
    assert abs(y[1, 0] - p0) < 1e-15 and abs(y[1, 1] - (1 - p0)) < 1e-15 and y[1, 2] == 0
    assert y[0, 0] == 1.0 and (y[0, 1:] == 0).all()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("scale,off,period", [(0.5, 0, 0), (4.0, 5, 0), (0.25, -1, 7), (1.0, 0, 16)])
def test_masked_equals_plain_softmax_of_the_masked_scaled_matrix(dtype, scale, off, period):
    # With a power-of-two scale, x * scale is exact in every storage type, so the
    # masked softmax must equal the plain softmax of the matrix whose kept entries
    # are pre-scaled and whose masked entries are -inf (a different code path).
    rows, cols = 40, 33
    x = W.make_random(rows, cols, dtype, seed=11, sigma=2.0)
    vals = oracle.decode(W.bits_view(x, dtype), dtype) if dtype != "f32" else x.astype(np.float64)
    pre = vals * scale
    for r in range(rows):
        q = r % period if period > 0 else r
        pre[r, max(0, min(cols, q + off + 1)):] = -np.inf
    xs = W.quantise(pre, dtype)
    back = oracle.decode(W.bits_view(xs, dtype), dtype) if dtype != "f32" else xs.astype(np.float64)
    assert np.array_equal(back, pre)  # the pre-scaled matrix is exact in storage
    want = oracle.softmax(xs, dtype)
    got = oracle.softmax_masked(x, dtype, scale, off, period)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_masked_inputs_are_never_read():
    rows, cols = 12, 10
    x = W.make_random(rows, cols, "f32", seed=4)
    poisoned = x.copy()
    for r in range(rows):
        poisoned[r, r + 1:] = np.nan
    a = oracle.softmax_masked(x, "f32", 0.3, 0)
    b = oracle.softmax_masked(poisoned, "f32", 0.3, 0)
    assert np.array_equal(a, b) and np.isfinite(a).all()


def test_masked_rejects_a_scale_that_is_not_positive():
    x = np.zeros((2, 3), np.float32)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(AssertionError):
            oracle.softmax_masked(x, "f32", bad, 0)


# -- one head of attention (groundwork for the fused attention forward) -------------------------

def _qkv(n_q, n_k, d, dtype, seed):
    q = W.make_random(n_q, d, dtype, seed=seed, sigma=1.0)
    k = W.make_random(n_k, d, dtype, seed=seed + 1, sigma=1.0)
    v = W.make_random(n_k, d, dtype, seed=seed + 2, sigma=1.0)
    return q, k, v


def _dec(a, dtype):
    return a.astype(np.float64) if dtype == "f32" else oracle.decode(W.bits_view(a, dtype), dtype)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_attention_with_zero_queries_averages_the_kept_values(dtype):
    # Q = 0: every score is 0, the weights are uniform over the kept keys, so
    # output row i is the mean of the first i + 1 value rows (causal) or of all
    q, k, v = _qkv(6, 9, 8, dtype, 21)
    q[:] = W.quantise(np.zeros((6, 8)), dtype)
    vd = _dec(v, dtype)
    full = oracle.attention_fwd(q, k, v, dtype, 0.25)
    assert np.abs(full - vd.mean(axis=0)).max() < 1e-14
    causal = oracle.attention_fwd(q, k, v, dtype, 0.25, causal=True)
    for i in range(6):
        assert np.abs(causal[i] - vd[:i + 1].mean(axis=0)).max() < 1e-14


def test_attention_causal_rows_see_exactly_their_prefix():
    # query 0 of a causal head sees key 0 only: its output is value row 0
    # exactly; with offset -1 it sees nothing (NaN) and query 1 sees key 0;
    # an offset past every key keeps them all (the unmasked head)
    q, k, v = _qkv(5, 7, 4, "f32", 31)
    o = oracle.attention_fwd(q, k, v, "f32", 1.0, causal=True)
    assert np.array_equal(o[0], v[0].astype(np.float64))
    o = oracle.attention_fwd(q, k, v, "f32", 1.0, causal=True, causal_offset=-1)
    assert np.isnan(o[0]).all() and np.array_equal(o[1], v[0].astype(np.float64))
    full = oracle.attention_fwd(q, k, v, "f32", 1.0)
    assert np.array_equal(oracle.attention_fwd(q, k, v, "f32", 1.0, causal=True, causal_offset=10), full)
    two = oracle.attention_fwd(q, k, v, "f32", 1.0, causal=True, causal_offset=1)
    assert np.array_equal(two[5 - 1], oracle.attention_fwd(q[4:5], k[:6], v[:6], "f32", 1.0)[0])


def test_attention_with_one_dominant_key_returns_its_value():
    # a key aligned with the query and far larger than the rest: its weight
    # is 1 up to e^-90, so the output is its value row
    d = 16
    q = np.zeros((1, d), np.float32)
    q[0, 3] = 10.0
    k = W.make_random(8, d, "f32", seed=5, sigma=0.1)
    k[6, 3] = 10.0                                      # score 100 against about 1 for the others
    v = W.make_random(8, d, "f32", seed=6)
    o = oracle.attention_fwd(q, k, v, "f32", 1.0)
    assert np.abs(o[0] - v[6]).max() < 1e-30


def test_attention_is_linear_in_the_values_and_invariant_to_key_order():
    q, k, v = _qkv(4, 10, 8, "f32", 41)
    v2 = W.make_random(10, 8, "f32", seed=99)
    a = oracle.attention_fwd(q, k, v, "f32", 0.3)
    b = oracle.attention_fwd(q, k, v2, "f32", 0.3)
    vs = (v.astype(np.float64) + v2.astype(np.float64)).astype(np.float32)
    assert np.allclose(oracle.attention_fwd(q, k, vs, "f32", 0.3), a + b, atol=1e-6)
    perm = np.random.default_rng(0).permutation(10)
    c = oracle.attention_fwd(q, k[perm], v[perm], "f32", 0.3)
    assert np.abs(c - a).max() < 1e-12


def test_attention_scale_is_the_same_as_scaling_the_queries():
    # scale 2 on the scores equals doubled queries (exact in fp32) at scale 1
    q, k, v = _qkv(5, 6, 8, "f32", 51)
    assert np.array_equal(oracle.attention_fwd(q, k, v, "f32", 2.0), oracle.attention_fwd(q * 2, k, v, "f32", 1.0))
