"""The seeded input generators: determinism, shapes and the stated distributions."""
import math

import numpy as np
import pytest

from memory_bound_row_softmax_gb300 import workloads as W


def test_splitmix_reference_values():
    # splitmix64 from state 0: the published first outputs of the generator
    # (Vigna's reference implementation, seed 0).
    gamma = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        z = np.arange(1, 4, dtype=np.uint64) * gamma
    got = [int(v) for v in W._mix64(z)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_streams_are_deterministic_and_independent():
    idx = np.arange(1000, dtype=np.uint64)
    a = W.uniform(3, 0, idx)
    assert (a == W.uniform(3, 0, idx)).all()
    assert not (a == W.uniform(3, 1, idx)).any()
    assert not (a == W.uniform(4, 0, idx)).any()
    assert ((a > 0) & (a < 1)).all()
    # any element can be regenerated alone
    assert W.uniform(3, 0, np.array([517], dtype=np.uint64))[0] == a[517]


def test_normal_moments():
    z = W.normal(1, 0, np.arange(400_000, dtype=np.uint64))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, np.inf, -np.inf, np.nan], dtype=np.float32)
    b = W.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 3*2^-8 is a tie -> even (1 + 2^-6)
    assert list(b[:6]) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F80, 0xFF80]
    assert b[6] & 0x7FFF == 0x7FC0


def test_config_shapes_and_padding():
    w = W.CONFIGS["c4"]
    x = W.make_input(w.with_rows(5))
    assert x.shape == (5, 4104) and x.dtype == np.uint16
    assert (x[:, 4096:] == W.PAD_IN["f16"]).all()
    # causal: entries past (r mod 4096) are -inf
    assert (x[3, 4:4096] == W.neg_inf_bits("f16")).all()
    assert not (x[3, :4] == W.neg_inf_bits("f16")).any()


def test_spike_rows():
    w = W.CONFIGS["c3"]
    rows, cols = W.spike_plan(w)
    assert len(rows) == 205 == round(0.05 * 4096)
    assert len(set(rows.tolist())) == 205
    small = w.with_rows(4096)
    assert small.rows == 4096


@pytest.mark.parametrize("dtype", W.DTYPES)
def test_make_random_dtype(dtype):
    x = W.make_random(3, 10, dtype, seed=1, row_stride=12)
    assert x.shape == (3, 12)
    assert x.dtype == (np.float32 if dtype == "f32" else np.uint16)


def test_vocab_ranks_are_permutations():
    w = W.Workload("v", 3, 64, "bf16", 4, "vocab", zipf_s=1.1)
    v = W._row_block_values(w, 0, 3)
    g = W.gumbel(4, 0, np.arange(3 * 64, dtype=np.uint64)).reshape(3, 64)
    ranks = np.exp((g - v) / 1.1)
    for r in range(3):
        assert sorted(np.rint(ranks[r]).astype(int).tolist()) == list(range(1, 65))


def test_sweep_widths():
    assert len(W.SWEEP_WIDTHS) == 20
    assert W.SWEEP_WIDTHS[0] == 32 and W.SWEEP_WIDTHS[-1] == 16384 + 7
    w = W.sweep_workload(4103)
    assert w.rows == 50_000_000 // 4103
    assert math.isclose(w.rows * w.cols * 4, 200e6, rel_tol=1e-3)


def test_attention_workloads_are_the_pages_shapes():
    # batch 4, 32 heads, head dim 128, fp16, causal (the pages' attention table)
    for key in ("a4k", "a16k"):
        w = W.ATTENTION_CONFIGS[key]
        assert (w.batch, w.heads, w.head_dim, w.dtype, w.causal) == (4, 32, 128, "f16", True)
    assert W.ATTENTION_CONFIGS["a4k"].n_ctx == 4096 and W.ATTENTION_CONFIGS["a16k"].n_ctx == 16384
    w = W.ATTENTION_CONFIGS["a4k"]
    assert w.flops() == 4.0 * 4 * 32 * 4096 * 4096 * 128 / 2


def test_qkv_heads_are_slices_of_the_whole():
    # any head range regenerates exactly the same bits as the whole tensor
    w = W.AttentionWorkload("t", 2, 3, 70, 128, "bf16", seed=3, causal=False)
    q, k, v = W.make_qkv(w, chunk_heads=4)
    assert q.shape == (2, 3, 70, 128) and q.dtype == np.uint16
    flat = {"q": q.reshape(6, 70, 128), "k": k.reshape(6, 70, 128), "v": v.reshape(6, 70, 128)}
    for which in ("q", "k", "v"):
        part = W.qkv_heads(w.seed, which, 2, 5, 70, 128, "bf16")
        assert (part == flat[which][2:5]).all()
    # Q, K and V come from different streams
    assert not (q == k).all() and not (k == v).all()
    vals = q.astype(np.uint32) << 16
    x = vals.view(np.float32)
    assert abs(float(x.mean())) < 0.05 and 0.9 < float(x.std()) < 1.1
