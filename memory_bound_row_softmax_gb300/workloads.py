"""Seeded synthetic inputs for the row-softmax workloads.

This module only makes input data: counter-based random numbers, their
quantisation to the storage dtype, and the shapes, strides and value
distributions of the workloads the pages measure.  It holds none of the
softmax arithmetic, so the GPU path, the CPU oracle, the tests and the bench
can all draw the same bits from it without sharing any of the method.

Random numbers come from the splitmix64 finaliser (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) applied to a
counter, so any element of any workload can be regenerated on its own and the
stream does not depend on numpy's generator versions.

Storage conventions (the same ones the C ABI takes):
  * f32 data is a ``numpy.float32`` array;
  * f16 and bf16 data are ``numpy.uint16`` arrays holding the raw bit patterns;
  * every matrix is row-major with shape ``(rows, row_stride)``; columns
    ``cols .. row_stride-1`` are padding and hold ``PAD_IN`` on input.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPES = ("f32", "f16", "bf16")
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

# Sentinels.  Input padding is a quiet NaN with a payload: a kernel that reads
# a padding column poisons its row.  Output padding is pre-filled with a
# different NaN payload that must survive the call bit for bit.
PAD_IN = {"f32": 0x7FE5A5A5, "f16": 0x7E5A, "bf16": 0x7FDA}
PAD_OUT = {"f32": 0xFFE5A5A5, "f16": 0xFE5A, "bf16": 0xFFDA}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    """Key of sub-stream ``stream`` of ``seed`` (each purpose draws its own)."""
    base = np.array([(seed * 0x100000001B3 + stream * 0x1F1F1F1F) & (2**64 - 1)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base * _GAMMA + _GAMMA)[0]


def u64(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """The 64-bit values at counter positions ``idx`` of one sub-stream."""
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        z = key + (idx.astype(np.uint64) + np.uint64(1)) * _GAMMA
    return _mix64(z)


def uniform(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1) from the top 53 bits."""
    return ((u64(seed, stream, idx) >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0**-53


def normal(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """Standard normal deviates by the Box-Muller transform (Box & Muller, 1958)."""
    idx = idx.astype(np.uint64)
    u1 = uniform(seed, stream, np.uint64(2) * idx)
    u2 = uniform(seed, stream, np.uint64(2) * idx + np.uint64(1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def gumbel(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    """Gumbel(0, 1) deviates: -ln(-ln U)."""
    return -np.log(-np.log(uniform(seed, stream, idx)))


# ---------------------------------------------------------------------------
# quantisation to storage bits
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns, round-to-nearest-even.

    NaN keeps its sign and becomes the quiet NaN 0x7FC0 (or 0xFFC0)."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x32)
    if nan.any():
        r[nan] = ((b[nan] >> np.uint32(16)).astype(np.uint16) & np.uint16(0x8000)) | np.uint16(0x7FC0)
    return r


def quantise(x: np.ndarray, dtype: str) -> np.ndarray:
    """float64 values -> storage array for ``dtype`` (see module doc)."""
    if dtype == "f32":
        return x.astype(np.float32)
    if dtype == "f16":
        with np.errstate(over="ignore"):
            return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        with np.errstate(over="ignore"):
            return f32_to_bf16_bits(x.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def bits_view(a: np.ndarray, dtype: str) -> np.ndarray:
    """Unsigned-integer view of a storage array (for bit-exact comparisons)."""
    return a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)


def neg_inf_bits(dtype: str) -> int:
    return {"f32": 0xFF800000, "f16": 0xFC00, "bf16": 0xFF80}[dtype]


def fill_bits(shape, dtype: str, bits: int) -> np.ndarray:
    """A storage array whose every element has the raw pattern ``bits``."""
    if dtype == "f32":
        return np.full(shape, bits, dtype=np.uint32).view(np.float32)
    return np.full(shape, bits, dtype=np.uint16)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One synthetic input matrix.

    kind:
      ``normal``   x ~ N(0, sigma^2)
      ``spike``    x ~ N(0, 1), then ``spike_rows`` seeded rows get one seeded
                   column set to (that row's max + 100)
      ``causal``   x ~ N(0,1)/sqrt(128)*8, entries with c > (r mod causal_period)
                   set to -inf
      ``vocab``    x = G - s*ln(pi_r(c)), G ~ Gumbel(0,1), pi_r a seeded per-row
                   permutation of the ranks 1..cols (Zipf(s) base probabilities)
      ``uniform``  x ~ U(lo, hi)
    """

    name: str
    rows: int
    cols: int
    dtype: str
    seed: int
    kind: str
    row_stride: int = 0
    sigma: float = 1.0
    spike_rows: int = 0
    causal_period: int = 0
    zipf_s: float = 0.0
    lo: float = 0.0
    hi: float = 0.0
    note: str = field(default="", compare=False)

    @property
    def stride(self) -> int:
        return self.row_stride or self.cols

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes a fused softmax must move: every valid element read once and written once."""
        return 2 * self.rows * self.cols * self.elem_bytes

    def with_rows(self, rows: int) -> "Workload":
        d = dict(self.__dict__)
        d["rows"] = rows
        return Workload(**d)


def _row_block_values(w: Workload, r0: int, r1: int) -> np.ndarray:
    """float64 values of rows [r0, r1) before quantisation (no spikes yet)."""
    n = r1 - r0
    idx = (np.arange(r0, r1, dtype=np.uint64)[:, None] * np.uint64(w.cols)
           + np.arange(w.cols, dtype=np.uint64)[None, :])
    if w.kind in ("normal", "spike"):
        return normal(w.seed, 0, idx) * w.sigma
    if w.kind == "causal":
        x = normal(w.seed, 0, idx) / math.sqrt(128.0) * 8.0
        r = np.arange(r0, r1)[:, None] % w.causal_period
        c = np.arange(w.cols)[None, :]
        x[c > r] = -np.inf
        return x
    if w.kind == "vocab":
        g = gumbel(w.seed, 0, idx)
        keys = uniform(w.seed, 1, idx)
        ranks = np.empty((n, w.cols), dtype=np.float64)
        order = np.argsort(keys, axis=1, kind="stable")
        rank_vals = np.arange(1, w.cols + 1, dtype=np.float64)
        np.put_along_axis(ranks, order, np.broadcast_to(rank_vals, (n, w.cols)), axis=1)
        return g - w.zipf_s * np.log(ranks)
    if w.kind == "uniform":
        return w.lo + (w.hi - w.lo) * uniform(w.seed, 0, idx)
    raise ValueError(f"unknown workload kind {w.kind!r}")


def spike_plan(w: Workload) -> tuple[np.ndarray, np.ndarray]:
    """(row indices, column indices) of the spiked entries of a ``spike`` workload.

    The rows are the first ``spike_rows`` of a seeded shuffle (sort by random
    key); each spiked row's column is uniform over [0, cols)."""
    keys = uniform(w.seed, 2, np.arange(w.rows, dtype=np.uint64))
    rows = np.sort(np.argsort(keys, kind="stable")[: w.spike_rows])
    cols = np.floor(uniform(w.seed, 3, rows.astype(np.uint64)) * w.cols).astype(np.int64)
    return rows, cols


def make_input(w: Workload, block_rows: int = 0) -> np.ndarray:
    """The quantised input of ``w`` as a (rows, stride) storage array."""
    out = fill_bits((w.rows, w.stride), w.dtype, PAD_IN[w.dtype])
    if w.rows == 0:
        return out
    if block_rows <= 0:
        block_rows = max(1, (1 << 22) // max(1, w.cols))
    for r0 in range(0, w.rows, block_rows):
        r1 = min(w.rows, r0 + block_rows)
        out[r0:r1, : w.cols] = quantise(_row_block_values(w, r0, r1), w.dtype)
    if w.kind == "spike" and w.spike_rows:
        assert w.dtype == "f32", "spike workloads are fp32"
        rows, cols = spike_plan(w)
        for r, c in zip(rows, cols):
            m = float(np.max(out[r, : w.cols].astype(np.float64)))
            out[r, c] = np.float32(m + 100.0)
    return out


def make_output(w: Workload) -> np.ndarray:
    """An output buffer for ``w``: every element, padding included, holds PAD_OUT."""
    return fill_bits((w.rows, w.stride), w.dtype, PAD_OUT[w.dtype])


def make_random(rows: int, cols: int, dtype: str, seed: int, *, row_stride: int = 0,
                kind: str = "normal", sigma: float = 1.0, lo: float = -100.0,
                hi: float = 100.0) -> np.ndarray:
    """A small seeded matrix for tests (``normal`` or ``uniform``)."""
    w = Workload(name="random", rows=rows, cols=cols, dtype=dtype, seed=seed, kind=kind,
                 row_stride=row_stride, sigma=sigma, lo=lo, hi=hi)
    return make_input(w)


# The workloads the pages measure, at the sizes and distributions they name.
CONFIGS: dict[str, Workload] = {
    "c1": Workload("c1_f32_64x1000", 64, 1000, "f32", 0, "normal",
                   note="fp32 64x1000, N(0,1): non-power-of-two width, launch-bound"),
    "c2": Workload("c2_f16_4096x2048", 4096, 2048, "f16", 1, "normal", sigma=3.0,
                   note="fp16 4096x2048, N(0,9): fp32 accumulation"),
    "c3": Workload("c3_f32_4096x4096_spike", 4096, 4096, "f32", 2, "spike", spike_rows=205,
                   note="fp32 4096x4096, N(0,1); 205 rows (5%) get one entry at row max + 100"),
    "c4": Workload("c4_f16_8192x4096_causal_s4104", 8192, 4096, "f16", 3, "causal",
                   row_stride=4104, causal_period=4096,
                   note="fp16 attention scores, causal -inf mask, row stride 4104"),
    "c5": Workload("c5_bf16_512x131072_vocab", 512, 131072, "bf16", 4, "vocab", zipf_s=1.1,
                   note="bf16 vocabulary logits: Gumbel(0,1) + Zipf(1.1) offsets"),
}

SWEEP_WIDTHS = tuple(sorted([2**k for k in range(5, 15)] + [2**k + 7 for k in range(5, 15)]))

# Shapes beside the pages' workloads that the benchmark also times: 16-bit
# rows just past a power of two whose byte stride is off the 16-byte grid
# (every row has its own alignment), and a few very long rows -- too few for
# a cluster of blocks per row to fill the GPU (decode-time vocabulary rows).
EXTRA_SHAPES: dict[str, Workload] = {
    "r1": Workload("ragged_f16_8192x2055", 8192, 2055, "f16", 41, "normal", sigma=3.0,
                   note="fp16 rows 4110 bytes apart: a different 16-byte phase per row"),
    "r2": Workload("ragged_bf16_16384x2049", 16384, 2049, "bf16", 42, "normal", sigma=3.0,
                   note="bf16 rows 4098 bytes apart: a different 16-byte phase per row"),
    "l1": Workload("few_f32_3x1000000", 3, 1_000_000, "f32", 43, "normal", sigma=3.0,
                   note="three fp32 rows of 10^6"),
    "l2": Workload("few_bf16_9x262144", 9, 262144, "bf16", 44, "normal", sigma=3.0,
                   note="nine bf16 vocabulary rows of 2^18"),
    "l3": Workload("few_f32_1x4000000", 1, 4_000_000, "f32", 45, "normal", sigma=3.0,
                   note="one fp32 row of 4 * 10^6"),
}


def sweep_workload(cols: int, total_elems: int = 50_000_000) -> Workload:
    """fp32 width-sweep matrix: about 200 MB per tensor, x ~ U(-100, 100)."""
    return Workload(f"sweep_f32_w{cols}", total_elems // cols, cols, "f32", 5 * 100003 + cols,
                    "uniform", lo=-100.0, hi=100.0,
                    note="fp32 width sweep, ~200 MB per tensor, U(-100,100)")


# ---------------------------------------------------------------------------
# attention inputs: Q, K, V of shape [batch, heads, n_ctx, head_dim]
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class AttentionWorkload:
    """The attention forward the pages benchmark (page "Dissecting Memory
    Bandwidth & SRAM Tiling in Triton", section "Benchmark Results": batch 4,
    32 heads, head dim 128, fp16, causal, context 1,024 .. 32,768).  Q, K and V
    are N(0, 1) quantised to ``dtype``, each from its own sub-stream."""
    name: str
    batch: int
    heads: int
    n_ctx: int
    head_dim: int
    dtype: str
    seed: int
    causal: bool = True

    @property
    def elems(self) -> int:
        return self.batch * self.heads * self.n_ctx * self.head_dim

    def flops(self) -> float:
        """Matmul FLOPs of the two products: 4 B H N^2 D, halved under a
        causal mask (the usual count for a causal attention forward)."""
        f = 4.0 * self.batch * self.heads * self.n_ctx * self.n_ctx * self.head_dim
        return f / 2 if self.causal else f


ATTENTION_CONFIGS: dict[str, AttentionWorkload] = {
    "a4k": AttentionWorkload("attn_f16_b4_h32_n4096_d128_causal", 4, 32, 4096, 128, "f16", 6),
    "a16k": AttentionWorkload("attn_f16_b4_h32_n16384_d128_causal", 4, 32, 16384, 128, "f16", 7),
    # a small case of the same kernel for detailed profiler captures
    "a4k_small": AttentionWorkload("attn_f16_b1_h8_n4096_d128_causal", 1, 8, 4096, 128, "f16", 8),
    # a profiler case of several full waves: 512 items on 152 persistent blocks
    "a4k_wave": AttentionWorkload("attn_f16_b2_h16_n4096_d128_causal", 2, 16, 4096, 128, "f16", 9),
}

QKV_STREAMS = {"q": 0, "k": 1, "v": 2}


def qkv_heads(seed: int, which: str, bh0: int, bh1: int, n_ctx: int, head_dim: int, dtype: str) -> np.ndarray:
    """Heads bh0 .. bh1-1 (flattened batch * heads index) of one of Q, K, V as
    a storage array of shape (bh1 - bh0, n_ctx, head_dim): element (bh, i, c)
    is normal deviate number (bh * n_ctx + i) * head_dim + c of its stream."""
    per_head = n_ctx * head_dim
    idx = np.arange(bh0 * per_head, bh1 * per_head, dtype=np.uint64)
    x = normal(seed, QKV_STREAMS[which], idx)
    return quantise(x, dtype).reshape(bh1 - bh0, n_ctx, head_dim)


def make_qkv(w: AttentionWorkload, chunk_heads: int = 8) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Q, K, V of a workload as storage arrays [batch, heads, n_ctx, head_dim]."""
    bh = w.batch * w.heads
    out = []
    for which in ("q", "k", "v"):
        parts = [qkv_heads(w.seed, which, h0, min(bh, h0 + chunk_heads), w.n_ctx, w.head_dim, w.dtype)
                 for h0 in range(0, bh, chunk_heads)]
        out.append(np.concatenate(parts).reshape(w.batch, w.heads, w.n_ctx, w.head_dim))
    return out[0], out[1], out[2]
