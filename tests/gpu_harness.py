"""Helpers for the GPU parity tests: guarded device buffers around the C-ABI
call and element-wise comparison with the CPU oracle.

Tolerances (absolute, against the double-precision oracle on the same
quantised inputs): fp32 1e-6 with |1 - row sum| <= 1e-5, fp16 1e-3,
bf16 4e-3.  fp16/bf16 outputs are rounded once to a grid whose spacing below
1.0 is 2^-11 / 2^-8, so their rounding alone is at most 4.9e-4 / 1.95e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from memory_bound_row_softmax_gb300 import binding as B
from memory_bound_row_softmax_gb300 import workloads as W

TOL = {"f32": 1e-6, "f16": 1e-3, "bf16": 4e-3}
SUM_TOL_F32 = 1e-5
GUARD = 96                       # guard elements on each side of a matrix
GUARD_BITS = {"f32": 0x7FB0B0B0, "f16": 0x7D0B, "bf16": 0x7FB0}  # NaN payloads


def _torch_bits(a: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32))
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _np_bits(t: torch.Tensor, dtype: str) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(np.uint32) if dtype == "f32" else a.view(np.uint16)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits -> float64 (outputs of the GPU)."""
    bits = np.ascontiguousarray(bits)
    if dtype == "f32":
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


class DeviceCase:
    """A (rows, stride) matrix on the device between guard regions."""

    def __init__(self, x: np.ndarray, dtype: str, *, in_off: int = 0, out_off: int = 0, inplace: bool = False,
                 device: str = "cuda:0"):
        self.dtype = dtype
        self.rows, self.stride = x.shape
        self.es = W.ELEM_BYTES[dtype]
        n = self.rows * self.stride
        self.n = n
        self.in_off, self.out_off, self.inplace = in_off, (in_off if inplace else out_off), inplace
        fill = np.full(GUARD * 2 + in_off + n, GUARD_BITS[dtype],
                       dtype=np.uint32 if dtype == "f32" else np.uint16)
        fill[GUARD + in_off: GUARD + in_off + n] = W.bits_view(np.ascontiguousarray(x), dtype).ravel()
        self.d_in = _torch_bits(fill, dtype).to(device)
        if inplace:
            self.d_out = self.d_in
            self.host_out0 = fill.copy()
        else:
            out0 = np.full(GUARD * 2 + out_off + n, GUARD_BITS[dtype], dtype=fill.dtype)
            out0[GUARD + out_off: GUARD + out_off + n] = W.PAD_OUT[dtype]
            self.host_out0 = out0
            self.d_out = _torch_bits(out0, dtype).to(device)

    @property
    def in_ptr(self) -> int:
        return self.d_in.data_ptr() + (GUARD + self.in_off) * self.es

    @property
    def out_ptr(self) -> int:
        return self.d_out.data_ptr() + (GUARD + self.out_off) * self.es

    def run(self, cols: int, *, path: int = 0, threads: int = 0, vpt: int = 0, group: int = 0) -> int:
        B.set_force_path(path, threads, vpt, group)
        try:
            stream = torch.cuda.current_stream().cuda_stream
            st = B.softmax_fwd_ptr(self.in_ptr, self.out_ptr, self.rows, cols, self.stride,
                                   B.DTYPE_CODES[self.dtype], stream)
        finally:
            B.set_force_path(0)
        return st

    def result(self, cols: int) -> np.ndarray:
        """Output bits (rows, cols) after checking guards and padding are untouched."""
        torch.cuda.synchronize()
        out = _np_bits(self.d_out, self.dtype)
        lo, hi = GUARD + self.out_off, GUARD + self.out_off + self.n
        assert (out[:lo] == self.host_out0[:lo]).all(), "guard before the matrix was written"
        assert (out[hi:] == self.host_out0[hi:]).all(), "guard after the matrix was written"
        mat = out[lo:hi].reshape(self.rows, self.stride)
        ref = self.host_out0[lo:hi].reshape(self.rows, self.stride)
        assert (mat[:, cols:] == ref[:, cols:]).all(), "padding columns were written"
        return mat[:, :cols].copy()


def compare(y_bits: np.ndarray, x: np.ndarray, dtype: str, cols: int, rows=None, threads: int = 8) -> dict:
    """Compare GPU output bits with the oracle on the given rows (default all)."""
    y = decode(y_bits, dtype)
    ref = oracle.softmax(x, dtype, cols=cols, rows=rows, threads=threads)
    if rows is not None and y.shape[0] != len(rows):
        y = y[np.asarray(rows)]
    nan_ref = np.isnan(ref)
    assert (np.isnan(y) == nan_ref).all(), "NaN pattern differs from the oracle"
    fin = ~nan_ref
    err = float(np.abs(y[fin] - ref[fin]).max()) if fin.any() else 0.0
    assert err <= TOL[dtype], f"max abs err {err:.3e} > {TOL[dtype]:.0e} ({dtype})"
    out = {"max_abs_err": err}
    if dtype == "f32":
        ok_rows = ~nan_ref.any(axis=1)
        if ok_rows.any():
            s = np.abs(y[ok_rows].sum(axis=1) - 1.0).max()
            assert s <= SUM_TOL_F32, f"|1 - row sum| {s:.3e} > {SUM_TOL_F32:.0e}"
            out["max_sum_err"] = float(s)
    return out


def run_and_compare(x: np.ndarray, dtype: str, cols: int | None = None, *, rows=None, in_off=0, out_off=0,
                    inplace=False, path=0, threads=0, vpt=0, group=0) -> dict:
    cols = x.shape[1] if cols is None else cols
    case = DeviceCase(x, dtype, in_off=in_off, out_off=out_off, inplace=inplace)
    st = case.run(cols, path=path, threads=threads, vpt=vpt, group=group)
    assert st == B.OK, f"softmax_fwd returned {st}: {B.status_string(st)}"
    assert B.check_device_error() == B.OK
    y = case.result(cols)
    res = compare(y, x, dtype, cols, rows=rows)
    res["path"] = B.last_path()
    return res
