"""ctypes binding over the C ABI in ``include/mbrs_softmax.h``.

Argument marshalling only: every step of the softmax runs in the CUDA kernels
of ``_build/libmbrs_softmax.so``.  If that library has not been built, the
first call raises -- there is no other implementation to fall back to.
PyTorch supplies device memory and the current stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmbrs_softmax.so")

OK, ERR_NULL, ERR_SHAPE, ERR_STRIDE, ERR_DTYPE, ERR_OVERLAP, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_ALIGN, \
    ERR_ARG, ERR_SCRATCH_LIMIT = range(12)
PATH_AUTO, PATH_WARP, PATH_CTA, PATH_CLUSTER, PATH_SPLIT = range(5)  # PATH_SPLIT: softmax_fwd_noalloc only
PATH_STREAM, PATH_PACKED, PATH_GRID = 6, 7, 8
PATH_NAMES = {PATH_WARP: "warp", PATH_CTA: "cta", PATH_CLUSTER: "cluster", PATH_SPLIT: "split",
              PATH_STREAM: "stream", PATH_PACKED: "packed", PATH_GRID: "grid"}
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}

_i64, _u64, _int, _vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p


class Plan(ctypes.Structure):
    _fields_ = [("path", _int), ("threads", _int), ("vpt", _int), ("group", _int), ("launches", _int),
                ("vec_store", _int), ("grid", _i64), ("smem_bytes", _i64), ("scratch_bytes", _i64),
                ("hbm_bytes", _i64), ("whole_vectors", _int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class TuneResult(ctypes.Structure):
    _fields_ = [("plan", Plan), ("best_us", ctypes.c_double), ("auto_us", ctypes.c_double), ("candidates", _int)]


class AttentionPlan(ctypes.Structure):
    _fields_ = [("items", _i64), ("grid", _i64), ("head_group", _int), ("threads", _int), ("smem_bytes", _i64),
                ("tmem_columns", _int), ("flops", ctypes.c_double)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class Shape(ctypes.Structure):
    _fields_ = [("path", _int), ("threads", _int), ("vpt", _int), ("group", _int)]

    def as_tuple(self) -> tuple:
        return (self.path, self.threads, self.vpt, self.group)


# Every function the header declares, with its ctypes signature.
SIGNATURES = {
    "softmax_fwd": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "softmax_status_string": (ctypes.c_char_p, [_int]),
    "softmax_last_path": (_int, []),
    "softmax_set_force_path": (_int, [_int, _int, _int, _int]),
    "softmax_plan": (_int, [_u64, _u64, _i64, _i64, _i64, _int, _int, ctypes.POINTER(Plan)]),
    "softmax_check_device_error": (_int, [_vp]),
    "softmax_set_wait_test": (_int, [_i64, _int]),
    "softmax_set_launch_overlap": (_int, [_int]),
    "softmax_fwd_host": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp, _i64, _vp]),
    "softmax_host_workspace_bytes": (_i64, [_i64, _i64, _i64, _int, _i64]),
    "softmax_autotune": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp, _int, ctypes.POINTER(TuneResult)]),
    "softmax_tune_candidates": (_int, [_u64, _u64, _i64, _i64, _i64, _int, _int, ctypes.POINTER(Shape), _int]),
    "softmax_autotune_size": (_int, []),
    "softmax_autotune_clear": (_int, []),
    "softmax_abi_version": (_int, []),
    "softmax_fwd_noalloc": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "softmax_fwd_masked": (_int, [_vp, _vp, _i64, _i64, _i64, _int, ctypes.c_float, _i64, _i64, _vp]),
    "softmax_masked_copy": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _i64, _i64, _int, _vp]),
    "softmax_attention_fwd": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, ctypes.c_float, _vp]),
    "softmax_attention_fwd_counter": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _int, _int, ctypes.c_float,
                                             _vp, _vp]),
    "softmax_attention_set_wait_test": (_int, [_int]),
    "softmax_attention_plan": (_int, [_i64, _i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(AttentionPlan)]),
}

_lib = None
_lock = threading.Lock()


class SoftmaxError(RuntimeError):
    def __init__(self, status: int, what: str = "softmax_fwd"):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {_LIB_PATH} is missing: build it with "
                    "`python -m memory_bound_row_softmax_gb300.build` (there is no fallback path)")
            handle = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().softmax_status_string(status).decode()


def _torch_dtype_code(t) -> int:
    import torch
    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in codes:
        raise TypeError(f"softmax_fwd takes float32, float16 or bfloat16, not {t.dtype}")
    return codes[t.dtype]


def softmax_fwd_ptr(in_ptr: int, out_ptr: int, rows: int, cols: int, row_stride: int, dtype: int,
                    stream: int = 0) -> int:
    """Raw call: device addresses and sizes in, status out (no exception)."""
    return lib().softmax_fwd(in_ptr, out_ptr, rows, cols, row_stride, dtype, stream)


def softmax_fwd_noalloc_ptr(in_ptr: int, out_ptr: int, rows: int, cols: int, row_stride: int, dtype: int,
                            stream: int = 0) -> int:
    """Raw call of the entry point that allocates nothing (for callers that
    cannot allocate device memory; its scratch is a fixed array in the
    library).  Status out, no exception."""
    return lib().softmax_fwd_noalloc(in_ptr, out_ptr, rows, cols, row_stride, dtype, stream)


def softmax_fwd_masked_ptr(in_ptr: int, out_ptr: int, rows: int, cols: int, row_stride: int, dtype: int,
                           scale: float, causal_offset: int, rows_per_seq: int = 0, stream: int = 0) -> int:
    """Raw call of the scaled, causally masked softmax (status out)."""
    return lib().softmax_fwd_masked(in_ptr, out_ptr, rows, cols, row_stride, dtype, scale, causal_offset,
                                    rows_per_seq, stream)


def masked_copy_ptr(in_ptr: int, out_ptr: int, rows: int, cols: int, row_stride: int, dtype: int,
                    causal_offset: int, rows_per_seq: int = 0, threads: int = 0, stream: int = 0) -> int:
    """Raw call of the diagnostic softmax_masked_copy: the masked call's
    traffic (kept entries copied, the rest zeroed) with no arithmetic."""
    return lib().softmax_masked_copy(in_ptr, out_ptr, rows, cols, row_stride, dtype, causal_offset, rows_per_seq,
                                     threads, stream)


def _prepare(x, out, what: str):
    """Check a 2-D CUDA tensor (last dimension contiguous) and its output;
    returns (rows, cols, row_stride, dtype code, out)."""
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise TypeError(f"{what} needs a CUDA tensor")
    if x.dim() != 2:
        raise ValueError(f"{what} needs a 2-D tensor, got {tuple(x.shape)}")
    rows, cols = x.shape
    if cols > 1 and x.stride(1) != 1:
        raise ValueError("the last dimension must be contiguous (stride 1)")
    row_stride = x.stride(0) if rows > 1 else max(cols, x.stride(0))
    code = _torch_dtype_code(x)
    if out is None:
        out = torch.empty_strided((rows, cols), (row_stride, 1), dtype=x.dtype, device=x.device)
    else:
        if out.shape != x.shape or out.dtype != x.dtype or out.device != x.device:
            raise ValueError("out must match x in shape, dtype and device")
        o_stride = out.stride(0) if rows > 1 else row_stride
        if (cols > 1 and out.stride(1) != 1) or o_stride != row_stride:
            raise ValueError("out must have x's row stride")
    return rows, cols, row_stride, code, out


def _stream_handle(x, stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def softmax_fwd(x, out=None, stream=None):
    """Row softmax of a 2-D CUDA tensor (last dimension contiguous).

    ``out`` (optional) must have x's shape, dtype, device and row stride; it
    may be ``x`` itself.  Launches on ``stream`` (default: the current stream of
    x's device) and returns ``out``.
    """
    import torch
    rows, cols, row_stride, code, out = _prepare(x, out, "softmax_fwd")
    with torch.cuda.device(x.device):
        st = lib().softmax_fwd(x.data_ptr(), out.data_ptr(), rows, cols, row_stride, code, _stream_handle(x, stream))
    if st != OK:
        raise SoftmaxError(st)
    return out


def softmax_fwd_masked(x, scale: float = 1.0, causal_offset: int = 0, rows_per_seq: int = 0, out=None,
                       stream=None):
    """Softmax of scaled, causally masked rows: row r keeps the columns
    c <= (r mod rows_per_seq) + causal_offset (rows_per_seq 0: r itself), its
    scores are x * scale, masked outputs are 0 and masked inputs are never
    read.  Arguments otherwise as ``softmax_fwd``; returns ``out``."""
    import torch
    rows, cols, row_stride, code, out = _prepare(x, out, "softmax_fwd_masked")
    with torch.cuda.device(x.device):
        st = lib().softmax_fwd_masked(x.data_ptr(), out.data_ptr(), rows, cols, row_stride, code, float(scale),
                                      int(causal_offset), int(rows_per_seq), _stream_handle(x, stream))
    if st != OK:
        raise SoftmaxError(st, "softmax_fwd_masked")
    return out


def attention_fwd_ptr(q: int, k: int, v: int, o: int, batch: int, heads: int, n_ctx: int, head_dim: int,
                      dtype: int, causal: bool, sm_scale: float, stream: int = 0) -> int:
    """Raw call of the fused attention forward (status out)."""
    return lib().softmax_attention_fwd(q, k, v, o, batch, heads, n_ctx, head_dim, dtype, 1 if causal else 0,
                                       sm_scale, stream)


def attention_fwd_counter_ptr(q: int, k: int, v: int, o: int, batch: int, heads: int, n_ctx: int, head_dim: int,
                              dtype: int, causal: bool, sm_scale: float, counter: int, stream: int = 0) -> int:
    """Raw call of the fused attention forward with the caller's two work
    counters at device address ``counter`` (status out)."""
    return lib().softmax_attention_fwd_counter(q, k, v, o, batch, heads, n_ctx, head_dim, dtype,
                                               1 if causal else 0, sm_scale, counter, stream)


def attention_fwd(q, k, v, causal: bool = True, sm_scale: float | None = None, out=None, stream=None):
    """Fused attention forward O = softmax(Q K^T * sm_scale [causal]) V of
    [batch, heads, n_ctx, 128] contiguous fp16 / bf16 CUDA tensors (sm_scale
    defaults to 1 / sqrt(head_dim)); returns ``out``."""
    import torch
    for t in (q, k, v):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError("attention_fwd needs CUDA tensors")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError("attention_fwd needs contiguous [batch, heads, n_ctx, head_dim] tensors")
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k and v must have one shape and dtype")
    batch, heads, n_ctx, head_dim = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / float(head_dim) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of q's shape and dtype")
    with torch.cuda.device(q.device):
        st = attention_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), batch, heads, n_ctx,
                               head_dim, _torch_dtype_code(q), causal, float(sm_scale), _stream_handle(q, stream))
    if st != OK:
        raise SoftmaxError(st, "attention_fwd")
    return out


def host_workspace_bytes(rows: int, cols: int, row_stride: int, dtype, chunk_bytes: int = 0) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype
    n = lib().softmax_host_workspace_bytes(rows, cols, row_stride, code, chunk_bytes)
    if n < 0:
        raise SoftmaxError(-n, "softmax_host_workspace_bytes")
    return n


def softmax_fwd_host(x, out=None, workspace=None, stream=None, zero_copy: bool = False):
    """Row softmax of a 2-D CPU tensor (pinned for overlapping copies),
    written to ``out`` (a CPU tensor, default a new pinned one) through the
    library's chunked copy / softmax / copy pipeline on the current CUDA
    device.  ``workspace`` (a CUDA tensor) defaults to a new one of
    softmax_host_workspace_bytes.  ``zero_copy=True`` passes no workspace:
    the kernels read and write the host buffers in place (they must be memory
    the device reaches directly).  Synchronises ``stream`` before returning."""
    import torch
    if not isinstance(x, torch.Tensor) or x.is_cuda or x.dim() != 2:
        raise TypeError("softmax_fwd_host needs a 2-D CPU tensor")
    rows, cols = x.shape
    if cols > 1 and x.stride(1) != 1:
        raise ValueError("the last dimension must be contiguous (stride 1)")
    row_stride = x.stride(0) if rows > 1 else max(cols, x.stride(0))
    code = _torch_dtype_code(x)
    if out is None:
        out = torch.empty_strided((rows, cols), (row_stride, 1), dtype=x.dtype, pin_memory=True)
    elif out.shape != x.shape or out.dtype != x.dtype or out.is_cuda or (rows > 1 and out.stride(0) != row_stride):
        raise ValueError("out must be a CPU tensor with x's shape, dtype and row stride")
    if zero_copy:
        ws_ptr, ws_bytes = None, 0
    else:
        if workspace is None:
            workspace = torch.empty(max(host_workspace_bytes(rows, cols, row_stride, code), 1), dtype=torch.uint8,
                                    device="cuda")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    s = stream if stream is not None else torch.cuda.current_stream()
    handle = s.cuda_stream if hasattr(s, "cuda_stream") else int(s)
    st = lib().softmax_fwd_host(x.data_ptr(), out.data_ptr(), rows, cols, row_stride, code, ws_ptr, ws_bytes,
                                handle)
    if st != OK:
        raise SoftmaxError(st, "softmax_fwd_host")
    torch.cuda.current_stream().synchronize() if stream is None else s.synchronize()
    return out


def autotune(x, out=None, stream=None, iters: int = 20) -> dict:
    """softmax_autotune on a tensor (``out`` must be another buffer): time the
    candidate launch shapes and cache the fastest for calls of this shape."""
    import torch
    rows, cols, row_stride, code, out = _prepare(x, out, "autotune")
    if out.data_ptr() == x.data_ptr():
        raise ValueError("autotune needs an out buffer other than x")
    with torch.cuda.device(x.device):
        return autotune_ptr(x.data_ptr(), out.data_ptr(), rows, cols, row_stride, code, _stream_handle(x, stream),
                            iters)


def plan(in_addr: int, out_addr: int, rows: int, cols: int, row_stride: int, dtype,
         num_sms: int = 0) -> dict:
    """The launch softmax_fwd would make (host only when num_sms > 0)."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype
    p = Plan()
    st = lib().softmax_plan(in_addr, out_addr, rows, cols, row_stride, code, num_sms, ctypes.byref(p))
    if st != OK:
        raise SoftmaxError(st, "softmax_plan")
    return p.as_dict()


def set_force_path(path: int, threads: int = 0, vpt: int = 0, group: int = 0) -> None:
    st = lib().softmax_set_force_path(path, threads, vpt, group)
    if st != OK:
        raise SoftmaxError(st, "softmax_set_force_path")


def last_path() -> int:
    return lib().softmax_last_path()


def check_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    handle = s.cuda_stream if hasattr(s, "cuda_stream") else int(s)
    return lib().softmax_check_device_error(handle)


def set_wait_test(wait_limit_ns: int = 0, starve: bool = False) -> None:
    lib().softmax_set_wait_test(wait_limit_ns, 1 if starve else 0)


def attention_plan(batch: int, heads: int, n_ctx: int, head_dim: int = 128, dtype="f16", causal: bool = True,
                   num_sms: int = 0) -> dict:
    """The launch softmax_attention_fwd makes for a shape (host only when
    num_sms > 0); raises SoftmaxError for arguments the call would refuse."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype
    p = AttentionPlan()
    st = lib().softmax_attention_plan(batch, heads, n_ctx, head_dim, code, 1 if causal else 0, num_sms,
                                      ctypes.byref(p))
    if st != OK:
        raise SoftmaxError(st, "softmax_attention_plan")
    return p.as_dict()


def set_attention_wait_test(starve: bool = False) -> None:
    """Attention forward test hook: leave the first Q barrier of every block
    unarmed so that its bounded wait runs out (see set_wait_test for the limit)."""
    lib().softmax_attention_set_wait_test(1 if starve else 0)


def set_launch_overlap(enable: bool = True) -> None:
    """Programmatic dependent launch on (default) or off, process-wide."""
    lib().softmax_set_launch_overlap(1 if enable else 0)


def autotune_ptr(in_ptr: int, out_ptr: int, rows: int, cols: int, row_stride: int, dtype: int, stream: int = 0,
                 iters: int = 20) -> dict:
    """Time the candidate launch shapes for this call and cache the fastest
    (raises on a bad status).  Returns the kept plan and the timings."""
    r = TuneResult()
    st = lib().softmax_autotune(in_ptr, out_ptr, rows, cols, row_stride, dtype, stream, iters, ctypes.byref(r))
    if st != OK:
        raise SoftmaxError(st, "softmax_autotune")
    return {"plan": r.plan.as_dict(), "best_us": r.best_us, "auto_us": r.auto_us, "candidates": r.candidates}


def tune_candidates(in_addr: int, out_addr: int, rows: int, cols: int, row_stride: int, dtype) -> list:
    """The (path, threads, vpt, group) shapes softmax_autotune would time."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype
    n = lib().softmax_tune_candidates(in_addr, out_addr, rows, cols, row_stride, code, 0, None, 0)
    if n < 0:
        raise SoftmaxError(-n, "softmax_tune_candidates")
    arr = (Shape * max(n, 1))()
    lib().softmax_tune_candidates(in_addr, out_addr, rows, cols, row_stride, code, 0, arr, n)
    return [arr[i].as_tuple() for i in range(n)]


def autotune_size() -> int:
    return lib().softmax_autotune_size()


def autotune_clear() -> None:
    lib().softmax_autotune_clear()


def abi_version() -> int:
    return lib().softmax_abi_version()
