"""Thin Python binding of ``libsparse_mla.so`` (ctypes; argument marshalling only).

The names mirror the C ABI in ``include/sparse_mla.h``.  Torch supplies the
device memory and the stream; every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
the calls raise.

Argument checks mirror the pages' public entry ("Tuned sparse MLA prefill for
DSv4.1-Flash TP4; fix attn_sink in Triton fallback", description: a clear
error for a q that is not bf16, a kv dtype mismatch and a non-contiguous
``out``; ``out`` on q's device with a unit-stride last dim; and "Sparse MLA
training backward", review reply on host tensors: a named device error).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libsparse_mla.so")

SMLA_IDX_INT32 = 0
SMLA_IDX_INT64 = 1
SMLA_OK = 0

STATUS = {
    0: "SMLA_OK", 1: "SMLA_ERR_NULL_PTR", 2: "SMLA_ERR_BAD_SHAPE", 3: "SMLA_ERR_UNSUPPORTED_H",
    4: "SMLA_ERR_BAD_INDEX_DTYPE", 5: "SMLA_ERR_MISALIGNED", 6: "SMLA_ERR_BAD_SCALE",
    7: "SMLA_ERR_ALIASING", 8: "SMLA_ERR_CUDA", 9: "SMLA_ERR_DEVICE_TIMEOUT",
    10: "SMLA_ERR_BAD_SPLITS", 11: "SMLA_ERR_SCRATCH_LIMIT", 12: "SMLA_ERR_WORKSPACE",
}

# exported symbol -> (restype, argtypes)
_P, _I32, _I64, _F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
_U64 = ctypes.c_uint64
_FWD_ARGS = [_P, _P, _P, _I32, _P, _F32, _P, _P, _I64, _I32, _I64, _I32, _P]
SIGNATURES = {
    "sparse_mla_fwd": (_I32, _FWD_ARGS),
    "sparse_mla_fwd_ex": (_I32, _FWD_ARGS + [_I32, _P]),
    "sparse_mla_fwd_static_scratch": (_I32, _FWD_ARGS + [_I32]),
    "sparse_mla_fwd_host": (_I32, _FWD_ARGS[:-1] + [_P, _U64, _P]),
    "sparse_mla_fwd_host_workspace": (_I32, [_I64, _I32, _I32, _I64, _I32, _I32, _P]),
    "sparse_mla_fwd_dims": (_I32, _FWD_ARGS[:-1] + [_I32, _I32, _P]),
    "sparse_mla_fwd_fp8kv": (_I32, [_P, _P, _P, _P, _I32, _P, _F32, _P, _P, _I64, _I32, _I64,
                                    _I32, _P]),
    "sparse_mla_bwd": (_I32, [_P, _P, _P, _I32, _P, _F32, _P, _P, _P, _P, _P, _P, _I64, _I32,
                              _I64, _I32, _P, _U64, _P]),
    "sparse_mla_bwd_workspace": (_I32, [_I64, _I32, _I32, _I64, _P]),
    "sparse_mla_plan": (_I32, [_I64, _I32, _I32, _I32, _P, _P, _P]),
    "sparse_mla_launch_config": (_I32, [_I64, _I32, _I32, _I64, _I32, _P, _P, _P, _P]),
    "sparse_mla_device_status": (_I32, [_P]),
    "sparse_mla_selftest_wait_timeout": (_I32, [_P]),
    "sparse_mla_strerror": (ctypes.c_char_p, [_I32]),
    "sparse_mla_last_cuda_error": (ctypes.c_char_p, []),
    "sparse_mla_abi_version": (_I32, []),
}

_lib: Optional[ctypes.CDLL] = None


class SparseMLAError(RuntimeError):
    """A non-OK status from the library (``status`` holds the code)."""

    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}: {strerror(status)}"
        if status == 8:
            msg += f" [{last_cuda_error()}]"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load the library once; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().sparse_mla_strerror(int(status)).decode()


def last_cuda_error() -> str:
    return lib().sparse_mla_last_cuda_error().decode()


def abi_version() -> int:
    return int(lib().sparse_mla_abi_version())


def sparse_mla_plan(T: int, H: int, topk: int, num_splits: int = 0):
    """(kernel_family, splits, launches) the library would use."""
    fam, sp, ln = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = lib().sparse_mla_plan(T, H, topk, num_splits, ctypes.byref(fam), ctypes.byref(sp),
                               ctypes.byref(ln))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_plan")
    return fam.value, sp.value, ln.value


def sparse_mla_launch_config(T: int, H: int, topk: int, num_kv: int, num_splits: int = 0):
    """Launch geometry on the current device: dict(grid_ctas, threads, cluster, smem)."""
    v = [ctypes.c_int32() for _ in range(4)]
    st = lib().sparse_mla_launch_config(T, H, topk, num_kv, num_splits,
                                        *[ctypes.byref(x) for x in v])
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_launch_config")
    return dict(zip(("grid_ctas", "threads", "cluster", "smem"), (x.value for x in v)))


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_dev(name, x, dev):
    if not x.is_cuda:
        raise RuntimeError(f"{name} must be a CUDA tensor, got device {x.device}")
    if x.device != dev:
        raise RuntimeError(f"{name} is on {x.device}, expected {dev}")


def sparse_mla_fwd(q, kv, topk_indices, attn_sink=None, scale: Optional[float] = None,
                   out=None, lse=None, num_splits: int = 0, read_trace=None, stream=None):
    """Sparse MLA prefill forward; returns ``(out, lse)``.

    q ``[T, H, 512]`` bf16; kv ``[num_kv, 512]`` bf16 (K == V); topk_indices
    ``[T, topk]`` int32/int64 (any value outside ``[0, num_kv)`` is an invalid
    slot); attn_sink ``[H]`` fp32 or None; scale defaults to 1/sqrt(512).
    ``out`` (bf16, q's shape) and ``lse`` (fp32 ``[T, H]``) are allocated when
    not given.  ``num_splits`` and ``read_trace`` are the test controls of
    ``sparse_mla_fwd_ex``.
    """
    import torch
    if q.dim() != 3 or q.shape[-1] != 512:
        raise RuntimeError(f"q must be [T, H, 512], got {tuple(q.shape)}")
    if q.dtype != torch.bfloat16:
        raise RuntimeError(f"q must be bfloat16, got {q.dtype}")
    if kv.dtype != q.dtype:
        raise RuntimeError(f"kv dtype mismatch: kv is {kv.dtype}, q is {q.dtype}")
    if kv.dim() != 2 or kv.shape[-1] != 512:
        raise RuntimeError(f"kv must be [num_kv, 512], got {tuple(kv.shape)}")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    T, H, _ = q.shape
    if topk_indices.dim() != 2 or topk_indices.shape[0] != T:
        raise RuntimeError(f"topk_indices must be [T, topk], got {tuple(topk_indices.shape)}")
    dev = q.device
    for n, x in (("q", q), ("kv", kv), ("topk_indices", topk_indices)):
        _check_dev(n, x, dev)
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if attn_sink is not None:
        _check_dev("attn_sink", attn_sink, dev)
        if attn_sink.dtype != torch.float32 or tuple(attn_sink.shape) != (H,):
            raise RuntimeError(f"attn_sink must be float32 [{H}], got {attn_sink.dtype} "
                               f"{tuple(attn_sink.shape)}")
        if not attn_sink.is_contiguous():
            raise RuntimeError("attn_sink must be contiguous")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_dev("out", out, dev)
        if out.shape != q.shape or out.dtype != q.dtype:
            raise RuntimeError(f"out must match q ({tuple(q.shape)}, {q.dtype}), got "
                               f"{tuple(out.shape)}, {out.dtype}")
        if not out.is_contiguous():
            raise RuntimeError("out must be contiguous with a unit-stride last dim")
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    else:
        _check_dev("lse", lse, dev)
        if tuple(lse.shape) != (T, H) or lse.dtype != torch.float32 or not lse.is_contiguous():
            raise RuntimeError(f"lse must be contiguous float32 [{T}, {H}]")
    if read_trace is not None:
        _check_dev("read_trace", read_trace, dev)
        if read_trace.dtype != torch.int64 or read_trace.shape != topk_indices.shape:
            raise RuntimeError("read_trace must be int64 with topk_indices' shape")
    if scale is None:
        scale = 512 ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(dev):
        st = lib().sparse_mla_fwd_ex(
            q.data_ptr(), kv.data_ptr() if kv.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), T, H, kv.shape[0], topk_indices.shape[1],
            _stream_ptr(stream), int(num_splits),
            read_trace.data_ptr() if read_trace is not None else None)
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd")
    return out, lse


def sparse_mla_selftest_wait_timeout(stream=None) -> None:
    """Queue the bounded-wait self-test (its wait always expires after ~1 ms)."""
    st = lib().sparse_mla_selftest_wait_timeout(_stream_ptr(stream))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_selftest_wait_timeout")


def sparse_mla_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    import torch
    return int(lib().sparse_mla_device_status(_stream_ptr(stream) if torch.cuda.is_available()
                                              else None))


def sparse_mla_fwd_static_scratch(q, kv, topk_indices, out, lse, attn_sink=None,
                                  scale: Optional[float] = None, num_splits: int = 0,
                                  stream=None):
    """The split-TOPK forward with no device allocation at all; returns ``(out, lse)``.

    For callers that may not allocate while they run (a fixed memory budget, a
    window in which no allocation may happen, an allocator owned by someone else):
    ``out`` and ``lse`` must be passed in, and the split partials live in the
    library's own 16 MiB static array.  ``num_splits * T * H`` may not exceed
    8192.  Calls that overlap on the GPU share that array and race; run them
    on one stream.  The first call on a device sets up the array's address.
    """
    import torch
    if q.dtype != torch.bfloat16 or kv.dtype != q.dtype:
        raise RuntimeError(f"q and kv must be bfloat16, got {q.dtype} / {kv.dtype}")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    T, H, _ = q.shape
    dev = q.device
    for n, x in (("q", q), ("kv", kv), ("topk_indices", topk_indices), ("out", out), ("lse", lse)):
        _check_dev(n, x, dev)
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise RuntimeError("out must match q's shape and dtype")
    if tuple(lse.shape) != (T, H) or lse.dtype != torch.float32:
        raise RuntimeError(f"lse must be float32 [{T}, {H}]")
    if attn_sink is not None:
        _check_dev("attn_sink", attn_sink, dev)
        if attn_sink.dtype != torch.float32 or tuple(attn_sink.shape) != (H,):
            raise RuntimeError(f"attn_sink must be float32 [{H}]")
    if scale is None:
        scale = 512 ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(dev):
        st = lib().sparse_mla_fwd_static_scratch(
            q.data_ptr(), kv.data_ptr() if kv.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), T, H, kv.shape[0], topk_indices.shape[1],
            _stream_ptr(stream), int(num_splits))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd_static_scratch")
    return out, lse


def sparse_mla_fwd_host_workspace(T: int, H: int, topk: int, num_kv: int,
                                  index_dtype: int = SMLA_IDX_INT32, has_sink: bool = True) -> int:
    """Device workspace bytes of :func:`sparse_mla_fwd_host` for these sizes."""
    n = ctypes.c_uint64(0)
    st = lib().sparse_mla_fwd_host_workspace(int(T), int(H), int(topk), int(num_kv),
                                             int(index_dtype), 1 if has_sink else 0, ctypes.byref(n))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd_host_workspace")
    return int(n.value)


def sparse_mla_fwd_host(q, kv, topk_indices, out, lse, attn_sink=None, workspace=None,
                        scale: Optional[float] = None, stream=None):
    """The forward on HOST tensors (copies in, compute, copies out, overlapped).

    ``q``, ``kv``, ``topk_indices``, ``attn_sink`` (or None), ``out`` and
    ``lse`` are CPU tensors, best page-locked (``pin_memory()``) so that the
    copies overlap; ``workspace`` is a CUDA uint8 tensor of at least
    :func:`sparse_mla_fwd_host_workspace` bytes on the current device.  The
    results are in ``out`` / ``lse`` once ``stream`` (default: the current
    stream) has passed the call.  Returns ``(out, lse)``.
    """
    import torch
    if q.dtype != torch.bfloat16 or kv.dtype != q.dtype:
        raise RuntimeError(f"q and kv must be bfloat16, got {q.dtype} / {kv.dtype}")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    for n, x in (("q", q), ("kv", kv), ("topk_indices", topk_indices), ("out", out), ("lse", lse)):
        if x.is_cuda:
            raise RuntimeError(f"{n} must be a host (CPU) tensor for the host-buffer call")
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if attn_sink is not None and (attn_sink.is_cuda or attn_sink.dtype != torch.float32):
        raise RuntimeError("attn_sink must be a float32 host tensor")
    T, H, _ = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise RuntimeError("out must match q's shape and dtype")
    if tuple(lse.shape) != (T, H) or lse.dtype != torch.float32:
        raise RuntimeError(f"lse must be float32 [{T}, {H}]")
    if workspace is None or not workspace.is_cuda:
        raise RuntimeError("workspace must be a CUDA tensor")
    if scale is None:
        scale = 512 ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(workspace.device):
        st = lib().sparse_mla_fwd_host(
            q.data_ptr(), kv.data_ptr() if kv.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), T, H, kv.shape[0], topk_indices.shape[1],
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_ptr(stream))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd_host")
    return out, lse


def sparse_mla_bwd_workspace(T: int, H: int, topk: int, num_kv: int) -> int:
    """Device workspace bytes of :func:`sparse_mla_bwd` for these sizes."""
    n = ctypes.c_uint64(0)
    st = lib().sparse_mla_bwd_workspace(int(T), int(H), int(topk), int(num_kv), ctypes.byref(n))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_bwd_workspace")
    return int(n.value)


def sparse_mla_bwd(q, kv, topk_indices, out, lse, dout, attn_sink=None,
                   scale: Optional[float] = None, dq=None, dkv=None, dsink=None, workspace=None,
                   stream=None):
    """Training backward; returns ``(dq, dkv, dsink)`` (fp32; dsink None without a sink).

    ``out`` and ``lse`` are the forward's outputs for the same inputs, ``dout``
    the output gradient (bf16, q's shape).  ``dq`` / ``dkv`` / ``dsink`` and the
    CUDA uint8 ``workspace`` (at least :func:`sparse_mla_bwd_workspace` bytes)
    are allocated when not given.
    """
    import torch
    if q.dtype != torch.bfloat16 or kv.dtype != q.dtype:
        raise RuntimeError(f"q and kv must be bfloat16, got {q.dtype} / {kv.dtype}")
    if out.dtype != torch.bfloat16 or dout.dtype != torch.bfloat16:
        raise RuntimeError("out and dout must be bfloat16")
    if out.shape != q.shape or dout.shape != q.shape:
        raise RuntimeError("out and dout must have q's shape")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    T, H, _ = q.shape
    dev = q.device
    if tuple(lse.shape) != (T, H) or lse.dtype != torch.float32:
        raise RuntimeError(f"lse must be float32 [{T}, {H}]")
    for n, x in (("q", q), ("kv", kv), ("topk_indices", topk_indices), ("out", out),
                 ("lse", lse), ("dout", dout)):
        _check_dev(n, x, dev)
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if attn_sink is not None:
        _check_dev("attn_sink", attn_sink, dev)
        if attn_sink.dtype != torch.float32 or tuple(attn_sink.shape) != (H,):
            raise RuntimeError(f"attn_sink must be float32 [{H}]")
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    if dkv is None:
        dkv = torch.empty(kv.shape, dtype=torch.float32, device=dev)
    if dsink is None and attn_sink is not None:
        dsink = torch.empty(H, dtype=torch.float32, device=dev)
    for n, x, shp in (("dq", dq, tuple(q.shape)), ("dkv", dkv, tuple(kv.shape))):
        _check_dev(n, x, dev)
        if x.dtype != torch.float32 or tuple(x.shape) != shp or not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous float32 {shp}")
    topk = topk_indices.shape[1]
    need = sparse_mla_bwd_workspace(T, H, topk, kv.shape[0])
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check_dev("workspace", workspace, dev)
    if scale is None:
        scale = 512 ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(dev):
        st = lib().sparse_mla_bwd(
            q.data_ptr(), kv.data_ptr() if kv.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), dout.data_ptr(), dq.data_ptr(),
            dkv.data_ptr() if dkv.numel() else None,
            dsink.data_ptr() if dsink is not None else None, T, H, kv.shape[0], topk,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(),
            _stream_ptr(stream))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_bwd")
    return dq, dkv, dsink


def sparse_mla_fwd_dims(q, kv, topk_indices, attn_sink=None, scale: Optional[float] = None,
                        d_v: Optional[int] = None, out=None, lse=None, stream=None):
    """The forward at head dim ``d_qk = q.shape[-1]`` with values the first ``d_v``
    columns of each kv row (default all); returns ``(out [T, H, d_v], lse)``.

    Supported (d_qk, d_v): (512, 512), (128, 128), (576, 576) and (576, 512)
    (rows ``[512 no-pe | 64 pe]``: the positional part enters the scores only).
    ``scale`` defaults to 1/sqrt(d_qk).
    """
    import torch
    if q.dim() != 3 or kv.dim() != 2 or kv.shape[-1] != q.shape[-1]:
        raise RuntimeError(f"q [T, H, D] and kv [num_kv, D] must share D, got "
                           f"{tuple(q.shape)} / {tuple(kv.shape)}")
    if q.dtype != torch.bfloat16 or kv.dtype != q.dtype:
        raise RuntimeError(f"kv dtype mismatch or not bfloat16: q {q.dtype}, kv {kv.dtype}")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    T, H, d_qk = q.shape
    dv = d_qk if d_v is None else int(d_v)
    dev = q.device
    for n, x in (("q", q), ("kv", kv), ("topk_indices", topk_indices)):
        _check_dev(n, x, dev)
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if attn_sink is not None:
        _check_dev("attn_sink", attn_sink, dev)
        if attn_sink.dtype != torch.float32 or tuple(attn_sink.shape) != (H,):
            raise RuntimeError(f"attn_sink must be float32 [{H}]")
    if out is None:
        out = torch.empty((T, H, dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if tuple(out.shape) != (T, H, dv) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise RuntimeError(f"out must be contiguous bfloat16 [{T}, {H}, {dv}]")
    if scale is None:
        scale = d_qk ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(dev):
        st = lib().sparse_mla_fwd_dims(
            q.data_ptr(), kv.data_ptr() if kv.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), T, H, kv.shape[0], topk_indices.shape[1],
            d_qk, dv, _stream_ptr(stream))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd_dims")
    return out, lse


def sparse_mla_fwd_fp8kv(q, kv_fp8, kv_scale, topk_indices, attn_sink=None,
                         scale: Optional[float] = None, out=None, lse=None, stream=None):
    """The forward on an fp8 KV cache; returns ``(out, lse)``.

    ``kv_fp8`` is ``[num_kv, 512]`` uint8 (or torch.float8_e4m3fn) e4m3 codes and
    ``kv_scale`` ``[num_kv, 4]`` float32, one scale per 128-column block.
    """
    import torch
    if q.dim() != 3 or q.shape[-1] != 512 or q.dtype != torch.bfloat16:
        raise RuntimeError(f"q must be bfloat16 [T, H, 512], got {q.dtype} {tuple(q.shape)}")
    if kv_fp8.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        raise RuntimeError(f"kv_fp8 must hold e4m3 codes (uint8 / float8_e4m3fn), got {kv_fp8.dtype}")
    if kv_fp8.dim() != 2 or kv_fp8.shape[-1] != 512:
        raise RuntimeError(f"kv_fp8 must be [num_kv, 512], got {tuple(kv_fp8.shape)}")
    if kv_scale.dtype != torch.float32 or tuple(kv_scale.shape) != (kv_fp8.shape[0], 4):
        raise RuntimeError(f"kv_scale must be float32 [{kv_fp8.shape[0]}, 4]")
    if topk_indices.dtype not in (torch.int32, torch.int64):
        raise RuntimeError(f"topk_indices must be int32 or int64, got {topk_indices.dtype}")
    T, H, _ = q.shape
    dev = q.device
    for n, x in (("q", q), ("kv_fp8", kv_fp8), ("kv_scale", kv_scale),
                 ("topk_indices", topk_indices)):
        _check_dev(n, x, dev)
        if not x.is_contiguous():
            raise RuntimeError(f"{n} must be contiguous")
    if attn_sink is not None:
        _check_dev("attn_sink", attn_sink, dev)
        if attn_sink.dtype != torch.float32 or tuple(attn_sink.shape) != (H,):
            raise RuntimeError(f"attn_sink must be float32 [{H}]")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    if scale is None:
        scale = 512 ** -0.5
    idt = SMLA_IDX_INT64 if topk_indices.dtype == torch.int64 else SMLA_IDX_INT32
    with torch.cuda.device(dev):
        st = lib().sparse_mla_fwd_fp8kv(
            q.data_ptr(), kv_fp8.data_ptr() if kv_fp8.numel() else None,
            kv_scale.data_ptr() if kv_scale.numel() else None,
            topk_indices.data_ptr() if topk_indices.numel() else None, idt,
            attn_sink.data_ptr() if attn_sink is not None else None, float(scale),
            out.data_ptr(), lse.data_ptr(), T, H, kv_fp8.shape[0], topk_indices.shape[1],
            _stream_ptr(stream))
    if st != SMLA_OK:
        raise SparseMLAError(st, "sparse_mla_fwd_fp8kv")
    return out, lse
