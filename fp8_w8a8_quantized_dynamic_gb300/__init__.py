"""FP8 (e4m3fn) W8A8 linear with dynamic per-tensor activation quantization, for sm_103a.

Thin ctypes binding over the C-ABI library libfp8w8a8.so (declared in include/fp8w8a8.h).
The functions carry the C names. PyTorch supplies device memory and the current CUDA
stream only; every step of the layer runs in the library's CUDA kernels. There is no CPU
fallback: a missing library raises.

Typical use::

    qw, s_w = fp8_quantize_weight(w)                 # once, at load (per-tensor)
    qw, s_w = fp8_quantize_weight(w, per_channel=True)
    y = fp8_linear(a, qw, s_w, bias)                 # every forward; dynamic s_a
    y = fp8_linear_channelwise(a, qw, s_w, bias)
    y = fp8_linear_static(a, s_a, qw, s_w)           # calibrated activation scale
    qw, s_w = fp8_quantize_weight(w, fmt="e5m2")     # the other FP8 format
    y = fp8_linear_ex(a, qw, s_w, fmt_a="e5m2", fmt_w="e5m2")
    y = fp8_linear_weight_only(a, qw, s_w, fmt_w="e5m2")  # bf16 A, FP8 weights up-converted
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

from ._build import LIB_PATH

FP8_OK = 0
FP8_ERR_INVALID_ARG = 1
FP8_ERR_MISALIGNED = 2
FP8_ERR_WORKSPACE = 3
FP8_ERR_CUDA = 4
FP8_ERR_TIMEOUT = 5
FP8_ERR_UNSUPPORTED_DEVICE = 6
FP8_QUANT_WORKSPACE_BYTES = 4352
FP8_E4M3, FP8_E5M2 = 0, 1
_FORMATS = {"e4m3": FP8_E4M3, "e5m2": FP8_E5M2}
FP8_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

_i64, _sz, _vp, _int = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int

_SIGNATURES = {
    "fp8_min_ld": (_i64, [_i64]),
    "fp8_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "fp8_uses_gemv": (_int, [_i64, _i64, _i64]),
    "fp8_set_gemv_max_m": (_int, [_int]),
    "fp8_quantize_weight": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _i64, _vp, _vp, _sz, _vp]),
    "fp8_quantize_act": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _sz, _vp]),
    "fp8_scaled_mm": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _int, _vp, _vp, _i64, _vp]),
    "fp8_linear": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "fp8_linear_channelwise": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "fp8_linear_noalloc": (_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _int, _vp, _vp, _i64, _vp]),
    "fp8_quantize_weight_ex": (_int, [_vp, _i64, _i64, _i64, _int, _int, _vp, _i64, _vp, _vp, _sz, _vp]),
    "fp8_quantize_act_ex": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _vp, _i64, _vp, _vp, _sz, _vp]),
    "fp8_scaled_mm_ex": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp,
                                _i64, _vp]),
    "fp8_linear_static": (_int, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _int, _vp, _vp, _i64, _vp,
                                 _sz, _vp]),
    "fp8_linear_ex": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp, _i64,
                             _vp, _sz, _vp]),
    "fp8_weight_only_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "fp8_linear_weight_only": (_int, [_vp, _i64, _i64, _i64, _vp, _int, _i64, _i64, _vp, _int, _vp, _vp, _i64,
                                      _vp, _sz, _vp]),
    "fp8_gemm_config": (_int, [_vp, _i64, _i64, _vp, _i64, _i64, _i64, _sz, _vp, _vp, _vp, _vp, _vp]),
    "fp8_gemm_plan_model": (_int, [_i64, _i64, _i64, _int, _int, _sz, _vp, _vp, _vp, _vp, _vp]),
    "fp8_gemv_plan_model": (_int, [_i64, _i64, _i64, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "fp8_last_device_status": (_int, [_vp]),
    "fp8_selftest_timeout": (_int, [_i64, _vp]),
    "fp8_status_string": (ctypes.c_char_p, [_int]),
}


class FP8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built (no fallback exists)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"FP8 CUDA library missing ({LIB_PATH}); build it with "
                                       "fp8_w8a8_quantized_dynamic_gb300._build.build()")
                L = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fp8_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != FP8_OK:
        raise FP8Error(status, where)


def min_ld(K: int) -> int:
    """Leading dimension (bytes) of the library's FP8 matrices: K rounded up to 16 (16 for K == 0)."""
    return (int(K) + 15) // 16 * 16 if K > 0 else 16


# ---------------------------------------------------------------------------
# torch-facing wrappers (torch is imported lazily: host-only users need none of it)
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_ptr(t) -> int:
    return _torch().cuda.current_stream(t.device).cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_bf16_2d(t, name: str):
    torch = _torch()
    if t.dtype != torch.bfloat16 or t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA bf16 matrix with unit column stride")


def _check_fp8_2d(t, K: int, name: str):
    torch = _torch()
    if t.dtype != torch.uint8 or t.dim() != 2 or t.stride(1) != 1 or not t.is_cuda or t.shape[1] < K:
        raise ValueError(f"{name}: expected a CUDA uint8 [rows, ld >= K] matrix")


def fp8_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().fp8_workspace_bytes(M, K, N))


def fp8_uses_gemv(M: int, K: int, N: int) -> bool:
    return bool(lib().fp8_uses_gemv(M, K, N))


def fp8_set_gemv_max_m(m: int) -> int:
    """Largest M that runs the decode GEMV (clamped to 0..16; m < 0 only queries); returns the previous value."""
    return int(lib().fp8_set_gemv_max_m(int(m)))


def fp8_min_ld(K: int) -> int:
    return int(lib().fp8_min_ld(K))


def fp8_status_string(status: int) -> str:
    return status_string(status)


def workspace(M: int, K: int, N: int, device):
    """Allocate a workspace big enough for fp8_linear on [M, K] x [N, K] (and any quantize call)."""
    torch = _torch()
    return torch.empty(fp8_workspace_bytes(M, K, N), dtype=torch.uint8, device=device)


def _fmt(name: str) -> int:
    if name not in _FORMATS:
        raise ValueError(f"unknown FP8 format {name!r} (expected 'e4m3' or 'e5m2')")
    return _FORMATS[name]


def fp8_quantize_weight(w, per_channel: bool = False, ws=None, fmt: str = "e4m3"
                        ) -> Tuple["torch.Tensor", "torch.Tensor"]:
    """W bf16 [N, K] -> (qW uint8 [N, min_ld(K)], s_w fp32 [1] or [N]); fmt 'e4m3' or 'e5m2'."""
    torch = _torch()
    _check_bf16_2d(w, "w")
    N, K = w.shape
    qw = torch.empty((N, min_ld(K)), dtype=torch.uint8, device=w.device)
    s_w = torch.empty((N if per_channel else 1,), dtype=torch.float32, device=w.device)
    if ws is None and not per_channel:
        ws = torch.empty(FP8_QUANT_WORKSPACE_BYTES, dtype=torch.uint8, device=w.device)
    args = (w.data_ptr(), N, K, w.stride(0), int(per_channel))
    tail = (qw.data_ptr(), qw.stride(0), s_w.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(), _stream_ptr(w))
    if fmt == "e4m3":
        _check(lib().fp8_quantize_weight(*args, *tail), "fp8_quantize_weight")
    else:
        _check(lib().fp8_quantize_weight_ex(*args, _fmt(fmt), *tail), "fp8_quantize_weight_ex")
    return qw, s_w


def fp8_quantize_act(a, ws=None, fmt: str = "e4m3", s_static=None):
    """A bf16 [M, K] -> (qA uint8 [M, min_ld(K)], s_a fp32 [1]).

    Dynamic s_a = amax(A) / max(fmt), or the given static scale s_static (device fp32 [1]).
    """
    torch = _torch()
    _check_bf16_2d(a, "a")
    M, K = a.shape
    qa = torch.empty((M, min_ld(K)), dtype=torch.uint8, device=a.device)
    s_a = torch.empty((1,), dtype=torch.float32, device=a.device)
    if ws is None and s_static is None:
        ws = torch.empty(FP8_QUANT_WORKSPACE_BYTES, dtype=torch.uint8, device=a.device)
    if fmt == "e4m3" and s_static is None:
        _check(lib().fp8_quantize_act(a.data_ptr(), M, K, a.stride(0), qa.data_ptr(), qa.stride(0), s_a.data_ptr(),
                                      ws.data_ptr(), ws.numel(), _stream_ptr(a)), "fp8_quantize_act")
    else:
        _check(lib().fp8_quantize_act_ex(a.data_ptr(), M, K, a.stride(0), _fmt(fmt), _ptr(s_static), qa.data_ptr(),
                                         qa.stride(0), s_a.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(),
                                         _stream_ptr(a)), "fp8_quantize_act_ex")
    return qa, s_a


def fp8_scaled_mm(qa, K: int, s_a, qw, s_w, per_channel: bool = False, bias=None, out=None,
                  fmt_a: str = "e4m3", fmt_w: str = "e4m3"):
    """Y = bf16(s_a * s_w * (qA @ qW^T) (+ bias)) on already-quantized operands."""
    torch = _torch()
    _check_fp8_2d(qa, K, "qa")
    _check_fp8_2d(qw, K, "qw")
    M, N = qa.shape[0], qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=qa.device)
    if fmt_a == "e4m3" and fmt_w == "e4m3":
        _check(lib().fp8_scaled_mm(qa.data_ptr(), M, K, qa.stride(0), s_a.data_ptr(), qw.data_ptr(), N,
                                   qw.stride(0), s_w.data_ptr(), int(per_channel), _ptr(bias), y.data_ptr(),
                                   y.stride(0), _stream_ptr(qa)), "fp8_scaled_mm")
    else:
        _check(lib().fp8_scaled_mm_ex(qa.data_ptr(), _fmt(fmt_a), M, K, qa.stride(0), s_a.data_ptr(), qw.data_ptr(),
                                      _fmt(fmt_w), N, qw.stride(0), s_w.data_ptr(), int(per_channel), _ptr(bias),
                                      y.data_ptr(), y.stride(0), _stream_ptr(qa)), "fp8_scaled_mm_ex")
    return y


def _linear(fn_name: str, a, qw, s_w, bias, out, ws):
    torch = _torch()
    _check_bf16_2d(a, "a")
    M, K = a.shape
    _check_fp8_2d(qw, K, "qw")
    N = qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    L = lib()
    if ws is None:
        need = L.fp8_workspace_bytes(M, K, N)
        ws = workspace(M, K, N, a.device) if need else None
    fn = getattr(L, fn_name)
    _check(fn(a.data_ptr(), M, K, a.stride(0), qw.data_ptr(), N, qw.stride(0), s_w.data_ptr(), _ptr(bias),
              y.data_ptr(), y.stride(0), _ptr(ws), 0 if ws is None else ws.numel(), _stream_ptr(a)), fn_name)
    return y


def fp8_linear(a, qw, s_w, bias=None, out=None, ws=None):
    """Dynamic W8A8 linear, per-tensor weight scale s_w [1]: Y = A W^T (+ bias), bf16 out."""
    return _linear("fp8_linear", a, qw, s_w, bias, out, ws)


def fp8_linear_channelwise(a, qw, s_w, bias=None, out=None, ws=None):
    """Dynamic W8A8 linear, per-output-channel weight scales s_w [N]."""
    return _linear("fp8_linear_channelwise", a, qw, s_w, bias, out, ws)


def fp8_quantize_weight_ex(w, fmt: str, per_channel: bool = False, ws=None):
    """fp8_quantize_weight with an explicit FP8 format."""
    return fp8_quantize_weight(w, per_channel=per_channel, ws=ws, fmt=fmt)


def fp8_quantize_act_ex(a, fmt: str, s_static=None, ws=None):
    """fp8_quantize_act with an explicit FP8 format and an optional static scale."""
    return fp8_quantize_act(a, ws=ws, fmt=fmt, s_static=s_static)


def fp8_scaled_mm_ex(qa, fmt_a: str, K: int, s_a, qw, fmt_w: str, s_w, per_channel: bool = False, bias=None,
                     out=None):
    """fp8_scaled_mm with the FP8 formats of both operands."""
    return fp8_scaled_mm(qa, K, s_a, qw, s_w, per_channel=per_channel, bias=bias, out=out, fmt_a=fmt_a,
                         fmt_w=fmt_w)


def _prologue(a, qw, out, ws):
    torch = _torch()
    _check_bf16_2d(a, "a")
    M, K = a.shape
    _check_fp8_2d(qw, K, "qw")
    N = qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if ws is None:
        need = lib().fp8_workspace_bytes(M, K, N)
        ws = workspace(M, K, N, a.device) if need else None
    return M, K, N, y, ws


def fp8_linear_static(a, s_a, qw, s_w, per_channel: bool = False, bias=None, out=None, ws=None):
    """W8A8 linear with a static (calibrated) activation scale s_a (device fp32 [1])."""
    M, K, N, y, ws = _prologue(a, qw, out, ws)
    _check(lib().fp8_linear_static(a.data_ptr(), M, K, a.stride(0), s_a.data_ptr(), qw.data_ptr(), N, qw.stride(0),
                                   s_w.data_ptr(), int(per_channel), _ptr(bias), y.data_ptr(), y.stride(0),
                                   _ptr(ws), 0 if ws is None else ws.numel(), _stream_ptr(a)), "fp8_linear_static")
    return y


def fp8_linear_ex(a, qw, s_w, per_channel: bool = False, bias=None, out=None, ws=None,
                  fmt_a: str = "e4m3", fmt_w: str = "e4m3", s_static=None):
    """The general linear: FP8 formats of A and W, dynamic (s_static None) or static activation scale."""
    M, K, N, y, ws = _prologue(a, qw, out, ws)
    _check(lib().fp8_linear_ex(a.data_ptr(), M, K, a.stride(0), _fmt(fmt_a), _ptr(s_static), qw.data_ptr(),
                               _fmt(fmt_w), N, qw.stride(0), s_w.data_ptr(), int(per_channel), _ptr(bias),
                               y.data_ptr(), y.stride(0), _ptr(ws), 0 if ws is None else ws.numel(),
                               _stream_ptr(a)), "fp8_linear_ex")
    return y


def fp8_weight_only_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().fp8_weight_only_workspace_bytes(M, K, N))


def fp8_linear_weight_only(a, qw, s_w, per_channel: bool = False, bias=None, out=None, ws=None,
                           fmt_w: str = "e4m3"):
    """Weight-only FP8 linear: bf16 A times the exactly up-converted FP8 weights, scaled by s_w."""
    torch = _torch()
    _check_bf16_2d(a, "a")
    M, K = a.shape
    _check_fp8_2d(qw, K, "qw")
    N = qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if ws is None:
        need = fp8_weight_only_workspace_bytes(M, K, N)
        ws = torch.empty(need, dtype=torch.uint8, device=a.device) if need else None
    _check(lib().fp8_linear_weight_only(a.data_ptr(), M, K, a.stride(0), qw.data_ptr(), _fmt(fmt_w), N,
                                        qw.stride(0), s_w.data_ptr(), int(per_channel), _ptr(bias), y.data_ptr(),
                                        y.stride(0), _ptr(ws), 0 if ws is None else ws.numel(), _stream_ptr(a)),
           "fp8_linear_weight_only")
    return y


def fp8_linear_noalloc(a, qw, s_w, per_channel: bool = False, bias=None, out=None):
    """The linear without a workspace, for callers that cannot allocate device memory.

    Uses the library's fixed scratch array (FP8_NOALLOC_SCRATCH_BYTES per GPU) instead of
    a caller workspace; calls that overlap on the GPU share it and race. Only `out` (when
    omitted) is allocated here, by torch, for convenience; pass `out` to allocate nothing.
    """
    torch = _torch()
    _check_bf16_2d(a, "a")
    M, K = a.shape
    _check_fp8_2d(qw, K, "qw")
    N = qw.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check(lib().fp8_linear_noalloc(a.data_ptr(), M, K, a.stride(0), qw.data_ptr(), N, qw.stride(0),
                                    s_w.data_ptr(), int(per_channel), _ptr(bias), y.data_ptr(), y.stride(0),
                                    _stream_ptr(a)), "fp8_linear_noalloc")
    return y


def fp8_selftest_timeout(limit_ns: int = 20_000_000, stream=None) -> int:
    """Enqueue the failure-path self-test (a bounded device wait made to run out); returns the status."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    return int(lib().fp8_selftest_timeout(int(limit_ns), s))


def fp8_last_device_status(stream=None) -> int:
    """Synchronizes the stream; returns FP8_OK or the device-side error the kernels recorded."""
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    return int(lib().fp8_last_device_status(s))


def fp8_gemm_config(qa, qw, K: Optional[int] = None, ws_bytes: int = 0) -> dict:
    """The GEMM launch the library would use for FP8 operands qa [M, ld] and qw [N, ld] (K columns;
    default: the row length) with a linear workspace of ws_bytes, on the current device:
    {"two_sm": bool, "grid": int, "group_n": int, "splits": int, "tail_split": int}. Enqueues nothing."""
    two, grid, gn, sp, ts = (ctypes.c_int(0) for _ in range(5))
    K = qa.shape[1] if K is None else int(K)
    st = lib().fp8_gemm_config(qa.data_ptr(), qa.shape[0], qa.stride(0), qw.data_ptr(), qw.shape[0], qw.stride(0),
                               K, int(ws_bytes), ctypes.byref(two), ctypes.byref(grid), ctypes.byref(gn),
                               ctypes.byref(sp), ctypes.byref(ts))
    if st != FP8_OK:
        raise FP8Error(st, "fp8_gemm_config")
    return {"two_sm": bool(two.value), "grid": grid.value, "group_n": gn.value, "splits": sp.value,
            "tail_split": ts.value}


def fp8_gemm_plan_model(M: int, N: int, K: int, num_sms: int = 152, pair_slots: int = 76, ws_bytes: int = 0) -> dict:
    """The GEMM launch plan fp8_gemm_config would report for gap-free FP8 operands in a GPU's own
    memory, computed on the host (no device): same keys."""
    two, grid, gn, sp, ts = (ctypes.c_int(0) for _ in range(5))
    st = lib().fp8_gemm_plan_model(int(M), int(N), int(K), int(num_sms), int(pair_slots), int(ws_bytes),
                                   ctypes.byref(two), ctypes.byref(grid), ctypes.byref(gn), ctypes.byref(sp),
                                   ctypes.byref(ts))
    if st != FP8_OK:
        raise FP8Error(st, "fp8_gemm_plan_model")
    return {"two_sm": bool(two.value), "grid": grid.value, "group_n": gn.value, "splits": sp.value,
            "tail_split": ts.value}


def fp8_gemv_plan_model(M: int, N: int, K: int, mode: int, clusters_of_size, smem_limit: int = 227 * 1024,
                        static_scale: bool = False) -> dict:
    """The decode GEMV's launch configuration computed on the host (no device): mode 0 activations
    pre-quantized, 1 quantized in the kernel, 2 bf16 (weight-only); clusters_of_size[s - 1] =
    co-resident clusters of s CTAs, s = 1..8."""
    occ = (ctypes.c_int * 8)(*[int(x) for x in clusters_of_size])
    outs = [ctypes.c_int(0) for _ in range(7)]
    st = lib().fp8_gemv_plan_model(int(M), int(N), int(K), int(mode), int(bool(static_scale)), int(smem_limit),
                                   ctypes.cast(occ, ctypes.c_void_p), *[ctypes.byref(o) for o in outs])
    if st != FP8_OK:
        raise FP8Error(st, "fp8_gemv_plan_model")
    keys = ("cluster", "clusters", "stages", "kslice", "scratch_a", "cluster_amax", "tcgen05")
    return {k: o.value for k, o in zip(keys, outs)}


def min_workspace_bytes(M: int, K: int, N: int) -> int:
    """The least workspace fp8_linear accepts for this shape (no K split): 0 for decode shapes of
    up to 16 tokens, which the GEMV quantizes itself."""
    if M <= 0 or K <= 0 or (M <= 16 and fp8_uses_gemv(M, K, N)):
        return 0
    return FP8_QUANT_WORKSPACE_BYTES + M * min_ld(K)
