"""Thin ctypes binding of libmoe.so (``include/moe.h``).

Argument marshalling only: every function below forwards device pointers,
sizes and the current CUDA stream to the C entry point of the same name and
raises :class:`MoeError` on a non-OK status.  All arithmetic runs in the
CUDA kernels of the library; there is no fallback.  The ``*_t`` helpers
allocate outputs with torch (plumbing) and call the same entry points.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_BF16, MOE_FP8_E4M3_B128 = 0, 1
MOE_EPI_STORE, MOE_EPI_SWIGLU, MOE_EPI_SWIGLU_QUANT_FP8 = 0, 1, 2
MOE_DEVERR_NONE, MOE_DEVERR_OFFSETS, MOE_DEVERR_TIMEOUT, MOE_DEVERR_ROUTE = 0, 1, 2, 3
MOE_FWD_HOST_IO = 1
MOE_FWD_GATHER = 2
MOE_FWD_FUSED_COMBINE = 4
MOE_FWD_STAGED_OUT = 8


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class ForwardArgs(C.Structure):
    _fields_ = [
        ("dtype", C.c_int), ("T", C.c_int), ("E", C.c_int), ("k", C.c_int), ("H", C.c_int),
        ("I", C.c_int), ("renormalize", C.c_int), ("flags", C.c_uint),
        ("logits", C.c_void_p), ("expert_bias", C.c_void_p), ("sentinel_mask", C.c_void_p),
        ("topk_ids", C.c_void_p), ("topk_w", C.c_void_p), ("x", C.c_void_p), ("W1", C.c_void_p),
        ("W1_scales", C.c_void_p), ("W2", C.c_void_p), ("W2_scales", C.c_void_p), ("out", C.c_void_p),
    ]


_P, _I, _S, _Z = C.c_void_p, C.c_int, C.c_int, C.c_size_t
_SIGS = {
    "moe_abi_version": (C.c_int, []),
    "moe_status_string": (C.c_char_p, [_I]),
    "moe_get_device_error": (_S, [_P, _P]),
    "moe_selftest_wait_timeout": (_S, [C.c_uint64, _P]),
    "moe_route_sort_workspace_size": (_Z, [_I, _I, _I]),
    "moe_route_sort": (_S, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P]),
    "moe_route_sort_noalloc": (_S, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_ep_local_ids": (_S, [_P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_act_quant_fp8": (_S, [_P, _I, _I, _P, _P, _P]),
    "moe_weight_quant_fp8": (_S, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_permute": (_S, [_I, _P, _P, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P]),
    "moe_grouped_gemm": (_S, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_gemm_gather": (_S, [_I, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "moe_grouped_gemm_dgrad_workspace_size": (C.c_size_t, [_I, _I, _I]),
    "moe_grouped_gemm_dgrad": (_S, [_P, _P, _P, _I, _I, _I, _I, _P, _P, C.c_size_t, _P]),
    "moe_grouped_gemm_wgrad_workspace_size": (C.c_size_t, [_I, _I, _I, _I]),
    "moe_grouped_gemm_wgrad": (_S, [_P, _P, _P, _I, _I, _I, _I, _P, _P, C.c_size_t, _P]),
    "moe_batched_matmul_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "moe_batched_matmul": (_S, [_I, _P, _P, _I, _I, _P, _I, _P, _P, _I, _I, _P, _P, _Z, _P]),
    "moe_grouped_gemm_combine_workspace_size": (_Z, [_I, _I]),
    "moe_grouped_gemm_combine": (_S, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_swiglu": (_S, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_combine": (_S, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_forward_workspace_size": (_Z, [C.POINTER(ForwardArgs)]),
    "moe_forward": (_S, [C.POINTER(ForwardArgs), _P, _Z, _P]),
}

_lib = None


def lib() -> C.CDLL:
    """Load libmoe.so (built in-tree by ``build.build()``); fails loudly if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m grouped_gemm_serving_gb300.build`")
        lb = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lb, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lb
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def status_string(status: int) -> str:
    """moe_status_string for error messages: never raises."""
    try:
        return moe_status_string(status)
    except Exception:  # noqa: BLE001 - used while reporting another error
        return "unknown"


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


# ---------------------------------------------------------------- raw entry points
def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_get_device_error(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word."""
    code = C.c_int32(0)
    st = lib().moe_get_device_error(C.addressof(code), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_CHECK, MOE_ERR_TIMEOUT):
        raise MoeError(st, "moe_get_device_error")
    return code.value


def moe_selftest_wait_timeout(limit_ns: int, stream=None):
    _check(lib().moe_selftest_wait_timeout(limit_ns, _stream(stream)), "moe_selftest_wait_timeout")


def moe_route_sort_workspace_size(T, E, k) -> int:
    return lib().moe_route_sort_workspace_size(T, E, k)


def moe_route_sort(logits, expert_bias, sentinel_mask, topk_ids, topk_w, T, E, k, renormalize,
                   sorted_rows, row_pos, offsets, ws, ws_bytes, stream=None):
    _check(lib().moe_route_sort(_p(logits), _p(expert_bias), _p(sentinel_mask), _p(topk_ids),
                                _p(topk_w), T, E, k, int(renormalize), _p(sorted_rows), _p(row_pos),
                                _p(offsets), _p(ws), ws_bytes, _stream(stream)), "moe_route_sort")


def moe_route_sort_noalloc(logits, expert_bias, sentinel_mask, topk_ids, topk_w, T, E, k, renormalize,
                           sorted_rows, row_pos, offsets, stream=None):
    """moe_route_sort with the histogram scratch in the library's static
    device array: for callers that cannot allocate device memory."""
    _check(lib().moe_route_sort_noalloc(_p(logits), _p(expert_bias), _p(sentinel_mask), _p(topk_ids),
                                        _p(topk_w), T, E, k, int(renormalize), _p(sorted_rows),
                                        _p(row_pos), _p(offsets), _stream(stream)),
           "moe_route_sort_noalloc")


def moe_ep_local_ids(topk_ids, T, k, E_global, first_expert, E_local, local_ids, stream=None):
    _check(lib().moe_ep_local_ids(_p(topk_ids), T, k, E_global, first_expert, E_local, _p(local_ids),
                                  _stream(stream)), "moe_ep_local_ids")


def moe_act_quant_fp8(x, M, K, q, scales, stream=None):
    _check(lib().moe_act_quant_fp8(_p(x), M, K, _p(q), _p(scales), _stream(stream)), "moe_act_quant_fp8")


def moe_weight_quant_fp8(w, E, N, K, q, scales, stream=None):
    _check(lib().moe_weight_quant_fp8(_p(w), E, N, K, _p(q), _p(scales), _stream(stream)),
           "moe_weight_quant_fp8")


def moe_permute(dtype, x, x_scales, T, H, k, sorted_rows, offsets, E, M_cap, xp, xp_scales, stream=None):
    _check(lib().moe_permute(dtype, _p(x), _p(x_scales), T, H, k, _p(sorted_rows), _p(offsets), E,
                             M_cap, _p(xp), _p(xp_scales), _stream(stream)), "moe_permute")


def moe_grouped_gemm(dtype, A, A_scales, B, B_scales, offsets, E, M_cap, N, K, epilogue, Cout,
                     C_scales, stream=None):
    _check(lib().moe_grouped_gemm(dtype, _p(A), _p(A_scales), _p(B), _p(B_scales), _p(offsets), E,
                                  M_cap, N, K, epilogue, _p(Cout), _p(C_scales), _stream(stream)),
           "moe_grouped_gemm")


def moe_grouped_gemm_gather(dtype, x, x_scales, T, k, sorted_rows, B, B_scales, offsets, E, M_cap, N, K,
                            epilogue, Cout, C_scales, stream=None):
    _check(lib().moe_grouped_gemm_gather(dtype, _p(x), _p(x_scales), T, k, _p(sorted_rows), _p(B), _p(B_scales),
                                         _p(offsets), E, M_cap, N, K, epilogue, _p(Cout), _p(C_scales),
                                         _stream(stream)),
           "moe_grouped_gemm_gather")


def moe_grouped_gemm_dgrad_workspace_size(E, N, K) -> int:
    return lib().moe_grouped_gemm_dgrad_workspace_size(E, N, K)


def moe_grouped_gemm_dgrad(dC, B, offsets, E, M_cap, N, K, dA, ws, ws_bytes, stream=None):
    _check(lib().moe_grouped_gemm_dgrad(_p(dC), _p(B), _p(offsets), E, M_cap, N, K, _p(dA), _p(ws), ws_bytes,
                                        _stream(stream)), "moe_grouped_gemm_dgrad")


def moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K) -> int:
    return lib().moe_grouped_gemm_wgrad_workspace_size(E, M_cap, N, K)


def moe_grouped_gemm_wgrad(A, dC, offsets, E, M_cap, N, K, dB, ws, ws_bytes, stream=None):
    _check(lib().moe_grouped_gemm_wgrad(_p(A), _p(dC), _p(offsets), E, M_cap, N, K, _p(dB), _p(ws), ws_bytes,
                                        _stream(stream)), "moe_grouped_gemm_wgrad")


def moe_batched_matmul_workspace_size(dtype, T, K, k, E, N) -> int:
    return lib().moe_batched_matmul_workspace_size(dtype, T, K, k, E, N)


def moe_batched_matmul(dtype, x, x_scales, T, K, topk_ids, k, W, W_scales, E, N, out, ws, ws_bytes, stream=None):
    _check(lib().moe_batched_matmul(dtype, _p(x), _p(x_scales), T, K, _p(topk_ids), k, _p(W), _p(W_scales), E, N,
                                    _p(out), _p(ws), ws_bytes, _stream(stream)), "moe_batched_matmul")


def moe_grouped_gemm_combine_workspace_size(T, H) -> int:
    return lib().moe_grouped_gemm_combine_workspace_size(T, H)


def moe_grouped_gemm_combine(h, W2, offsets, E, M_cap, H, I, topk_ids, topk_w, sorted_rows, row_pos, T, k, Y2, out,
                             ws, ws_bytes, stream=None):
    _check(lib().moe_grouped_gemm_combine(_p(h), _p(W2), _p(offsets), E, M_cap, H, I, _p(topk_ids), _p(topk_w),
                                          _p(sorted_rows), _p(row_pos), T, k, _p(Y2), _p(out), _p(ws), ws_bytes,
                                          _stream(stream)), "moe_grouped_gemm_combine")


def moe_swiglu(Y1, offsets, E, M_cap, I, h, stream=None):
    _check(lib().moe_swiglu(_p(Y1), _p(offsets), E, M_cap, I, _p(h), _stream(stream)), "moe_swiglu")


def moe_combine(Y2, topk_ids, topk_w, row_pos, T, k, H, E, out, stream=None):
    _check(lib().moe_combine(_p(Y2), _p(topk_ids), _p(topk_w), _p(row_pos), T, k, H, E, _p(out),
                             _stream(stream)), "moe_combine")


def moe_forward_workspace_size(args: ForwardArgs) -> int:
    return lib().moe_forward_workspace_size(C.byref(args))


def moe_forward(args: ForwardArgs, ws, ws_bytes, stream=None):
    _check(lib().moe_forward(C.byref(args), _p(ws), ws_bytes, _stream(stream)), "moe_forward")


# ---------------------------------------------------------------- torch helpers
def _dev(t):
    return t.device if isinstance(t, torch.Tensor) else torch.device("cuda")


def route_sort_t(E: int, k: int, *, logits=None, expert_bias=None, sentinel_mask=None,
                 topk_ids=None, renormalize=True, stream=None):
    """Routing + sort with torch-allocated outputs.  Returns dict of tensors."""
    src = logits if logits is not None else topk_ids
    T = src.shape[0]
    dev = _dev(src)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    sr = torch.empty(T * k, dtype=torch.int32, device=dev)
    rp = torch.empty(T * k, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    wsb = moe_route_sort_workspace_size(T, E, k)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
    moe_route_sort(logits, expert_bias, sentinel_mask, ids, w if logits is not None else None, T, E, k,
                   renormalize, sr, rp, off, ws, wsb, stream)
    return dict(ids=ids, w=w, sorted_rows=sr, row_pos=rp, offsets=off)


def forward_args(*, dtype, T, E, k, H, I, x, W1, W2, out, logits=None, expert_bias=None,
                 sentinel_mask=None, topk_ids=None, topk_w=None, W1_scales=None, W2_scales=None,
                 renormalize=True, host_io=False, gather=False, fused_combine=False,
                 staged_out=False) -> ForwardArgs:
    """Fill a ForwardArgs from tensors (or raw addresses); ``gather`` sets
    MOE_FWD_GATHER.  The returned struct keeps the given tensors alive for as
    long as it lives."""
    a = ForwardArgs()
    a._keepalive = [logits, expert_bias, sentinel_mask, topk_ids, topk_w, x, W1, W1_scales, W2,
                    W2_scales, out]
    a.dtype, a.T, a.E, a.k, a.H, a.I = dtype, T, E, k, H, I
    a.renormalize = int(renormalize)
    a.flags = ((MOE_FWD_HOST_IO if host_io else 0) | (MOE_FWD_GATHER if gather else 0) |
               (MOE_FWD_FUSED_COMBINE if fused_combine else 0) | (MOE_FWD_STAGED_OUT if staged_out else 0))
    a.logits, a.expert_bias, a.sentinel_mask = _p(logits), _p(expert_bias), _p(sentinel_mask)
    a.topk_ids, a.topk_w = _p(topk_ids), _p(topk_w)
    a.x, a.W1, a.W1_scales, a.W2, a.W2_scales, a.out = (_p(x), _p(W1), _p(W1_scales), _p(W2),
                                                       _p(W2_scales), _p(out))
    return a
