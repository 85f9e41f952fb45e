"""ctypes wrapper of the C++ oracle (``moe_oracle.cpp``) -- test infrastructure.

Arrays are numpy; bf16 tensors are passed as their ``uint16`` bit patterns.
Every function returns fresh fp32 / int32 / uint8 arrays.  Nothing here runs
on, or is reachable from, the CUDA path.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIBS = {False: os.path.join(_HERE, "libmoe_oracle.so"),       # one core
         True: os.path.join(_HERE, "libmoe_oracle_omp.so")}    # OpenMP over rows

__all__ = [
    "build", "use_openmp", "threads", "e4m3_encode", "e4m3_decode", "bf16_round", "route_topk",
    "mark_sentinels", "ep_local_ids", "sort_by_expert", "quant_act_fp8", "quant_weight_fp8", "permute",
    "grouped_gemm_bf16", "grouped_gemm_fp8", "swiglu", "combine", "moe_forward",
    "grouped_gemm_dgrad_bf16", "grouped_gemm_wgrad_bf16", "batched_matmul",
]


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction).  With
    openmp, the same source with -fopenmp: its row loops run on all cores,
    each output element still computed by one thread in the same order."""
    lib = _LIBS[bool(openmp)]
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
               "-shared"] + (["-fopenmp"] if openmp else []) + [_SRC, "-o", lib + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(lib + ".tmp", lib)
    return lib


_lib = {}
_openmp = False


def use_openmp(on: bool = True) -> bool:
    """Route every function of this module to the OpenMP build (on) or the
    one-core build (off); returns the previous setting."""
    global _openmp
    prev, _openmp = _openmp, bool(on)
    return prev


def _L():
    lib = _lib.get(_openmp)
    if lib is None:
        lib = _lib[_openmp] = C.CDLL(build(openmp=_openmp))
    return lib


def threads() -> int:
    """Threads the active build runs its row loops on (1 for the one-core build)."""
    return int(_L().orc_threads())


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


def e4m3_encode(v) -> np.ndarray:
    v = _c(v, np.float32)
    q = np.empty(v.shape, np.uint8)
    _L().orc_e4m3_encode(_p(v), C.c_int64(v.size), _p(q))
    return q


def e4m3_decode(q) -> np.ndarray:
    q = _c(q, np.uint8)
    v = np.empty(q.shape, np.float32)
    _L().orc_e4m3_decode(_p(q), C.c_int64(q.size), _p(v))
    return v


def bf16_round(v) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    _L().orc_bf16_round(_p(v), C.c_int64(v.size), _p(out))
    return out


def route_topk(logits, bias, k: int, renormalize: bool = True):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _L().orc_route_topk(_p(logits), _p(_c(bias, np.float32)), T, E, k, int(renormalize),
                        _p(ids), _p(w))
    return ids, w


def mark_sentinels(ids, mask, E: int):
    ids = np.array(ids, dtype=np.int32, copy=True)
    mask = _c(mask, np.uint8)
    _L().orc_mark_sentinels(_p(ids), _p(mask), C.c_int64(ids.size), E)
    return ids


def ep_local_ids(ids, E_global: int, first: int, E_local: int):
    """Global expert ids -> the ids of the rank holding experts [first,
    first + E_local); every other pick becomes the local sentinel E_local."""
    ids = _c(ids, np.int32)
    out = np.empty(ids.shape, np.int32)
    _L().orc_ep_local_ids(_p(ids), C.c_int64(ids.size), E_global, first, E_local, _p(out))
    return out


def sort_by_expert(ids, E: int):
    ids = _c(ids, np.int32)
    R = ids.size
    sr = np.empty(R, np.int32)
    rp = np.empty(R, np.int32)
    off = np.empty(E + 1, np.int32)
    _L().orc_sort_by_expert(_p(ids), C.c_int64(R), E, _p(sr), _p(rp), _p(off))
    return sr, rp, off


def quant_act_fp8(x_bf16):
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((M, K // 128), np.float32)
    _L().orc_quant_act_fp8(_p(x), C.c_int64(M), K, _p(q), _p(s))
    return q, s


def quant_weight_fp8(w_bf16):
    w = _c(w_bf16, np.uint16)
    E, N, K = w.shape
    q = np.empty((E, N, K), np.uint8)
    s = np.empty((E, (N + 127) // 128, K // 128), np.float32)
    _L().orc_quant_weight_fp8(_p(w), E, N, K, _p(q), _p(s))
    return q, s


def permute(x, k: int, sorted_rows, L: int, x_scales=None, M_cap: int | None = None):
    """bf16 rows (uint16) or e4m3 rows (uint8, with x_scales).  Rows >= L of
    the result are zero-initialised here (the definition leaves them as they are)."""
    x = np.ascontiguousarray(x)
    T, H = x.shape
    sr = _c(sorted_rows, np.int32)
    M_cap = sr.size if M_cap is None else M_cap
    xp = np.zeros((M_cap, H), x.dtype)
    xs = None
    if x_scales is not None:
        x_scales = _c(x_scales, np.float32)
        xs = np.zeros((M_cap, H // 128), np.float32)
    _L().orc_permute(_p(x), _p(x_scales), x.dtype.itemsize, C.c_int64(T), H, k, _p(sr),
                     C.c_int64(L), _p(xp), _p(xs))
    return (xp, xs) if x_scales is not None else xp


def grouped_gemm_bf16(A, B, offsets, rows=None):
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    off = _c(offsets, np.int32)
    M_cap, K = A.shape
    E, N, K2 = B.shape
    assert K == K2 and off.size == E + 1
    rows = _c(rows, np.int32)
    nout = M_cap if rows is None else rows.size
    Cm = np.empty((nout, N), np.float32)
    _L().orc_grouped_gemm_bf16(_p(A), _p(B), _p(off), E, C.c_int64(M_cap), N, K, _p(rows),
                               C.c_int64(0 if rows is None else rows.size), _p(Cm))
    return Cm


def grouped_gemm_dgrad_bf16(dC, B, offsets, rows=None):
    """dA [M_cap, K] fp32 of C = A B[e]^T given dC (bf16 bits [M_cap, N]);
    with rows, only those rows ([len(rows), K])."""
    dC = _c(dC, np.uint16)
    B = _c(B, np.uint16)
    off = _c(offsets, np.int32)
    M_cap, N = dC.shape
    E, N2, K = B.shape
    assert N == N2 and off.size == E + 1
    rows = _c(rows, np.int32)
    nout = M_cap if rows is None else rows.size
    dA = np.empty((nout, K), np.float32)
    _L().orc_grouped_gemm_dgrad_bf16(_p(dC), _p(B), _p(off), E, C.c_int64(M_cap), N, K, _p(rows),
                                     C.c_int64(0 if rows is None else rows.size), _p(dA))
    return dA


def grouped_gemm_wgrad_bf16(A, dC, offsets, E: int, pairs=None):
    """dB [E, N, K] fp32 of C = A B[e]^T given A and dC (bf16 bits); with
    pairs (int32 [n, 2] of (expert, row of B)) only those rows, [n, K]."""
    A = _c(A, np.uint16)
    dC = _c(dC, np.uint16)
    off = _c(offsets, np.int32)
    M_cap, K = A.shape
    M2, N = dC.shape
    assert M_cap == M2 and off.size == E + 1
    pr = _c(pairs, np.int32)
    n = 0 if pr is None else pr.shape[0]
    dB = np.empty((n, K) if pr is not None else (E, N, K), np.float32)
    _L().orc_grouped_gemm_wgrad_bf16(_p(A), _p(dC), _p(off), E, C.c_int64(M_cap), N, K, _p(pr),
                                     C.c_int64(n), _p(dB))
    return dB


def grouped_gemm_fp8(qa, sa, qb, sb, offsets, rows=None):
    qa = _c(qa, np.uint8)
    sa = _c(sa, np.float32)
    qb = _c(qb, np.uint8)
    sb = _c(sb, np.float32)
    off = _c(offsets, np.int32)
    M_cap, K = qa.shape
    E, N, K2 = qb.shape
    assert K == K2 and off.size == E + 1 and sa.shape == (M_cap, K // 128)
    assert sb.shape == (E, (N + 127) // 128, K // 128)
    rows = _c(rows, np.int32)
    nout = M_cap if rows is None else rows.size
    Cm = np.empty((nout, N), np.float32)
    _L().orc_grouped_gemm_fp8(_p(qa), _p(sa), _p(qb), _p(sb), _p(off), E, C.c_int64(M_cap), N, K,
                              _p(rows), C.c_int64(0 if rows is None else rows.size), _p(Cm))
    return Cm


def batched_matmul(x, ids, W, E: int, x_scales=None, W_scales=None):
    """out [T*k, N] fp32: for slot f = t*k + j with expert e = ids[t, j] < E,
    out[f] = W[e] x[t] (bf16 bits, or e4m3 bytes with their scales); sentinel
    slots give zero rows."""
    fp8 = W_scales is not None
    x = np.ascontiguousarray(x, np.uint8 if fp8 else np.uint16)
    W = np.ascontiguousarray(W, np.uint8 if fp8 else np.uint16)
    ids = _c(ids, np.int32)
    T, K = x.shape
    k = ids.shape[1]
    E2, N, K2 = W.shape
    assert K == K2 and ids.shape[0] == T
    out = np.empty((T * k, N), np.float32)
    _L().orc_batched_matmul(int(fp8), _p(x), _p(_c(x_scales, np.float32)), _p(ids), C.c_int64(T), k, E, _p(W),
                            _p(_c(W_scales, np.float32)), N, K, _p(out))
    return out


def swiglu(Y1, L: int):
    Y1 = _c(Y1, np.float32)
    M_cap, I2 = Y1.shape
    h = np.empty((M_cap, I2 // 2), np.float32)
    _L().orc_swiglu(_p(Y1), C.c_int64(M_cap), I2 // 2, C.c_int64(L), _p(h))
    return h


def combine(Y2, ids, w, row_pos, E: int):
    Y2 = _c(Y2, np.float32)
    ids = _c(ids, np.int32)
    w = _c(w, np.float32)
    rp = _c(row_pos, np.int32)
    T, k = ids.shape
    H = Y2.shape[1]
    out = np.empty((T, H), np.float32)
    _L().orc_combine(_p(Y2), _p(ids), _p(w), _p(rp), C.c_int64(T), k, H, E, _p(out))
    return out


def moe_forward(x, W1, W2, *, E: int, k: int, logits=None, bias=None, sentinel_mask=None,
                ids=None, w=None, renormalize: bool = True, W1_scales=None, W2_scales=None):
    """The full expert layer.  bf16 mode: W1/W2 are uint16 bf16 bits.  FP8 mode
    (W1_scales given): W1/W2 are e4m3 bytes with 128x128 block scales.
    Returns dict(out, ids, w, sorted_rows, row_pos, offsets)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    fp8 = W1_scales is not None
    I = W2.shape[2]
    if logits is not None:
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
    else:
        ids = np.array(ids, dtype=np.int32, copy=True)
        w = np.array(w, dtype=np.float32, copy=True)
    W1 = np.ascontiguousarray(W1)
    W2 = np.ascontiguousarray(W2)
    out = np.empty((T, H), np.float32)
    sr = np.empty(T * k, np.int32)
    rp = np.empty(T * k, np.int32)
    off = np.empty(E + 1, np.int32)
    rc = _L().orc_moe_forward(
        int(fp8), _p(_c(logits, np.float32)), _p(_c(bias, np.float32)),
        _p(_c(sentinel_mask, np.uint8)), _p(ids), _p(w), C.c_int64(T), E, k, H, I,
        int(renormalize), _p(x), _p(W1), _p(_c(W1_scales, np.float32)), _p(W2),
        _p(_c(W2_scales, np.float32)), _p(out), _p(sr), _p(rp), _p(off))
    if rc:
        raise ValueError("oracle: unsupported shape for the FP8 layer")
    return dict(out=out, ids=ids, w=w, sorted_rows=sr, row_pos=rp, offsets=off)
