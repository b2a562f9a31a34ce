"""CPU oracle for the BF16 TN GEMM — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it.

The arithmetic lives in ``gemm_ref.c`` (plain C, FP64, one dot product per
output element, rows split over POSIX threads).  This module builds that file
with gcc, calls it through ctypes, and holds the accuracy bound the GPU
results are judged against.

Accuracy bound, per output element (the FP32-accumulation bound of the
workload statement, widened for a general beta):

* FP32 output: ``|D - ref| <= 1e-4 * (absdot + |beta * c|)``
* BF16 output: the same plus ``ulp_bf16(|ref|)``

where ``absdot = |alpha| * sum_k |a_ik * b_jk|`` (returned by the oracle) and
``ulp_bf16(x) = 2**(floor(log2 x) - 7)`` for ``x >= 2**-126``, else
``2**-133``.  On inputs whose every partial sum is an integer below 2**24 the
comparison is bit-exact instead: ``D == float32(ref)``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_LIB = os.path.join(_HERE, "_build", "libgemm_ref.so")
_lock = threading.Lock()
_lib = None

C_BF16 = 0
C_F32 = 1


def build(force: bool = False) -> str:
    """Compile gemm_ref.c into a shared library (gcc, -O2, pthreads)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p, d, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
            lib.oracle_gemm_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, i32,
                                            d, d, p, p, i64, i32]
            lib.oracle_gemm_f64.restype = i32
            lib.oracle_gemm_f64_sampled.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64,
                                                    i32, d, d, i64, p, p, p, p, i32]
            lib.oracle_gemm_f64_sampled.restype = i32
            lib.oracle_nthreads_default.restype = i32
            lib.oracle_gemm_fp8_f64.argtypes = [i64, i64, i64, p, i64, p, i64, i32, p, i64, i32,
                                                d, d, p, p, i64, i32]
            lib.oracle_gemm_fp8_f64.restype = i32
            lib.oracle_gemm_fp8_f64_sampled.argtypes = [i64, i64, i64, p, i64, p, i64, i32, p, i64, i32,
                                                        d, d, i64, p, p, p, p, i32]
            lib.oracle_gemm_fp8_f64_sampled.restype = i32
            lib.oracle_epilogue_f64.argtypes = [i64, i64, p, i64, p, i32, i32]
            lib.oracle_epilogue_f64.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_nthreads_default())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c_args(C, ldc):
    if C is None:
        return None, 0, C_BF16
    if C.dtype == np.uint16:
        return C, ldc if ldc is not None else C.shape[1], C_BF16
    if C.dtype == np.float32:
        return C, ldc if ldc is not None else C.shape[1], C_F32
    raise TypeError("C must hold bf16 bits (uint16) or float32")


def gemm_ref(A, B, C=None, alpha=1.0, beta=0.0, M=None, N=None, K=None,
             lda=None, ldb=None, ldc=None, nthreads=0):
    """Full FP64 reference: returns (ref, absdot), both M x N float64.

    A: uint16 bf16 bits, M x lda; B: uint16, N x ldb; C: uint16 (bf16) or
    float32, M x ldc, or None.  M/N/K default to the array shapes.
    """
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M = A.shape[0] if M is None else M
    N = B.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    if C is not None:
        C = np.ascontiguousarray(C)
    Cc, ldc_, cd = _c_args(C, ldc)
    ref = np.empty((M, N), dtype=np.float64)
    absdot = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(Cc), ldc_, cd,
                                 float(alpha), float(beta), _ptr(ref), _ptr(absdot), N,
                                 int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_f64 rejected its arguments")
    return ref, absdot


def gemm_ref_sampled(A, B, rows, cols, C=None, alpha=1.0, beta=0.0, M=None, N=None,
                     K=None, lda=None, ldb=None, ldc=None, nthreads=0):
    """FP64 reference at the listed (rows[s], cols[s]) only: (ref, absdot) 1-D."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M = A.shape[0] if M is None else M
    N = B.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if C is not None:
        C = np.ascontiguousarray(C)
    Cc, ldc_, cd = _c_args(C, ldc)
    ref = np.empty(rows.shape, dtype=np.float64)
    absdot = np.empty(rows.shape, dtype=np.float64)
    rc = _load().oracle_gemm_f64_sampled(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(Cc), ldc_,
                                         cd, float(alpha), float(beta), rows.size,
                                         _ptr(rows), _ptr(cols), _ptr(ref), _ptr(absdot),
                                         int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_f64_sampled rejected its arguments")
    return ref, absdot


def gemm_ref_fp8(A, B, fmt, C=None, alpha=1.0, beta=0.0, M=None, N=None, K=None, lda=None, ldb=None,
                 ldc=None, nthreads=0):
    """FP64 reference for fp8 operands (uint8 codes; fmt 0 = e4m3, 1 = e5m2): (ref, absdot)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M = A.shape[0] if M is None else M
    N = B.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    if C is not None:
        C = np.ascontiguousarray(C)
    Cc, ldc_, cd = _c_args(C, ldc)
    ref = np.empty((M, N), dtype=np.float64)
    absdot = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_fp8_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, int(fmt), _ptr(Cc), ldc_, cd,
                                     float(alpha), float(beta), _ptr(ref), _ptr(absdot), N, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_fp8_f64 rejected its arguments")
    return ref, absdot


def gemm_ref_fp8_sampled(A, B, fmt, rows, cols, C=None, alpha=1.0, beta=0.0, M=None, N=None, K=None,
                         lda=None, ldb=None, ldc=None, nthreads=0):
    """FP64 fp8 reference at the listed (rows[s], cols[s]) only: (ref, absdot) 1-D."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    M = A.shape[0] if M is None else M
    N = B.shape[0] if N is None else N
    K = A.shape[1] if K is None else K
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if C is not None:
        C = np.ascontiguousarray(C)
    Cc, ldc_, cd = _c_args(C, ldc)
    ref = np.empty(rows.shape, dtype=np.float64)
    absdot = np.empty(rows.shape, dtype=np.float64)
    rc = _load().oracle_gemm_fp8_f64_sampled(M, N, K, _ptr(A), lda, _ptr(B), ldb, int(fmt), _ptr(Cc), ldc_,
                                             cd, float(alpha), float(beta), rows.size, _ptr(rows),
                                             _ptr(cols), _ptr(ref), _ptr(absdot), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_fp8_f64_sampled rejected its arguments")
    return ref, absdot


def epilogue(ref, bias=None, act=0):
    """act(ref + bias[n]) in FP64 (see gemm_ref.c); returns a new array.

    bias: N values as bf16 bits (uint16) or float32, or None.
    act: 0 none, 1 ReLU, 2 GELU (erf), 3 GELU (tanh), 4 SiLU.
    """
    out = np.array(ref, dtype=np.float64, order="C", copy=True)
    if out.ndim != 2:
        raise ValueError("ref must be 2-D")
    M, N = out.shape
    bd = 0
    if bias is not None:
        bias = np.ascontiguousarray(bias)
        if bias.shape != (N,):
            raise ValueError("bias must hold N values")
        if bias.dtype == np.float32:
            bd = 1
        elif bias.dtype != np.uint16:
            raise TypeError("bias must be bf16 bits (uint16) or float32")
    rc = _load().oracle_epilogue_f64(M, N, _ptr(out), N, _ptr(bias), bd, int(act))
    if rc != 0:
        raise ValueError("oracle_epilogue_f64 rejected its arguments")
    return out


# Largest slope of each activation (bounds how a pre-activation error grows).
ACT_LIPSCHITZ = {0: 1.0, 1: 1.0, 2: 1.13, 3: 1.13, 4: 1.1}


def bound_act(z, fz, absdot, out_dtype, act, beta=0.0, c=None):
    """Allowed |D - act(z)| when D = act(alpha A B^T + beta C + bias) is computed
    with fp32 accumulation and an fp32 activation: the pre-activation bound
    (1e-4 (absdot + |beta c|) plus fp32 rounding of the epilogue sums) times the
    activation's slope, plus the fp32 evaluation error of the activation
    (cancellation in 1 + erf / 1 + tanh costs up to ~2^-22 |z|), plus one bf16
    ulp of |act(z)| for bf16 output."""
    z = np.asarray(z, dtype=np.float64)
    pre = 1e-4 * np.asarray(absdot, dtype=np.float64) + 2.0 ** -22 * np.abs(z)
    if beta != 0.0 and c is not None:
        pre = pre + 1e-4 * np.abs(beta * np.asarray(c, dtype=np.float64))
    b = ACT_LIPSCHITZ[act] * pre + 2.0 ** -21 * (np.abs(z) + np.abs(fz))
    if out_dtype == 0:
        b = b + ulp_bf16(fz)
    return b


# ---------------------------------------------------------------------------
# accuracy bound
# ---------------------------------------------------------------------------

def ulp_bf16(x):
    """One bf16 ulp at |x|: 2**(floor(log2|x|) - 7) for |x| >= 2**-126, else 2**-133."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    out = np.full(x.shape, 2.0 ** -133)
    big = x >= 2.0 ** -126
    if np.any(big):
        e = np.floor(np.log2(x[big]))
        out[big] = np.exp2(e - 7)
    return out


def bound(ref, absdot, out_dtype, beta=0.0, c=None):
    """Per-element allowed |D - ref| (see module docstring)."""
    b = 1e-4 * np.asarray(absdot, dtype=np.float64)
    if beta != 0.0 and c is not None:
        b = b + 1e-4 * np.abs(beta * np.asarray(c, dtype=np.float64))
    if out_dtype == 0:  # bf16 output
        b = b + ulp_bf16(ref)
    return b


def decode_out(D, out_dtype):
    """GPU output as float64: D holds bf16 bits (uint16) or float32 values."""
    D = np.asarray(D)
    if out_dtype == 0:
        return (D.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return D.astype(np.float64)


def check(D, ref, absdot, out_dtype, beta=0.0, c=None):
    """Return (ok, worst_ratio, index_of_worst) with ratio = |D-ref| / bound."""
    d = decode_out(D, out_dtype)
    err = np.abs(d - ref)
    bnd = bound(ref, absdot, out_dtype, beta, c)
    bad_nan = ~np.isfinite(d) & np.isfinite(ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bnd > 0, err / bnd, np.where(err == 0, 0.0, np.inf))
    ratio = np.where(bad_nan, np.inf, ratio)
    if ratio.size == 0:
        return True, 0.0, None
    idx = int(np.argmax(ratio))
    worst = float(ratio.reshape(-1)[idx])
    return worst <= 1.0, worst, np.unravel_index(idx, ratio.shape)


def exact_f32(ref):
    """float32(ref) — the bit-exact expectation on integer-valued inputs."""
    return np.asarray(ref, dtype=np.float64).astype(np.float32)
