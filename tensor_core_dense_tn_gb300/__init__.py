"""Python binding of the GB300 BF16 TN GEMM library (libgemm_tn.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/gemm_tn.h``.  There is no CPU
fallback — if the library is missing, every call raises.

Raw entry points take integers (device pointers, a ``cudaStream_t`` handle):

    gemm_bf16_tn(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream)

``gemm()`` is a convenience wrapper over torch tensors (torch supplies device
memory and the current stream).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgemm_tn.so")

OUT_BF16 = 0
OUT_F32 = 1

PATH_AUTO, PATH_1SM, PATH_2SM, PATH_SKINNY = 0, 1, 2, 3

GEMM_OK = 0
GEMM_ERR_INVALID_VALUE = -1
GEMM_ERR_MISALIGNED = -2
GEMM_ERR_UNSUPPORTED_DEVICE = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_NOT_IMPLEMENTED = -6
GEMM_ERR_OUT_OF_MEMORY = -7
GEMM_ERR_CUDA = -8

EXPORTED = ["gemm_bf16_tn", "gemm_bf16_tn_ex", "gemm_get_status", "gemm_get_status_detail",
            "gemm_last_error_string", "gemm_last_launch_info", "gemm_shutdown", "gemm_version",
            "gemm_bf16_tn_skinny_noalloc", "gemm_bf16_tn_bias_act", "gemm_fp8_tn", "gemm_fp8_tn_ex",
            "gemm_bf16_tn_grouped", "gemm_bf16_tn_batched", "gemm_plan", "gemm_stream_read",
            "gemm_mma_rate", "gemm_fp8_tn_bias_act"]

FP8_E4M3, FP8_E5M2 = 0, 1
SCHED_DEFAULT, SCHED_STATIC, SCHED_CLC = 0, 1, 2

ACT_NONE, ACT_RELU, ACT_GELU, ACT_GELU_TANH, ACT_SILU = 0, 1, 2, 3, 4


class GemmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"gemm error {code}: {msg}")
        self.code = code


class GemmConfig(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("grid", ctypes.c_int), ("raster_group", ctypes.c_int),
                ("skinny_grid", ctypes.c_int), ("wait_timeout_ns", ctypes.c_uint64),
                ("test_fault", ctypes.c_int), ("disable_pdl", ctypes.c_int),
                ("skinny_skew_kb", ctypes.c_int), ("scheduler", ctypes.c_int), ("skinny_bm", ctypes.c_int),
                ("skinny_kgroup", ctypes.c_int), ("tiled_k_parts", ctypes.c_int), ("l2_hints", ctypes.c_int),
                ("cluster_pref", ctypes.c_int), ("b_static", ctypes.c_int), ("skinny_pair", ctypes.c_int),
                ("tail_slices", ctypes.c_int)]


class GemmPlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("skinny_kgroup", ctypes.c_int), ("skinny_stages", ctypes.c_int), ("skinny_grid", ctypes.c_int),
                ("k_parts", ctypes.c_int), ("skinny_skew", ctypes.c_int), ("tail_slices", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmProblem(ctypes.Structure):
    """One problem of gemm_bf16_tn_grouped (device pointers as integers)."""
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64), ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("grid", ctypes.c_int), ("cluster", ctypes.c_int),
                ("block", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("stages", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("kernel", ctypes.c_char_p),
                ("scheduler", ctypes.c_int), ("k_parts", ctypes.c_int), ("cluster_pref", ctypes.c_int),
                ("tail_slices", ctypes.c_int)]

    def as_dict(self):
        return {f: (getattr(self, f).decode() if f == "kernel" and getattr(self, f) else getattr(self, f))
                for f, _ in self._fields_}


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m tensor_core_dense_tn_gb300.build`")
        lib = ctypes.CDLL(path)
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        args = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, f32, i32, vp]
        lib.gemm_bf16_tn.argtypes = args
        lib.gemm_bf16_tn.restype = i32
        lib.gemm_fp8_tn.argtypes = [i64, i64, i64, vp, i64, vp, i64, i32, f32, f32, vp, i64, vp, i64,
                                    f32, f32, i32, vp]
        lib.gemm_fp8_tn.restype = i32
        lib.gemm_fp8_tn_bias_act.argtypes = lib.gemm_fp8_tn.argtypes[:-1] + [vp, i32, i32, vp]
        lib.gemm_fp8_tn_bias_act.restype = i32
        lib.gemm_fp8_tn_ex.argtypes = lib.gemm_fp8_tn.argtypes + [ctypes.POINTER(GemmConfig)]
        lib.gemm_fp8_tn_ex.restype = i32
        lib.gemm_plan.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(GemmConfig), ctypes.POINTER(GemmPlanInfo)]
        lib.gemm_plan.restype = i32
        lib.gemm_bf16_tn_bias_act.argtypes = args[:-1] + [vp, i32, i32, vp]
        lib.gemm_bf16_tn_bias_act.restype = i32
        lib.gemm_bf16_tn_skinny_noalloc.argtypes = args
        lib.gemm_bf16_tn_skinny_noalloc.restype = i32
        lib.gemm_stream_read.argtypes = [vp, i64, i64, i32, i32, i32, vp]
        lib.gemm_stream_read.restype = i32
        lib.gemm_mma_rate.argtypes = [i32, i32, i32, i32, i32, vp, vp]
        lib.gemm_mma_rate.restype = i32
        lib.gemm_bf16_tn_grouped.argtypes = [i32, ctypes.POINTER(GemmProblem), f32, f32, i32, vp]
        lib.gemm_bf16_tn_grouped.restype = i32
        lib.gemm_bf16_tn_batched.argtypes = [i64, i64, i64, i64, vp, i64, i64, vp, i64, i64, vp, i64, i64,
                                             vp, i64, i64, f32, f32, i32, vp]
        lib.gemm_bf16_tn_batched.restype = i32
        lib.gemm_bf16_tn_ex.argtypes = args + [ctypes.POINTER(GemmConfig)]
        lib.gemm_bf16_tn_ex.restype = i32
        lib.gemm_get_status.argtypes = [vp]
        lib.gemm_get_status.restype = i32
        lib.gemm_get_status_detail.restype = i32
        lib.gemm_last_error_string.restype = ctypes.c_char_p
        lib.gemm_last_launch_info.argtypes = [ctypes.POINTER(LaunchInfo)]
        lib.gemm_last_launch_info.restype = i32
        lib.gemm_shutdown.restype = None
        lib.gemm_version.restype = i32
        _lib = lib
        return lib


def last_error() -> str:
    s = load().gemm_last_error_string()
    return s.decode() if s else ""


def _check(rc: int) -> int:
    if rc != GEMM_OK:
        raise GemmError(rc, last_error())
    return rc


def gemm_bf16_tn(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream) -> int:
    """Raw C-ABI call; returns the gemm_status code (does not raise)."""
    return load().gemm_bf16_tn(M, N, K, A, lda, B, ldb, C or None, ldc, D, ldd, alpha, beta,
                               out_dtype, stream or None)


def gemm_bf16_tn_ex(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, stream,
                    config: GemmConfig | None = None) -> int:
    cfg = ctypes.byref(config) if config is not None else None
    return load().gemm_bf16_tn_ex(M, N, K, A, lda, B, ldb, C or None, ldc, D, ldd, alpha, beta,
                                  out_dtype, stream or None, cfg)


def gemm_bf16_tn_skinny_noalloc(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype,
                                stream) -> int:
    """Raw C-ABI call of the allocation-free skinny entry point (1 <= M <= 64)."""
    return load().gemm_bf16_tn_skinny_noalloc(M, N, K, A, lda, B, ldb, C or None, ldc, D, ldd, alpha,
                                              beta, out_dtype, stream or None)


def gemm_stream_read(src, rows, row_bytes, box_rows, kgroup, grid, stream) -> int:
    """Raw C-ABI call of the TMA streaming-read ceiling kernel (reads rows x
    row_bytes bytes at src in the skinny kernel's box shape, discards them)."""
    return load().gemm_stream_read(src, rows, row_bytes, box_rows, kgroup, grid, stream or None)


def gemm_mma_rate(n, cta_group, fp8, reps, grid, out_ns, stream) -> int:
    """Raw C-ABI call of the tcgen05.mma rate kernel (out_ns: device pointer to two uint64)."""
    return load().gemm_mma_rate(n, cta_group, fp8, reps, grid, out_ns, stream or None)


def gemm_bf16_tn_grouped(problems, alpha, beta, out_dtype, stream) -> int:
    """Raw C-ABI call: `problems` is a sequence of GemmProblem (or of dicts with its fields)."""
    arr = (GemmProblem * max(1, len(problems)))()
    for i, q in enumerate(problems):
        arr[i] = q if isinstance(q, GemmProblem) else GemmProblem(**q)
    return load().gemm_bf16_tn_grouped(len(problems), arr, alpha, beta, out_dtype, stream or None)


def gemm_bf16_tn_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C, ldc, stride_c, D, ldd, stride_d,
                         alpha, beta, out_dtype, stream) -> int:
    """Raw C-ABI call of the strided batched GEMM (strides in elements)."""
    return load().gemm_bf16_tn_batched(batch, M, N, K, A, lda, stride_a, B, ldb, stride_b, C or None, ldc,
                                       stride_c, D, ldd, stride_d, alpha, beta, out_dtype, stream or None)


def gemm_bf16_tn_bias_act(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, alpha, beta, out_dtype, bias,
                          bias_dtype, activation, stream) -> int:
    """Raw C-ABI call: D = act(alpha * A B^T + beta * C + bias)."""
    return load().gemm_bf16_tn_bias_act(M, N, K, A, lda, B, ldb, C or None, ldc, D, ldd, alpha, beta,
                                        out_dtype, bias or None, bias_dtype, activation, stream or None)


def gemm_fp8_tn_bias_act(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C, ldc, D, ldd, alpha, beta,
                         out_dtype, bias, bias_dtype, activation, stream) -> int:
    """Raw C-ABI call: D = act(alpha * scale_a * scale_b * A B^T + beta * C + bias), fp8 A and B."""
    return load().gemm_fp8_tn_bias_act(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C or None, ldc, D,
                                       ldd, alpha, beta, out_dtype, bias or None, bias_dtype, activation,
                                       stream or None)


def gemm_fp8_tn(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C, ldc, D, ldd, alpha, beta,
                out_dtype, stream) -> int:
    """Raw C-ABI call: D = alpha * scale_a * scale_b * A B^T + beta * C, fp8 A and B."""
    return load().gemm_fp8_tn(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C or None, ldc, D,
                              ldd, alpha, beta, out_dtype, stream or None)


def gemm_fp8_tn_ex(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C, ldc, D, ldd, alpha, beta,
                   out_dtype, stream, config=None) -> int:
    """gemm_fp8_tn with a GemmConfig of overrides (None = library defaults)."""
    cfg = ctypes.byref(config) if config is not None else None
    return load().gemm_fp8_tn_ex(M, N, K, A, lda, B, ldb, fp8_format, scale_a, scale_b, C or None, ldc, D,
                                 ldd, alpha, beta, out_dtype, stream or None, cfg)


def gemm_plan(M, N, K, fp8_inputs=0, num_sms=152, config=None):
    """Host-only plan of a call: (status, dict of GemmPlanInfo fields)."""
    out = GemmPlanInfo()
    cfg = ctypes.byref(config) if config is not None else None
    rc = load().gemm_plan(M, N, K, fp8_inputs, num_sms, cfg, ctypes.byref(out))
    return rc, out.as_dict()


def gemm_get_status(stream=None) -> int:
    return load().gemm_get_status(stream or None)


def gemm_get_status_detail() -> int:
    return load().gemm_get_status_detail()


def last_launch_info() -> dict:
    info = LaunchInfo()
    load().gemm_last_launch_info(ctypes.byref(info))
    return info.as_dict()


def shutdown() -> None:
    load().gemm_shutdown()


def version() -> int:
    return load().gemm_version()


def gemm(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, out_dtype=None, out=None,
         config: GemmConfig | None = None, stream=None):
    """D = alpha * A @ B.T + beta * C on the current CUDA stream (torch tensors).

    A: (M, K) bf16, B: (N, K) bf16, both with unit stride along K.
    C/out: (M, N) of out_dtype (torch.bfloat16 default, or torch.float32).
    """
    import torch

    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    for name, t in (("A", A), ("B", B)):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda or t.stride(1) != 1:
            raise ValueError(f"{name} must be a 2-D bf16 CUDA tensor with unit stride along K")
    M, K = A.shape
    N, Kb = B.shape
    if Kb != K:
        raise ValueError("A and B must have the same K")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if out.shape != (M, N) or out.dtype != out_dtype or out.stride(1) != 1:
        raise ValueError("out must be (M, N), out_dtype, unit column stride")
    c_ptr, ldc = 0, 0
    if beta != 0.0:
        if C is None or C.shape != (M, N) or C.dtype != out_dtype or C.stride(1) != 1:
            raise ValueError("beta != 0 needs C of shape (M, N) and out_dtype")
        c_ptr, ldc = C.data_ptr(), C.stride(0)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    code = OUT_F32 if out_dtype == torch.float32 else OUT_BF16
    args = (M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), c_ptr, ldc,
            out.data_ptr(), out.stride(0), float(alpha), float(beta), code, stream)
    rc = gemm_bf16_tn_ex(*args, config=config) if config is not None else gemm_bf16_tn(*args)
    _check(rc)
    return out
