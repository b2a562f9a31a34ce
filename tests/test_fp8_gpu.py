"""GPU parity of the FP8 TN GEMM, D = alpha * scale_a * scale_b * A B^T + beta * C.

A and B are one-byte e4m3 or e5m2 codes (the same format for both); products
are formed on the tensor cores with FP32 accumulation.  Against the FP64
oracle, which decodes every code by the formats' definitions:
* integer inputs in [-4, 4] (exact in both formats): bit-exact on all three
  kernel paths, ragged M, N and K, and with power-of-two scales;
* normal inputs, real scales, beta with C: within the oracle's accumulation
  bound (1e-4 of sum |alpha' a b| plus the output rounding).
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import check_every_element, empty_out, from_dev, to_dev_bf16, to_dev_f32  # noqa: E402

# M picks the kernel path: 48 -> skinny, 100 -> 1-SM tiled, 2200 -> 2-SM tiled
# (with N at least 1040: more than 64 tiles of 128 x 256, so pair tiles)
PATH_M = {"skinny": 24, "1sm": 100, "2sm": 2200}
PATH_CODE = {"skinny": 3, "1sm": 1, "2sm": 2}


def shape_n(path, n):
    """N for a test on `path`: the 2-SM case needs enough tiles to use pair tiles."""
    return max(n, 1040) if path == "2sm" else n


def check_path(path):
    assert g.last_launch_info()["path"] == PATH_CODE[path], g.last_launch_info()
FMTS = [gi.FP8_E4M3, gi.FP8_E5M2]


def to_dev_u8(codes):
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).to("cuda:0")


def _run(M, N, K, A, B, fmt, out_dtype, scale_a=1.0, scale_b=1.0, alpha=1.0, beta=0.0, C=None,
         lda=None, ldb=None):
    import torch
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    dC = None
    if C is not None:
        dC = to_dev_bf16(C) if out_dtype == gi.OUT_BF16 else to_dev_f32(C)
    dD, ldd = empty_out(M, N, out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_fp8_tn(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), ldb, fmt, scale_a, scale_b,
                       dC.data_ptr() if dC is not None else 0, N if dC is not None else 0,
                       dD.data_ptr(), ldd, alpha, beta, out_dtype, s)
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(s) == 0, g.last_error()
    return from_dev(dD, out_dtype)


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("N,K", [(520, 320), (264, 1040), (300, 1152)])
def test_integer_exact(path, fmt, N, K):
    M, N = PATH_M[path], shape_n(path, N)
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5000 + fmt, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5010 + fmt, fmt)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
    got = _run(M, N, K, A, B, fmt, gi.OUT_F32)
    check_path(path)
    assert np.array_equal(got, oracle.exact_f32(ref))


@pytest.mark.parametrize("path", list(PATH_M))
def test_integer_exact_scales_and_padding(path):
    # power-of-two scales keep the result exact; padded rows (ld > K) hold NaN codes
    M, N, K, ld = PATH_M[path] + 3, shape_n(path, 392), 208, 256
    fmt = gi.FP8_E4M3
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5100, fmt, ld=ld)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5101, fmt, ld=ld)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt, M=M, N=N, K=K, lda=ld, ldb=ld, alpha=0.5 * 0.25 * 8.0)
    got = _run(M, N, K, A, B, fmt, gi.OUT_F32, scale_a=0.25, scale_b=8.0, alpha=0.5, lda=ld, ldb=ld)
    check_path(path)
    assert np.array_equal(got, oracle.exact_f32(ref))


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("out_dtype", [gi.OUT_BF16, gi.OUT_F32])
def test_normal_within_bound(path, fmt, out_dtype):
    M, N, K = PATH_M[path], shape_n(path, 776), 1536
    A = gi.draw_fp8(M, K, gi.Dist("normal", 4.0), 5200 + fmt, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("normal", 4.0), 5210 + fmt, fmt)
    C = (gi.draw_bf16(M, N, gi.Dist("normal", 1.0), 5220) if out_dtype == gi.OUT_BF16
         else gi.draw_f32(M, N, gi.Dist("normal", 1.0), 5220))
    sa, sb, alpha, beta = 0.37, 0.011, 1.25, 0.5
    c64 = gi.bf16_bits_to_f32(C) if out_dtype == gi.OUT_BF16 else C
    ref, absdot = oracle.gemm_ref_fp8(A, B, fmt, C=C, alpha=alpha * np.float32(sa) * np.float32(sb),
                                      beta=beta)
    got = _run(M, N, K, A, B, fmt, out_dtype, scale_a=sa, scale_b=sb, alpha=alpha, beta=beta, C=C)
    check_path(path)
    ok, worst, idx = oracle.check(got, ref, absdot, out_dtype, beta, c64)
    assert ok, (worst, idx)


@pytest.mark.parametrize("idx", [4, 3])
def test_bench_shapes_every_element(idx):
    """The two FP8 bench steps (the 16 x 8192 x 8192 decode and the
    8192 x 28672 x 4096 up-projection, e4m3 codes with per-tensor scales, the
    same operands the benchmark draws): every output against the oracle."""
    w = gi.WORKLOADS[idx]
    fmt = gi.FP8_E4M3
    A, B, sa, sb = gi.fp8_operands(w, fmt)
    got = _run(w.M, w.N, w.K, A, B, fmt, gi.OUT_BF16, scale_a=sa, scale_b=sb)
    alpha = float(np.float32(sa) * np.float32(sb))   # the scales fold into alpha in FP32
    ok, worst, where = check_every_element(
        got, lambda r0, r1: oracle.gemm_ref_fp8(A[r0:r1], B, fmt, alpha=alpha), gi.OUT_BF16, w.M)
    assert ok, (worst, where)


def test_fp8_matches_bf16_path_on_common_values():
    """Small integers are exact in bf16 and both fp8 formats: all three inputs
    kinds must give the same bits through their own kernels."""
    import torch
    M, N, K = 300, 520, 512
    Ai = np.random.default_rng(5400).integers(-4, 5, size=(M, K))
    Bi = np.random.default_rng(5401).integers(-4, 5, size=(N, K))
    outs = []
    for fmt in FMTS:
        outs.append(_run(M, N, K, gi.f32_to_fp8_bits(Ai, fmt), gi.f32_to_fp8_bits(Bi, fmt), fmt, gi.OUT_F32))
    dA = to_dev_bf16(gi.f32_to_bf16_bits(Ai.astype(np.float32)))
    dB = to_dev_bf16(gi.f32_to_bf16_bits(Bi.astype(np.float32)))
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0, dD.data_ptr(), ldd,
                        1.0, 0.0, gi.OUT_F32, s)
    assert rc == 0 and g.gemm_get_status(s) == 0
    outs.append(from_dev(dD, gi.OUT_F32))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_fp8_argument_errors():
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64)
    tail = (1.0, 1.0, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_fp8_tn(*a, 2, *tail) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_fp8_tn(*a, -1, *tail) == g.GEMM_ERR_INVALID_VALUE
    # lda must be a multiple of 16 one-byte elements
    assert g.gemm_fp8_tn(64, 64, 64, 0x1000, 72, 0x2000, 64, 0, *tail) == g.GEMM_ERR_MISALIGNED
    assert g.gemm_fp8_tn(64, 64, 64, 0x1008, 64, 0x2000, 64, 0, *tail) == g.GEMM_ERR_MISALIGNED


@pytest.mark.parametrize("fmt", FMTS)
def test_wide_streaming_integer_exact(fmt):
    """96 tokens against an 8192 x 4096 fp8 weight (32 MiB): the auto path is the
    streaming kernel's wide form (128 whole 64-row tiles).  Every row at
    sampled columns, tile edges included."""
    M, N, K = 96, 8192, 4096
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5500 + fmt, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5510 + fmt, fmt)
    got = _run(M, N, K, A, B, fmt, gi.OUT_F32)
    assert g.last_launch_info()["path"] == 3 and g.last_launch_info()["tile_m"] == 64
    cols_1 = sorted(set(np.random.default_rng(5520 + fmt).integers(0, N, 200).tolist())
                    | {0, 63, 64, 127, 128, N - 65, N - 64, N - 1})
    rows = np.repeat(np.arange(M), len(cols_1))
    cols = np.tile(np.array(cols_1), M)
    ref, _ = oracle.gemm_ref_fp8_sampled(A, B, fmt, rows, cols)
    assert np.array_equal(got[rows, cols], oracle.exact_f32(ref))


@pytest.mark.parametrize("path,bm,kg", [(1, 0, 0), (2, 0, 0), (3, 64, 1), (3, 64, 4), (3, 128, 2), (3, 128, 4)])
@pytest.mark.parametrize("fmt", FMTS)
def test_forced_path_and_kgroups(path, bm, kg, fmt):
    """gemm_fp8_tn_ex: every path, tile height and k-group on one shape whose
    K = 1408 is 11 k-blocks of 128 (the last group partly zero-filled)."""
    import torch
    M, N, K = 40, 648, 1408
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5600 + fmt, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5610 + fmt, fmt)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=path, skinny_bm=bm, skinny_kgroup=kg)
    rc = g.gemm_fp8_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, fmt, 1.0, 1.0, 0, 0,
                          dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_F32, s, cfg)
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(s) == 0, g.last_error()
    info = g.last_launch_info()
    assert info["path"] == path and (bm == 0 or info["tile_m"] == bm)
    assert np.array_equal(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("parts", [2, 3])
def test_fp8_tiled_k_split_exact(path, parts):
    """fp8 inputs on split tiles (k-blocks of 128 elements: K = 1408 is 11)."""
    import torch
    fmt = gi.FP8_E4M3
    M, N, K = 300, 520, 1408
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5700 + parts, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5710 + parts, fmt)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=path, tiled_k_parts=parts)
    rc = g.gemm_fp8_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, fmt, 1.0, 1.0, 0, 0,
                          dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_F32, s, cfg)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    info = g.last_launch_info()
    assert info["path"] == path and info["k_parts"] == parts and "split" in info["kernel"]
    assert np.array_equal(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("M,N,K", [(16, 8192, 2048), (40, 648, 1408), (96, 2048, 1024)])
@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_skinny_pair_exact(M, N, K, fmt):
    """fp8 inputs through the pair form of the streaming kernel."""
    import torch
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5800 + fmt + M, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5810 + fmt + N, fmt)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=3, skinny_pair=2)
    rc = g.gemm_fp8_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, fmt, 1.0, 1.0, 0, 0,
                          dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_F32, s, cfg)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    assert g.last_launch_info()["cluster"] == 2
    assert np.array_equal(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


def _run_fused(M, N, K, A, B, fmt, bias, bias_dtype, act, out_dtype, scale_a=1.0, scale_b=1.0):
    import torch
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    dbias = to_dev_bf16(bias) if bias_dtype == 0 else to_dev_f32(bias)
    dD, ldd = empty_out(M, N, out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_fp8_tn_bias_act(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, fmt, scale_a, scale_b, 0, 0,
                                dD.data_ptr(), ldd, 1.0, 0.0, out_dtype, dbias.data_ptr(), bias_dtype, act, s)
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(s) == 0, g.last_error()
    return from_dev(dD, out_dtype)


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("act", [0, 1])
def test_fp8_bias_act_integer_exact(path, fmt, act):
    """gemm_fp8_tn_bias_act: integer codes and bias, no activation or ReLU, bit-exact on every path."""
    M, N, K = PATH_M[path], shape_n(path, 520), 384
    A = gi.draw_fp8(M, K, gi.Dist("int", -4, 4), 5900 + fmt, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("int", -4, 4), 5910 + fmt, fmt)
    bias = gi.draw_bf16(N, 1, gi.Dist("int", -50, 50), 5920).reshape(N)
    ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
    want = oracle.epilogue(ref, bias, act)
    got = _run_fused(M, N, K, A, B, fmt, bias, 0, act, gi.OUT_F32)
    check_path(path)
    assert np.array_equal(got, oracle.exact_f32(want))


@pytest.mark.parametrize("path", list(PATH_M))
def test_fp8_bias_gelu_within_bound(path):
    """e4m3 with real per-tensor scales, fp32 bias and tanh-GELU: within the
    oracle's activation bound (the pre-activation bound times the slope plus
    fp32 evaluation error and one bf16 ulp)."""
    fmt = gi.FP8_E4M3
    M, N, K = PATH_M[path], shape_n(path, 776), 1024
    A = gi.draw_fp8(M, K, gi.Dist("normal", 1.0), 5930, fmt)
    B = gi.draw_fp8(N, K, gi.Dist("normal", 1.0), 5931, fmt)
    bias = gi.draw_f32(N, 1, gi.Dist("normal", 1.0), 5932).reshape(N)
    sa, sb = 1.0, 1.0 / 32.0
    alpha = float(np.float32(sa) * np.float32(sb))
    ref, absdot = oracle.gemm_ref_fp8(A, B, fmt, alpha=alpha)
    z = oracle.epilogue(ref, bias, 0)
    fz = oracle.epilogue(ref, bias, 3)
    got = oracle.decode_out(_run_fused(M, N, K, A, B, fmt, bias, 1, 3, gi.OUT_BF16, sa, sb), 0)
    check_path(path)
    bnd = oracle.bound_act(z, fz, absdot, 0, 3)
    assert np.all(np.abs(got - fz) <= bnd), float(np.max(np.abs(got - fz) / bnd))


def test_fp8_bias_act_argument_errors():
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64)
    tail = (1.0, 1.0, 0, 0, 0x3000, 64, 1.0, 0.0, 0)
    assert g.gemm_fp8_tn_bias_act(*a, 2, *tail, 0x4000, 0, 1, 0) == g.GEMM_ERR_INVALID_VALUE   # format
    assert g.gemm_fp8_tn_bias_act(*a, 0, *tail, 0x4000, 0, 7, 0) == g.GEMM_ERR_INVALID_VALUE   # activation
    assert g.gemm_fp8_tn_bias_act(*a, 0, *tail, 0x4000, 5, 1, 0) == g.GEMM_ERR_INVALID_VALUE   # bias dtype
    assert g.gemm_fp8_tn_bias_act(*a, 0, *tail, 0x4002, 1, 1, 0) == g.GEMM_ERR_MISALIGNED      # fp32 bias at 2 B
