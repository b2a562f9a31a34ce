"""GPU parity of the fused MLP epilogue, D = act(alpha A B^T + beta C + bias).

Against the FP64 oracle (GEMM then epilogue):
* integer inputs, integer bias, no activation or ReLU: bit-exact (pins the
  per-column bias indexing on all three kernel paths, ragged N included);
* real inputs, every activation: within the pre-activation bound times the
  activation's slope plus fp32 evaluation error (oracle.bound_act).
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import empty_out, from_dev, to_dev_bf16, to_dev_f32  # noqa: E402

# M picks the kernel path: 48 -> skinny, 100 -> 1-SM tiled, 2200 -> 2-SM tiled
# (with N at least 1040: more than 64 tiles of 128 x 256, so pair tiles)
PATH_M = {"skinny": 24, "1sm": 100, "2sm": 2200}
PATH_CODE = {"skinny": 3, "1sm": 1, "2sm": 2}


def shape_n(path, n):
    """N for a test on `path`: the 2-SM case needs enough tiles to use pair tiles."""
    return max(n, 1040) if path == "2sm" else n


def check_path(path):
    assert g.last_launch_info()["path"] == PATH_CODE[path], g.last_launch_info()


def _run(M, N, K, A, B, bias, bias_dtype, act, out_dtype, C=None, beta=0.0):
    import torch
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dbias = None
    if bias is not None:
        dbias = to_dev_bf16(bias) if bias_dtype == 0 else to_dev_f32(bias)
    dC = None
    if C is not None:
        dC = to_dev_bf16(C) if out_dtype == gi.OUT_BF16 else to_dev_f32(C)
    dD, ldd = empty_out(M, N, out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_tn_bias_act(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K,
                                 dC.data_ptr() if dC is not None else 0, N if dC is not None else 0,
                                 dD.data_ptr(), ldd, 1.0, beta, out_dtype,
                                 dbias.data_ptr() if dbias is not None else 0, bias_dtype, act, s)
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(s) == 0, g.last_error()
    return from_dev(dD, out_dtype)


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("bias_dtype", [0, 1])
def test_integer_bias_exact(path, act, bias_dtype):
    M, N, K = PATH_M[path], shape_n(path, 520), 192
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 4000)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 4001)
    bias = gi.draw_bf16(N, 1, gi.Dist("int", -50, 50), 4002).reshape(N)
    if bias_dtype == 1:
        bias = gi.bf16_bits_to_f32(bias)
    ref, _ = oracle.gemm_ref(A, B)
    want = oracle.epilogue(ref, bias, act)
    got = _run(M, N, K, A, B, bias, bias_dtype, act, gi.OUT_F32)
    check_path(path)
    assert np.array_equal(got, oracle.exact_f32(want))


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("act", [1, 2, 3, 4])
@pytest.mark.parametrize("out_dtype", [gi.OUT_BF16, gi.OUT_F32])
def test_activations_within_bound(path, act, out_dtype):
    M, N, K = PATH_M[path], shape_n(path, 776), 512
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 4100 + act)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 4.0 / K), 4200 + act)       # z ~ N(0, 4)
    bias = gi.draw_bf16(N, 1, gi.Dist("normal", 1.0), 4300).reshape(N)
    ref, absdot = oracle.gemm_ref(A, B)
    z = oracle.epilogue(ref, bias, 0)
    fz = oracle.epilogue(ref, bias, act)
    got = oracle.decode_out(_run(M, N, K, A, B, bias, 0, act, out_dtype), out_dtype)
    check_path(path)
    bnd = oracle.bound_act(z, fz, absdot, out_dtype, act)
    err = np.abs(got - fz)
    assert np.all(err <= bnd), float(np.max(err / bnd))


@pytest.mark.parametrize("path", list(PATH_M))
@pytest.mark.parametrize("act", [3, 4])
def test_logistic_activations_in_the_tails(path, act):
    """Pre-activations spread over [-130, 130] by an fp32 bias: the saturated
    tails of tanh-GELU and SiLU, and below -80 (SiLU) or about -9.7
    (tanh-GELU), where the kernel caps the exponent of its logistic form."""
    M, N, K = PATH_M[path], shape_n(path, 520), 128
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 4700 + act)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 4710 + act)
    bias = gi.draw_f32(N, 1, gi.Dist("uniform", -130.0, 130.0), 4720 + act).reshape(N)
    ref, absdot = oracle.gemm_ref(A, B)
    z = oracle.epilogue(ref, bias, 0)
    fz = oracle.epilogue(ref, bias, act)
    assert np.any(z < -90.0) and np.any(z > 90.0)
    for out_dtype in (gi.OUT_F32, gi.OUT_BF16):
        got = oracle.decode_out(_run(M, N, K, A, B, bias, 1, act, out_dtype), out_dtype)
        check_path(path)
        bnd = oracle.bound_act(z, fz, absdot, out_dtype, act)
        err = np.abs(got - fz)
        assert np.all(err <= bnd), float(np.max(err / bnd))


@pytest.mark.parametrize("path", list(PATH_M))
def test_gelu_with_c_and_fp32_bias(path):
    M, N, K = PATH_M[path], shape_n(path, 264), 320
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 4400)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 4401)
    C = gi.draw_bf16(M, N, gi.Dist("normal", 1.0), 4402)
    bias = gi.draw_f32(N, 1, gi.Dist("normal", 1.0), 4403).reshape(N)
    ref, absdot = oracle.gemm_ref(A, B, C, 1.0, 0.5)
    z = oracle.epilogue(ref, bias, 0)
    fz = oracle.epilogue(ref, bias, 2)
    got = oracle.decode_out(_run(M, N, K, A, B, bias, 1, 2, gi.OUT_BF16, C=C, beta=0.5), 0)
    check_path(path)
    bnd = oracle.bound_act(z, fz, absdot, 0, 2, 0.5, gi.bf16_bits_to_f32(C))
    assert np.all(np.abs(got - fz) <= bnd)


def test_no_bias_no_activation_equals_plain_gemm():
    import torch
    M, N, K = 300, 520, 256
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 4500)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 4501)
    fused = _run(M, N, K, A, B, None, 0, 0, gi.OUT_BF16)
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    s = torch.cuda.current_stream().cuda_stream
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)   # keep the buffers alive across the call
    rc = g.gemm_bf16_tn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0,
                        dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_BF16, s)
    assert rc == 0 and g.gemm_get_status(s) == 0
    assert np.array_equal(fused, from_dev(dD, gi.OUT_BF16))


def test_bias_act_argument_errors():
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0)
    assert g.gemm_bf16_tn_bias_act(*a, 0x4000, 0, 7, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_bf16_tn_bias_act(*a, 0x4000, 5, 1, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_bf16_tn_bias_act(*a, 0x4002, 1, 1, 0) == g.GEMM_ERR_MISALIGNED


@pytest.mark.parametrize("act", [0, 1, 3])
def test_wide_streaming_epilogue(act):
    """96 tokens against a 4608 x 8192 weight (72 MiB): the auto path is the
    streaming kernel's wide form (64-row tiles, two k-parts each).  Checked on
    every row at sampled columns, tile edges included."""
    M, N, K = 96, 4608, 8192
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 4600 + act)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 4610 + act)
    bias = gi.draw_bf16(N, 1, gi.Dist("int", -50, 50), 4620).reshape(N)
    got = _run(M, N, K, A, B, bias, 0, act, gi.OUT_F32)
    assert g.last_launch_info()["path"] == 3 and g.last_launch_info()["tile_m"] == 64
    cols_1 = sorted(set(np.random.default_rng(4630).integers(0, N, 200).tolist())
                    | {0, 63, 64, 127, 128, N - 65, N - 64, N - 1})
    rows = np.repeat(np.arange(M), len(cols_1))
    cols = np.tile(np.array(cols_1), M)
    ref, absdot = oracle.gemm_ref_sampled(A, B, rows, cols)
    g_s = got[rows, cols]
    if act in (0, 1):
        exp = oracle.exact_f32(oracle.epilogue(ref[None, :], bias[cols], act))[0]
        assert np.array_equal(g_s, exp)
    else:
        z = oracle.epilogue(ref[None, :], bias[cols], 0)[0]
        fz = oracle.epilogue(ref[None, :], bias[cols], act)[0]
        bnd = oracle.bound_act(z, fz, absdot, gi.OUT_F32, act)
        assert np.all(np.abs(g_s.astype(np.float64) - fz) <= bnd)
