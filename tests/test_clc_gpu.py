"""The cluster-launch-control tile scheduler (GEMM_SCHED_CLC) of the tiled paths.

One CTA (pair) is launched per tile; running CTAs cancel CTAs that have not
started and take over their tiles.  The schedule changes which CTA computes
a tile, never how: integer inputs stay bit-exact against the oracle, and
real inputs give the same bits as the static persistent schedule.
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import call, empty_out, from_dev, sample_positions, to_dev_bf16, to_dev_f32  # noqa: E402
from test_gemm_gpu import TILED_SHAPES, assert_same, run_int  # noqa: E402

P1, P2 = 1, 2
CLC, STATIC = 2, 1


@pytest.mark.parametrize("shape", TILED_SHAPES)
@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_integer_ragged_clc(shape, path, out_dtype):
    M, N, K = shape
    got, exp = run_int(M, N, K, path, out_dtype, seed=300 + M + 7 * N + 13 * K, scheduler=CLC)
    assert_same(got, exp)


@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("M,N,K", [(4096, 4096, 64), (2048, 6144, 8), (1536, 2560, 1000)])
def test_many_tiles_short_k(path, M, N, K):
    """Hundreds of tiles with one or a few k-blocks: the producer runs many
    tiles ahead of the epilogue, so the answer ring wraps and throttles."""
    got, exp = run_int(M, N, K, path, gi.OUT_F32, seed=400 + K, scheduler=CLC)
    assert_same(got, exp)


@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_same_bits_as_static(path, out_dtype):
    M, N, K = 1000, 1504, 704
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 1200)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 1201)
    C = gi.draw_bf16(M, N, gi.Dist("normal", 1.0), 1202) if out_dtype == gi.OUT_BF16 else \
        gi.draw_f32(M, N, gi.Dist("normal", 1.0), 1202)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dC = to_dev_bf16(C) if out_dtype == gi.OUT_BF16 else to_dev_f32(C)
    outs = []
    for sched in (STATIC, CLC):
        dD, ldd = empty_out(M, N, out_dtype)
        rc, st = call(M, N, K, dA, K, dB, K, dC, N, dD, ldd, 0.75, -0.5, out_dtype, path=path, scheduler=sched)
        assert rc == 0 and st == 0, g.last_error()
        outs.append(from_dev(dD, out_dtype))
    assert np.array_equal(outs[0], outs[1])
    ref, absdot = oracle.gemm_ref(A, B, C, 0.75, -0.5)
    cvals = gi.bf16_bits_to_f32(C) if out_dtype == gi.OUT_BF16 else C
    ok, worst, where = oracle.check(outs[1], ref, absdot, out_dtype, -0.5, cvals)
    assert ok, (worst, where)


@pytest.mark.parametrize("path,cg", [(P1, 1), (P2, 2)])
def test_launch_info(path, cg):
    M, N, K = 1000, 1504, 128
    dA = to_dev_bf16(gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 1))
    dB = to_dev_bf16(gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 2))
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    tiles = -(-M // (128 * cg)) * -(-N // 256)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_BF16, path=path, scheduler=CLC)
    assert rc == 0 and st == 0
    info = g.last_launch_info()
    assert info["scheduler"] == CLC and info["grid"] == tiles * cg and info["cluster"] == cg
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_BF16, path=path, scheduler=STATIC)
    assert rc == 0 and st == 0
    assert g.last_launch_info()["scheduler"] == STATIC


def test_mlp_up_projection_clc_same_bits_as_static():
    """8192 x 28672 x 4096 under cluster launch control: every tile is the same
    computation whichever CTA takes it, so all 235 M outputs must carry the bits
    of the static schedule (which test_gemm_gpu checks against the oracle
    element by element), and sampled outputs are checked against the oracle
    directly as well."""
    w = gi.WORKLOADS[3]
    A, B, _ = gi.operands(w)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    outs = []
    for sched in (CLC, STATIC):
        dD, ldd = empty_out(w.M, w.N, w.out_dtype)
        rc, st = call(w.M, w.N, w.K, dA, w.K, dB, w.K, None, 0, dD, ldd,
                      w.alpha, w.beta, w.out_dtype, scheduler=sched)
        assert rc == 0 and st == 0, g.last_error()
        assert g.last_launch_info()["scheduler"] == sched
        outs.append(from_dev(dD, w.out_dtype))
        del dD
    assert np.array_equal(outs[0], outs[1])
    rows, cols = sample_positions(w.M, w.N, n_random=4000, seed=31)
    ref, absdot = oracle.gemm_ref_sampled(A, B, rows, cols)
    ok, worst, where = oracle.check(outs[0][rows, cols], ref, absdot, w.out_dtype)
    assert ok, (worst, where)


def test_unknown_scheduler_rejected():
    dA = to_dev_bf16(gi.draw_bf16(256, 64, gi.Dist("int", -4, 4), 1))
    dD, ldd = empty_out(256, 256, gi.OUT_F32)
    rc, _ = call(256, 256, 64, dA, 64, dA, 64, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_F32, scheduler=7)
    assert rc == g.GEMM_ERR_INVALID_VALUE


def test_clc_scheduler_never_splits():
    """A k-split request under cluster launch control runs unsplit."""
    got, exp = run_int(300, 520, 640, 2, gi.OUT_F32, seed=930, scheduler=2, tiled_k_parts=2)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["scheduler"] == 2 and info["k_parts"] == 1
