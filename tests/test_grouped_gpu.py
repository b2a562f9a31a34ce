"""GPU parity of the grouped and the strided batched GEMM entry points.

Every problem of a group or batch is checked against the FP64 oracle:
integer inputs bit-exact (ragged shapes, K = 0 with beta * C, empty
problems, groups of more than 32 problems that take several launches),
real inputs within the bound.  A batch must also give the same bits as the
same GEMMs called one at a time.
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import empty_out, from_dev, to_dev_bf16, to_dev_f32  # noqa: E402


def up8(x):
    return (x + 7) // 8 * 8


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check_exact(got, ref, out_dtype):
    want = oracle.exact_f32(ref)
    if out_dtype == gi.OUT_BF16:
        want = gi.f32_to_bf16_bits(want)
    assert np.array_equal(got, want)


def _int_problem(M, N, K, seed, out_dtype, with_c):
    lda, ldb, ldd = up8(max(K, 1)), up8(max(K, 1)), up8(N)
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), seed, ld=lda) if K else np.zeros((M, lda), np.uint16)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), seed + 1, ld=ldb) if K else np.zeros((N, ldb), np.uint16)
    C = None
    if with_c:
        C = gi.draw_bf16(M, ldd, gi.Dist("int", -8, 8), seed + 2) if out_dtype == gi.OUT_BF16 else \
            gi.draw_f32(M, ldd, gi.Dist("int", -8, 8), seed + 2)
    return dict(M=M, N=N, K=K, A=A, B=B, C=C, lda=lda, ldb=ldb, ldd=ldd)


GROUP_SHAPES = [(256, 256, 256), (1, 7, 64), (100, 300, 130), (129, 257, 65), (300, 520, 200), (64, 64, 8),
                (7, 1000, 1), (0, 50, 64), (513, 40, 320), (255, 129, 0)]


@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_grouped_integer_exact(out_dtype, beta):
    probs = [_int_problem(M, N, K, 500 + 17 * i, out_dtype, beta != 0) for i, (M, N, K) in enumerate(GROUP_SHAPES)]
    dev = []
    for q in probs:
        dA, dB = to_dev_bf16(q["A"]), to_dev_bf16(q["B"])
        dC = None
        if q["C"] is not None:
            dC = to_dev_bf16(q["C"]) if out_dtype == gi.OUT_BF16 else to_dev_f32(q["C"])
        dD, _ = empty_out(max(q["M"], 1), q["N"], out_dtype, ld=q["ldd"])
        dev.append((dA, dB, dC, dD))
    arg = [dict(M=q["M"], N=q["N"], K=q["K"], A=dA.data_ptr(), lda=q["lda"], B=dB.data_ptr(), ldb=q["ldb"],
                C=dC.data_ptr() if dC is not None else 0, ldc=q["ldd"] if dC is not None else 0,
                D=dD.data_ptr(), ldd=q["ldd"]) for q, (dA, dB, dC, dD) in zip(probs, dev)]
    rc = g.gemm_bf16_tn_grouped(arg, 1.0, beta, out_dtype, _stream())
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(_stream()) == 0
    assert g.last_launch_info()["cluster"] == 1          # 30 tiles of 128 x 256: one wave
    for q, (_, _, _, dD) in zip(probs, dev):
        if q["M"] == 0:
            continue
        C = None if q["C"] is None else q["C"][:, :q["N"]]
        ref, _ = oracle.gemm_ref(q["A"], q["B"], C, 1.0, beta, M=q["M"], N=q["N"], K=q["K"],
                                 lda=q["lda"], ldb=q["ldb"])
        _check_exact(from_dev(dD, out_dtype)[:, :q["N"]], ref, out_dtype)


def test_grouped_pair_tiles():
    """Problems taller than 128 rows needing more than one wave of 1-SM tiles run
    on pair tiles: three 1024 x 2048 problems (64 tiles of 128 x 256 each)."""
    probs, dev = [], []
    for i in range(3):
        q = _int_problem(1024 - 3 * i, 2048, 192, 1500 + 5 * i, gi.OUT_F32, False)
        dA, dB = to_dev_bf16(q["A"]), to_dev_bf16(q["B"])
        dD, _ = empty_out(q["M"], q["N"], gi.OUT_F32, ld=q["ldd"])
        probs.append(q)
        dev.append((dA, dB, dD))
    arg = [dict(M=q["M"], N=q["N"], K=q["K"], A=dA.data_ptr(), lda=q["lda"], B=dB.data_ptr(), ldb=q["ldb"],
                C=0, ldc=0, D=dD.data_ptr(), ldd=q["ldd"]) for q, (dA, dB, dD) in zip(probs, dev)]
    assert g.gemm_bf16_tn_grouped(arg, 1.0, 0.0, gi.OUT_F32, _stream()) == 0, g.last_error()
    assert g.gemm_get_status(_stream()) == 0
    assert g.last_launch_info()["cluster"] == 2
    for q, (_, _, dD) in zip(probs, dev):
        ref, _ = oracle.gemm_ref(q["A"], q["B"], M=q["M"], N=q["N"], K=q["K"], lda=q["lda"], ldb=q["ldb"])
        _check_exact(from_dev(dD, gi.OUT_F32)[:, :q["N"]], ref, gi.OUT_F32)


def test_grouped_many_problems_several_launches():
    """70 problems of 256^3 with M <= 128 in some: 3 launches of <= 32 problems, 1-SM tiles."""
    probs, dev = [], []
    for i in range(70):
        M = 128 if i % 2 else 96
        q = _int_problem(M, 256, 256, 900 + 3 * i, gi.OUT_F32, False)
        dA, dB = to_dev_bf16(q["A"]), to_dev_bf16(q["B"])
        dD, _ = empty_out(M, 256, gi.OUT_F32, ld=q["ldd"])
        probs.append(q)
        dev.append((dA, dB, dD))
    arg = [dict(M=q["M"], N=q["N"], K=q["K"], A=dA.data_ptr(), lda=q["lda"], B=dB.data_ptr(), ldb=q["ldb"],
                C=0, ldc=0, D=dD.data_ptr(), ldd=q["ldd"]) for q, (dA, dB, dD) in zip(probs, dev)]
    assert g.gemm_bf16_tn_grouped(arg, 1.0, 0.0, gi.OUT_F32, _stream()) == 0, g.last_error()
    assert g.gemm_get_status(_stream()) == 0
    assert g.last_launch_info()["cluster"] == 1
    for q, (_, _, dD) in zip(probs, dev):
        ref, _ = oracle.gemm_ref(q["A"], q["B"])
        _check_exact(from_dev(dD, gi.OUT_F32), ref, gi.OUT_F32)


def test_grouped_real_within_bound():
    shapes = [(1000, 1504, 704), (64, 256, 4096), (333, 776, 1000)]
    dev, host = [], []
    for i, (M, N, K) in enumerate(shapes):
        A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 1300 + i)
        B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 1310 + i)
        C = gi.draw_bf16(M, N, gi.Dist("normal", 1.0), 1320 + i)
        host.append((A, B, C))
        dD, _ = empty_out(M, N, gi.OUT_BF16)
        dev.append((to_dev_bf16(A), to_dev_bf16(B), to_dev_bf16(C), dD))
    arg = [dict(M=M, N=N, K=K, A=dA.data_ptr(), lda=K, B=dB.data_ptr(), ldb=K, C=dC.data_ptr(), ldc=N,
                D=dD.data_ptr(), ldd=N) for (M, N, K), (dA, dB, dC, dD) in zip(shapes, dev)]
    assert g.gemm_bf16_tn_grouped(arg, 0.75, -0.5, gi.OUT_BF16, _stream()) == 0, g.last_error()
    assert g.gemm_get_status(_stream()) == 0
    for (A, B, C), (_, _, _, dD) in zip(host, dev):
        ref, absdot = oracle.gemm_ref(A, B, C, 0.75, -0.5)
        ok, worst, where = oracle.check(from_dev(dD, gi.OUT_BF16), ref, absdot, gi.OUT_BF16, -0.5,
                                        gi.bf16_bits_to_f32(C))
        assert ok, (worst, where)


def _batched(batch, M, N, K, out_dtype, beta, pad, seed):
    """Integer strided batch with `pad` extra elements between problems."""
    lda, ldd = up8(K), up8(N)
    sa, sb, sd = M * lda + pad, N * lda + pad, M * ldd + pad
    A = gi.draw_bf16(1, batch * sa, gi.Dist("int", -4, 4), seed).reshape(-1)
    B = gi.draw_bf16(1, batch * sb, gi.Dist("int", -4, 4), seed + 1).reshape(-1)
    C = None
    if beta:
        C = gi.draw_bf16(1, batch * sd, gi.Dist("int", -8, 8), seed + 2).reshape(-1) if out_dtype == gi.OUT_BF16 \
            else gi.draw_f32(1, batch * sd, gi.Dist("int", -8, 8), seed + 2).reshape(-1)
    return dict(A=A, B=B, C=C, lda=lda, ldd=ldd, sa=sa, sb=sb, sd=sd)


@pytest.mark.parametrize("batch,M,N,K", [(5, 300, 520, 200), (7, 100, 129, 65), (64, 256, 256, 256),
                                         (3, 1, 7, 64), (2, 513, 40, 0)])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_batched_integer_exact(batch, M, N, K, out_dtype):
    beta = 0.5 if (M + N) % 2 else 0.0
    h = _batched(batch, M, N, K, out_dtype, beta, pad=24, seed=2000 + M + N + K)
    dA, dB = to_dev_bf16(h["A"]), to_dev_bf16(h["B"])
    dC = None if h["C"] is None else (to_dev_bf16(h["C"]) if out_dtype == gi.OUT_BF16 else to_dev_f32(h["C"]))
    dD, _ = empty_out(1, batch * h["sd"], out_dtype)
    rc = g.gemm_bf16_tn_batched(batch, M, N, K, dA.data_ptr(), h["lda"], h["sa"], dB.data_ptr(), h["lda"], h["sb"],
                                dC.data_ptr() if dC is not None else 0, h["ldd"] if dC is not None else 0, h["sd"],
                                dD.data_ptr(), h["ldd"], h["sd"], 1.0, beta, out_dtype, _stream())
    assert rc == 0, g.last_error()
    assert g.gemm_get_status(_stream()) == 0
    D = from_dev(dD, out_dtype).reshape(-1)
    for b in range(batch):
        Ab = h["A"][b * h["sa"]: b * h["sa"] + M * h["lda"]].reshape(M, h["lda"])
        Bb = h["B"][b * h["sb"]: b * h["sb"] + N * h["lda"]].reshape(N, h["lda"])
        Cb = None if h["C"] is None else h["C"][b * h["sd"]: b * h["sd"] + M * h["ldd"]].reshape(M, h["ldd"])[:, :N]
        ref, _ = oracle.gemm_ref(Ab, Bb, Cb, 1.0, beta, M=M, N=N, K=K, lda=h["lda"], ldb=h["lda"])
        got = D[b * h["sd"]: b * h["sd"] + M * h["ldd"]].reshape(M, h["ldd"])[:, :N]
        _check_exact(got, ref, out_dtype)
        # the padding between problems is untouched (NaN pattern)
        gap = D[b * h["sd"] + M * h["ldd"]: (b + 1) * h["sd"]]
        fill = 0x7FC3 if out_dtype == gi.OUT_BF16 else None
        if fill is not None:
            assert np.all(gap == fill)
        else:
            assert np.all(np.isnan(gap))


def test_batched_matches_single_calls():
    batch, M, N, K = 6, 384, 512, 320
    A = gi.draw_bf16(batch * M, K, gi.Dist("normal", 1.0), 2100)
    B = gi.draw_bf16(batch * N, K, gi.Dist("normal", 1.0 / K), 2101)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, _ = empty_out(batch * M, N, gi.OUT_BF16)
    assert g.gemm_bf16_tn_batched(batch, M, N, K, dA.data_ptr(), K, M * K, dB.data_ptr(), K, N * K, 0, 0, 0,
                                  dD.data_ptr(), N, M * N, 1.0, 0.0, gi.OUT_BF16, _stream()) == 0, g.last_error()
    dS, _ = empty_out(batch * M, N, gi.OUT_BF16)
    for b in range(batch):
        rc = g.gemm_bf16_tn(M, N, K, dA.data_ptr() + 2 * b * M * K, K, dB.data_ptr() + 2 * b * N * K, K, 0, 0,
                            dS.data_ptr() + 2 * b * M * N, N, 1.0, 0.0, gi.OUT_BF16, _stream())
        assert rc == 0
    assert g.gemm_get_status(_stream()) == 0
    assert np.array_equal(from_dev(dD, gi.OUT_BF16), from_dev(dS, gi.OUT_BF16))
