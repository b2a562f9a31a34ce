"""Pins for the CPU oracle, each fixed by something other than the oracle itself.

* bf16 decoding against values fixed by the binary32 format (golden file);
* A = I gives D = B^T exactly; A = P (a permutation) permutes the rows of B^T;
* rank-1 closed form (u 1^T)(v 1^T)^T = K u v^T, exact for bf16 u, v and K = 2^p;
* transpose symmetry ref(A, B) = ref(B, A)^T;
* brute force on tiny shapes with exact rational arithmetic (independent decode);
* integer-valued inputs against an exact int64 matrix product;
* K = 0 gives beta * C; alpha linearity; row padding (lda/ldb/ldc > K/N) is not read;
* the sampled entry point agrees with the full one;
* a planted mistake (operands swapped = transposed product) fails the identity pin.
"""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import gemm_inputs as gi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def py_dec(h):
    """bf16 bits -> float through struct (independent of the oracle's decoder)."""
    return struct.unpack(">f", bytes([(h >> 8) & 0xFF, h & 0xFF, 0, 0]))[0]


def rand_bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return gi.f32_to_bf16_bits(x)


ONE = 0x3F80


def test_bf16_decode_golden():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                b, v = line.split()
                rows.append((int(b, 16), float(v)))
    A = np.array([[b] for b, _ in rows], dtype=np.uint16)   # M x 1
    B = np.array([[ONE]], dtype=np.uint16)                  # 1 x 1, value 1.0
    ref, absdot = oracle.gemm_ref(A, B)
    for (b, v), r, a in zip(rows, ref[:, 0], absdot[:, 0]):
        assert r == v, (hex(b), r, v)  # a sum started at +0 gives +0 for -0.0
        assert a == abs(v)
        assert py_dec(b) == v and np.signbit(py_dec(b)) == np.signbit(v)


def test_identity_gives_b_transpose():
    rng = np.random.default_rng(1)
    K, N = 40, 23
    A = np.zeros((K, K), dtype=np.uint16)
    A[np.arange(K), np.arange(K)] = ONE
    B = rand_bits(rng, (N, K))
    ref, _ = oracle.gemm_ref(A, B)
    Bf = gi.bf16_bits_to_f32(B).astype(np.float64)
    assert np.array_equal(ref, Bf.T)


def test_permutation_permutes_rows():
    rng = np.random.default_rng(2)
    K, N = 33, 17
    perm = rng.permutation(K)
    A = np.zeros((K, K), dtype=np.uint16)
    A[np.arange(K), perm] = ONE
    B = rand_bits(rng, (N, K))
    ref, _ = oracle.gemm_ref(A, B)
    Bf = gi.bf16_bits_to_f32(B).astype(np.float64)
    assert np.array_equal(ref, Bf.T[perm, :])


@pytest.mark.parametrize("K", [1, 16, 256, 1024])
def test_rank1_closed_form(K):
    rng = np.random.default_rng(3 + K)
    M, N = 19, 13
    u = rand_bits(rng, (M,))
    v = rand_bits(rng, (N,))
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[:, None], K, axis=1)
    ref, absdot = oracle.gemm_ref(A, B)
    uf = gi.bf16_bits_to_f32(u).astype(np.float64)
    vf = gi.bf16_bits_to_f32(v).astype(np.float64)
    expect = K * np.outer(uf, vf)
    assert np.array_equal(ref, expect)
    assert np.array_equal(absdot, np.abs(expect))


def test_transpose_symmetry():
    rng = np.random.default_rng(4)
    M, N, K = 21, 34, 57
    A = rand_bits(rng, (M, K))
    B = rand_bits(rng, (N, K))
    r1, _ = oracle.gemm_ref(A, B)
    r2, _ = oracle.gemm_ref(B, A)
    assert np.array_equal(r1, r2.T)


@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 4), (3, 5, 7), (4, 2, 9)])
@pytest.mark.parametrize("with_c", [False, True])
def test_brute_force_tiny(shape, with_c):
    M, N, K = shape
    rng = np.random.default_rng(sum(shape) + 10 * with_c)
    lda, ldb, ldc = K + 3, K + 1, N + 2
    A = rand_bits(rng, (M, lda))
    B = rand_bits(rng, (N, ldb))
    C = rand_bits(rng, (M, ldc)) if with_c else None
    alpha, beta = 0.75, (-1.5 if with_c else 0.0)
    ref, absdot = oracle.gemm_ref(A, B, C, alpha, beta, M=M, N=N, K=K,
                                  lda=lda, ldb=ldb, ldc=ldc)
    for i in range(M):
        for j in range(N):
            exact = Fraction(0)
            mag = Fraction(0)
            for k in range(K):
                p = Fraction(py_dec(int(A[i, k]))) * Fraction(py_dec(int(B[j, k])))
                exact += p
                mag += abs(p)
            exact *= Fraction(alpha)
            if with_c:
                exact += Fraction(beta) * Fraction(py_dec(int(C[i, j])))
            tol = float(mag) * abs(alpha) * K * 2.0 ** -52 + 2.0 ** -1000
            assert abs(ref[i, j] - float(exact)) <= tol, (i, j)
            assert abs(absdot[i, j] - float(abs(Fraction(alpha)) * mag)) <= tol


def test_integer_exact_against_int64():
    rng = np.random.default_rng(5)
    M, N, K = 70, 45, 300
    Ai = rng.integers(-4, 5, size=(M, K))
    Bi = rng.integers(-4, 5, size=(N, K))
    A = gi.f32_to_bf16_bits(Ai.astype(np.float32))
    B = gi.f32_to_bf16_bits(Bi.astype(np.float32))
    ref, absdot = oracle.gemm_ref(A, B)
    assert np.array_equal(ref, (Ai @ Bi.T).astype(np.float64))
    assert np.array_equal(absdot, (np.abs(Ai) @ np.abs(Bi).T).astype(np.float64))


def test_k_zero_gives_beta_c():
    rng = np.random.default_rng(6)
    M, N = 9, 11
    A = np.zeros((M, 1), dtype=np.uint16)
    B = np.zeros((N, 1), dtype=np.uint16)
    C = rand_bits(rng, (M, N))
    ref, absdot = oracle.gemm_ref(A, B, C, alpha=3.0, beta=0.5, K=0)
    assert np.array_equal(ref, 0.5 * gi.bf16_bits_to_f32(C).astype(np.float64))
    assert np.all(absdot == 0)
    Cf = gi.bf16_bits_to_f32(C)
    ref32, _ = oracle.gemm_ref(A, B, Cf, alpha=3.0, beta=-2.0, K=0)
    assert np.array_equal(ref32, -2.0 * Cf.astype(np.float64))


def test_beta_zero_ignores_nan_c():
    rng = np.random.default_rng(7)
    A = rand_bits(rng, (5, 8))
    B = rand_bits(rng, (6, 8))
    C = np.full((5, 6), 0x7FC0, dtype=np.uint16)  # NaN everywhere
    r1, _ = oracle.gemm_ref(A, B, C, 1.0, 0.0)
    r2, _ = oracle.gemm_ref(A, B)
    assert np.array_equal(r1, r2) and np.all(np.isfinite(r1))


def test_alpha_linearity():
    rng = np.random.default_rng(8)
    A = rand_bits(rng, (12, 40))
    B = rand_bits(rng, (15, 40))
    r1, a1 = oracle.gemm_ref(A, B, alpha=1.0)
    r2, a2 = oracle.gemm_ref(A, B, alpha=2.0)
    r3, a3 = oracle.gemm_ref(A, B, alpha=-0.5)
    assert np.array_equal(r2, 2 * r1) and np.array_equal(a2, 2 * a1)
    assert np.array_equal(r3, -0.5 * r1) and np.array_equal(a3, 0.5 * a1)


def test_padding_is_not_read():
    rng = np.random.default_rng(9)
    M, N, K = 7, 9, 13
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 11, ld=K + 8)   # NaN-padded
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0), 12, ld=K + 16)
    ref, _ = oracle.gemm_ref(A, B, M=M, N=N, K=K, lda=K + 8, ldb=K + 16)
    ref2, _ = oracle.gemm_ref(A[:, :K].copy(), B[:, :K].copy())
    assert np.all(np.isfinite(ref)) and np.array_equal(ref, ref2)


def test_sampled_matches_full():
    rng = np.random.default_rng(10)
    M, N, K = 37, 29, 65
    A = rand_bits(rng, (M, K))
    B = rand_bits(rng, (N, K))
    C = rand_bits(rng, (M, N))
    ref, absdot = oracle.gemm_ref(A, B, C, 1.25, 0.5)
    rows = rng.integers(0, M, 200)
    cols = rng.integers(0, N, 200)
    rs, as_ = oracle.gemm_ref_sampled(A, B, rows, cols, C, 1.25, 0.5)
    assert np.array_equal(rs, ref[rows, cols]) and np.array_equal(as_, absdot[rows, cols])
    with pytest.raises(ValueError):
        oracle.gemm_ref_sampled(A, B, [M], [0])


def test_thread_count_does_not_change_result():
    rng = np.random.default_rng(11)
    A = rand_bits(rng, (50, 77))
    B = rand_bits(rng, (31, 77))
    r1, _ = oracle.gemm_ref(A, B, nthreads=1)
    r7, _ = oracle.gemm_ref(A, B, nthreads=7)
    assert np.array_equal(r1, r7)


def test_planted_transpose_mistake_fails_identity_pin():
    """Swapping the operands (the product transposed) must break the A = I pin."""
    rng = np.random.default_rng(12)
    K = N = 24
    A = np.zeros((K, K), dtype=np.uint16)
    A[np.arange(K), np.arange(K)] = ONE
    B = rand_bits(rng, (N, K))
    good, _ = oracle.gemm_ref(A, B)
    planted, _ = oracle.gemm_ref(B, A)  # the mistake: B A^T instead of A B^T
    Bf = gi.bf16_bits_to_f32(B).astype(np.float64)
    assert np.array_equal(good, Bf.T)
    assert not np.array_equal(planted, Bf.T)


def test_tolerance_helpers():
    assert oracle.ulp_bf16(1.0) == 2.0 ** -7
    assert oracle.ulp_bf16(1.5) == 2.0 ** -7
    assert oracle.ulp_bf16(2.0) == 2.0 ** -6
    assert oracle.ulp_bf16(-0.75) == 2.0 ** -8
    assert oracle.ulp_bf16(0.0) == 2.0 ** -133
    ref = np.array([1.0, 1.0])
    ab = np.array([0.0, 0.0])
    D = gi.f32_to_bf16_bits(np.array([1.0, 1.0 + 2 ** -7], dtype=np.float32))
    ok, worst, _ = oracle.check(D, ref, ab, 0)
    assert ok and worst == 1.0
    D2 = gi.f32_to_bf16_bits(np.array([1.0, 1.0 + 2 ** -6], dtype=np.float32))
    ok, worst, _ = oracle.check(D2, ref, ab, 0)
    assert not ok


def test_workload_inputs_are_seeded_and_shaped():
    w = gi.WORKLOADS[0]
    A1, B1, C1 = gi.operands(w)
    A2, B2, _ = gi.operands(w)
    assert A1.shape == (256, 256) and B1.shape == (256, 256) and C1 is None
    assert np.array_equal(A1, A2) and np.array_equal(B1, B2)
    vals = gi.bf16_bits_to_f32(A1)
    assert set(np.unique(vals).tolist()) <= set(range(-4, 5))
    assert len(np.unique(vals)) == 9
    assert not np.array_equal(A1, B1)


def test_rne_rounding_of_inputs():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -1.0 - 2 ** -8],
                 dtype=np.float32)
    got = gi.bf16_bits_to_f32(gi.f32_to_bf16_bits(x))
    assert got.tolist() == [1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -1.0]


# ----------------------------------------------------------------------------- fused epilogue


def test_epilogue_matches_library_activations():
    """The FP64 activations against torch's own (float64, CPU) implementations."""
    torch = pytest.importorskip("torch")
    x = np.concatenate([np.linspace(-12, 12, 4001), [0.0, -0.0, 1e-8, -1e-8, 30.0, -30.0]])
    ref = x[None, :]
    t = torch.from_numpy(x)
    lib = {1: torch.relu(t), 2: torch.nn.functional.gelu(t),
           3: torch.nn.functional.gelu(t, approximate="tanh"), 4: torch.nn.functional.silu(t)}
    for act, want in lib.items():
        got = oracle.epilogue(ref, act=act)[0]
        # 1 + erf and 1 + tanh cancel for x < 0: agreement to FP64 rounding of the formula
        assert np.allclose(got, want.numpy(), rtol=1e-12, atol=1e-14), act
    assert np.array_equal(oracle.epilogue(ref, act=0)[0], x)


def test_epilogue_gelu_is_x_times_normal_cdf():
    """GELU(x) = x * Phi(x), Phi from scipy's normal distribution."""
    stats = pytest.importorskip("scipy.stats")
    x = np.linspace(-8, 8, 1601)
    got = oracle.epilogue(x[None, :], act=2)[0]
    assert np.allclose(got, x * stats.norm.cdf(x), rtol=1e-13, atol=1e-15)


def test_epilogue_bias_is_per_column_and_exact():
    rng = np.random.default_rng(21)
    ref = rng.standard_normal((5, 7))
    b16 = gi.f32_to_bf16_bits(rng.standard_normal(7).astype(np.float32))
    b32 = rng.standard_normal(7).astype(np.float32)
    assert np.array_equal(oracle.epilogue(ref, b16, 0), ref + gi.bf16_bits_to_f32(b16).astype(np.float64)[None, :])
    assert np.array_equal(oracle.epilogue(ref, b32, 0), ref + b32.astype(np.float64)[None, :])
    relu = oracle.epilogue(ref, b32, 1)
    assert np.array_equal(relu, np.maximum(ref + b32.astype(np.float64)[None, :], 0.0))
    with pytest.raises(ValueError):
        oracle.epilogue(ref, b32[:3], 0)


def test_epilogue_special_values():
    x = np.array([[0.0, 50.0, -50.0]])
    for act in (2, 3, 4):
        y = oracle.epilogue(x, act=act)[0]
        assert y[0] == 0.0 and y[1] == 50.0 and abs(y[2]) < 1e-20


# ----------------------------------------------------------------------------- fp8 operands


def _fp8_golden():
    rows = []
    with open(os.path.join(GOLDEN, "fp8_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                fmt, code, val = line.split()
                rows.append((0 if fmt == "e4m3" else 1, int(code, 16), float(val)))
    return rows


def test_fp8_decode_golden():
    for fmt, code, val in _fp8_golden():
        A = np.array([[code]], dtype=np.uint8)
        one = 0x38 if fmt == 0 else 0x3C
        B = np.array([[one]], dtype=np.uint8)
        ref, _ = oracle.gemm_ref_fp8(A, B, fmt)
        assert ref[0, 0] == val, (fmt, hex(code), ref[0, 0], val)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_decode_all_codes_against_torch(fmt):
    torch = pytest.importorskip("torch")
    dt = torch.float8_e4m3fn if fmt == 0 else torch.float8_e5m2
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(dt).to(torch.float64).numpy()
    one = 0x38 if fmt == 0 else 0x3C
    ref, _ = oracle.gemm_ref_fp8(codes[:, None], np.array([[one]], dtype=np.uint8), fmt)
    got = ref[:, 0]
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert np.all(same), codes[~same]
    # the input encoder inverts the decoder on every finite code
    fin = np.isfinite(want)
    enc = gi.f32_to_fp8_bits(want[fin], fmt)
    assert np.array_equal(gi.fp8_bits_to_f64(enc, fmt), want[fin])


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_integer_gemm_exact_and_identity(fmt):
    rng = np.random.default_rng(31 + fmt)
    M, N, K = 23, 17, 96
    Ai = rng.integers(-4, 5, size=(M, K))
    Bi = rng.integers(-4, 5, size=(N, K))
    A = gi.f32_to_fp8_bits(Ai, fmt)
    B = gi.f32_to_fp8_bits(Bi, fmt)
    ref, absdot = oracle.gemm_ref_fp8(A, B, fmt)
    assert np.array_equal(ref, (Ai @ Bi.T).astype(np.float64))
    eye = gi.f32_to_fp8_bits(np.eye(K), fmt)
    ref, _ = oracle.gemm_ref_fp8(eye, B, fmt)
    assert np.array_equal(ref, gi.fp8_bits_to_f64(B, fmt).T)


def test_fp8_rounding_ties_and_saturation():
    # e4m3 around 1: spacing 1/8; 1 + 1/16 ties to the even code (1.0)
    x = np.array([1.0 + 1 / 16, 1.0 + 3 / 16, 1000.0, -1000.0, 1e-9])
    got = gi.fp8_bits_to_f64(gi.f32_to_fp8_bits(x, 0), 0)
    assert got.tolist() == [1.0, 1.25, 448.0, -448.0, 0.0]


def test_fp8_sampled_matches_full():
    rng = np.random.default_rng(77)
    M, N, K = 37, 29, 160
    for fmt in (0, 1):
        A = gi.draw_fp8(M, K, gi.Dist("normal", 1.0), 900 + fmt, fmt)
        B = gi.draw_fp8(N, K, gi.Dist("normal", 1.0), 910 + fmt, fmt)
        C = gi.draw_f32(M, N, gi.Dist("normal", 1.0), 920)
        full, fabs_ = oracle.gemm_ref_fp8(A, B, fmt, C=C, alpha=0.75, beta=-0.5)
        r, c = rng.integers(0, M, 50), rng.integers(0, N, 50)
        s, sabs = oracle.gemm_ref_fp8_sampled(A, B, fmt, r, c, C=C, alpha=0.75, beta=-0.5)
        assert np.array_equal(s, full[r, c]) and np.array_equal(sabs, fabs_[r, c])
        # beta * C is the only other term: against the decoded operands' plain product
        a64 = gi.fp8_bits_to_f64(A, fmt)
        b64 = gi.fp8_bits_to_f64(B, fmt)
        assert np.allclose(full, 0.75 * (a64 @ b64.T) - 0.5 * C, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_encoder_is_nearest_ties_even(fmt):
    """The input encoder against a brute-force search over every finite code."""
    rng = np.random.default_rng(88 + fmt)
    top = 448.0 if fmt == 0 else 57344.0
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-4, 1e-2, 1.0, 30.0, top / 3)]).astype(np.float32)
    # exact midpoints between neighbouring finite values, and just past the top
    codes = np.arange(256, dtype=np.uint8)
    vals = gi.fp8_bits_to_f64(codes, fmt)
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, [top * 1.01, -top * 1.5, 1e30, 0.0]]).astype(np.float32)
    got = gi.fp8_bits_to_f64(gi.f32_to_fp8_bits(x, fmt), fmt)
    fin_codes = codes[np.isfinite(vals)]
    fin_vals = vals[np.isfinite(vals)]
    for xi, gv in zip(x.astype(np.float64), got):
        xc = min(max(xi, -top), top)
        d = np.abs(fin_vals - xc)
        best = fin_codes[d == d.min()]
        # among equally near codes, ties go to the even one (+0 and -0 both fine)
        want = {float(gi.fp8_bits_to_f64(np.uint8(c), fmt)) for c in best if c % 2 == 0 or len(best) == 1}
        assert gv in want or (xc == 0 and gv == 0), (xi, gv, want)
