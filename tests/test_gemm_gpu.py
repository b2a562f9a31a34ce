"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* integer-valued inputs: bit-exact (every partial sum is an integer < 2^24);
* real-valued inputs: |D - ref| <= 1e-4 (sum_k |a b| + |beta c|) (+ 1 bf16 ulp);
* the five workloads at full size, every element against the oracle, in the
  launch configuration the benchmark uses;
* edge cases: ragged M/N/K, K = 0, NaN in an unread C, in-place C == D,
  padding and rows beyond M untouched, determinism, small persistent grids,
  stream-K splits of the skinny path.
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import call, check_every_element, empty_out, from_dev, to_dev_bf16, to_dev_f32  # noqa: E402

P1, P2, PS = 1, 2, 3


def expect_exact(ref, out_dtype):
    f = oracle.exact_f32(ref)
    if out_dtype == gi.OUT_F32:
        return f
    return gi.f32_to_bf16_bits(f)


def up8(x):
    """Leading dimensions must be multiples of 16 bytes: pad to 8 elements."""
    return (x + 7) // 8 * 8


def run_int(M, N, K, path, out_dtype, seed, lda=None, ldb=None, grid=0, skinny_grid=0, alpha=1.0,
            disable_pdl=0, scheduler=0, skinny_bm=0, skinny_kgroup=0, tiled_k_parts=0, b_static=0,
            skinny_pair=0):
    lda = up8(K) if lda is None else lda
    ldb = up8(K) if ldb is None else ldb
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), seed, ld=lda)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), seed + 1, ld=ldb)
    ref, _ = oracle.gemm_ref(A, B, alpha=alpha, M=M, N=N, K=K, lda=lda, ldb=ldb)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, out_dtype, ld=up8(N))
    rc, st = call(M, N, K, dA, lda, dB, ldb, None, 0, dD, ldd, alpha, 0.0, out_dtype, path=path,
                  grid=grid, skinny_grid=skinny_grid, disable_pdl=disable_pdl, scheduler=scheduler,
                  skinny_bm=skinny_bm, skinny_kgroup=skinny_kgroup, tiled_k_parts=tiled_k_parts,
                  b_static=b_static, skinny_pair=skinny_pair)
    assert rc == 0, g.last_error()
    assert st == 0, g.last_error()
    return from_dev(dD, out_dtype)[:, :N], expect_exact(ref, out_dtype)


def assert_same(got, exp):
    if not np.array_equal(got.view(np.uint32) if got.dtype == np.float32 else got,
                          exp.view(np.uint32) if exp.dtype == np.float32 else exp):
        bad = np.argwhere(got != exp)
        pytest.fail(f"{len(bad)} mismatches; first {bad[:5].tolist()}: got {got[tuple(bad[0])]} "
                    f"expected {exp[tuple(bad[0])]}")


# ----------------------------------------------------------------------------- exact


@pytest.mark.parametrize("path", [P1, P2, 0])
def test_tiny_exact_workload(path):
    w = gi.WORKLOADS[0]
    A, B, _ = gi.operands(w)
    ref, _ = oracle.gemm_ref(A, B)
    dD, ldd = empty_out(w.M, w.N, w.out_dtype)
    rc, st = call(w.M, w.N, w.K, to_dev_bf16(A), w.K, to_dev_bf16(B), w.K, None, 0, dD, ldd,
                  w.alpha, w.beta, w.out_dtype, path=path)
    assert rc == 0 and st == 0, g.last_error()
    assert_same(from_dev(dD, w.out_dtype), oracle.exact_f32(ref))


TILED_SHAPES = [(128, 256, 64), (129, 257, 65), (127, 255, 63), (255, 129, 130), (257, 300, 1),
                (7, 9, 17), (513, 520, 200), (384, 1024, 320), (1, 1, 1), (96, 40, 8)]


@pytest.mark.parametrize("shape", TILED_SHAPES)
@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_integer_ragged_tiled(shape, path, out_dtype):
    M, N, K = shape
    got, exp = run_int(M, N, K, path, out_dtype, seed=100 + M + 7 * N + 13 * K)
    assert_same(got, exp)


SKINNY_SHAPES = [(16, 256, 256), (1, 300, 70), (16, 1000, 640), (33, 129, 1000), (64, 260, 513),
                 (5, 8192, 64), (48, 128, 8192)]


@pytest.mark.parametrize("shape", SKINNY_SHAPES)
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_integer_ragged_skinny(shape, out_dtype):
    M, N, K = shape
    got, exp = run_int(M, N, K, PS, out_dtype, seed=200 + M + 7 * N + 13 * K)
    assert_same(got, exp)


@pytest.mark.parametrize("shape", SKINNY_SHAPES)
@pytest.mark.parametrize("bm", [64, 128])
def test_integer_ragged_skinny_tile_rows(shape, bm):
    """Both B-tile heights (MMA M = 64 or 128) on every skinny shape."""
    M, N, K = shape
    got, exp = run_int(M, N, K, PS, gi.OUT_F32, seed=250 + M + 7 * N + 13 * K, skinny_bm=bm)
    assert_same(got, exp)


@pytest.mark.parametrize("skinny_grid", [0, 1, 7, 33, 100, 151])
@pytest.mark.parametrize("K", [64, 1344, 4160])
def test_skinny_bm64_partitions(skinny_grid, K):
    """64-row tiles split between CTAs (stream-K ranges): only lanes 0..15 of
    each epilogue warp hold rows, in partials and fix-ups alike."""
    got, exp = run_int(16, 1000, K, PS, gi.OUT_BF16, seed=700 + skinny_grid + K, skinny_grid=skinny_grid,
                       skinny_bm=64)
    assert_same(got, exp)


def test_decode_shape_launch():
    M, N, K = 16, 8192, 512
    got, exp = run_int(M, N, K, 0, gi.OUT_BF16, seed=777)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["path"] == PS and info["tile_m"] == 128 and info["grid"] == 128
    got, exp = run_int(M, N, K, 0, gi.OUT_BF16, seed=777, skinny_bm=64)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["tile_m"] == 64 and info["grid"] == 128      # 128 whole 64-row tiles, one per CTA


KGROUP_SHAPES = [(16, 1000, 640), (1, 300, 1344), (64, 260, 4160), (33, 8192, 256), (16, 129, 64),
                 (7, 520, 1000)]


@pytest.mark.parametrize("shape", KGROUP_SHAPES)
@pytest.mark.parametrize("bm", [64, 128])
@pytest.mark.parametrize("kg", [1, 2, 4])
def test_skinny_kgroups(shape, bm, kg):
    """kg k-blocks per ring stage, loaded as one 3D box per operand.  K = 640,
    1344 and 4160 leave the last group short (its missing k-blocks are
    zero-filled); K = 1000 is not a whole number of k-blocks, so the path
    falls back to one k-block per stage."""
    M, N, K = shape
    got, exp = run_int(M, N, K, PS, gi.OUT_BF16, seed=330 + M + 7 * N + K + bm + kg, skinny_bm=bm,
                       skinny_kgroup=kg)
    assert_same(got, exp)


@pytest.mark.parametrize("kg", [2, 4])
@pytest.mark.parametrize("bm", [64, 128])
def test_skinny_kgroups_padded_leading_dims(kg, bm):
    got, exp = run_int(40, 270, 640, PS, gi.OUT_F32, seed=340 + kg + bm, lda=704, ldb=768, skinny_bm=bm,
                       skinny_kgroup=kg)
    assert_same(got, exp)


@pytest.mark.parametrize("bm", [64, 128])
def test_skinny_kgroups_wide(bm):
    """144 tokens with two k-blocks per stage (forced; automatic keeps one here)."""
    got, exp = run_int(144, 700, 1344, PS, gi.OUT_BF16, seed=350 + bm, skinny_bm=bm, skinny_kgroup=2)
    assert_same(got, exp)


def test_skinny_kgroups_too_large_for_the_ring():
    M, N, K = 144, 256, 1024
    dA, dB = to_dev_bf16(np.zeros((M, K), np.uint16)), to_dev_bf16(np.zeros((N, K), np.uint16))
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    rc, _ = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_BF16, path=PS, skinny_bm=128,
                 skinny_kgroup=4)
    assert rc == g.GEMM_ERR_INVALID_VALUE and "ring stages" in g.last_error()


@pytest.mark.parametrize("M", [1, 17, 32])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_skinny_two_part_tiles(M, out_dtype):
    """N = 8192 splits each 128-row tile in two k-parts (128 CTAs); with up to
    32 tokens the finisher fetches the other part's partial before its own
    accumulator is ready."""
    got, exp = run_int(M, 8192, 1088, PS, out_dtype, seed=360 + M)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["grid"] == 128 and info["tile_m"] == 128


@pytest.mark.parametrize("M,N,tile_m,grid", [(64, 8192, 64, 128), (48, 8192, 64, 128), (32, 8192, 128, 128),
                                             (24, 4096, 64, 128), (8, 4096, 128, 128), (64, 16384, 128, 128),
                                             (128, 4096, 64, 128)])
def test_skinny_automatic_tile_rows(M, N, tile_m, grid):
    """64-row tiles where they fit one wave and cut the parts per tile, else 128 rows."""
    got, exp = run_int(M, N, 2048, PS, gi.OUT_BF16, seed=370 + M + N)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert (info["tile_m"], info["grid"]) == (tile_m, grid), info


WIDE_SHAPES = [(65, 300, 256), (80, 1000, 640), (128, 520, 2048), (200, 130, 1000), (256, 384, 300),
               (97, 8192, 128)]


@pytest.mark.parametrize("shape", WIDE_SHAPES)
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_integer_ragged_skinny_wide(shape, out_dtype):
    """65..256 tokens on the streaming kernel (tokens as MMA N up to 256, chunked epilogue)."""
    M, N, K = shape
    got, exp = run_int(M, N, K, PS, out_dtype, seed=260 + M + 7 * N + 13 * K)
    assert_same(got, exp)
    assert g.last_launch_info()["tile_n"] == -(-M // 16) * 16


@pytest.mark.parametrize("skinny_grid", [1, 7, 33, 100, 151])
@pytest.mark.parametrize("bm", [64, 128])
def test_skinny_wide_partitions(skinny_grid, bm):
    """Wide accumulators split between CTAs: partials published and added chunk by chunk."""
    for rep in range(2):
        got, exp = run_int(144, 700, 1344, PS, gi.OUT_BF16, seed=310 + rep + bm, skinny_grid=skinny_grid,
                           skinny_bm=bm)
        assert_same(got, exp)


def test_mid_batch_decode_streams():
    """128 tokens against an 8192 x 4096 weight: auto path is the streaming kernel."""
    M, N, K = 128, 8192, 4096
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 320)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 321)
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_BF16)
    assert rc == 0 and st == 0, g.last_error()
    assert g.last_launch_info()["path"] == PS
    ref, absdot = oracle.gemm_ref(A, B)
    ok, worst, where = oracle.check(from_dev(dD, gi.OUT_BF16), ref, absdot, gi.OUT_BF16)
    assert ok, (worst, where)


@pytest.mark.parametrize("skinny_grid", [1, 3, 7, 64, 100, 151, 1000])
@pytest.mark.parametrize("K", [64, 1344, 4160])
def test_skinny_stream_k_partitions(skinny_grid, K):
    # every split of the (n-tile, k-block) units gives the same exact result, and the
    # arrival counters are left clean for the next call
    for rep in range(2):
        got, exp = run_int(16, 640, K, PS, gi.OUT_F32, seed=300 + rep, skinny_grid=skinny_grid)
        assert_same(got, exp)


@pytest.mark.parametrize("skew", [-1, 1, 5, 1000])
def test_skinny_equal_split_skew(skew):
    # default grid on 16 x 1024 x 4096 is the equal-split mode (8 tiles x 4 parts);
    # every skew (clamped so each part keeps a k-group) gives the exact result
    import torch
    M, N, K = 16, 1024, 4096
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 320)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 321)
    ref, _ = oracle.gemm_ref(A, B)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)   # keep the buffers alive across the calls
    for rep in range(2):
        dD, ldd = empty_out(M, N, gi.OUT_F32)
        cfg = g.GemmConfig(path=PS, skinny_skew_kb=skew)
        rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0,
                               dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_F32,
                               torch.cuda.current_stream().cuda_stream, cfg)
        assert rc == 0, g.last_error()
        assert g.gemm_get_status(torch.cuda.current_stream().cuda_stream) == 0
        assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_without_programmatic_launch(path):
    M = 16 if path == PS else 300
    got, exp = run_int(M, 520, 640, path, gi.OUT_BF16, seed=310, disable_pdl=1)
    assert_same(got, exp)


@pytest.mark.parametrize("path,grid", [(P1, 1), (P1, 3), (P2, 2), (P2, 6)])
def test_small_persistent_grid(path, grid):
    # few CTAs, many tiles each: ring wrap-around and accumulator double buffering
    got, exp = run_int(700, 1100, 448, path, gi.OUT_F32, seed=400, grid=grid)
    assert_same(got, exp)


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_padded_leading_dims(path):
    M = 40 if path == PS else 300
    got, exp = run_int(M, 270, 150, path, gi.OUT_BF16, seed=500, lda=168, ldb=256)
    assert_same(got, exp)


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_alpha_scaling_exact(path):
    M = 24 if path == PS else 260
    got1, _ = run_int(M, 300, 200, path, gi.OUT_F32, seed=600)
    got2, _ = run_int(M, 300, 200, path, gi.OUT_F32, seed=600, alpha=2.0)
    assert np.array_equal(got2, 2 * got1)


# ----------------------------------------------------------------------------- edge cases


@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_k_zero_gives_beta_c(out_dtype):
    M, N = 300, 264
    rng = np.random.default_rng(1)
    Cb = gi.f32_to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    Cf = gi.bf16_bits_to_f32(Cb)
    dC = to_dev_bf16(Cb) if out_dtype == gi.OUT_BF16 else to_dev_f32(Cf)
    dD, ldd = empty_out(M, N, out_dtype)
    rc, st = call(M, N, 0, None, 0, None, 0, dC, N, dD, ldd, 1.0, 0.5, out_dtype)
    assert rc == 0 and st == 0, g.last_error()
    got = oracle.decode_out(from_dev(dD, out_dtype), out_dtype)
    assert np.array_equal(got, 0.5 * Cf.astype(np.float64))
    dD2, _ = empty_out(M, N, out_dtype)
    rc, st = call(M, N, 0, None, 0, None, 0, None, 0, dD2, ldd, 1.0, 0.0, out_dtype)
    assert rc == 0 and st == 0
    assert np.all(oracle.decode_out(from_dev(dD2, out_dtype), out_dtype) == 0)


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_beta_zero_does_not_read_nan_c(path):
    M, N, K = (32 if path == PS else 300), 264, 128
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 700)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 701)
    ref, _ = oracle.gemm_ref(A, B)
    dC = to_dev_bf16(np.full((M, N), 0x7FC0, dtype=np.uint16))
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, dC, N, dD, ldd, 1.0, 0.0,
                  gi.OUT_BF16, path=path)
    assert rc == 0 and st == 0
    assert_same(from_dev(dD, gi.OUT_BF16), expect_exact(ref, gi.OUT_BF16))


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_in_place_c_equals_d(path):
    M, N, K = (20 if path == PS else 260), 296, 96
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 800)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 801)
    Cb = gi.draw_bf16(M, N, gi.Dist("int", -8, 8), 802)
    ref, _ = oracle.gemm_ref(A, B, Cb, 1.0, 0.5)
    dCD = to_dev_bf16(Cb)
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, dCD, N, dCD, N, 1.0, 0.5,
                  gi.OUT_BF16, path=path)
    assert rc == 0 and st == 0
    assert_same(from_dev(dCD, gi.OUT_BF16), expect_exact(ref, gi.OUT_BF16))


@pytest.mark.parametrize("path", [P1, P2, PS])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_guard_bands_untouched(path, out_dtype):
    """Row padding (ldd > N) and rows past M keep their canary bits."""
    import torch
    M, N, K = (40 if path == PS else 300), 200, 136
    extra_rows, ldd = 9, 264
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 900)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 901)
    ref, _ = oracle.gemm_ref(A, B)
    dD, _ = empty_out(M + extra_rows, N, out_dtype, ld=ldd)
    canary = from_dev(dD, out_dtype).copy()
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, None, 0, dD, ldd, 1.0, 0.0,
                  out_dtype, path=path)
    assert rc == 0 and st == 0
    torch.cuda.synchronize()
    got = from_dev(dD, out_dtype)
    assert_same(got[:M, :N], expect_exact(ref, out_dtype))
    as_bits = (lambda x: x.view(np.uint32)) if out_dtype == gi.OUT_F32 else (lambda x: x)
    assert np.array_equal(as_bits(got[:M, N:]), as_bits(canary[:M, N:]))
    assert np.array_equal(as_bits(got[M:]), as_bits(canary[M:]))


@pytest.mark.parametrize("path", [P1, P2, PS])
def test_deterministic(path):
    M, N, K = (16 if path == PS else 520), 1024, 2048
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 1000)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 1001)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    outs = []
    for _ in range(3):
        dD, ldd = empty_out(M, N, gi.OUT_F32)
        rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_F32, path=path)
        assert rc == 0 and st == 0
        outs.append(from_dev(dD, gi.OUT_F32).view(np.uint32))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_argument_errors():
    import torch
    dA = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    dD = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    base = dict(M=64, N=64, K=64, A=dA.data_ptr(), lda=64, B=dA.data_ptr(), ldb=64, C=0, ldc=0,
                D=dD.data_ptr(), ldd=64, alpha=1.0, beta=0.0, out_dtype=0, stream=s)

    def rc(**kw):
        a = dict(base, **kw)
        return g.gemm_bf16_tn(*a.values())

    assert rc() == g.GEMM_OK
    assert rc(A=dA.data_ptr() + 2) == g.GEMM_ERR_MISALIGNED
    assert rc(lda=65) == g.GEMM_ERR_MISALIGNED
    assert rc(lda=32) == g.GEMM_ERR_INVALID_VALUE
    assert rc(beta=1.0) == g.GEMM_ERR_INVALID_VALUE
    assert rc(out_dtype=2) == g.GEMM_ERR_INVALID_VALUE
    assert rc(M=0) == g.GEMM_OK
    cfg = g.GemmConfig(path=g.PATH_SKINNY)
    a = dict(base, M=257)
    assert g.gemm_bf16_tn_ex(*a.values(), cfg) == g.GEMM_ERR_NOT_IMPLEMENTED
    torch.cuda.synchronize()
    assert g.gemm_get_status(s) == 0


# ----------------------------------------------------------------------------- tolerance


@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_random_with_beta_tolerance(path, out_dtype):
    M, N, K = 1000, 1504, 704
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 1100)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0), 1101)
    if out_dtype == gi.OUT_BF16:
        C = gi.draw_bf16(M, N, gi.Dist("normal", 1.0), 1102)
        dC = to_dev_bf16(C)
        cvals = gi.bf16_bits_to_f32(C)
    else:
        C = gi.draw_f32(M, N, gi.Dist("normal", 1.0), 1102)
        dC = to_dev_f32(C)
        cvals = C
    ref, absdot = oracle.gemm_ref(A, B, C, 0.75, -1.25)
    dD, ldd = empty_out(M, N, out_dtype)
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, dC, N, dD, ldd, 0.75, -1.25,
                  out_dtype, path=path)
    assert rc == 0 and st == 0
    ok, worst, where = oracle.check(from_dev(dD, out_dtype), ref, absdot, out_dtype, -1.25, cvals)
    assert ok, (worst, where)


# ----------------------------------------------------------------------------- workloads


def _run_workload(w, path=0):
    A, B, C = gi.operands(w)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dC = None
    if C is not None:
        dC = to_dev_bf16(C) if w.out_dtype == gi.OUT_BF16 else to_dev_f32(C)
    dD, ldd = empty_out(w.M, w.N, w.out_dtype)
    rc, st = call(w.M, w.N, w.K, dA, w.K, dB, w.K, dC, w.N if C is not None else 0, dD, ldd,
                  w.alpha, w.beta, w.out_dtype, path=path)
    assert rc == 0 and st == 0, g.last_error()
    return A, B, C, from_dev(dD, w.out_dtype)


def _cvals(w, C):
    if C is None:
        return None
    return gi.bf16_bits_to_f32(C) if w.out_dtype == gi.OUT_BF16 else C


def test_workload_square_full():
    w = gi.WORKLOADS[1]
    A, B, C, D = _run_workload(w)
    ref, absdot = oracle.gemm_ref(A, B, C, w.alpha, w.beta)
    ok, worst, where = oracle.check(D, ref, absdot, w.out_dtype, w.beta, _cvals(w, C))
    assert ok, (worst, where)


def test_workload_ragged_full():
    w = gi.WORKLOADS[2]
    A, B, C, D = _run_workload(w)
    ref, absdot = oracle.gemm_ref(A, B, C, w.alpha, w.beta)
    ok, worst, where = oracle.check(D, ref, absdot, w.out_dtype)
    assert ok, (worst, where)


def test_workload_mlp_up_projection_full():
    """8192 x 28672 x 4096, the benchmark's main step: all 235 M outputs
    against the FP64 oracle, a block of rows at a time."""
    w = gi.WORKLOADS[3]
    A, B, C, D = _run_workload(w)
    ok, worst, where = check_every_element(
        D, lambda r0, r1: oracle.gemm_ref(A[r0:r1], B, None, w.alpha, w.beta), w.out_dtype, w.M)
    assert ok, (worst, where)


def test_workload_decode_full():
    w = gi.WORKLOADS[4]
    A, B, C, D = _run_workload(w)
    ref, absdot = oracle.gemm_ref(A, B, C, w.alpha, w.beta)
    ok, worst, where = oracle.check(D, ref, absdot, w.out_dtype)
    assert ok, (worst, where)


@pytest.mark.parametrize("M,N,K", [(16, 8192, 1024), (64, 8192, 2048), (24, 4096, 4096), (7, 520, 1000),
                                    (96, 1024, 2048), (300, 1100, 448), (224, 8192, 2048)])
def test_plan_matches_the_launch(M, N, K):
    """gemm_plan (host only) predicts the path and skinny geometry the call takes."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, plan = g.gemm_plan(M, N, K, 0, sms)
    assert rc == 0
    got, exp = run_int(M, N, K, 0, gi.OUT_BF16, seed=380 + M)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["path"] == plan["path"]
    if plan["path"] == PS:
        assert (info["tile_m"], info["tile_n"], info["grid"], info["stages"]) == \
            (plan["tile_m"], plan["tile_n"], plan["skinny_grid"], plan["skinny_stages"])
    else:
        assert info["tile_m"] == plan["tile_m"]


# ----------------------------------------------------------------------------- tiled k-split

SPLIT_SHAPES = [(129, 257, 1000), (300, 520, 640), (40, 300, 2048), (257, 1100, 96), (7, 9, 17), (128, 256, 512)]


@pytest.mark.parametrize("shape", SPLIT_SHAPES)
@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("parts", [2, 3, 4])
def test_tiled_k_split_exact(shape, path, parts):
    """Tiles split into k-parts: parts > 0 publish fp32 partials, part 0 adds
    them in part order (exact on integers; K = 17 and 96 leave parts of one
    or two k-blocks, K = 17 with 4 parts is capped at its single k-block)."""
    M, N, K = shape
    got, exp = run_int(M, N, K, path, gi.OUT_F32, seed=390 + M + N + K + parts, tiled_k_parts=parts)
    assert_same(got, exp)
    info = g.last_launch_info()
    assert info["k_parts"] == min(parts, -(-K // 64))


@pytest.mark.parametrize("path", [P1, P2])
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_tiled_k_split_with_c(path, out_dtype):
    """beta C on a split tile (part 0's epilogue only)."""
    import torch
    M, N, K = 300, 520, 1024
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 395)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 396)
    Cb = gi.draw_bf16(M, N, gi.Dist("int", -8, 8), 397)
    ref, _ = oracle.gemm_ref(A, B, Cb, 1.0, 0.5)
    Cf = gi.bf16_bits_to_f32(Cb)
    dC = to_dev_bf16(Cb) if out_dtype == gi.OUT_BF16 else to_dev_f32(Cf)
    dD, ldd = empty_out(M, N, out_dtype)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=path, tiled_k_parts=3)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)   # alive until the kernel has run
    rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, dC.data_ptr(), N,
                           dD.data_ptr(), ldd, 1.0, 0.5, out_dtype, s, cfg)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    assert g.last_launch_info()["k_parts"] == 3
    assert_same(from_dev(dD, out_dtype), expect_exact(ref, out_dtype))


def test_tiled_k_split_automatic():
    """Few tiles and a long K split automatically (300 x 1100 x 8192: 15 tiles
    of 128 x 256 on 152 SMs, 128 k-blocks -> 4 parts), deterministically."""
    outs = []
    for _ in range(3):
        got, exp = run_int(300, 1100, 8192, 0, gi.OUT_F32, seed=399)
        assert_same(got, exp)
        outs.append(got.view(np.uint32))
        info = g.last_launch_info()
        assert info["path"] == P1 and info["k_parts"] == 4 and info["grid"] == 60
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_tiled_k_split_normal_inputs_within_bound():
    M, N, K = 224, 2048, 8192
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 400)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 401)
    dD, ldd = empty_out(M, N, gi.OUT_BF16)
    rc, st = call(M, N, K, to_dev_bf16(A), K, to_dev_bf16(B), K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_BF16)
    assert rc == 0 and st == 0, g.last_error()
    info = g.last_launch_info()
    assert info["path"] == P2 and info["k_parts"] == 4
    ref, absdot = oracle.gemm_ref(A, B)
    ok, worst, where = oracle.check(from_dev(dD, gi.OUT_BF16), ref, absdot, gi.OUT_BF16)
    assert ok, (worst, where)


@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_skinny_whole_tiles_beyond_one_wave(out_dtype):
    """More 128-row tiles than SMs (304 at N = 38912): each CTA takes whole
    tiles, no partial sums; exact, and the grid is the one gemm_plan gives."""
    import torch
    M, N, K = 16, 38912, 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rc, plan = g.gemm_plan(M, N, K, 0, sms)
    assert rc == 0
    got, exp = run_int(M, N, K, PS, out_dtype, seed=410)
    assert_same(got, exp)
    assert g.last_launch_info()["grid"] == plan["skinny_grid"]


def test_tiled_split_first_used_inside_graph_capture():
    """A split-eligible shape first called while a fresh stream is captured:
    its workspace cannot grow then, so the call runs unsplit instead of
    failing, and the replayed graph is exact."""
    import torch
    M, N, K = 300, 1104, 8192
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 420)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 421)
    ref, _ = oracle.gemm_ref(A, B)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0, dD.data_ptr(), ldd, 1.0, 0.0,
                               gi.OUT_F32, stream.cuda_stream, None)
    assert rc == 0, g.last_error()
    assert g.last_launch_info()["k_parts"] == 1
    graph.replay()
    torch.cuda.synchronize()
    assert g.gemm_get_status(stream.cuda_stream) == 0
    assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))
    # outside capture the same shape splits
    got, exp = run_int(M, N, K, 0, gi.OUT_F32, seed=422)
    assert_same(got, exp)
    assert g.last_launch_info()["k_parts"] == 4


@pytest.mark.parametrize("M,N,K,parts", [
    (300, 1104, 8192, 4),   # 15 1-SM tiles, 128 k-blocks: four parts of 32
    (192, 4096, 4096, 1),   # plain calls split in four here, fused ones (64 k-blocks) do not
])
def test_fused_epilogue_split_rule(M, N, K, parts):
    """Fused bias + ReLU splits only into four parts of at least 32 k-blocks;
    exact either way (the bias and activation run on the finisher's sums)."""
    import torch
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 430)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 431)
    bias = gi.draw_bf16(N, 1, gi.Dist("int", -50, 50), 432).reshape(N)
    ref, _ = oracle.gemm_ref(A, B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    dA, dB, dbias = to_dev_bf16(A), to_dev_bf16(B), to_dev_bf16(bias)   # alive until the kernel has run
    s = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_bf16_tn_bias_act(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0,
                                 dD.data_ptr(), ldd, 1.0, 0.0, gi.OUT_F32, dbias.data_ptr(), 0, 1, s)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    assert g.last_launch_info()["k_parts"] == parts
    assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(oracle.epilogue(ref, bias, 1)))


def test_fused_gelu_on_split_tiles_within_bound():
    """bias + tanh-GELU on tiles split in four parts (256 x 1024 x 8192: 1-SM
    tiles), real inputs, within the oracle's activation bound, bf16 and fp32
    outputs."""
    import torch
    M, N, K = 256, 1024, 8192
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 440)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 4.0 / K), 441)
    bias = gi.draw_bf16(N, 1, gi.Dist("normal", 1.0), 442).reshape(N)
    ref, absdot = oracle.gemm_ref(A, B)
    z = oracle.epilogue(ref, bias, 0)
    fz = oracle.epilogue(ref, bias, 3)
    dA, dB, dbias = to_dev_bf16(A), to_dev_bf16(B), to_dev_bf16(bias)
    s = torch.cuda.current_stream().cuda_stream
    for out_dtype in (gi.OUT_BF16, gi.OUT_F32):
        dD, ldd = empty_out(M, N, out_dtype)
        rc = g.gemm_bf16_tn_bias_act(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0,
                                     dD.data_ptr(), ldd, 1.0, 0.0, out_dtype, dbias.data_ptr(), 0, 3, s)
        assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
        info = g.last_launch_info()
        assert info["k_parts"] == 4, info
        got = oracle.decode_out(from_dev(dD, out_dtype), out_dtype)
        bnd = oracle.bound_act(z, fz, absdot, out_dtype, 3)
        err = np.abs(got - fz)
        assert np.all(err <= bnd), float(np.max(err / bnd))


@pytest.mark.parametrize("pref", [4, 8])
@pytest.mark.parametrize("shape", [(513, 520, 200), (1024, 2048, 640), (300, 1100, 448)])
def test_preferred_cluster_exact(pref, shape):
    """Pair tiles launched with a preferred cluster of 4 or 8 CTAs (pairs as the
    fallback): each pair addresses its own leader inside the larger cluster."""
    import torch
    M, N, K = shape
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 990 + M)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 991 + N)
    ref, _ = oracle.gemm_ref(A, B)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    for grid in (0, 2 * pref):   # the persistent grid, and one that makes every pair loop over tiles
        cfg = g.GemmConfig(path=P2, cluster_pref=pref, grid=grid)
        rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0, dD.data_ptr(), ldd,
                               1.0, 0.0, gi.OUT_F32, s, cfg)
        assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
        info = g.last_launch_info()
        assert info["path"] == P2 and info["cluster_pref"] in (0, pref)
        assert info["cluster_pref"] == (pref if info["grid"] % pref == 0 else 0)
        assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


# Shapes whose last round of tiles can be cut into slices: (M, N, K, path,
# slices with tail_slices = 0, which slices only grids of less than one
# round).  2-SM: 76 pair slots, 1-SM: 152 CTAs.
SLICE_SHAPES = [
    (2300, 2248, 320, P2, 1),    # 81 pair tiles: 76 whole + 5 in the last round, ragged M and N
    (600, 696, 448, P2, 4),      # 9 pair tiles, less than one round
    (4096, 4096, 256, P2, 1),    # 256 tiles: 28 in the last round
    (1000, 5000, 192, P1, 1),    # 160 1-SM tiles: 8 in the last round
    (130, 296, 72, P1, 4),       # 4 tiles, K not a whole k-block
]


def expected_slices(M, N, path, slices, auto):
    """Slices a launch takes: the automatic count, or a forced one where the
    last round's tiles times it still fit one round of clusters."""
    import torch
    if slices == 0:
        return auto
    clusters = torch.cuda.get_device_properties(0).multi_processor_count // path
    tiles = -(-M // (128 * path)) * -(-N // 256)
    r = tiles % clusters
    return slices if r and r * slices <= clusters else 1


@pytest.mark.parametrize("M,N,K,path,auto", SLICE_SHAPES)
@pytest.mark.parametrize("slices", [0, 2, 4])
def test_tail_slices_exact(M, N, K, path, auto, slices):
    """The last round's tiles computed as 2 or 4 column slices, one cluster
    each (narrower MMAs and B boxes), give the same bits as the oracle, with
    beta * C through the epilogue, fp32 and bf16 outputs."""
    import torch
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 1300 + M % 97)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 1310 + N % 89)
    C = gi.draw_f32(M, N, gi.Dist("int", -4, 4), 1320 + K % 83)
    ref, _ = oracle.gemm_ref(A, B, C, 1.0, 0.5)
    dA, dB, dC = to_dev_bf16(A), to_dev_bf16(B), to_dev_f32(C)
    for out_dtype in (gi.OUT_F32, gi.OUT_BF16):
        dD, ldd = empty_out(M, N, out_dtype)
        dCo = dC if out_dtype == gi.OUT_F32 else to_dev_bf16(gi.f32_to_bf16_bits(C))
        rc, st = call(M, N, K, dA, K, dB, K, dCo, N, dD, ldd, 1.0, 0.5, out_dtype, path=path,
                      tail_slices=slices)
        assert rc == 0 and st == 0, g.last_error()
        info = g.last_launch_info()
        assert info["tail_slices"] == expected_slices(M, N, path, slices, auto), info
        assert_same(from_dev(dD, out_dtype)[:, :N], expect_exact(ref, out_dtype))
    # and switched off
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, dC, N, dD, ldd, 1.0, 0.5, gi.OUT_F32, path=path, tail_slices=1)
    assert rc == 0 and st == 0 and g.last_launch_info()["tail_slices"] == 1, g.last_error()
    assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("hints", [1, 2, 4, 7])
@pytest.mark.parametrize("path", [P1, P2])
def test_l2_hints_exact(hints, path):
    """Cache-hinted loads and stores (evict-last A, evict-first B, evict-first
    D) give the same bits, with beta * C read through the epilogue as well."""
    import torch
    M, N, K = 520, 1100, 448
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 1200 + hints)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 1210 + hints)
    C = gi.draw_f32(M, N, gi.Dist("int", -4, 4), 1220 + hints)
    ref, _ = oracle.gemm_ref(A, B, C, 1.0, 0.5)
    dA, dB, dC = to_dev_bf16(A), to_dev_bf16(B), to_dev_f32(C)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=path, l2_hints=hints)
    rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, dC.data_ptr(), N, dD.data_ptr(), ldd,
                           1.0, 0.5, gi.OUT_F32, s, cfg)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("M,N,K,skinny_grid,kg", [
    (16, 8192, 1024, 0, 0),      # two parts per tile, 4 k-blocks per box
    (16, 2048, 4096, 0, 0),      # four parts
    (16, 1000, 4160, 37, 0),     # stream-K ranges
    (5, 300, 70, 0, 0),          # ragged, K below one k-block (2D maps)
    (48, 4096, 2048, 0, 2),      # 64-row tiles, 2 k-blocks per box
    (96, 8192, 4096, 0, 0),      # wide form
])
def test_skinny_b_static_exact(M, N, K, skinny_grid, kg):
    """B loaded before the dependency wait (gemm_tn_config.b_static): the same
    bits, with the previous call on the stream writing the D this one writes."""
    for rep in range(2):
        got, exp = run_int(M, N, K, PS, gi.OUT_F32, seed=1400 + M + N + K + rep, skinny_grid=skinny_grid,
                           skinny_kgroup=kg, b_static=1)
        assert_same(got, exp)


PAIR_SHAPES = [
    (16, 8192, 1024, 0, 0),     # 32 pair tiles in two parts (equal split)
    (16, 2048, 4096, 0, 0),     # 8 pair tiles in four parts
    (1, 300, 70, 0, 0),         # ragged: one token, K below one k-block (2D maps), last tile partial
    (5, 1000, 4160, 23, 0),     # stream-K ranges over 23 pairs
    (32, 1000, 640, 0, 2),      # 32 tokens (16 per CTA), 2 k-blocks per box
    (48, 520, 1408, 7, 1),      # 48 tokens (24 per CTA), one k-block per box, stream-K
    (64, 4096, 2048, 0, 0),     # 64 tokens (32 per CTA)
    (80, 1100, 1000, 0, 0),     # wide form: 80 tokens (40 per CTA)
    (128, 8192, 2048, 0, 0),    # wide form, 64 tokens per CTA
    (224, 2048, 1024, 11, 0),   # wide form, 112 tokens per CTA, stream-K
    (256, 600, 512, 0, 0),      # wide form, the largest token count
]


@pytest.mark.parametrize("M,N,K,grid,kg", PAIR_SHAPES)
@pytest.mark.parametrize("out_dtype", [gi.OUT_F32, gi.OUT_BF16])
def test_skinny_pair_exact(M, N, K, grid, kg, out_dtype):
    """The pair form of the streaming kernel (gemm_tn_config.skinny_pair = 2):
    clusters of two CTAs on 256-row tiles of B, cta_group::2 MMAs, the tokens
    split between the CTAs; bit-exact on integers, twice in a row."""
    for rep in range(2):
        got, exp = run_int(M, N, K, PS, out_dtype, seed=1500 + M + N + K + rep, skinny_grid=grid, skinny_kgroup=kg,
                           skinny_pair=2)
        info = g.last_launch_info()
        assert info["path"] == PS and info["cluster"] == 2 and info["tile_m"] == 256 and "pair" in info["kernel"]
        assert_same(got, exp)


def test_skinny_pair_with_c_and_b_static():
    """beta * C read in the pair form's epilogue, with the early weight loads."""
    import torch
    M, N, K = 24, 3000, 2048
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 1601)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 1602)
    C = gi.draw_f32(M, N, gi.Dist("int", -4, 4), 1603)
    ref, _ = oracle.gemm_ref(A, B, C, 1.0, 0.5)
    dA, dB, dC = to_dev_bf16(A), to_dev_bf16(B), to_dev_f32(C)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    s = torch.cuda.current_stream().cuda_stream
    cfg = g.GemmConfig(path=PS, skinny_pair=2, b_static=1)
    rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, dC.data_ptr(), N, dD.data_ptr(), ldd,
                           1.0, 0.5, gi.OUT_F32, s, cfg)
    assert rc == 0 and g.gemm_get_status(s) == 0, g.last_error()
    assert_same(from_dev(dD, gi.OUT_F32), oracle.exact_f32(ref))


def test_skinny_pair_decode_normal_within_bound():
    """The 16 x 8192 x 8192 decode's own operands through the pair form, every output."""
    w = gi.WORKLOADS[4]
    A, B, C = gi.operands(w)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(w.M, w.N, w.out_dtype)
    rc, st = call(w.M, w.N, w.K, dA, w.K, dB, w.K, None, 0, dD, ldd, w.alpha, w.beta, w.out_dtype, path=PS,
                  skinny_pair=2)
    assert rc == 0 and st == 0, g.last_error()
    ref, absdot = oracle.gemm_ref(A, B, C, w.alpha, w.beta)
    ok, worst, where = oracle.check(from_dev(dD, w.out_dtype), ref, absdot, w.out_dtype)
    assert ok, (worst, where)
