"""Host-only planning (gemm_plan): the automatic path and skinny geometry for
shapes whose best choice was measured on GB300 (152 SMs), without a GPU.

Each expected value is the choice the shape sweeps found fastest (or within
a few percent of it); the comments give the measured times."""
import pytest

import tensor_core_dense_tn_gb300 as g
from tensor_core_dense_tn_gb300 import build as gbuild

P1, P2, S = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    gbuild.build()
    return g.load()


def plan(M, N, K, fp8=0, sms=152, **cfg):
    rc, info = g.gemm_plan(M, N, K, fp8, sms, g.GemmConfig(**cfg) if cfg else None)
    assert rc == 0, g.last_error()
    return info


@pytest.mark.parametrize("M,N,K,fp8,path", [
    (16, 8192, 8192, 0, S),      # decode: skinny 25.6 us
    (16, 8192, 8192, 1, S),
    (1, 256, 256, 0, S),         # skinny 3.9 us against 5.9 (1-SM)
    (32, 1024, 1024, 0, P1),     # short rows, small B: sliced 1-SM 7.4 us; skinny 10.9
    (16, 4096, 1024, 0, P1),     # 7.6 us; skinny 8.9
    (16, 8192, 1024, 0, S),
    (64, 8192, 8192, 0, S),      # 64-row whole tiles 31.4 us; 2-SM 43.1
    (64, 4096, 4096, 0, P2),     # tiles in 4 k-parts about 21 us; skinny 22.3
    (64, 1024, 4096, 0, P1),     # 1-SM in 4 k-parts 17.6 us; skinny 22.6
    (64, 1024, 8192, 0, P1),     # 1-SM in 4 k-parts 22.8 us; skinny 26.3
    (64, 4096, 8192, 0, P2),     # pair tiles in 4 k-parts 27.1 us; skinny 28.9
    (64, 16384, 4096, 0, S),     # skinny 27.1 us
    (64, 1024, 2048, 0, P1),     # K short: 1-SM 13.4 us
    (64, 4096, 1024, 0, P1),     # 8 MiB B: 1-SM 9.3 us; skinny 13.1
    (64, 28672, 4096, 0, P1),    # stream-K skinny 49.9 us; 1-SM 44.5
    (96, 1024, 2048, 0, P1),     # 1-SM 13.5 us; skinny 49.7
    (96, 8192, 2048, 0, S),      # 32 MiB: skinny 14.7 us; 2-SM 15.5
    (96, 8192, 4096, 1, S),      # fp8, 32 MiB
    (96, 8192, 2048, 1, P1),     # fp8, 16 MiB stays in L2
    (96, 16384, 8192, 0, P2),    # N > 8192: 2-SM 53.0 us, skinny 53.0
    (128, 16384, 2048, 0, P1),   # sliced 1-SM 17.4 us; 2-SM 18.4; skinny 19.9
    (128, 16384, 4096, 0, P2),   # 2-SM 30.5 us
    (128, 4096, 4096, 0, P2),    # 2-SM 23.7 us; skinny 29.5
    (128, 4096, 8192, 0, P2),    # pair tiles in 4 k-parts 27.5 us; skinny 37.5
    (128, 8192, 2048, 0, P1),    # 1-SM 14.6 us; skinny 16.0
    (128, 8192, 8192, 0, S),     # skinny 38.5 us; 2-SM 43.6; 1-SM 56.6
    (96, 28672, 8192, 0, P1),    # 1-SM 83.1 us; skinny 90.6
    (160, 8192, 8192, 0, P2),    # 2-SM 43.8 us; skinny 46.9
    (224, 8192, 8192, 0, P2),    # 2-SM 44.0 us; 1-SM 56.6
    (256, 4096, 4096, 0, P2),    # 2-SM 23.7 us; 1-SM 29.9
    (256, 4096, 2048, 0, P1),    # B in L2: 1-SM 13.9 us; 2-SM 14.5
    (256, 256, 256, 0, P1),      # 6.0 us against 6.6
    (384, 8192, 2048, 0, P2),    # 16.5 us against 18.3
    (3000, 5000, 2000, 0, P2),
    (4096, 4096, 4096, 0, P2),
    (8192, 28672, 4096, 0, P2),  # the up-projection
    (8192, 28672, 4096, 1, P2),
    (300, 264, 0, 0, P1),        # K = 0: D = beta C on the 1-SM kernel
])
def test_automatic_path(M, N, K, fp8, path):
    assert plan(M, N, K, fp8)["path"] == path


@pytest.mark.parametrize("M,N,K,fp8,geometry", [
    # tile rows, k-group, stages, grid, parts, skew (k-groups)
    (16, 8192, 8192, 0, (128, 4, 3, 128, 2, 2)),
    (16, 8192, 8192, 1, (128, 4, 3, 128, 2, 2)),
    (1, 8192, 8192, 0, (128, 4, 3, 128, 2, 2)),
    (32, 8192, 8192, 0, (128, 2, 5, 128, 2, 4)),  # 4 k-blocks would leave 2 stages; skew 8 k-blocks
    (64, 8192, 8192, 0, (64, 4, 3, 128, 1, 0)),
    (24, 4096, 4096, 0, (64, 4, 4, 128, 2, 2)),   # 64 rows: two parts instead of four
    (8, 4096, 8192, 0, (128, 4, 3, 128, 4, 2)),
    (128, 8192, 8192, 0, (64, 2, 4, 128, 1, 0)),  # wide form
    (16, 8192, 1000, 0, (128, 1, 12, 128, 2, 7)), # K not a whole number of k-blocks: 2D maps; skew capped
    (16, 2048, 8192, 0, (128, 4, 3, 64, 4, 2)),   # at most 4 parts: 15.2 us against 16.8 with 9
    (16, 1024, 8192, 1, (128, 4, 3, 32, 4, 2)),   # e4m3: 11.1 us against 15.5 with 16
])
def test_skinny_geometry(M, N, K, fp8, geometry):
    p = plan(M, N, K, fp8)
    assert p["path"] == S
    got = (p["tile_m"], p["skinny_kgroup"], p["skinny_stages"], p["skinny_grid"], p["k_parts"],
           p["skinny_skew"])
    assert got == geometry
    assert p["tile_n"] == -(-M // 16) * 16


@pytest.mark.parametrize("N,K,fp8,grid", [
    (32768, 8192, 0, 128),    # 256 tiles: 2 whole tiles per CTA (83.2 against 86.1 us stream-K)
    (28672, 8192, 1, 112),    # 224 tiles: 2 per CTA
    (57344, 4096, 1, 112),    # 448 tiles: 4 per CTA
    (131072, 4096, 0, 128),   # 1024 tiles: 8 per CTA
    (20480, 8192, 0, 152),    # 160 tiles: 80 CTAs would idle too many SMs: stream-K
])
def test_skinny_whole_tiles_when_tiles_exceed_sms(N, K, fp8, grid):
    p = plan(16, N, K, fp8)
    assert (p["path"], p["tile_m"], p["skinny_grid"], p["k_parts"]) == (S, 128, grid, 0)


def test_skinny_partition_follows_the_sm_count():
    # 148 SMs: 64 tiles x 2 parts still keep >= 80% of the SMs busy
    assert plan(16, 8192, 8192, sms=148)["skinny_grid"] == 128
    # 100 SMs: 64 tiles x 1 part leave 36% idle: stream-K over all 100
    p = plan(16, 8192, 8192, sms=100)
    assert p["skinny_grid"] == 100 and p["k_parts"] == 0


def test_overrides_reach_the_plan():
    p = plan(16, 8192, 8192, path=S, skinny_bm=64, skinny_kgroup=2, skinny_skew_kb=-1)
    assert (p["tile_m"], p["skinny_kgroup"], p["k_parts"], p["skinny_skew"]) == (64, 2, 1, 0)
    p = plan(16, 8192, 8192, path=S, skinny_grid=37)
    assert p["skinny_grid"] == 37 and p["k_parts"] == 0
    assert plan(16, 8192, 8192, path=P2)["tile_m"] == 256
    assert plan(8192, 8192, 8192, path=P1)["tile_m"] == 128


def test_tiled_tile_shape():
    p = plan(8192, 28672, 4096)
    assert (p["tile_m"], p["tile_n"], p["skinny_grid"], p["k_parts"]) == (256, 256, 0, 1)


@pytest.mark.parametrize("M,N,K,path,parts", [
    (256, 2048, 8192, P2, 4),     # 24.6 us; 2 parts 31.7, none 40.0
    (224, 8192, 8192, P2, 2),     # 32 pair tiles: 38.4 against 41.8 (4 parts would not fit)
    (300, 1100, 8192, P1, 4),
    (192, 4096, 4096, P2, 4),     # 64 k-blocks: 21.2 against 22.7
    (512, 4096, 4096, P2, 1),     # 32 tiles, 64 k-blocks: 2 parts 23.8 against 23.5
    (256, 2048, 2048, P1, 1),     # 32 k-blocks: 4 parts 17.6 against 13.3
    (1024, 2048, 2048, P1, 1),
    (96, 28672, 8192, P1, 1),     # 112 tiles: more than half of the SMs
])
def test_tiled_k_split_choice(M, N, K, path, parts):
    p = plan(M, N, K)
    assert (p["path"], p["k_parts"]) == (path, parts)
    # forced parts are capped at K's k-blocks
    assert plan(M, N, 128, path=path, tiled_k_parts=4)["k_parts"] == 2


@pytest.mark.parametrize("M,N,K,path,slices", [
    (256, 256, 256, P1, 4),        # two 128 x 256 tiles: 6.1 -> 3.8 us
    (512, 3072, 4096, P1, 2),      # 48 1-SM tiles: 96 halves fit one round (32.1 -> 26.4 us)
    (600, 696, 448, P1, 4),        # 15 1-SM tiles: 60 quarters
    (2048, 2048, 2048, P2, 1),     # 64 tiles: less than one round, but 128 halves would not fit it
    (4096, 4096, 4096, P2, 1),     # 256 tiles: several rounds, no automatic slices
    (3000, 5000, 2000, P2, 1),
    (8192, 28672, 4096, P2, 1),
    (256, 2048, 8192, P2, 1),      # k-split instead
])
def test_tail_slices_choice(M, N, K, path, slices):
    p = plan(M, N, K)
    assert (p["path"], p["tail_slices"]) == (path, slices)
    assert p["tail_slices"] == 1 or p["k_parts"] == 1
    assert plan(M, N, K, tail_slices=1)["tail_slices"] == 1
    # a forced count applies, at any number of rounds, where the round's tiles
    # times it still fit one round
    if path == P2 and p["k_parts"] == 1:
        r = (((M + 255) // 256) * ((N + 255) // 256)) % 76
        for want in (2, 4):
            got = plan(M, N, K, tail_slices=want)["tail_slices"]
            assert got == (want if r and r * want <= 76 else 1)
    # with the cluster-launch-control scheduler or a grid override there are none
    assert plan(M, N, K, scheduler=2)["tail_slices"] == 1
    assert plan(M, N, K, grid=64)["tail_slices"] == 1


@pytest.mark.parametrize("args,cfg,code,text", [
    ((257, 64, 64), dict(path=3), g.GEMM_ERR_NOT_IMPLEMENTED, "skinny"),
    ((16, 64, 0), dict(path=3), g.GEMM_ERR_NOT_IMPLEMENTED, "skinny"),
    ((144, 256, 1024), dict(path=3, skinny_bm=128, skinny_kgroup=4), g.GEMM_ERR_INVALID_VALUE, "ring stages"),
    ((-1, 64, 64), {}, g.GEMM_ERR_INVALID_VALUE, "negative"),
    ((16, 64, 64), dict(skinny_kgroup=5), g.GEMM_ERR_INVALID_VALUE, "skinny_kgroup"),
    ((16, 64, 64), dict(path=9), g.GEMM_ERR_INVALID_VALUE, "path"),
    ((512, 512, 64), dict(tail_slices=3), g.GEMM_ERR_INVALID_VALUE, "tail_slices"),
])
def test_plan_errors(args, cfg, code, text):
    rc, _ = g.gemm_plan(*args, 0, 152, g.GemmConfig(**cfg) if cfg else None)
    assert rc == code and text in g.last_error()


def test_plan_argument_errors():
    assert g.gemm_plan(16, 64, 64, 0, 0)[0] == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_plan(16, 64, 64, 2, 152)[0] == g.GEMM_ERR_INVALID_VALUE
    rc, info = g.gemm_plan(0, 64, 64)
    assert rc == 0 and info["path"] == 0


# The automatic path as the header (gemm_path) states it, restated here so
# that the documentation and the code cannot drift apart.
def _split_parts(tiles, sms):
    if tiles < 1 or tiles > sms:
        return 0
    s = sms // tiles
    if s >= 4:
        return 4
    return s if 5 * tiles * s >= 4 * sms else 0


def _equal_parts(N, np_, sms):
    s64 = _split_parts(-(-N // 64), sms)
    s128 = _split_parts(-(-N // 128), sms)
    bm = 64 if (s64 >= 1 and np_ >= 48) or (s64 >= 1 and np_ >= 32 and s128 >= 4) else 128
    return _split_parts(-(-N // bm), sms)


def _documented_path(M, N, K, fp8, sms=152):
    if K == 0:
        return P1
    kb = -(-K // (128 if fp8 else 64))
    large = N * K * (1 if fp8 else 2) >= 32 << 20
    parts = _equal_parts(N, -(-M // 16) * 16, sms) if M <= 256 else 0
    tiles = -(-M // 128) * -(-N // 256)
    if M <= 32:
        return P1 if kb <= 16 and 1024 <= N <= 4096 else S
    if M <= 64 and parts >= 1 and ((large and parts <= 2 and not (N <= 4096 and kb >= 64)) or
                                   (kb >= 64 and N > 4096)):
        return S
    if 64 < M <= 128 and large and 1 <= parts <= 2 and 4096 < N <= 8192 and (kb >= 64 or (M <= 96 and kb >= 32)):
        return S
    if M > 128 and (large or tiles > 64):
        return P2
    if M <= 128 and large and 2 * tiles <= sms and kb > 32:
        return P2
    return P1


def test_automatic_path_follows_the_documented_rule():
    bad = []
    for fp8 in (0, 1):
        for M in (1, 16, 31, 32, 33, 48, 64, 65, 80, 96, 97, 112, 128, 129, 192, 256, 257, 1024):
            for N in (256, 1024, 2048, 4096, 4352, 6144, 8192, 8448, 16384, 28672):
                for K in (0, 256, 1000, 1024, 2048, 2056, 4096, 8192):
                    got = plan(M, N, K, fp8)["path"]
                    want = _documented_path(M, N, K, fp8)
                    if got != want:
                        bad.append((M, N, K, fp8, got, want))
    assert not bad, bad[:10]


def test_tiled_split_and_slices_follow_the_documented_rules():
    """gemm_tn_config.tiled_k_parts and .tail_slices at 0 (automatic), as the
    header states them: four k-parts when four per tile fit one round of
    clusters and K holds at least 64 k-blocks, else two when two fit and K
    holds at least 128, else none; without a split, tiles that fill less than
    one round are cut into the most slices (4, then 2) that still fit it."""
    bad = []
    for fp8 in (0, 1):
        for M in (129, 256, 300, 512, 1024, 2048, 4096):
            for N in (256, 1024, 2048, 4096, 8192, 28672):
                for K in (64, 1024, 4096, 8192, 16384):
                    p = plan(M, N, K, fp8)
                    if p["path"] not in (P1, P2):
                        continue
                    cg = p["path"]
                    clusters = 152 // cg
                    tiles = -(-M // (128 * cg)) * -(-N // 256)
                    kb = -(-K // (128 if fp8 else 64))
                    parts = 4 if 4 * tiles <= clusters and kb >= 64 else (
                        2 if 2 * tiles <= clusters and kb >= 128 else 1)
                    slices = 1
                    if parts == 1 and tiles < clusters:
                        slices = 4 if 4 * tiles <= clusters else (2 if 2 * tiles <= clusters else 1)
                    if (p["k_parts"], p["tail_slices"]) != (parts, slices):
                        bad.append((M, N, K, fp8, cg, p["k_parts"], p["tail_slices"], parts, slices))
    assert not bad, bad[:10]


def test_skinny_tile_rows_and_kgroup_follow_the_documented_rules():
    """gemm_tn_config.skinny_bm and .skinny_kgroup at 0, as the header states
    them: 64-row tiles where they fit one wave and M > 32 (or M > 16 with
    128-row tiles split into 4 or more parts); k-groups of 4, 2 or 1 k-blocks
    that leave at least 3 ring stages and do not exceed K's k-blocks, 1 for a
    partial last k-block and for 128-row tiles of more than 64 tokens."""
    bad = []
    for fp8 in (0, 1):
        kbe = 128 if fp8 else 64
        for M in (1, 16, 17, 32, 33, 48, 64, 65, 96, 128, 160, 256):
            for N in (1024, 2048, 4096, 8192, 16384, 28672):
                for K in (64, 128, 256, 1000, 4096, 8192):
                    p = plan(M, N, K, fp8, path=S)
                    np_ = -(-M // 16) * 16
                    s64 = _split_parts(-(-N // 64), 152)
                    s128 = _split_parts(-(-N // 128), 152)
                    bm = 64 if (s64 >= 1 and np_ >= 48) or (s64 >= 1 and np_ >= 32 and s128 >= 4) else 128
                    kg, kb = p["skinny_kgroup"], -(-K // kbe)
                    ok = p["tile_m"] == bm and kg in (1, 2, 4) and kg <= max(1, kb) and p["skinny_stages"] >= 2
                    if K % kbe or (np_ > 64 and bm == 128):
                        ok = ok and kg == 1
                    elif kg > 1:
                        ok = ok and p["skinny_stages"] >= 3
                    if not ok:
                        bad.append((M, N, K, fp8, p["tile_m"], kg, p["skinny_stages"], bm))
    assert not bad, bad[:10]
