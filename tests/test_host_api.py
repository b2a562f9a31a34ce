"""Host-side checks that need no GPU: the library builds, loads, exports every
entry point the header declares, and rejects bad arguments before touching a
device."""
import ctypes
import os
import re

import pytest

import tensor_core_dense_tn_gb300 as g
from tensor_core_dense_tn_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_tn.h")


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(g.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version(lib):
    assert g.version() == 100


def test_no_torch_or_oracle_in_product_sources():
    csrc = os.path.join(ROOT, "tensor_core_dense_tn_gb300", "csrc")
    for f in os.listdir(csrc):
        src = open(os.path.join(csrc, f)).read()
        assert "torch" not in src and "oracle" not in src, f
    pkg = open(os.path.join(ROOT, "tensor_core_dense_tn_gb300", "__init__.py")).read()
    assert "import oracle" not in pkg and "from oracle" not in pkg


@pytest.mark.parametrize("kw,code", [
    (dict(out_dtype=2), g.GEMM_ERR_INVALID_VALUE),
    (dict(M=-1), g.GEMM_ERR_INVALID_VALUE),
    (dict(D=0), g.GEMM_ERR_INVALID_VALUE),
    (dict(ldd=8), g.GEMM_ERR_INVALID_VALUE),
    (dict(beta=1.0), g.GEMM_ERR_INVALID_VALUE),         # C is NULL
    (dict(lda=32), g.GEMM_ERR_INVALID_VALUE),           # lda < K
    (dict(A=0x1008), g.GEMM_ERR_MISALIGNED),
    (dict(lda=68), g.GEMM_ERR_MISALIGNED),              # 136 B rows
    (dict(D=0x3004), g.GEMM_ERR_MISALIGNED),
    (dict(ldd=20, N=20), g.GEMM_ERR_MISALIGNED),        # 40 B rows of bf16
    (dict(M=0), g.GEMM_OK),                             # empty: no launch
    (dict(N=0), g.GEMM_OK),
    (dict(M=1 << 31), g.GEMM_ERR_INVALID_VALUE),        # sizes below 2^31
    (dict(K=1 << 31, lda=1 << 31, ldb=1 << 31), g.GEMM_ERR_INVALID_VALUE),
    (dict(B=0), g.GEMM_ERR_INVALID_VALUE),              # K > 0 needs A and B
    (dict(ldb=48), g.GEMM_ERR_INVALID_VALUE),           # ldb < K
    (dict(beta=0.5, C=0x4000, ldc=32), g.GEMM_ERR_INVALID_VALUE),   # ldc < N
    (dict(beta=0.5, C=0x4008, ldc=64), g.GEMM_ERR_MISALIGNED),      # C read: 16-byte base
    (dict(beta=0.5, C=0x4000, ldc=68), g.GEMM_ERR_MISALIGNED),      # C rows of 136 B
    (dict(out_dtype=1, ldd=66), g.GEMM_ERR_MISALIGNED), # fp32 rows of 264 B
    (dict(B=0x2004), g.GEMM_ERR_MISALIGNED),
])
def test_validation_before_any_device_call(lib, kw, code):
    a = dict(M=64, N=64, K=64, A=0x1000, lda=64, B=0x2000, ldb=64, C=0, ldc=0, D=0x3000, ldd=64,
             alpha=1.0, beta=0.0, out_dtype=0, stream=0)
    a.update(kw)
    assert g.gemm_bf16_tn(*a.values()) == code
    if code != g.GEMM_OK:
        assert g.last_error() != ""


def test_forced_unknown_path_rejected(lib):
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(path=9)) == g.GEMM_ERR_INVALID_VALUE


def test_gemm_wrapper_checks_types():
    torch = pytest.importorskip("torch")
    A = torch.zeros((4, 8), dtype=torch.float32)
    with pytest.raises(ValueError):
        g.gemm(A, A)


def test_unknown_scheduler_rejected(lib):
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(scheduler=3)) == g.GEMM_ERR_INVALID_VALUE
    assert "scheduler" in g.last_error()


def _struct_fields(name):
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct " + name + r" \{(.*?)\}", text, flags=re.S).group(1)
    names = []
    for decl in body.split(";"):
        parts = [q for q in decl.split(",") if q.strip()]
        names += [re.findall(r"\w+", q)[-1] for q in parts]
    return names


@pytest.mark.parametrize("name,cls", [("gemm_tn_config", g.GemmConfig), ("gemm_launch_info", g.LaunchInfo),
                                      ("gemm_problem", g.GemmProblem), ("gemm_plan_info", g.GemmPlanInfo)])
def test_ctypes_structs_follow_the_header(name, cls):
    assert _struct_fields(name) == [f for f, _ in cls._fields_]


def _problem(**kw):
    q = dict(M=64, N=64, K=64, A=0x1000, lda=64, B=0x2000, ldb=64, C=0, ldc=0, D=0x3000, ldd=64)
    q.update(kw)
    return q


@pytest.mark.parametrize("problems,out_dtype,code,text", [
    ([_problem()], 2, g.GEMM_ERR_INVALID_VALUE, "out_dtype"),
    ([_problem(), _problem(M=-1)], 0, g.GEMM_ERR_INVALID_VALUE, "problem 1"),
    ([_problem(), _problem(), _problem(A=0x1008)], 0, g.GEMM_ERR_MISALIGNED, "problem 2"),
    ([_problem(ldd=8)], 0, g.GEMM_ERR_INVALID_VALUE, "problem 0"),
    ([_problem(M=0), _problem(N=0)], 0, g.GEMM_OK, ""),
    ([], 0, g.GEMM_OK, ""),
])
def test_grouped_validation_before_any_device_call(lib, problems, out_dtype, code, text):
    assert g.gemm_bf16_tn_grouped(problems, 1.0, 0.0, out_dtype, 0) == code
    assert text in g.last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(batch=-1), g.GEMM_ERR_INVALID_VALUE),
    (dict(batch=0), g.GEMM_OK),
    (dict(stride_a=64 * 64 - 8), g.GEMM_ERR_INVALID_VALUE),     # problems would overlap
    (dict(stride_d=64 * 64 - 8), g.GEMM_ERR_INVALID_VALUE),
    (dict(stride_b=64 * 64 + 4), g.GEMM_ERR_MISALIGNED),        # 8-byte step
    (dict(lda=68), g.GEMM_ERR_MISALIGNED),
    (dict(beta=1.0), g.GEMM_ERR_INVALID_VALUE),                 # C is NULL
])
def test_batched_validation_before_any_device_call(lib, kw, code):
    a = dict(batch=3, M=64, N=64, K=64, A=0x1000, lda=64, stride_a=64 * 64, B=0x2000, ldb=64, stride_b=64 * 64,
             C=0, ldc=0, stride_c=0, D=0x3000, ldd=64, stride_d=64 * 64, alpha=1.0, beta=0.0, out_dtype=0, stream=0)
    a.update(kw)
    assert g.gemm_bf16_tn_batched(*a.values()) == code


@pytest.mark.parametrize("bm", [32, 96, -64, 256])
def test_unknown_skinny_tile_rows_rejected(lib, bm):
    a = (16, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(skinny_bm=bm)) == g.GEMM_ERR_INVALID_VALUE
    assert "skinny_bm" in g.last_error()


@pytest.mark.parametrize("kg", [5, 8, -1])
def test_unknown_skinny_kgroup_rejected(lib, kg):
    a = (16, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(skinny_kgroup=kg)) == g.GEMM_ERR_INVALID_VALUE
    assert "skinny_kgroup" in g.last_error()


@pytest.mark.parametrize("parts", [5, -1])
def test_unknown_tiled_k_parts_rejected(lib, parts):
    a = (300, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(tiled_k_parts=parts)) == g.GEMM_ERR_INVALID_VALUE
    assert "tiled_k_parts" in g.last_error()


@pytest.mark.parametrize("args,code", [
    ((0x1008, 128, 512, 128, 4, 0), g.GEMM_ERR_MISALIGNED),      # src not 16-byte aligned
    ((0, 128, 512, 128, 4, 0), g.GEMM_ERR_MISALIGNED),           # NULL src
    ((0x1000, 128, 512, 96, 4, 0), g.GEMM_ERR_INVALID_VALUE),    # box_rows not 32/64/128/256
    ((0x1000, 128, 512, 128, 3, 0), g.GEMM_ERR_INVALID_VALUE),   # kgroup not 1/2/4
    ((0x1000, 100, 512, 64, 4, 0), g.GEMM_ERR_INVALID_VALUE),    # rows not a multiple of box_rows
    ((0x1000, 128, 640, 128, 4, 0), g.GEMM_ERR_INVALID_VALUE),   # row_bytes not a multiple of 512
    ((0x1000, 128, 512, 128, 4, -1), g.GEMM_ERR_INVALID_VALUE),  # negative grid
    ((0x1000, 256, 1024, 256, 4, 0), g.GEMM_ERR_INVALID_VALUE),  # 128 KiB box: no two-stage ring
])
def test_stream_read_argument_errors(lib, args, code):
    assert g.gemm_stream_read(*args, 0) == code
    assert g.last_error() != ""


@pytest.mark.parametrize("field,value", [("l2_hints", 8), ("l2_hints", -2), ("cluster_pref", 2),
                                         ("cluster_pref", 6), ("cluster_pref", 16)])
def test_unknown_l2_hints_and_cluster_pref_rejected(lib, field, value):
    a = (300, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(**{field: value})) == g.GEMM_ERR_INVALID_VALUE
    assert field in g.last_error()


@pytest.mark.parametrize("value", [-1, 2])
def test_unknown_b_static_rejected(lib, value):
    a = (16, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(b_static=value)) == g.GEMM_ERR_INVALID_VALUE
    assert "b_static" in g.last_error()


@pytest.mark.parametrize("args,code", [
    ((8, 1, 0, 16, 1, 0x1000), g.GEMM_ERR_INVALID_VALUE),      # n below 16
    ((24, 1, 0, 16, 1, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # n not a multiple of 16
    ((272, 1, 0, 16, 1, 0x1000), g.GEMM_ERR_INVALID_VALUE),    # n above 256
    ((16, 3, 0, 16, 3, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # cta_group
    ((16, 2, 0, 16, 3, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # grid not a multiple of the pair
    ((16, 1, 0, 0, 1, 0x1000), g.GEMM_ERR_INVALID_VALUE),      # reps
    ((16, 1, 0, 16, 1, 0x1004), g.GEMM_ERR_MISALIGNED),        # out_ns not 8-byte aligned
])
def test_mma_rate_argument_errors(lib, args, code):
    assert g.gemm_mma_rate(*args, 0) == code
    assert g.last_error() != ""


@pytest.mark.parametrize("kw", [dict(skinny_pair=3), dict(skinny_pair=-1)])
def test_unknown_skinny_pair_rejected(lib, kw):
    a = (16, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0, 0)
    assert g.gemm_bf16_tn_ex(*a, config=g.GemmConfig(**kw)) == g.GEMM_ERR_INVALID_VALUE
    assert "skinny_pair" in g.last_error()


def test_plan_reports_the_pair_form(lib):
    rc, plan = g.gemm_plan(16, 8192, 8192, 0, 152, g.GemmConfig(path=3, skinny_pair=2))
    assert rc == 0
    assert plan["tile_m"] == 256 and plan["skinny_grid"] % 2 == 0
    rc, _ = g.gemm_plan(16, 8192, 8192, 0, 152, g.GemmConfig(path=3, skinny_pair=2, skinny_bm=64))
    assert rc == g.GEMM_ERR_INVALID_VALUE


def test_fp8_bias_act_rejects_before_any_device_call(lib):
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64)
    tail = (1.0, 1.0, 0, 0, 0x3000, 64, 1.0, 0.0, 0)
    assert g.gemm_fp8_tn_bias_act(*a, 2, *tail, 0x4000, 0, 1, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_fp8_tn_bias_act(*a, 0, *tail, 0x4000, 0, 9, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_fp8_tn_bias_act(*a, 0, *tail, 0x4002, 1, 1, 0) == g.GEMM_ERR_MISALIGNED


_BASE = (64, 64, 64, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 64, 1.0, 0.0, 0)


@pytest.mark.parametrize("bias,bias_dtype,act,code", [
    (0x4000, 0, 7, g.GEMM_ERR_INVALID_VALUE),     # unknown activation
    (0x4000, 0, -1, g.GEMM_ERR_INVALID_VALUE),
    (0x4000, 5, 1, g.GEMM_ERR_INVALID_VALUE),     # unknown bias dtype
    (0x4002, 1, 1, g.GEMM_ERR_MISALIGNED),        # fp32 bias on a 2-byte boundary
    (0x4001, 0, 1, g.GEMM_ERR_MISALIGNED),        # bf16 bias on an odd address
])
def test_bias_act_validation_before_any_device_call(lib, bias, bias_dtype, act, code):
    assert g.gemm_bf16_tn_bias_act(*_BASE, bias, bias_dtype, act, 0) == code
    assert g.last_error() != ""


@pytest.mark.parametrize("kw,code", [
    (dict(fp8_format=2), g.GEMM_ERR_INVALID_VALUE),
    (dict(fp8_format=-1), g.GEMM_ERR_INVALID_VALUE),
    (dict(lda=72), g.GEMM_ERR_MISALIGNED),          # one-byte rows must be multiples of 16 elements
    (dict(ldb=88), g.GEMM_ERR_MISALIGNED),
    (dict(lda=32), g.GEMM_ERR_INVALID_VALUE),       # lda < K
    (dict(A=0x1008), g.GEMM_ERR_MISALIGNED),
    (dict(out_dtype=3), g.GEMM_ERR_INVALID_VALUE),
])
def test_fp8_validation_before_any_device_call(lib, kw, code):
    a = dict(M=64, N=64, K=64, A=0x1000, lda=64, B=0x2000, ldb=64, fp8_format=0, scale_a=1.0, scale_b=1.0,
             C=0, ldc=0, D=0x3000, ldd=64, alpha=1.0, beta=0.0, out_dtype=0, stream=0)
    a.update(kw)
    assert g.gemm_fp8_tn(*a.values()) == code
    assert g.last_error() != ""


def test_fp8_bias_act_validation_before_any_device_call(lib):
    a = (64, 64, 64, 0x1000, 64, 0x2000, 64, 0, 1.0, 1.0, 0, 0, 0x3000, 64, 1.0, 0.0, 0)
    assert g.gemm_fp8_tn_bias_act(*a, 0x4000, 0, 9, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_fp8_tn_bias_act(*a, 0x4000, 2, 1, 0) == g.GEMM_ERR_INVALID_VALUE
    assert g.gemm_fp8_tn_bias_act(*a, 0x4002, 1, 1, 0) == g.GEMM_ERR_MISALIGNED
    b = list(a)
    b[7] = 3                                        # fp8_format
    assert g.gemm_fp8_tn_bias_act(*b, 0, 0, 0, 0) == g.GEMM_ERR_INVALID_VALUE


@pytest.mark.parametrize("kw,code", [
    (dict(M=65), g.GEMM_ERR_INVALID_VALUE),          # 1 <= M <= 64
    (dict(M=0), g.GEMM_ERR_INVALID_VALUE),
    (dict(N=131072 + 16, ldd=131072 + 16), g.GEMM_ERR_INVALID_VALUE),   # fixed scratch: N <= 131072
    (dict(K=0), g.GEMM_ERR_INVALID_VALUE),
    (dict(out_dtype=2), g.GEMM_ERR_INVALID_VALUE),
    (dict(B=0), g.GEMM_ERR_INVALID_VALUE),
    (dict(beta=1.0), g.GEMM_ERR_INVALID_VALUE),        # C is NULL
    (dict(ldd=32), g.GEMM_ERR_INVALID_VALUE),
    (dict(lda=68), g.GEMM_ERR_MISALIGNED),
    (dict(D=0x3008), g.GEMM_ERR_MISALIGNED),
])
def test_noalloc_validation_before_any_device_call(lib, kw, code):
    a = dict(M=16, N=64, K=64, A=0x1000, lda=64, B=0x2000, ldb=64, C=0, ldc=0, D=0x3000, ldd=64,
             alpha=1.0, beta=0.0, out_dtype=0, stream=0)
    a.update(kw)
    assert g.gemm_bf16_tn_skinny_noalloc(*a.values()) == code
    assert g.last_error() != ""


@pytest.mark.parametrize("args,code", [
    ((64, 3, 0, 16, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # cta_group not 1 or 2
    ((8, 1, 0, 16, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),      # n below 16
    ((72, 1, 0, 16, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # n not a multiple of 16
    ((272, 1, 0, 16, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),    # n above 256
    ((64, 1, 0, 0, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),      # reps below 1
    ((64, 1, 0, (1 << 24) + 1, 2, 0x1000), g.GEMM_ERR_INVALID_VALUE),
    ((64, 2, 0, 16, 3, 0x1000), g.GEMM_ERR_INVALID_VALUE),     # grid not a multiple of the pair
    ((64, 1, 0, 16, 1025, 0x1000), g.GEMM_ERR_INVALID_VALUE),
    ((64, 1, 0, 16, 2, 0), g.GEMM_ERR_MISALIGNED),             # NULL output
    ((64, 1, 0, 16, 2, 0x1004), g.GEMM_ERR_MISALIGNED),        # output not 8-byte aligned
])
def test_mma_rate_argument_errors(lib, args, code):
    n, cg, fp8, reps, grid, out = args
    assert g.gemm_mma_rate(n, cg, fp8, reps, grid, out, 0) == code
    assert g.last_error() != ""
