"""Seeded synthetic inputs for the BF16 TN GEMM workloads.

This module only draws random numbers and stores them as bf16 bit patterns
(or, for the FP8 variant, as e4m3/e5m2 codes).
It holds none of the GEMM's arithmetic, so both the CPU oracle's tests and the
GPU path's tests/bench can take their operands from it without sharing any of
the computation.

Generator: numpy's PCG64 (O'Neill 2014), seeded per tensor with
``seed = 0x5EED0000 + 16 * workload_index + tensor_id`` (tensor_id 0 = A,
1 = B, 2 = C).  Normals are drawn in float32 (numpy's ziggurat), scaled, and
rounded to bf16 with round-to-nearest-even on the float32 bit pattern.

Distributions follow the five workloads: ``N(0, v)`` is read as a normal with
variance ``v`` (standard deviation sqrt(v)); ``int[-4,4]`` is the inclusive
integer range (9 values); ``uniform(-1,1)`` is continuous.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

SEED_BASE = 0x5EED0000
TENSOR_A, TENSOR_B, TENSOR_C = 0, 1, 2

OUT_BF16 = 0
OUT_F32 = 1

_CHUNK = 1 << 22  # elements converted per pass (bounds temporary memory)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).reshape(-1)
    out = np.empty(u.shape, dtype=np.uint16)
    for s in range(0, u.size, _CHUNK):
        v = u[s:s + _CHUNK].astype(np.uint64)
        v = (v + 0x7FFF + ((v >> 16) & 1)) >> 16
        out[s:s + _CHUNK] = v.astype(np.uint16)
    return out.reshape(x.shape)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


FP8_E4M3 = 0
FP8_E5M2 = 1


def _fp8_positive_table(fmt: int):
    """(codes, values) of the non-negative finite fp8 codes, ascending."""
    codes = np.arange(0x80, dtype=np.int64)
    if fmt == FP8_E4M3:          # 4 exponent bits (bias 7), 3 mantissa bits, 0x7F = NaN
        e, m = codes >> 3, codes & 7
        vals = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7))
        keep = codes != 0x7F
    else:                        # 5 exponent bits (bias 15), 2 mantissa bits, e = 31 inf/NaN
        e, m = codes >> 2, codes & 3
        vals = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1 + m / 4.0) * 2.0 ** (e - 15))
        keep = e != 31
    return codes[keep], vals[keep]


def f32_to_fp8_bits(x: np.ndarray, fmt: int) -> np.ndarray:
    """Round float32 values to fp8 codes: nearest value, ties to the even code,
    saturating at the largest finite value (448 e4m3, 57344 e5m2).

    Normal results round the float32 bit pattern's mantissa to 3 (e4m3) or 2
    (e5m2) bits, the carry moving into the exponent; results below the smallest
    normal (2^-6 e4m3, 2^-14 e5m2) are whole multiples of the subnormal step,
    rounded with numpy's half-to-even rint."""
    mbits, bias, max_code = (3, 7, 0x7E) if fmt == FP8_E4M3 else (2, 15, 0x7B)
    shift = 23 - mbits
    min_normal = np.float32(2.0 ** (1 - bias))
    sub_scale = np.float32(2.0 ** (bias - 1 + mbits))   # 1 / subnormal step
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for s in range(0, flat.size, _CHUNK):
        v = flat[s:s + _CHUNK]
        u = v.view(np.uint32)
        sign = ((u >> 31) << 7).astype(np.uint8)
        a = (u & 0x7FFFFFFF).astype(np.int64)
        r = (a + ((1 << (shift - 1)) - 1) + ((a >> shift) & 1)) >> shift
        code = r - ((127 - bias) << mbits)
        av = np.abs(v)
        sub = av < min_normal
        code = np.where(sub, np.rint(np.where(sub, av, 0) * sub_scale).astype(np.int64), code)
        code = np.minimum(code, max_code)
        out[s:s + _CHUNK] = np.where(code == 0, 0, code.astype(np.uint8) | sign)
    return out.reshape(x.shape)


def fp8_bits_to_f64(b: np.ndarray, fmt: int) -> np.ndarray:
    """Decode finite fp8 codes to float64 (exact)."""
    codes, vals = _fp8_positive_table(fmt)
    lut = np.full(256, np.nan)
    lut[codes] = vals
    lut[codes | 0x80] = -vals
    return lut[np.asarray(b, dtype=np.uint8)]


def draw_fp8(rows: int, cols: int, dist: "Dist", seed: int, fmt: int, ld: Optional[int] = None) -> np.ndarray:
    """A rows x ld array of fp8 codes drawn from dist in float32, then rounded
    to the format (padding filled with 0x7F, a NaN in e4m3 and e5m2)."""
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    rng = np.random.Generator(np.random.PCG64(seed))
    n = rows * cols
    if dist.kind == "int":
        vals = rng.integers(int(dist.a), int(dist.b) + 1, size=n, dtype=np.int64).astype(np.float32)
    elif dist.kind == "normal":
        vals = rng.standard_normal(size=n, dtype=np.float32)
        if dist.a != 1.0:
            vals *= np.float32(math.sqrt(dist.a))
    elif dist.kind == "uniform":
        vals = rng.uniform(dist.a, dist.b, size=n).astype(np.float32)
    else:
        raise ValueError(dist.kind)
    bits = f32_to_fp8_bits(vals, fmt).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7F, dtype=np.uint8)
    out[:, :cols] = bits
    return out


@dataclasses.dataclass(frozen=True)
class Dist:
    kind: str            # "int", "normal", "uniform"
    a: float = 0.0       # int: lo / normal: variance / uniform: lo
    b: float = 0.0       # int: hi (inclusive) / uniform: hi

    def describe(self) -> str:
        if self.kind == "int":
            return f"int[{int(self.a)},{int(self.b)}]"
        if self.kind == "normal":
            return f"N(0,{self.a:g})"
        return f"uniform({self.a:g},{self.b:g})"


def draw_bf16(rows: int, cols: int, dist: Dist, seed: int, ld: Optional[int] = None) -> np.ndarray:
    """A rows x ld array of bf16 bits; columns >= cols (row padding) are NaN-patterned.

    Padding is filled with 0x7FC1 (a quiet NaN) so that any read of it shows up.
    """
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    rng = np.random.Generator(np.random.PCG64(seed))
    n = rows * cols
    if dist.kind == "int":
        vals = rng.integers(int(dist.a), int(dist.b) + 1, size=n, dtype=np.int64).astype(np.float32)
    elif dist.kind == "normal":
        vals = rng.standard_normal(size=n, dtype=np.float32)
        std = math.sqrt(dist.a)
        if std != 1.0:
            vals *= np.float32(std)
    elif dist.kind == "uniform":
        vals = rng.uniform(dist.a, dist.b, size=n).astype(np.float32)
    else:
        raise ValueError(dist.kind)
    bits = f32_to_bf16_bits(vals).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7FC1, dtype=np.uint16)
    out[:, :cols] = bits
    return out


def draw_f32(rows: int, cols: int, dist: Dist, seed: int) -> np.ndarray:
    """float32 values (bf16-representable) for an FP32 C operand."""
    return bf16_bits_to_f32(draw_bf16(rows, cols, dist, seed))


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    M: int
    N: int
    K: int
    dist_a: Dist
    dist_b: Dist
    dist_c: Optional[Dist]
    alpha: float
    beta: float
    out_dtype: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def seed(self, tensor_id: int) -> int:
        return SEED_BASE + 16 * self.index + tensor_id

    def describe(self) -> dict:
        return {
            "workload": self.name, "M": self.M, "N": self.N, "K": self.K,
            "A": self.dist_a.describe(), "B": self.dist_b.describe(),
            "C": self.dist_c.describe() if self.dist_c else None,
            "alpha": self.alpha, "beta": self.beta,
            "out": "bf16" if self.out_dtype == OUT_BF16 else "f32",
            "seeds": [self.seed(i) for i in range(3)],
        }


WORKLOADS = [
    Workload(0, "tiny exact 256^3 int", 256, 256, 256,
             Dist("int", -4, 4), Dist("int", -4, 4), None, 1.0, 0.0, OUT_F32),
    Workload(1, "square 4096^3 beta=0.5", 4096, 4096, 4096,
             Dist("normal", 1.0), Dist("normal", 1.0), Dist("normal", 1.0), 1.0, 0.5, OUT_BF16),
    Workload(2, "ragged 3000x5000x2000", 3000, 5000, 2000,
             Dist("uniform", -1, 1), Dist("uniform", -1, 1), None, 1.0, 0.0, OUT_BF16),
    Workload(3, "MLP up-projection 8192x28672x4096", 8192, 28672, 4096,
             Dist("normal", 1.0), Dist("normal", 1.0 / 4096), None, 1.0, 0.0, OUT_BF16),
    Workload(4, "decode skinny 16x8192x8192", 16, 8192, 8192,
             Dist("normal", 1.0), Dist("normal", 1.0 / 8192), None, 1.0, 0.0, OUT_BF16),
]


def operands(w: Workload):
    """(A bits MxK, B bits NxK, C or None) for a workload; C dtype follows out_dtype."""
    A = draw_bf16(w.M, w.K, w.dist_a, w.seed(TENSOR_A))
    B = draw_bf16(w.N, w.K, w.dist_b, w.seed(TENSOR_B))
    C = None
    if w.dist_c is not None:
        if w.out_dtype == OUT_BF16:
            C = draw_bf16(w.M, w.N, w.dist_c, w.seed(TENSOR_C))
        else:
            C = draw_f32(w.M, w.N, w.dist_c, w.seed(TENSOR_C))
    return A, B, C


TENSOR_A_FP8, TENSOR_B_FP8 = 3, 4


def fp8_operands(w: Workload, fmt: int = FP8_E4M3):
    """(A codes MxK, B codes NxK, scale_a, scale_b) for workload w in fp8.

    Per-tensor scaling: an operand drawn from N(0, v) is stored as codes of
    N(0, 1) values with scale sqrt(v), so that scale * code has the
    workload's distribution while the codes use the format's normal range;
    integer and uniform operands are stored as they are with scale 1."""
    out = []
    for dist, tid, rows in ((w.dist_a, TENSOR_A_FP8, w.M), (w.dist_b, TENSOR_B_FP8, w.N)):
        if dist.kind == "normal":
            out.append((draw_fp8(rows, w.K, Dist("normal", 1.0), w.seed(tid), fmt), math.sqrt(dist.a)))
        else:
            out.append((draw_fp8(rows, w.K, dist, w.seed(tid), fmt), 1.0))
    (A, sa), (B, sb) = out
    return A, B, sa, sb
