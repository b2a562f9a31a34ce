"""Roofline arithmetic used by the benchmark (host-side, no GPU).

Algorithmic work and traffic of one GEMM launch, as the H100 Nsight Compute
page defines them (section 7, "connecting reuse, capacity and throughput
with GEMM"): F = 2MNK useful FLOPs, and the ideal HBM traffic when each
operand is read once and the output written once, Q = 2(MK + KN) + e*MN
(+ e*MN more when beta != 0 makes C an input; e = output element size).
The attainable rate is min(P_compute, BW * F/Q).

The same page's worked tile numbers (shared memory per stage, CTA input
intensity) and the SemiAnalysis Blackwell page's SMEM-vs-MMA cycle example
are reproduced by the helpers at the bottom; tests pin them against the
values the pages print.
"""
from __future__ import annotations

import json
import os

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, out_bytes: int = 2, beta_nonzero: bool = False,
               in_bytes: int = 2) -> int:
    q = in_bytes * (M * K + N * K) + out_bytes * M * N
    if beta_nonzero:
        q += out_bytes * M * N
    return q


def intensity(M, N, K, out_bytes=2, beta_nonzero=False) -> float:
    return gemm_flops(M, N, K) / gemm_bytes(M, N, K, out_bytes, beta_nonzero)


def attainable_tflops(M, N, K, peak_tflops, hbm_gbs, out_bytes=2, beta_nonzero=False) -> float:
    """min(P_tc, BW * I) in TFLOP/s."""
    return min(peak_tflops, hbm_gbs * 1e9 * intensity(M, N, K, out_bytes, beta_nonzero) / 1e12)


def roofline_entry(M, N, K, seconds, tensor_peak_tflops, hbm_gbs, out_bytes=2, beta_nonzero=False,
                   in_bytes=2) -> dict:
    """One launch of M x N x K taking `seconds` against the roofline
    min(P_tc, BW * F/Q): achieved TFLOP/s and GB/s (algorithmic F and Q), the
    attainable rate, which roof binds, and achieved / attainable."""
    f = gemm_flops(M, N, K)
    q = gemm_bytes(M, N, K, out_bytes, beta_nonzero, in_bytes)
    ai = f / q
    bw_roof = hbm_gbs * 1e9 * ai / 1e12
    roof = min(tensor_peak_tflops, bw_roof)
    tf = f / seconds / 1e12
    gbs = q / seconds / 1e9
    bound = "tensor" if tensor_peak_tflops <= bw_roof else "hbm"
    return {"bound": bound, "achieved_tflops": round(tf, 3), "achieved_gbs": round(gbs, 1),
            "algorithmic_flops": f, "algorithmic_bytes": q, "intensity_flop_per_byte": round(ai, 2),
            "attainable_tflops": round(roof, 2), "tensor_peak_tflops": tensor_peak_tflops, "hbm_peak_gbs": hbm_gbs,
            "frac": round(tf / roof, 4)}


def load_peaks(path: str | None = None) -> dict:
    """Measured peaks (HBM GB/s, bf16 TFLOP/s burst and sustained) with their source."""
    if path is None:
        path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED, "source": "fallback"}


# --------------------------------------------------------------------------
# the pages' worked numbers
# --------------------------------------------------------------------------

def smem_bytes_per_stage(bm: int, bn: int, bk: int, elem_bytes: int = 2) -> int:
    """A and B shared-memory bytes of one pipeline stage: e*(BM*BK + BK*BN)."""
    return elem_bytes * (bm * bk + bk * bn)


def cta_input_intensity(bm: int, bn: int) -> float:
    """FLOP per input byte of one CTA k-step with bf16 inputs: BM*BN/(BM+BN) (BK cancels)."""
    return bm * bn / (bm + bn)


def ss_mma_cycles(m: int, n: int, k: int, flops_per_clk: int = 8192, smem_bytes_per_clk: int = 128,
                  elem_bytes: int = 2):
    """(SMEM-read cycles, MMA cycles) of one SS-mode MMA on one SM."""
    smem = (elem_bytes * m * k + elem_bytes * n * k) / smem_bytes_per_clk
    mma = 2 * m * n * k / flops_per_clk
    return smem, mma


def ridge_point(peak_tflops: float, hbm_tbs: float) -> float:
    """FLOP per byte where the compute and bandwidth roofs meet."""
    return peak_tflops / hbm_tbs
