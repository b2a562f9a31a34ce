"""Roofline arithmetic pinned by the pages' printed numbers and closed forms."""
import json
import os

import pytest

from tensor_core_dense_tn_gb300 import roofline as rl

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_numbers.json")))


def test_stage_bytes():
    assert rl.smem_bytes_per_stage(128, 128, 64) == G["smem_stage_bytes_128_128_64"]["value"]


def test_cta_intensity():
    assert rl.cta_input_intensity(128, 128) == G["cta_input_intensity_128_128"]["value"]


def test_ss_mma_cycles():
    smem, mma = rl.ss_mma_cycles(128, 64, 16)
    assert smem == G["ss_mma_m128_n64_k16_smem_cycles"]["value"]
    assert mma == G["ss_mma_m128_n64_k16_mma_cycles"]["value"]
    n0 = G["ss_mma_compute_bound_from_n"]["value"]
    s, m = rl.ss_mma_cycles(128, n0, 16)
    assert s <= m
    s, m = rl.ss_mma_cycles(128, n0 - 16, 16)
    assert s > m


@pytest.mark.parametrize("key", ["h100_ridge_flop_per_byte", "a100_ridge_flop_per_byte"])
def test_ridge(key):
    e = G[key]
    assert round(rl.ridge_point(e["peak_tflops"], e["hbm_tbs"])) == e["value"]


def test_workload_flops_and_bytes():
    # 8192 x 28672 x 4096 up-projection: bf16 A, B and D
    assert rl.gemm_flops(8192, 28672, 4096) == 1_924_145_348_608
    assert rl.gemm_bytes(8192, 28672, 4096) == 771_751_936
    # decode 16 x 8192 x 8192
    assert rl.gemm_bytes(16, 8192, 8192) == 134_742_016
    # square with beta: C read as well
    assert rl.gemm_bytes(4096, 4096, 4096, beta_nonzero=True) == 4 * 32 * 2 ** 20
    # tiny, fp32 out
    assert rl.gemm_bytes(256, 256, 256, out_bytes=4) == 524_288


def test_attainable_is_min_of_roofs():
    assert rl.attainable_tflops(8192, 28672, 4096, 1900, 6800) == 1900
    t = rl.attainable_tflops(16, 8192, 8192, 1900, 6800)
    assert abs(t - 6800e9 * rl.intensity(16, 8192, 8192) / 1e12) < 1e-9


def test_peaks_fallback(tmp_path):
    p = rl.load_peaks(str(tmp_path / "missing.json"))
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0
    f = tmp_path / "peaks.json"
    f.write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0}))
    p = rl.load_peaks(str(f))
    assert p == {"hbm_gbs": 1.0, "bf16_tflops": 2.0, "bf16_tflops_sustained": 2.0, "source": "measured"}


def test_roofline_entry_picks_the_binding_roof():
    # 16 x 8192 x 8192 bf16: intensity ~15.9 FLOP/B, far left of the ridge -> HBM roof
    e = rl.roofline_entry(16, 8192, 8192, 25e-6, 1922.1, 6668.5)
    q = 2 * (16 * 8192 + 8192 * 8192) + 2 * 16 * 8192
    assert e["bound"] == "hbm" and e["algorithmic_bytes"] == q
    assert e["achieved_gbs"] == pytest.approx(q / 25e-6 / 1e9, rel=1e-3)
    # on the HBM roof, achieved / attainable is the fraction of the bandwidth
    assert e["frac"] == pytest.approx(q / 25e-6 / 1e9 / 6668.5, rel=1e-3)
    # 4096^3 with beta: C is read as well; intensity 2*4096^3 / (4 * 32 MiB) = 1024
    e = rl.roofline_entry(4096, 4096, 4096, 1e-4, 1922.1, 6668.5, beta_nonzero=True)
    assert e["intensity_flop_per_byte"] == 1024.0 and e["bound"] == "tensor"
    assert e["frac"] == pytest.approx(2 * 4096 ** 3 / 1e-4 / 1e12 / 1922.1, rel=1e-3)
