"""Bounded device waits: a dropped TMA load must end in GEMM_ERR_TIMEOUT, not a hang.

The test-only fault makes CTA 0's producer arm a stage's transaction count
without issuing its loads, so the consumer's wait on that stage can never
complete.  With a short wait limit every role of the kernel gives up, frees
Tensor Memory and returns; the host reads the status word, and the context
stays usable for a correct GEMM right after.
"""
import numpy as np
import pytest

import gemm_inputs as gi
import oracle

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")
from gpu_util import call, empty_out, from_dev, to_dev_bf16  # noqa: E402


@pytest.mark.parametrize("path,scheduler", [(1, 0), (2, 0), (3, 0), (1, 2), (2, 2)])
def test_dropped_load_times_out_then_recovers(path, scheduler):
    import torch
    M = 32 if path == 3 else 512
    N, K = 768, 512
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 77)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 78)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_F32, path=path,
                  timeout_ns=20_000_000, fault=1, scheduler=scheduler)
    assert rc == 0
    assert st == g.GEMM_ERR_TIMEOUT, (st, g.last_error())
    assert (g.gemm_get_status_detail() >> 24) in (1, 2, 3, 4)
    # status is cleared by the read, and the next call is correct
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_get_status(s) == 0
    ref, _ = oracle.gemm_ref(A, B)
    dD2, _ = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD2, ldd, 1.0, 0.0, gi.OUT_F32, path=path,
                  scheduler=scheduler)
    assert rc == 0 and st == 0
    assert np.array_equal(from_dev(dD2, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("b_static,pair", [(0, 0), (1, 0), (0, 2), (1, 2)])
def test_dropped_load_in_two_part_decode_tile(b_static, pair):
    """16 x 8192: CTA 0 finishes tile 0 and takes the other part's partial
    before its own accumulator; its dropped stage must still end in a timeout
    and leave the counters clean for the next call."""
    import torch
    M, N, K = 16, 8192, 1024
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 79)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 80)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_F32, path=3,
                  timeout_ns=20_000_000, fault=1, b_static=b_static, skinny_pair=pair)
    assert rc == 0
    assert st == g.GEMM_ERR_TIMEOUT, (st, g.last_error())
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_get_status(s) == 0
    ref, _ = oracle.gemm_ref(A, B)
    dD2, _ = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD2, ldd, 1.0, 0.0, gi.OUT_F32, path=3, skinny_pair=pair)
    assert rc == 0 and st == 0
    assert np.array_equal(from_dev(dD2, gi.OUT_F32), oracle.exact_f32(ref))


@pytest.mark.parametrize("path", [1, 2])
def test_dropped_load_in_split_tile(path):
    """A split tile whose publishing part (CTA 0) loses a stage: that part
    aborts without publishing, part 0 gives up its bounded wait for it, and
    the next call (counters cleared by the status read) is exact."""
    import torch
    M, N, K = 300, 520, 1024
    A = gi.draw_bf16(M, K, gi.Dist("int", -4, 4), 81)
    B = gi.draw_bf16(N, K, gi.Dist("int", -4, 4), 82)
    dA, dB = to_dev_bf16(A), to_dev_bf16(B)
    dD, ldd = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD, ldd, 1.0, 0.0, gi.OUT_F32, path=path,
                  timeout_ns=20_000_000, fault=1, tiled_k_parts=2)
    assert rc == 0
    assert st == g.GEMM_ERR_TIMEOUT, (st, g.last_error())
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_get_status(s) == 0
    ref, _ = oracle.gemm_ref(A, B)
    dD2, _ = empty_out(M, N, gi.OUT_F32)
    rc, st = call(M, N, K, dA, K, dB, K, None, 0, dD2, ldd, 1.0, 0.0, gi.OUT_F32, path=path, tiled_k_parts=2)
    assert rc == 0 and st == 0
    assert np.array_equal(from_dev(dD2, gi.OUT_F32), oracle.exact_f32(ref))
