"""The allocation-free skinny entry point, gemm_bf16_tn_skinny_noalloc.

It serves callers that cannot allocate device memory when they call a GEMM
(a serving process that owns all of HBM through its own pool, latency-critical
code that cannot take cudaMalloc's implicit synchronisation, plug-ins whose
host framework owns every allocation).  Its scratch is a fixed device array in
the library, so these tests check that:

* two calls in a row (different shapes, output types and beta, so the shared
  scratch carries the first call's leftovers into the second) give the same
  result as gemm_bf16_tn, within the accuracy bound every GPU test uses;
* in a fresh process that calls nothing but this entry point, a second pass
  of the same calls on a stream the library has never seen leaves the
  device's free memory unchanged (the regular entry point would allocate a
  workspace for that stream), and its results match the oracle;
* sizes beyond the fixed scratch are rejected with an error, not run.

This file is collected last so that a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import gemm_inputs as gi
import oracle

g = pytest.importorskip("tensor_core_dense_tn_gb300")


def _call(fn, M, N, K, dA, dB, dC, dD, alpha, beta, out_dtype, stream):
    return fn(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, dC.data_ptr() if dC is not None else 0,
              N if dC is not None else 0, dD.data_ptr(), N, alpha, beta, out_dtype, stream)


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    import torch
    from gpu_util import empty_out, from_dev, to_dev_bf16, to_dev_f32

    stream = torch.cuda.current_stream().cuda_stream
    cases = [  # (M, N, K, out, beta)
        (16, 2112, 4096, gi.OUT_BF16, 0.0),     # two k-parts per tile, 4 k-blocks per box
        (40, 1000, 3000, gi.OUT_F32, -0.5),     # K not a whole number of k-blocks
        (64, 8192, 1024, gi.OUT_BF16, 0.0),     # 128 whole 64-row tiles
        (16, 38912, 256, gi.OUT_F32, 0.0),      # 304 tiles: whole tiles, two per CTA
        (16, 1024, 2048, gi.OUT_BF16, 0.0),     # 8 tiles in four parts (the cap)
    ]
    for i, (M, N, K, out, beta) in enumerate(cases):
        A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 5100 + 3 * i)
        B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 5101 + 3 * i)
        C = None
        dC = None
        if beta != 0.0:
            C = gi.draw_f32(M, N, gi.Dist("normal", 1.0), 5102 + 3 * i)
            dC = to_dev_f32(C)
        dA, dB = to_dev_bf16(A), to_dev_bf16(B)
        d_new, _ = empty_out(M, N, out)
        d_old, _ = empty_out(M, N, out)
        rc = _call(g.gemm_bf16_tn_skinny_noalloc, M, N, K, dA, dB, dC, d_new, 1.0, beta, out, stream)
        assert rc == g.GEMM_OK, g.last_error()
        rc = _call(g.gemm_bf16_tn, M, N, K, dA, dB, dC, d_old, 1.0, beta, out, stream)
        assert rc == g.GEMM_OK, g.last_error()
        assert g.gemm_get_status(stream) == g.GEMM_OK
        got_new, got_old = from_dev(d_new, out), from_dev(d_old, out)
        ref, absdot = oracle.gemm_ref(A, B, C, 1.0, beta)
        bound = oracle.bound(ref, absdot, out, beta, C)
        diff = np.abs(oracle.decode_out(got_new, out) - oracle.decode_out(got_old, out))
        assert np.all(diff <= bound), float(np.max(diff / bound))
        ok, worst, where = oracle.check(got_new, ref, absdot, out, beta, C)
        assert ok, (worst, where)


_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Run in a child process: only gemm_bf16_tn_skinny_noalloc is called there.
_CHILD = r"""
import json
import numpy as np
import torch
import gemm_inputs as gi
import oracle
import tensor_core_dense_tn_gb300 as g
from gpu_util import empty_out, from_dev, to_dev_bf16

g.load()
cases = [(16, 2112, 4096, gi.OUT_BF16), (64, 8192, 1024, gi.OUT_F32), (16, 38912, 256, gi.OUT_BF16),
         (40, 1000, 3000, gi.OUT_F32)]
data = []
for i, (M, N, K, out) in enumerate(cases):
    A = gi.draw_bf16(M, K, gi.Dist("normal", 1.0), 5400 + 2 * i)
    B = gi.draw_bf16(N, K, gi.Dist("normal", 1.0 / K), 5401 + 2 * i)
    data.append((M, N, K, out, A, B, to_dev_bf16(A), to_dev_bf16(B), empty_out(M, N, out)[0]))
s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
torch.cuda.synchronize()

def run_all(stream):
    for M, N, K, out, A, B, dA, dB, dD in data:
        rc = g.gemm_bf16_tn_skinny_noalloc(M, N, K, dA.data_ptr(), K, dB.data_ptr(), K, 0, 0, dD.data_ptr(), N,
                                           1.0, 0.0, out, stream.cuda_stream)
        assert rc == g.GEMM_OK, g.last_error()
    assert g.gemm_get_status(stream.cuda_stream) == g.GEMM_OK, g.last_error()

run_all(s1)                  # loads the kernels and the scratch array's module
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
run_all(s2)                  # a stream the library has not seen before
torch.cuda.synchronize()
free2 = torch.cuda.mem_get_info()[0]
worst = 0.0
for M, N, K, out, A, B, dA, dB, dD in data:
    ref, absdot = oracle.gemm_ref(A, B)
    ok, w, _ = oracle.check(from_dev(dD, out), ref, absdot, out)
    worst = max(worst, w)
print(json.dumps({"free_before": free1, "free_after": free2, "worst": worst}))
"""


@pytest.mark.gpu
def test_noalloc_allocates_nothing_in_a_fresh_process():
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([_ROOT, os.path.join(_ROOT, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", _CHILD], cwd=_ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    # The regular skinny path would allocate at least 4 MiB for the new
    # stream (the 64-token case's partial sums); allow 1 MiB of unrelated noise.
    assert res["free_after"] >= res["free_before"] - (1 << 20), res
    assert res["worst"] <= 1.0, res


@pytest.mark.parametrize("M,N,K", [(65, 128, 64), (0, 128, 64), (16, 131073, 64), (16, 128, 0)])
def test_noalloc_rejects_sizes_beyond_its_scratch(M, N, K):
    g.load()
    rc = g.gemm_bf16_tn_skinny_noalloc(M, N, K, 0x1000, 64, 0x2000, 64, 0, 0, 0x3000, 131080, 1.0, 0.0, 0, 0)
    assert rc == g.GEMM_ERR_INVALID_VALUE
    assert g.last_error() != ""
