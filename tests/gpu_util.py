"""Helpers shared by the GPU tests: host<->device copies of bf16 bit arrays,
the C-ABI call on raw pointers, and sample positions for full-size checks."""
from __future__ import annotations

import numpy as np

import gemm_inputs as gi


def torch_dev():
    import torch
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(torch_dev()).view(torch.bfloat16)


def to_dev_f32(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch_dev())


def from_dev(D, out_dtype: int) -> np.ndarray:
    """Device output -> host array (uint16 bf16 bits, or float32)."""
    import torch
    if out_dtype == gi.OUT_BF16:
        return D.view(torch.int16).cpu().numpy().view(np.uint16)
    return D.cpu().numpy()


def empty_out(M, N, out_dtype, ld=None, fill_bits=None):
    """D buffer (rows x ld) pre-filled with a NaN pattern; returns (tensor, ld)."""
    import torch
    ld = N if ld is None else ld
    if out_dtype == gi.OUT_BF16:
        D = torch.empty((M, ld), dtype=torch.int16, device=torch_dev())
        D.fill_(int(np.uint16(0x7FC3 if fill_bits is None else fill_bits).view(np.int16)))
        return D.view(torch.bfloat16), ld
    D = torch.empty((M, ld), dtype=torch.int32, device=torch_dev())
    D.fill_(int(np.uint32(0x7FC00003 if fill_bits is None else fill_bits).view(np.int32)))
    return D.view(torch.float32), ld


def call(M, N, K, dA, lda, dB, ldb, dC, ldc, dD, ldd, alpha, beta, out_dtype, path=0, grid=0,
         skinny_grid=0, timeout_ns=0, fault=0, stream=None, disable_pdl=0, scheduler=0, skinny_bm=0,
         skinny_kgroup=0, tiled_k_parts=0, b_static=0, skinny_pair=0, tail_slices=0):
    """C-ABI call on device tensors; returns (rc, status)."""
    import torch
    import tensor_core_dense_tn_gb300 as g
    cfg = g.GemmConfig(path=path, grid=grid, raster_group=0, skinny_grid=skinny_grid,
                       wait_timeout_ns=timeout_ns, test_fault=fault, disable_pdl=disable_pdl,
                       scheduler=scheduler, skinny_bm=skinny_bm, skinny_kgroup=skinny_kgroup,
                       tiled_k_parts=tiled_k_parts, b_static=b_static, skinny_pair=skinny_pair,
                       tail_slices=tail_slices)
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = g.gemm_bf16_tn_ex(M, N, K, dA.data_ptr() if dA is not None else 0, lda,
                           dB.data_ptr() if dB is not None else 0, ldb,
                           dC.data_ptr() if dC is not None else 0, ldc,
                           dD.data_ptr(), ldd, alpha, beta, out_dtype, s, cfg)
    st = g.gemm_get_status(s) if rc == 0 else None
    return rc, st


def sample_positions(M, N, n_random=4096, seed=0, tile_m=256, tile_n=256):
    """Random (row, col) pairs plus rows/cols at tile edges and the ragged tail."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, M, n_random))
    cols = list(rng.integers(0, N, n_random))
    edge_r = sorted({r for t in range(0, M, tile_m // 2) for r in (t, t - 1) if 0 <= r < M} | {M - 1})
    edge_c = sorted({c for t in range(0, N, tile_n // 2) for c in (t, t - 1) if 0 <= c < N} | {N - 1})
    er = rng.choice(edge_r, size=min(len(edge_r), 64), replace=False)
    ec = rng.choice(edge_c, size=min(len(edge_c), 64), replace=False)
    for r in er:
        for c in rng.choice(ec, size=min(8, len(ec)), replace=False):
            rows.append(int(r))
            cols.append(int(c))
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)


def check_every_element(D, ref_rows, out_dtype, M, chunk_rows=512, beta=0.0, c_rows=None):
    """Compare every element of the host result D (M rows) with the oracle, a
    block of rows at a time so that the FP64 reference never needs more than
    chunk_rows x N doubles at once.  ref_rows(r0, r1) returns the oracle's
    (ref, absdot) for rows r0..r1-1; c_rows(r0, r1) the matching C values
    (or None).  Returns (ok, worst |D - ref| / bound, (row, col) of the worst)."""
    import oracle
    worst, where = 0.0, None
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        ref, absdot = ref_rows(r0, r1)
        c = None if c_rows is None else c_rows(r0, r1)
        ok, w, idx = oracle.check(D[r0:r1], ref, absdot, out_dtype, beta, c)
        if w > worst or where is None:
            worst, where = w, (r0 + int(idx[0]), int(idx[1])) if idx is not None else None
        del ref, absdot
    return worst <= 1.0, worst, where
