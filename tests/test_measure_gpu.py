"""The measurement kernels through the C ABI: gemm_stream_read (the skinny
path's weight stream with nothing else done) and gemm_mma_rate (the
tcgen05.mma cost at the skinny path's shapes).  They compute nothing to
compare with the oracle; these tests check that every box shape and operand
kind runs to completion without a device error, that the stream reads every
byte of the matrix it is given (through the time it takes against a bound),
and that the MMA timings are ordered the way the instruction's work is."""
import pytest

pytestmark = pytest.mark.gpu

g = pytest.importorskip("tensor_core_dense_tn_gb300")


@pytest.mark.parametrize("box_rows,kgroup", [(32, 1), (64, 2), (128, 4), (256, 1), (128, 2)])
@pytest.mark.parametrize("grid", [0, 1, 37])
def test_stream_read_runs(box_rows, kgroup, grid):
    import torch
    rows, row_bytes = 1024, 8192
    buf = torch.zeros(rows * row_bytes, dtype=torch.uint8, device="cuda:0")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_stream_read(buf.data_ptr(), rows, row_bytes, box_rows, kgroup, grid, s) == 0, g.last_error()
    assert g.gemm_get_status(s) == 0, g.last_error()


def test_stream_read_time_grows_with_the_bytes():
    """Reading 16x the bytes takes clearly longer (the kernel really streams them)."""
    import torch
    s = torch.cuda.Stream()
    times = []
    for rows in (1024, 16384):
        buf = torch.zeros(rows * 16384, dtype=torch.uint8, device="cuda:0")
        with torch.cuda.stream(s):
            for _ in range(3):
                assert g.gemm_stream_read(buf.data_ptr(), rows, 16384, 128, 4, 0, s.cuda_stream) == 0
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(10):
                assert g.gemm_stream_read(buf.data_ptr(), rows, 16384, 128, 4, 0, s.cuda_stream) == 0
            e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / 10)
        del buf
    assert g.gemm_get_status(s.cuda_stream) == 0
    assert times[1] > 4 * times[0], times


@pytest.mark.parametrize("fp8", [0, 1])
@pytest.mark.parametrize("cta_group", [1, 2])
def test_mma_rate_runs_and_orders(fp8, cta_group):
    """Every N runs; N = 256 costs at least as much per instruction as N = 16."""
    import torch
    out = torch.zeros(2, dtype=torch.int64, device="cuda:0")
    s = torch.cuda.current_stream().cuda_stream
    ns = {}
    for n in (16, 64, 256):
        for _ in range(2):
            assert g.gemm_mma_rate(n, cta_group, fp8, 1024, 2 * cta_group, out.data_ptr(), s) == 0, g.last_error()
        assert g.gemm_get_status(s) == 0, g.last_error()
        total, issue = (int(x) for x in out.cpu().tolist())
        assert total > 0 and 0 < issue <= total
        ns[n] = total / (1024 * 4)
    assert ns[256] >= ns[16] * 0.9, ns
