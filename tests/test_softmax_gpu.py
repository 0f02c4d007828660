"""Row softmax on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import online_softmax_06_gb300 as fa
import oracle
import workloads
from gpu_common import SOFTMAX_F32_TOL, device_error_clear, max_abs, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_gpu()


def run(x_np, dev, inplace=False, offset=0):
    """Run fa_softmax_rows on x_np; `offset` floats of padding misalign the rows."""
    rows, N = x_np.shape
    buf = torch.empty(rows * N + offset, dtype=torch.float32, device=dev)
    xg = buf[offset:].view(rows, N)
    xg.copy_(torch.from_numpy(x_np))
    if inplace:
        out = xg
    else:
        out_buf = torch.empty(rows * N + offset, dtype=torch.float32, device=dev)
        out = out_buf[offset:].view(rows, N)
    fa.fa_set_stream(torch.cuda.current_stream(dev).cuda_stream)
    rc = fa.fa_softmax_rows(xg.data_ptr(), out.data_ptr(), rows, N)
    assert rc == 0, fa.strerror(rc)
    torch.cuda.synchronize(dev)
    return out.cpu().numpy()


@pytest.mark.parametrize("N", workloads.SOFTMAX_NS)
def test_softmax_workload_rows(dev, N):
    """The 4096 x N workload at every row length, every element against the oracle
    (rows 0, 64, 128, ... carry the +1000 shift)."""
    x = workloads.softmax_workload(N)
    y = run(x, dev)
    ref = oracle.softmax_rows(x)
    err = max_abs(y, ref)
    assert err <= SOFTMAX_F32_TOL, f"N={N}: max abs err {err:.3e}"
    assert np.all(y >= 0)
    device_error_clear()


@pytest.mark.parametrize("N", [1, 2, 3, 5, 31, 33, 63, 100, 127, 129, 255, 1000, 1023, 1025,
                               2047, 4097, 5000, 9000, 20000, 40000, 70000, 131072, 131073,
                               200003])
def test_softmax_edge_lengths(dev, N):
    rows = 7 if N < 100000 else 3
    x = workloads.softmax_rows_input(rows, N, seed=77 + N, shift_every=2)
    y = run(x, dev)
    assert max_abs(y, oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


@pytest.mark.parametrize("rows", [1, 5, 31, 33, 257])
@pytest.mark.parametrize("N", [32, 64, 128, 96])
def test_softmax_ragged_row_counts(dev, rows, N):
    """Row counts that leave the last CTA of a multi-row launch partly empty."""
    x = workloads.softmax_rows_input(rows, N, seed=rows * 1000 + N)
    assert max_abs(run(x, dev), oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


@pytest.mark.parametrize("N", [64, 4096, 32768])
def test_softmax_in_place(dev, N):
    x = workloads.softmax_rows_input(64, N, seed=5 + N)
    assert max_abs(run(x, dev, inplace=True), oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


@pytest.mark.parametrize("N", [4, 64, 4096, 32768])
def test_softmax_misaligned_rows(dev, N):
    """Pointers off a 16-byte boundary take the scalar-access variant."""
    x = workloads.softmax_rows_input(9, N, seed=9 + N)
    assert max_abs(run(x, dev, offset=1), oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


def test_softmax_overflow_rows_exact(dev):
    """1000, 999, 998 gives the same as 2, 1, 0 and no inf/NaN."""
    x = np.array([[1000.0, 999.0, 998.0], [2.0, 1.0, 0.0]], dtype=np.float32)
    y = run(x, dev)
    assert np.all(np.isfinite(y))
    assert max_abs(y[0], y[1]) == 0.0
    assert max_abs(y, oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


def test_softmax_masked_entries(dev):
    """-inf entries get probability exactly 0."""
    x = workloads.softmax_rows_input(4, 300, seed=3)
    x[:, ::3] = -np.inf
    y = run(x, dev)
    assert np.all(y[:, ::3] == 0)
    assert max_abs(y, oracle.softmax_rows(x)) <= SOFTMAX_F32_TOL


def test_softmax_rows_sum_to_one(dev):
    x = workloads.softmax_workload(4096)
    y = run(x, dev).astype(np.float64)
    assert np.max(np.abs(y.sum(axis=1) - 1.0)) < 1e-4


def test_softmax_bad_arguments(dev):
    x = torch.zeros(4, 4, device=dev)
    assert fa.fa_softmax_rows(x.data_ptr(), None, 4, 4) == -1
    assert fa.fa_softmax_rows(x.data_ptr() + 2, x.data_ptr(), 1, 4) == -4
    assert fa.fa_softmax_rows(x.data_ptr(), x.data_ptr(), -1, 4) == -2
