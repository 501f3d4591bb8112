"""GPU parity of the CSR sparse matrix-vector product against the CPU oracle.

y <- alpha * A @ x + beta * y for A in CSR form ("AI Programming: Matrix
Product", sections "CSR" and "SpMV").  Every row is compared with the oracle
within its bound (1e-4 * sum |a x| + |beta y| * 2^-22); integer-valued inputs
whose sums stay below 2^24 must match bit for bit.  Structures cover the
page's worked example, power-law row lengths, empty rows (leading, trailing,
long runs), rows much longer than one CTA's share, unsorted and repeated
columns, and malformed arrays (reported, never read out of bounds).
"""
import ctypes
import json
import os

import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(offs, cols, vals, x, y=None, alpha=1.0, beta=0.0, n_cols=None, expect_sync=dga.OK):
    """Copy host CSR arrays to the GPU, call dga_spmv_csr through the C ABI
    and return y on the host."""
    dev = torch.device("cuda")
    rows = offs.numel() - 1
    nnz = vals.numel()
    n_cols = x.numel() if n_cols is None else n_cols
    o, c, v, xd = offs.to(dev), cols.to(dev), vals.to(dev), x.to(dev)
    yd = (y if y is not None else torch.full((rows,), float("nan"))).to(dev)
    ws_bytes = dga.dga_spmv_csr_workspace_size(rows, nnz)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    a, b = ctypes.c_float(alpha), ctypes.c_float(beta)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_spmv_csr(rows, n_cols, nnz, o.data_ptr(), c.data_ptr(), v.data_ptr(),
                          ctypes.byref(a), xd.data_ptr(), ctypes.byref(b), yd.data_ptr(),
                          ws.data_ptr(), ws_bytes, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    sync = dga.dga_sync_status(stream)
    assert sync == expect_sync, dga.dga_status_string(sync)
    return yd.cpu()


def _check(offs, cols, vals, x, y=None, alpha=1.0, beta=0.0, what=""):
    got = _run(offs, cols, vals, x, y, alpha, beta)
    ref, bound = oracle.spmv_csr(offs.numel() - 1, x.numel(), offs, cols, vals, x, alpha, beta,
                                 y)
    err = np.abs(got.double().numpy() - ref)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} rows outside the bound, first {np.argwhere(bad)[:5].ravel().tolist()}"
    return got, ref


def _from_lengths(lengths, n_cols, g, window=None):
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    offs = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(lengths, 0)
    nnz = int(offs[-1])
    cols = torch.randint(0, n_cols, (nnz,), generator=g, dtype=torch.int32)
    vals = torch.rand(nnz, generator=g) * 2 - 1
    return offs.to(torch.int32), cols, vals


def test_page_example():
    with open(os.path.join(HERE, "golden", "csr_example.json")) as f:
        ex = json.load(f)
    csr = ex["csr"]
    offs = torch.tensor(csr["row_offsets"], dtype=torch.int32)
    cols = torch.tensor(csr["column_indices"], dtype=torch.int32)
    vals = torch.tensor(csr["values"], dtype=torch.float32)
    x = torch.tensor([1.0, 2.0, 3.0, 4.0])
    got = _run(offs, cols, vals, x)
    # rows of the dense matrix the page's COO triplets describe, times x
    assert got.tolist() == [10.0, 30.0, 9.0]


@pytest.mark.parametrize("rows,cols,seed", [(1, 1, 0), (7, 5, 1), (2000, 3000, 2),
                                            (20000, 30000, 3), (65537, 1000, 4)])
def test_powerlaw(rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    offs, ci, vals = gen.csr_powerlaw(rows, cols, g, window=max(1, cols // 4))
    x = torch.rand(cols, generator=g) * 2 - 1
    y = torch.rand(rows, generator=g) * 2 - 1
    _check(offs, ci, vals, x, what=f"{rows}x{cols}")
    _check(offs, ci, vals, x, y, alpha=-1.5, beta=0.75, what=f"{rows}x{cols} alpha beta")


def test_workload_small_and_bit_exact_integers():
    w = gen.WORKLOADS["spmv_small"]
    offs, ci, vals, x, _ = gen.make_csr_inputs(w)
    _check(offs, ci, vals, x, what="spmv_small")
    # small integers: every partial sum is an exact fp32 integer
    g = torch.Generator().manual_seed(5)
    vi = torch.randint(-3, 4, vals.shape, generator=g).float()
    xi = torch.randint(-3, 4, x.shape, generator=g).float()
    got, ref = _check(offs, ci, vi, xi, what="integers")
    assert np.array_equal(got.double().numpy(), ref)


def test_long_rows_cross_ctas():
    # one row longer than many CTAs' shares, next to short and empty rows
    g = torch.Generator().manual_seed(6)
    lengths = [3, 0, 400000, 0, 0, 1, 250000, 5] + [2] * 1000 + [300000]
    offs, ci, vals = _from_lengths(lengths, 5000, g)
    x = torch.rand(5000, generator=g) * 2 - 1
    y = torch.rand(len(lengths), generator=g)
    _check(offs, ci, vals, x, what="long rows")
    _check(offs, ci, vals, x, y, alpha=2.0, beta=-1.0, what="long rows alpha beta")


def test_empty_rows_everywhere():
    g = torch.Generator().manual_seed(7)
    lengths = [0] * 5000 + [4, 0, 9] + [0] * 70000 + [1] + [0] * 3000
    offs, ci, vals = _from_lengths(lengths, 64, g)
    x = torch.rand(64, generator=g)
    y = torch.rand(len(lengths), generator=g)
    got, ref = _check(offs, ci, vals, x, y, alpha=1.0, beta=0.5, what="empty rows")
    empty = torch.tensor(lengths) == 0
    assert torch.equal(got[empty], (0.5 * y)[empty])


def test_repeated_and_unsorted_columns():
    # entries of a row in any order, one column repeated: the repeats add up
    offs = torch.tensor([0, 4, 6], dtype=torch.int32)
    cols = torch.tensor([3, 0, 3, 1, 2, 2], dtype=torch.int32)
    vals = torch.tensor([1.0, 2.0, 4.0, 8.0, 16.0, 32.0])
    x = torch.tensor([1.0, 10.0, 100.0, 1000.0])
    got = _run(offs, cols, vals, x)
    assert got.tolist() == [1000 + 2 + 4000 + 80, 1600 + 3200]


def test_beta_zero_never_reads_y_and_alpha_zero_never_reads_a():
    g = torch.Generator().manual_seed(8)
    offs, ci, vals = _from_lengths([2, 3, 0, 1], 6, g)
    x = torch.rand(6, generator=g)
    got = _run(offs, ci, vals, x)  # y starts as NaN
    assert torch.isfinite(got).all()
    y = torch.tensor([1.0, -2.0, 3.0, 4.0])
    nan_vals = torch.full_like(vals, float("nan"))
    got = _run(offs, ci, nan_vals, torch.full_like(x, float("nan")), y, alpha=0.0, beta=-0.5)
    assert torch.equal(got, -0.5 * y)
    assert dga.dga_last_launch_count() == 1


def test_no_entries():
    offs = torch.zeros(10, dtype=torch.int32)
    got = _run(offs, torch.zeros(0, dtype=torch.int32), torch.zeros(0), torch.rand(4))
    assert torch.equal(got, torch.zeros(9))


def test_deterministic():
    g = torch.Generator().manual_seed(9)
    offs, ci, vals = gen.csr_powerlaw(50000, 50000, g)
    x = torch.rand(50000, generator=g)
    a = _run(offs, ci, vals, x)
    b = _run(offs, ci, vals, x)
    assert torch.equal(a, b)


@pytest.mark.parametrize("case", ["column", "offsets_decrease", "last_offset"])
def test_malformed_arrays_are_reported(case):
    # the kernel clamps or skips what is out of range (never reading outside
    # the arrays) and dga_sync_status reports DGA_ERR_BAD_INDEX
    offs = torch.tensor([0, 2, 3, 5], dtype=torch.int32)
    cols = torch.tensor([0, 1, 2, 0, 1], dtype=torch.int32)
    vals = torch.ones(5)
    x = torch.ones(3)
    if case == "column":
        cols[3] = 7
    elif case == "offsets_decrease":
        offs[2] = 1
        offs[1] = 3
    else:
        offs[3] = 4
    _run(offs, cols, vals, x, expect_sync=dga.ERR_BAD_INDEX)
    # the next call is clean again
    _run(torch.tensor([0, 2, 3, 5], dtype=torch.int32), torch.tensor([0, 1, 2, 0, 1], dtype=torch.int32),
         vals, x)


def test_full_size_workload():
    w = gen.WORKLOADS["spmv_powerlaw"]
    offs, ci, vals, x, _ = gen.make_csr_inputs(w)
    dev = torch.device("cuda")
    y = dga.spmv_csr(offs.to(dev), ci.to(dev), vals.to(dev), x.to(dev))
    torch.cuda.synchronize()
    ref, bound = oracle.spmv_csr(w.M, w.N, offs, ci, vals, x)
    err = np.abs(y.cpu().double().numpy() - ref)
    assert (err <= bound).all(), f"{int((err > bound).sum())} rows outside the bound"


@pytest.mark.parametrize("length", [1, 5, 8, 16, 17, "mixed"])
def test_row_lengths_at_lane_boundaries(length):
    # a lane of a chunk holds 16 consecutive entries: rows of 8 close exactly
    # two rows in every lane (the branch-free path), rows of 5 close three in
    # some lanes (the general loop), rows of 16 and 17 end on and just past
    # lane boundaries, rows of 1 give chunks of more than 32 row ends (each
    # lane then takes 16 consecutive merge items); mixed lengths 0-40 combine
    # them within a warp
    g = torch.Generator().manual_seed(40 + (length if isinstance(length, int) else 0))
    n_rows = 30000
    if length == "mixed":
        lengths = torch.randint(0, 41, (n_rows,), generator=g).tolist()
    else:
        lengths = [length] * n_rows
    offs, ci, vals = _from_lengths(lengths, 7000, g)
    x = torch.rand(7000, generator=g) * 2 - 1
    y = torch.rand(n_rows, generator=g)
    _check(offs, ci, vals, x, what=f"rows of {length}")
    _check(offs, ci, vals, x, y, alpha=-1.5, beta=0.25, what=f"rows of {length}, alpha beta")
    # integer-valued inputs: every order of the sums gives the same exact value
    vi = torch.randint(-3, 4, vals.shape, generator=g).float()
    xi = torch.randint(-3, 4, x.shape, generator=g).float()
    got, ref = _check(offs, ci, vi, xi, what=f"rows of {length}, integers")
    assert np.array_equal(got.double().numpy(), ref)


def test_infinite_values_stay_in_their_rows():
    # every other row holds +inf entries (x > 0, so each of its products is
    # +inf): those rows are +inf and no NaN or inf reaches the rows between
    # them, wherever the chunk boundaries fall
    g = torch.Generator().manual_seed(50)
    lengths = torch.randint(1, 30, (40000,), generator=g).tolist()
    offs, ci, vals = _from_lengths(lengths, 3000, g)
    row_of = torch.repeat_interleave(torch.arange(len(lengths)), torch.tensor(lengths))
    inf_rows = row_of % 2 == 0
    vals[inf_rows] = float("inf")
    x = torch.rand(3000, generator=g) * 0.5 + 0.5
    got = _run(offs, ci, vals, x)
    even = torch.arange(len(lengths)) % 2 == 0
    assert torch.isinf(got[even]).all() and (got[even] > 0).all()
    finite_vals = vals.clone()
    finite_vals[inf_rows] = 0.0
    ref, bound = oracle.spmv_csr(len(lengths), 3000, offs, ci, finite_vals, x)
    odd = ~even.numpy()
    err = np.abs(got.double().numpy()[odd] - ref[odd])
    assert np.isfinite(got.numpy()[odd]).all() and (err <= bound[odd]).all()
