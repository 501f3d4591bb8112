"""The oracle on the worked example the pages print.

The sparse-matrix section of "AI Programming: Matrix Product" prints one 3 x 4
matrix twice, as COO and as CSR arrays.  Both encodings must describe the same
dense matrix; the oracle's A @ I must reproduce it exactly, and A @ X must
equal the row-wise sums that the page's SpMV description defines over the CSR
arrays (a different evaluation order of the same products, exact here because
every value is a small integer).
"""
import json
import os

import numpy as np

F32, ROW = 0, 0
HERE = os.path.dirname(os.path.abspath(__file__))


def _example():
    with open(os.path.join(HERE, "golden", "csr_example.json")) as f:
        return json.load(f)


def _dense_from_coo(ex):
    m, n = ex["shape"]
    A = np.zeros((m, n), np.float32)
    coo = ex["coo"]
    for v, r, c in zip(coo["values"], coo["rows"], coo["cols"]):
        A[r, c] += v
    return A


def _spmv_csr(ex, x):
    csr = ex["csr"]
    offs = csr["row_offsets"]
    y = []
    for i in range(len(offs) - 1):
        s = 0
        for p in range(offs[i], offs[i + 1]):
            s += csr["values"][p] * x[csr["column_indices"][p]]
        y.append(s)
    return y


def test_coo_and_csr_agree():
    ex = _example()
    A = _dense_from_coo(ex)
    csr = ex["csr"]
    assert csr["row_offsets"][-1] == len(csr["values"])
    B = np.zeros_like(A)
    offs = csr["row_offsets"]
    for i in range(len(offs) - 1):
        for p in range(offs[i], offs[i + 1]):
            B[i, csr["column_indices"][p]] = csr["values"][p]
    assert np.array_equal(A, B)


def test_oracle_identity_on_example(oracle_lib):
    ex = _example()
    A = _dense_from_coo(ex)
    m, n = A.shape
    ref, _ = oracle_lib.gemm_fp(F32, F32, ROW, m, n, n, 1.0, A, n, np.eye(n, dtype=np.float32),
                                n, 0.0)
    assert np.array_equal(ref, A.astype(np.float64))


def test_oracle_matches_csr_spmv(oracle_lib):
    ex = _example()
    A = _dense_from_coo(ex)
    m, n = A.shape
    X = np.array([[1, -2], [2, 5], [3, 0], [4, 7]], np.float32)     # K x 2
    ref, _ = oracle_lib.gemm_fp(F32, F32, ROW, m, 2, n, 1.0, A, n, X, 2, 0.0)
    for col in range(2):
        assert ref[:, col].tolist() == _spmv_csr(ex, X[:, col].tolist())
