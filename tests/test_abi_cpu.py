"""The C ABI without a GPU: the library loads, exports every entry point that
include/dga.h declares, and rejects invalid arguments before touching the
device (BLAS-style codes: -position of the bad argument)."""
import ctypes
import os
import re

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import build as dga_build
from dense_gemm_accelerator_gb300 import inputs as gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dga_build.build()
    return dga.lib()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(dga_[a-z0-9_]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert {"dga_gemm", "dga_gemm_ex", "dga_sync_status"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert declared <= set(dga.SIGNATURES), "binding lacks a declared entry point"


def test_version_and_strings(lib):
    assert dga.dga_version() >= 100
    for st in (0, 1, 2, 3, 4, 5, 6, 7, -4):
        assert dga.dga_status_string(st)


def _call(**over):
    one, zero = ctypes.c_float(1.0), ctypes.c_float(0.0)
    args = dict(in_dtype=gen.F32, out_dtype=gen.F32, layout_b=gen.ROW_MAJOR, M=4, N=4, K=4,
                alpha=ctypes.byref(one), A=0x1000, lda=4, B=0x2000, ldb=4, beta=ctypes.byref(zero),
                C=0x3000, ldc=4, workspace=None, workspace_bytes=0, path=dga.PATH_AUTO, stream=None)
    args.update(over)
    return dga.dga_gemm_ex(*args.values())


@pytest.mark.parametrize("over,code", [
    (dict(M=-1), -4), (dict(N=-1), -5), (dict(K=-1), -6), (dict(alpha=None), -7),
    (dict(A=None), -8), (dict(lda=3), -9), (dict(B=None), -10), (dict(ldb=3), -11),
    (dict(beta=None), -12), (dict(C=None), -13), (dict(ldc=3), -14),
    (dict(workspace=None, workspace_bytes=16), -15), (dict(path=9), -17),
    (dict(in_dtype=gen.F32, out_dtype=gen.BF16), dga.ERR_UNSUPPORTED),
    (dict(in_dtype=gen.I8, out_dtype=gen.F32), dga.ERR_UNSUPPORTED),
    (dict(in_dtype=gen.TF32, out_dtype=gen.BF16), dga.ERR_UNSUPPORTED),
    (dict(in_dtype=gen.F32, out_dtype=gen.TF32), dga.ERR_UNSUPPORTED),
    (dict(in_dtype=6, out_dtype=gen.F32), dga.ERR_UNSUPPORTED),
    (dict(layout_b=5), dga.ERR_UNSUPPORTED),
    (dict(C=0x1004), dga.ERR_OVERLAP),
])
def test_argument_errors(lib, over, code):
    assert _call(**over) == code


def test_col_major_ldb_rule(lib):
    # column-major B needs ldb >= K, not >= N
    assert _call(layout_b=gen.COL_MAJOR, K=8, lda=8, ldb=4) == -11


def test_selftest_limit_validated(lib):
    assert dga.dga_selftest_bounded_wait(0, None) == -1
    assert dga.dga_selftest_bounded_wait(3_000_000_000, None) == -1


def test_m_zero_is_a_no_op_without_device(lib):
    assert _call(M=0, A=None, C=None) == dga.OK
    assert _call(N=0, B=None, C=None) == dga.OK


def test_workspace_size_query(lib):
    W = gen.WORKLOADS
    # INT8 on the tensor cores packs A and B as bf16: 2 bytes x (M + N) x K8
    w = W["int8_ragged"]
    ws = dga.dga_gemm_workspace_size(w.in_dtype, w.out_dtype, w.layout_b, w.M, w.N, w.K, w.K,
                                     w.N, w.N, dga.PATH_TCGEN05)
    assert ws >= 2 * (w.M + w.N) * w.K
    # ... both K-major whatever B's layout: K padded to 8, each copy to 256
    # bytes (INT8 does not split its last wave, so nothing more)
    def ru(x, m):
        return (x + m - 1) // m * m
    for M, N, K in ((4093, 4099, 4096), (77, 91, 601), (5, 3, 1)):
        want = ru(M * ru(K, 8) * 2, 256) + ru(N * ru(K, 8) * 2, 256)
        for layout, ldb in ((gen.ROW_MAJOR, N + 3), (gen.COL_MAJOR, K + 5)):
            assert dga.dga_gemm_workspace_size(gen.I8, gen.I32, layout, M, N, K, K, ldb, N,
                                               dga.PATH_TCGEN05) == want, (M, N, K, layout)
    # column-major bf16 with aligned leading dimensions needs nothing; the
    # query reports the optional room for the split last wave of the CTA-pair
    # kernel (two 256 x 256 32-bit slots per pair: 76 pairs on the default 152
    # SMs), nothing for a single wave or a K too shallow to split
    w = W["bf16_8192"]
    assert dga.dga_gemm_workspace_size(w.in_dtype, w.out_dtype, w.layout_b, w.M, w.N, w.K, w.K,
                                       w.K, w.N, dga.PATH_TCGEN05) == 2 * 76 * 256 * 256 * 4
    assert dga.dga_gemm_workspace_size(gen.BF16, gen.F32, gen.COL_MAJOR, 512, 512, 8192, 8192,
                                       8192, 512, dga.PATH_TCGEN05) == 0
    assert dga.dga_gemm_workspace_size(gen.BF16, gen.F32, gen.COL_MAJOR, 8192, 8192, 512, 512,
                                       512, 8192, dga.PATH_TCGEN05) == 0
    # row-major B is read in place (MN-major) unless TMA cannot express its
    # leading dimension; then it is copied row by row (K rows of N, padded to
    # 8 elements) and still read MN-major
    assert dga.dga_gemm_workspace_size(gen.BF16, gen.F32, gen.ROW_MAJOR, 256, 512, 100, 104,
                                       512, 512, dga.PATH_TCGEN05) == 0
    assert dga.dga_gemm_workspace_size(gen.BF16, gen.F32, gen.ROW_MAJOR, 256, 512, 100, 104,
                                       513, 512, dga.PATH_TCGEN05) == 100 * 512 * 2
    assert dga.dga_gemm_workspace_size(gen.BF16, gen.F32, gen.ROW_MAJOR, 256, 510, 100, 104,
                                       513, 510, dga.PATH_TCGEN05) == 100 * 512 * 2
    assert dga.dga_gemm_workspace_size(gen.F32, gen.F32, gen.ROW_MAJOR, 64, 64, 64, 64, 64, 64,
                                       dga.PATH_SIMT) == 0
    # TF32 reads K-major only: column-major B in place (only the split last
    # wave's optional slots), a row-major B is transposed into the workspace
    # as fp32 (4 bytes x N x K4)
    w = W["tf32_8192"]
    assert dga.dga_gemm_workspace_size(w.in_dtype, w.out_dtype, w.layout_b, w.M, w.N, w.K, w.K,
                                       w.K, w.N, dga.PATH_TCGEN05) == 2 * 76 * 256 * 256 * 4
    assert dga.dga_gemm_workspace_size(gen.TF32, gen.F32, gen.ROW_MAJOR, 256, 512, 100, 100,
                                       512, 512, dga.PATH_TCGEN05) >= 512 * 100 * 4
    assert dga.dga_gemm_workspace_size(gen.TF32, gen.F32, gen.COL_MAJOR, 256, 512, 100, 102,
                                       100, 512, dga.PATH_TCGEN05) >= 256 * 100 * 4


def test_fp32_path_by_k(lib):
    # the SIMT kernels count K-slices in 32 bits: from K = 2^33 on, FP32 goes
    # to the generic kernel (addresses far apart: nothing is dereferenced)
    A, B, C = 0x100000000000, 0x200000000000, 0x300000000000
    for K, want in ((4096, dga.PATH_SIMT), ((1 << 33) - 1, dga.PATH_SIMT),
                    (1 << 33, dga.PATH_GENERIC)):
        assert dga.dga_select_path(gen.F32, gen.F32, gen.COL_MAJOR, 2, 3, K, A, K, B, K, C,
                                   3) == want, K


def test_binding_layout_from_strides():
    A = torch.empty(6, 5)
    C = torch.empty(6, 7)
    lda, layout, ldb, ldc = dga.operand_layout(A, torch.empty(5, 7), C)
    assert (lda, layout, ldb, ldc) == (5, gen.ROW_MAJOR, 7, 7)
    lda, layout, ldb, ldc = dga.operand_layout(A, torch.empty(7, 5).t(), C)
    assert (layout, ldb) == (gen.COL_MAJOR, 5)
    with pytest.raises(ValueError):
        dga.operand_layout(A.t(), torch.empty(5, 7), torch.empty(5, 7))
    with pytest.raises(ValueError):
        dga.operand_layout(A, torch.empty(10, 14)[::2, ::2], C)


def _call_general(**over):
    one, zero = ctypes.c_float(1.0), ctypes.c_float(0.0)
    args = dict(in_dtype=gen.F32, out_dtype=gen.F32, layout_a=gen.ROW_MAJOR,
                layout_b=gen.ROW_MAJOR, M=4, N=4, K=4, alpha=ctypes.byref(one), A=0x1000, lda=4,
                B=0x2000, ldb=4, beta=ctypes.byref(zero), C=0x3000, ldc=4, bias=None,
                workspace=None, workspace_bytes=0, path=dga.PATH_AUTO, stream=None)
    args.update(over)
    return dga.dga_gemm_general(*args.values())


@pytest.mark.parametrize("over,code", [
    (dict(M=-1), -5), (dict(N=-1), -6), (dict(K=-1), -7), (dict(alpha=None), -8),
    (dict(A=None), -9), (dict(lda=3), -10), (dict(B=None), -11), (dict(ldb=3), -12),
    (dict(beta=None), -13), (dict(C=None), -14), (dict(ldc=3), -15),
    (dict(workspace=None, workspace_bytes=16), -17), (dict(path=9), -19),
    (dict(layout_a=5), dga.ERR_UNSUPPORTED),
    (dict(C=0x1004), dga.ERR_OVERLAP),
    (dict(bias=0x3008), dga.ERR_OVERLAP),   # bias inside C
])
def test_general_argument_errors(lib, over, code):
    assert _call_general(**over) == code


def test_general_col_major_lda_rule(lib):
    # column-major A is stored K x M: lda >= M, not >= K
    assert _call_general(layout_a=gen.COL_MAJOR, M=8, K=4, lda=4, ldc=4, C=0x9000) == -10


def test_general_m_zero_is_a_no_op(lib):
    assert _call_general(M=0, A=None, C=None, layout_a=gen.COL_MAJOR) == dga.OK


def test_general_workspace_size_query(lib):
    # column-major A on the tensor cores is read in place (MN-major), or
    # transposed into the workspace when lda is not a multiple of 16 bytes
    assert dga.dga_gemm_general_workspace_size(gen.BF16, gen.F32, gen.COL_MAJOR, gen.COL_MAJOR,
                                               256, 512, 1024, 256, 1024, 512,
                                               dga.PATH_TCGEN05) == 0
    ws = dga.dga_gemm_general_workspace_size(gen.BF16, gen.F32, gen.COL_MAJOR, gen.COL_MAJOR,
                                             256, 512, 1024, 257, 1024, 512, dga.PATH_TCGEN05)
    assert ws >= 256 * 1024 * 2
    assert dga.dga_gemm_general_workspace_size(gen.BF16, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR,
                                               256, 512, 1024, 1024, 1024, 512,
                                               dga.PATH_TCGEN05) == 0
    # the row-major-A query agrees with the older entry point
    assert dga.dga_gemm_general_workspace_size(
        gen.I8, gen.I32, gen.ROW_MAJOR, gen.ROW_MAJOR, 100, 200, 300, 300, 200, 200,
        dga.PATH_TCGEN05) == dga.dga_gemm_workspace_size(
        gen.I8, gen.I32, gen.ROW_MAJOR, 100, 200, 300, 300, 200, 200, dga.PATH_TCGEN05)


@pytest.mark.parametrize("args,code", [
    ((gen.I8, 4, 4, 0x1000, 4, 0x2000), dga.ERR_UNSUPPORTED),
    ((gen.F32, -1, 4, 0x1000, 4, 0x2000), -2),
    ((gen.F32, 4, -1, 0x1000, 4, 0x2000), -3),
    ((gen.F32, 4, 4, None, 4, 0x2000), -4),
    ((gen.F32, 4, 4, 0x1000, 3, 0x2000), -5),
    ((gen.F32, 4, 4, 0x1000, 4, None), -6),
    ((gen.BF16, 4, 0, None, 1, None), dga.OK),   # no columns: nothing to do
])
def test_sum_rows_argument_errors(lib, args, code):
    assert dga.dga_sum_rows(*args, None) == code


def test_binding_general_layouts():
    # a transposed view is column-major with its storage row length as ld
    W = torch.empty(7, 5)
    assert dga._layout_of(W, "W") == (gen.ROW_MAJOR, 5)
    assert dga._layout_of(W.t(), "W") == (gen.COL_MAJOR, 5)
    assert dga._layout_of(torch.empty(10, 14)[:, :6], "W") == (gen.ROW_MAJOR, 14)
    with pytest.raises(ValueError):
        dga._layout_of(torch.empty(10, 14)[::2, ::2], "W")


def _spmv(**over):
    import ctypes
    one = ctypes.c_float(1.0)
    args = dict(rows=4, cols=4, nnz=8, row_offsets=0x1000, column_indices=0x2000, values=0x3000,
                alpha=ctypes.byref(one), x=0x4000, beta=ctypes.byref(one), y=0x5000,
                workspace=0x6000, workspace_bytes=1 << 20, stream=None)
    args.update(over)
    return dga.dga_spmv_csr(*args.values())


@pytest.mark.parametrize("over,code", [
    (dict(rows=-1), -1), (dict(cols=-1), -2), (dict(nnz=-1), -3), (dict(nnz=1 << 31), -3),
    (dict(alpha=None), -7), (dict(beta=None), -9), (dict(row_offsets=None), -4),
    (dict(column_indices=None), -5), (dict(values=None), -6), (dict(x=None), -8),
    (dict(y=None), -10), (dict(workspace=None), -11),
    (dict(y=0x4008), dga.ERR_OVERLAP), (dict(y=0x0ffc), dga.ERR_OVERLAP),
])
def test_spmv_argument_errors(lib, over, code):
    assert _spmv(**over) == code


def test_spmv_quick_returns_and_workspace(lib):
    import ctypes
    zero = ctypes.c_float(0.0)
    # no rows: nothing to do, nothing touched
    assert _spmv(rows=0, row_offsets=None, y=None) == dga.OK
    # alpha == 0 reads neither A nor x: their pointers may be NULL (the call
    # then needs the device, absent here, so it stops at the device check)
    st = _spmv(alpha=ctypes.byref(zero), column_indices=None, values=None, x=None)
    assert st in (dga.ERR_CUDA, dga.ERR_DEVICE)
    # one row index and one float per warp: at most 8 CTAs of 8 warps per SM
    ws = dga.dga_spmv_csr_workspace_size(1 << 22, 1 << 26)
    assert 8 * 8 * 152 * 8 <= ws <= 8 * 8 * 152 * 8 + 512
    assert dga.dga_spmv_csr_workspace_size(0, 10) == 0


def test_fma_probe_argument_errors(lib):
    import ctypes
    flops = ctypes.c_double(0.0)
    out_floats = dga.dga_probe_fp32_fma_out_floats()
    assert out_floats == 152 * 4 * 256  # no device here: 152 SMs assumed
    assert dga.dga_probe_fp32_fma(2, 10, 0x1000, out_floats, ctypes.byref(flops), None) == -1
    assert dga.dga_probe_fp32_fma(0, 0, 0x1000, out_floats, ctypes.byref(flops), None) == -2
    assert dga.dga_probe_fp32_fma(1, (1 << 20) + 1, 0x1000, out_floats, ctypes.byref(flops),
                                  None) == -2
    assert dga.dga_probe_fp32_fma(0, 10, None, out_floats, ctypes.byref(flops), None) == -3
    assert dga.dga_probe_fp32_fma(0, 10, 0x1000, out_floats, None, None) == -5
    # valid arguments need the device, absent here
    assert dga.dga_probe_fp32_fma(0, 10, 0x1000, out_floats, ctypes.byref(flops),
                                  None) in (dga.ERR_CUDA, dga.ERR_DEVICE)


def test_int8_mma_probe_argument_errors(lib):
    import ctypes
    ops = ctypes.c_double(0.0)
    n = dga.dga_probe_fp32_fma_out_floats()
    f = dga.dga_probe_int8_mma
    assert f(0, 0x1000, n, ctypes.byref(ops), None) == -1
    assert f((1 << 17) + 1, 0x1000, n, ctypes.byref(ops), None) == -1
    assert f(10, None, n, ctypes.byref(ops), None) == -2
    assert f(10, 0x1000, n, None, None) == -4
    # valid arguments need the device, absent here (the out size is checked
    # against the device's SM count, after the device)
    assert f(10, 0x1000, n, ctypes.byref(ops), None) in (dga.ERR_CUDA, dga.ERR_DEVICE)


def test_naive_probe_argument_errors_before_the_device():
    # the counter-calibration probe checks its arguments before touching a device
    f = dga.dga_probe_naive_sgemm
    assert f(0, 8, 8, 0x1000, 0x2000, 0x3000, None) == -1
    assert f(8, 65537, 8, 0x1000, 0x2000, 0x3000, None) == -2
    assert f(8, 8, 0, 0x1000, 0x2000, 0x3000, None) == -3
    assert f(65536, 8, 65536, 0x1000, 0x2000, 0x3000, None) == -3  # M * K = 2^32 elements
    assert f(8, 8, 8, None, 0x2000, 0x3000, None) == -4
    assert f(8, 8, 8, 0x1000, None, 0x3000, None) == -5
    assert f(8, 8, 8, 0x1000, 0x2000, None, None) == -6
