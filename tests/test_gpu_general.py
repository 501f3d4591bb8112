"""GPU parity of the general entry point (both operand layouts, bias row) and
of the fully-connected layer built on it ("AI Programming: Matrix Product",
section "Fully-connected layer"): every kernel family against the oracle,
through the C ABI, element by element.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, assert_exact

pytestmark = pytest.mark.gpu

S, T, K_, GEN = dga.PATH_SIMT, dga.PATH_TCGEN05, dga.PATH_SKINNY, dga.PATH_GENERIC


def _operands(in_dtype, out_dtype, layout_a, layout_b, M, N, K, seed, with_bias, pad=0):
    """Host operands in the stored shapes: A is M x lda (row) or K x lda
    (column-major), B is K x ldb (row) or N x ldb (column-major)."""
    g = torch.Generator().manual_seed(seed)
    dist = ("int8",) if in_dtype == gen.I8 else ("uniform",)
    a_shape = (M, K + pad) if layout_a == gen.ROW_MAJOR else (K, M + pad)
    b_shape = (K, N + pad) if layout_b == gen.ROW_MAJOR else (N, K + pad)
    A = gen.random_matrix(a_shape, in_dtype, g, dist)
    B = gen.random_matrix(b_shape, in_dtype, g, dist)
    cdist = ("int8",) if out_dtype == gen.I32 else ("uniform",)
    C = gen.random_matrix((M, N + pad), out_dtype, g, cdist)
    bias = gen.random_matrix((1, N), out_dtype, g, cdist).reshape(N) if with_bias else None
    return A, B, C, bias


def run_general(path, in_dtype, out_dtype, layout_a, layout_b, M, N, K, A, B, C, bias, alpha,
                beta, expect=dga.OK):
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    bd = bias.to(dev) if bias is not None else None
    lda, ldb, ldc = A.shape[1], B.shape[1], C.shape[1]
    ws_bytes = dga.dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N,
                                                   K, lda, ldb, ldc, path)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = dga.scalar(alpha, in_dtype), dga.scalar(beta, in_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_general(in_dtype, out_dtype, layout_a, layout_b, M, N, K, ctypes.byref(al),
                              Ad.data_ptr(), lda, Bd.data_ptr(), ldb, ctypes.byref(be),
                              Cd.data_ptr(), ldc, bd.data_ptr() if bd is not None else None,
                              ws.data_ptr() if ws_bytes else None, ws_bytes, path, stream)
    assert st == expect, f"dga_gemm_general returned {st} ({dga.dga_status_string(st)})"
    if st != dga.OK:
        return None
    sync = dga.dga_sync_status(stream)
    assert sync == dga.OK, dga.dga_status_string(sync)
    return Cd.cpu()


def check_general(path, in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha=1.0, beta=0.0,
                  with_bias=True, seed=0, pad=0):
    A, B, C, bias = _operands(in_dtype, out_dtype, layout_a, layout_b, M, N, K, seed, with_bias,
                              pad)
    got = run_general(path, in_dtype, out_dtype, layout_a, layout_b, M, N, K, A, B, C, bias,
                      alpha, beta)
    if path != dga.PATH_AUTO:
        assert dga.dga_last_path() == path
    lda, ldb, ldc = A.shape[1], B.shape[1], C.shape[1]
    what = (f"path={dga.PATH_NAMES.get(path, path)} in={in_dtype} out={out_dtype} "
            f"A={layout_a} B={layout_b} {M}x{N}x{K} bias={with_bias}")
    if in_dtype == gen.I8:
        ref = oracle.gemm_i8_ex(layout_a, layout_b, M, N, K, int(alpha), A, lda, B, ldb,
                                int(beta), C, ldc, bias)
        assert_exact(got[:, :N], ref, gen.I32, what)
    else:
        ref, bound = oracle.gemm_fp_ex(in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha,
                                       A, lda, B, ldb, beta, C, ldc, bias)
        assert_close(got[:, :N], ref, bound, out_dtype, what)
    if pad:
        assert torch.equal(got[:, N:], C[:, N:]), "wrote outside C"


# ------------------------------------------------------- column-major A --

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 33), (256, 256, 256), (300, 200, 1001),
                                   (1152, 1152, 1024), (1000, 1100, 1500)])
def test_simt_col_major_a(M, N, K):
    # the last two shapes take the split-K tail and the interior fast path
    check_general(S, gen.F32, gen.F32, gen.COL_MAJOR, gen.ROW_MAJOR, M, N, K, 1.5, 0.5,
                  with_bias=False)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 33), (256, 512, 256), (300, 200, 1001),
                                   (1152, 1152, 1024)])
@pytest.mark.parametrize("layout_a", [gen.ROW_MAJOR, gen.COL_MAJOR])
def test_simt_col_major_b(M, N, K, layout_a):
    check_general(S, gen.F32, gen.F32, layout_a, gen.COL_MAJOR, M, N, K, 0.5, 2.0,
                  with_bias=False)


def test_simt_col_major_a_unaligned_lda():
    # lda = M + 1 (odd): the float4 loads of A give way to scalar loads
    check_general(S, gen.F32, gen.F32, gen.COL_MAJOR, gen.COL_MAJOR, 130, 140, 70, pad=1)


@pytest.mark.parametrize("M,N,K", [(77, 300, 264), (128, 256, 512), (259, 515, 1100),
                                   (1024, 768, 640)])
@pytest.mark.parametrize("layout_b", [gen.COL_MAJOR, gen.ROW_MAJOR])
def test_tc_col_major_a(M, N, K, layout_b):
    # M <= 128 runs the single-CTA kernel, larger M the CTA-pair kernel
    check_general(T, gen.BF16, gen.F32, gen.COL_MAJOR, layout_b, M, N, K, with_bias=False)


def test_tc_col_major_a_f16_bf16_out():
    check_general(T, gen.F16, gen.F16, gen.COL_MAJOR, gen.COL_MAJOR, 300, 200, 136, 0.75, 0.25,
                  with_bias=False)
    check_general(T, gen.BF16, gen.BF16, gen.COL_MAJOR, gen.ROW_MAJOR, 200, 300, 264, 1.0, 1.0,
                  with_bias=False)


@pytest.mark.parametrize("M", [77, 260])
def test_tc_repack_keeps_mn_major(M):
    # leading dimensions TMA cannot express (M + 3, N + 3: not multiples of 8)
    # on a column-major A and a row-major B: each is copied row by row into
    # the workspace in its own layout and read MN-major (single-CTA and
    # CTA-pair kernels)
    check_general(T, gen.BF16, gen.F32, gen.COL_MAJOR, gen.ROW_MAJOR, M, 140, 99, 1.0, 0.5,
                  with_bias=False, pad=3)
    check_general(T, gen.F16, gen.F16, gen.COL_MAJOR, gen.ROW_MAJOR, M, 140, 99, 1.0, 0.0,
                  with_bias=True, pad=3, seed=1)


@pytest.mark.parametrize("M,N,K", [(77, 91, 600), (259, 515, 1100)])
def test_tc_int8_col_major_a(M, N, K):
    check_general(T, gen.I8, gen.I32, gen.COL_MAJOR, gen.ROW_MAJOR, M, N, K, 3, -2,
                  with_bias=False)


@pytest.mark.parametrize("M,N,K,pad", [(5, 3, 1, 0), (130, 7, 9, 3), (129, 129, 65, 0),
                                       (131, 300, 200, 3), (257, 136, 72, 1), (70, 1025, 130, 5)])
@pytest.mark.parametrize("layout_a,layout_b", [(gen.ROW_MAJOR, gen.ROW_MAJOR),
                                               (gen.COL_MAJOR, gen.ROW_MAJOR),
                                               (gen.COL_MAJOR, gen.COL_MAJOR),
                                               (gen.ROW_MAJOR, gen.COL_MAJOR)])
def test_tc_int8_transposing_repack_edges(M, N, K, pad, layout_a, layout_b):
    # int8 operands are re-encoded K-major: a column-major A and a row-major B
    # are transposed in 64 (k) x 128 (row) tiles.  The shapes put ragged edges
    # in both tile directions (N, M one past or short of 128-row tiles; K one,
    # a few, or past 64-deep tiles, padded to 8), and the padded leading
    # dimensions make source rows that are not 8-byte aligned (the
    # funnel-shifted loads and the bytewise ones at the operand's end)
    check_general(T, gen.I8, gen.I32, layout_a, layout_b, M, N, K, 3, -2, with_bias=True,
                  seed=M + N + K, pad=pad)


@pytest.mark.parametrize("pair", [(gen.F32, gen.F32), (gen.BF16, gen.BF16), (gen.F16, gen.F32),
                                  (gen.I8, gen.I32)])
def test_generic_col_major_a(pair):
    check_general(GEN, pair[0], pair[1], gen.COL_MAJOR, gen.COL_MAJOR, 70, 45, 50, 2.0, 0.5,
                  pad=3)


def test_skinny_rejects_col_major_a():
    A, B, C, _ = _operands(gen.BF16, gen.BF16, gen.COL_MAJOR, gen.COL_MAJOR, 8, 256, 256, 0,
                           False)
    run_general(K_, gen.BF16, gen.BF16, gen.COL_MAJOR, gen.COL_MAJOR, 8, 256, 256, A, B, C, None,
                1.0, 0.0, expect=dga.ERR_PATH)
    # AUTO then picks a family that takes it
    check_general(dga.PATH_AUTO, gen.BF16, gen.BF16, gen.COL_MAJOR, gen.COL_MAJOR, 8, 256, 256)


def test_col_major_a_detects_transpose():
    # a permutation matrix as A: a transposed read of A would permute rows
    M = K = 160
    N = 96
    perm = torch.randperm(M, generator=torch.Generator().manual_seed(3))
    P = torch.zeros(M, K)
    P[torch.arange(M), perm] = 1.0
    g = torch.Generator().manual_seed(4)
    B = gen.random_matrix((K, N), gen.F32, g)
    for path in (S, GEN):
        C = torch.zeros(M, N)
        got = run_general(path, gen.F32, gen.F32, gen.COL_MAJOR, gen.ROW_MAJOR, M, N, K,
                          P.t().contiguous(), B, C, None, 1.0, 0.0)
        assert torch.equal(got, B[perm]), dga.PATH_NAMES[path]


def test_col_major_b_detects_transpose():
    # a permutation matrix as B (stored N x K): columns of A come out permuted
    K = N = 160
    M = 96
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(5))
    P = torch.zeros(K, N)
    P[perm, torch.arange(N)] = 1.0          # (A P)[:, j] = A[:, perm[j]]
    g = torch.Generator().manual_seed(6)
    A = gen.random_matrix((M, K), gen.F32, g)
    for path in (S, GEN):
        C = torch.zeros(M, N)
        got = run_general(path, gen.F32, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, A,
                          P.t().contiguous(), C, None, 1.0, 0.0)
        assert torch.equal(got, A[:, perm]), dga.PATH_NAMES[path]


# ------------------------------------------------------------ bias row --

@pytest.mark.parametrize("path,in_dtype,out_dtype,layout_b,M,N,K", [
    (S, gen.F32, gen.F32, gen.ROW_MAJOR, 300, 200, 1001),
    (S, gen.F32, gen.F32, gen.ROW_MAJOR, 1152, 1152, 1024),   # split-K tail reduction
    (S, gen.F32, gen.F32, gen.COL_MAJOR, 256, 512, 256),      # interior kernel
    (T, gen.BF16, gen.F32, gen.COL_MAJOR, 100, 300, 264),     # single-CTA kernel
    (T, gen.BF16, gen.BF16, gen.COL_MAJOR, 600, 520, 520),    # CTA-pair kernel
    (T, gen.F16, gen.F16, gen.ROW_MAJOR, 259, 515, 200),
    (T, gen.I8, gen.I32, gen.ROW_MAJOR, 259, 515, 1100),
    (K_, gen.BF16, gen.BF16, gen.COL_MAJOR, 1, 1000, 1024),
    (K_, gen.BF16, gen.F32, gen.COL_MAJOR, 16, 96, 256),
    (K_, gen.F16, gen.F16, gen.COL_MAJOR, 8, 333, 520),
    (GEN, gen.F32, gen.F32, gen.ROW_MAJOR, 70, 45, 50),
    (GEN, gen.I8, gen.I32, gen.COL_MAJOR, 70, 45, 50),
])
@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_bias_every_family(path, in_dtype, out_dtype, layout_b, M, N, K, beta):
    if in_dtype == gen.I8:
        beta = int(beta * 4)
    check_general(path, in_dtype, out_dtype, gen.ROW_MAJOR, layout_b, M, N, K, 1.0, beta,
                  with_bias=True)


@pytest.mark.parametrize("in_dtype", [gen.F32, gen.BF16])
@pytest.mark.parametrize("alpha,K", [(0.0, 64), (1.0, 0)])
def test_bias_without_product(in_dtype, alpha, K):
    # alpha == 0 or K == 0: C <- beta*C + bias, which only the generic family
    # runs (AUTO picks it; a forced fast family is refused)
    # (pad = 1 keeps every leading dimension >= 1 when K == 0)
    check_general(dga.PATH_AUTO, in_dtype, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, 130, 140, K,
                  alpha, 0.5, pad=1)
    assert dga.dga_last_path() == GEN
    A, B, C, bias = _operands(in_dtype, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, 130, 140, K, 0,
                              True, pad=1)
    run_general(T if in_dtype == gen.BF16 else S, in_dtype, gen.F32, gen.ROW_MAJOR,
                gen.ROW_MAJOR, 130, 140, K, A, B, C, bias, alpha, 0.5, expect=dga.ERR_PATH)


# ------------------------------------------------- fully-connected layer --

FC_SHAPES = [(256, 1024, 512), (200, 300, 264), (1, 512, 256), (1000, 520, 776)]


@pytest.mark.parametrize("batch,n_in,n_out", FC_SHAPES)
@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_linear_forward_backward(batch, n_in, n_out, dtype):
    """Y = X W^T + b; dX = G W; dW = G^T X; db = the batch sum of G -- each
    element against the oracle on the same operands."""
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(batch + n_in)
    X = gen.random_matrix((batch, n_in), dtype, g)
    W = gen.random_matrix((n_out, n_in), dtype, g)
    b = gen.random_matrix((1, n_out), dtype, g).reshape(n_out)
    G = gen.random_matrix((batch, n_out), dtype, g)
    Xd, Wd, bd, Gd = (t.to(dev) for t in (X, W, b, G))

    Y = dga.linear_forward(Xd, Wd, bd)
    dX, dW, db = dga.linear_backward(Xd, Wd, Gd)
    torch.cuda.synchronize()

    # forward: A = X row-major, B = W^T (column-major, stored as W)
    ref, bound = oracle.gemm_fp_ex(dtype, dtype, gen.ROW_MAJOR, gen.COL_MAJOR, batch, n_out, n_in,
                                   1.0, X, n_in, W, n_in, 0.0, None, n_out, b)
    assert_close(Y.cpu(), ref, bound, dtype, "forward")
    # dX = G W: both row-major
    ref, bound = oracle.gemm_fp_ex(dtype, dtype, gen.ROW_MAJOR, gen.ROW_MAJOR, batch, n_in, n_out,
                                   1.0, G, n_out, W, n_in, 0.0)
    assert_close(dX.cpu(), ref, bound, dtype, "dX")
    # dW = G^T X: A = G^T column-major (stored as G), B = X row-major
    ref, bound = oracle.gemm_fp_ex(dtype, dtype, gen.COL_MAJOR, gen.ROW_MAJOR, n_out, n_in, batch,
                                   1.0, G, n_out, X, n_in, 0.0)
    assert_close(dW.cpu(), ref, bound, dtype, "dW")
    ref, bound = oracle.sum_rows(dtype, batch, n_out, G)
    assert_close(db.cpu(), ref, bound, gen.F32, "db")


# ------------------------------------------------------------- sum_rows --

@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16, gen.F16])
@pytest.mark.parametrize("rows,cols", [(1, 1), (0, 40), (7, 33), (1000, 4099), (8192, 64),
                                       (4097, 520)])
@pytest.mark.parametrize("aligned_ld", [False, True])
def test_sum_rows(dtype, rows, cols, aligned_ld):
    # aligned_ld: rows start on 16-byte boundaries (whole 16-byte loads, with
    # element-wise loads only for the ragged last columns); else every load
    # is element-wise
    g = torch.Generator().manual_seed(rows * 7 + cols)
    ldg = (cols + 7) // 8 * 8 if aligned_ld else cols + 5
    Gh = gen.random_matrix((max(rows, 1), ldg), dtype, g)
    out = torch.full((cols,), float("nan"), device="cuda")
    st = dga.dga_sum_rows(dtype, rows, cols, Gh.cuda().data_ptr(), ldg, out.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert st == dga.OK
    torch.cuda.synchronize()
    ref, bound = oracle.sum_rows(dtype, rows, cols, Gh, ldg)
    assert_close(out.cpu(), ref, bound, gen.F32, f"sum_rows {rows}x{cols}")


def test_sum_rows_deterministic():
    g = torch.Generator().manual_seed(9)
    Gd = gen.random_matrix((4096, 1000), gen.F32, g).cuda()
    first = dga.sum_rows(Gd).clone()
    for _ in range(3):
        assert torch.equal(dga.sum_rows(Gd), first)


def test_linear_full_size_sampled():
    """The bf16 fully-connected step at batch 8192, 8192 -> 8192 (the size the
    benchmark times, through the same calls): sampled rows and columns of Y,
    dX and dW against the oracle on the matching sub-problems, and every
    element of db."""
    dev = torch.device("cuda")
    b = n_in = n_out = 8192
    g = torch.Generator(device=dev).manual_seed(11)
    X = (torch.randn(b, n_in, generator=g, device=dev)).to(torch.bfloat16)
    W = (torch.randn(n_out, n_in, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    bias = (torch.randn(n_out, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    G = (torch.randn(b, n_out, generator=g, device=dev)).to(torch.bfloat16)
    Y = dga.linear_forward(X, W, bias)
    dX, dW, db = dga.linear_backward(X, W, G)
    torch.cuda.synchronize()
    pick = torch.Generator().manual_seed(12)
    rows = torch.cat([torch.tensor([0, 8191]), torch.randint(0, 8192, (14,), generator=pick)])
    cols = torch.cat([torch.tensor([0, 8191]), torch.randint(0, 8192, (62,), generator=pick)])
    Xh, Wh, Gh = X.cpu(), W.cpu(), G.cpu()
    BF = gen.BF16
    # Y[rows, cols] = X[rows] W[cols]^T + bias[cols]
    ref, bound = oracle.gemm_fp_ex(BF, BF, gen.ROW_MAJOR, gen.COL_MAJOR, len(rows), len(cols), n_in,
                                   1.0, Xh[rows], n_in, Wh[cols], n_in, 0.0, None, len(cols),
                                   bias.cpu()[cols])
    assert_close(Y.cpu()[rows][:, cols], ref, bound, BF, "Y sampled")
    # dX[rows, cols] = G[rows] W[:, cols]
    ref, bound = oracle.gemm_fp_ex(BF, BF, gen.ROW_MAJOR, gen.ROW_MAJOR, len(rows), len(cols),
                                   n_out, 1.0, Gh[rows], n_out, Wh[:, cols].contiguous(), len(cols),
                                   0.0)
    assert_close(dX.cpu()[rows][:, cols], ref, bound, BF, "dX sampled")
    # dW[rows, cols] = G[:, rows]^T X[:, cols]: A = G[:, rows] stored batch x len(rows)
    ref, bound = oracle.gemm_fp_ex(BF, BF, gen.COL_MAJOR, gen.ROW_MAJOR, len(rows), len(cols), b,
                                   1.0, Gh[:, rows].contiguous(), len(rows),
                                   Xh[:, cols].contiguous(), len(cols), 0.0)
    assert_close(dW.cpu()[rows][:, cols], ref, bound, BF, "dW sampled")
    ref, bound = oracle.sum_rows(BF, b, n_out, Gh)
    assert_close(db.cpu(), ref, bound, gen.F32, "db")
