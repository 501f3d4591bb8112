"""GPU parity of the INT8 tensor-core path a few tiles past one wave of
clusters, through the C ABI, bit for bit against the int64 CPU oracle.

On the CTA-pair kernel (M > 128) each cluster of two CTAs walks 256 x 256
tiles; the shapes here hold a few tiles more than one wave of clusters (76
on a GB300), so that most clusters take one tile and a few take two, with K
of one 64-deep K block, of a ragged 1000 and of 1024 and 2048 (one and two
exact 1024-deep chunks), alpha, beta and a bias row, including values that
wrap modulo 2^32.  Integer sums in any order are exact (mod 2^32), so the
result must equal the oracle's exactly: the BLAS update of "AI Programming:
Matrix Product", section "Dense matrix multiplication", with the bias row of
its section "Fully-connected layer".
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

T = dga.PATH_TCGEN05


def _clusters():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def _shape(K):
    # tile rows x tile columns of 256: a few tiles past one wave of clusters
    cl = _clusters()
    rows = 10
    cols = -(-(cl + 4) // rows)  # ceil
    return rows * 256 - 60, cols * 256 - 56, K


def _run(layout_a, layout_b, M, N, K, A, B, C, bias, alpha, beta):
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    bd = bias.to(dev) if bias is not None else None
    lda, ldb, ldc = A.shape[1], B.shape[1], C.shape[1]
    ws_bytes = dga.dga_gemm_general_workspace_size(gen.I8, gen.I32, layout_a, layout_b, M, N, K,
                                                   lda, ldb, ldc, T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = ctypes.c_int32(alpha), ctypes.c_int32(beta)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_general(gen.I8, gen.I32, layout_a, layout_b, M, N, K, ctypes.byref(al),
                              Ad.data_ptr(), lda, Bd.data_ptr(), ldb, ctypes.byref(be),
                              Cd.data_ptr(), ldc, bd.data_ptr() if bd is not None else None,
                              ws.data_ptr() if ws_bytes else None, ws_bytes, T, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    assert dga.dga_last_path() == T
    return Cd.cpu()


def _operands(layout_a, layout_b, M, N, K, seed, extreme=False):
    g = torch.Generator().manual_seed(seed)
    a_shape = (M, K) if layout_a == gen.ROW_MAJOR else (K, M)
    b_shape = (K, N) if layout_b == gen.ROW_MAJOR else (N, K)
    if extreme:
        A = torch.full(a_shape, -128, dtype=torch.int8)
        B = torch.full(b_shape, -128, dtype=torch.int8)
    else:
        A = torch.randint(-128, 128, a_shape, generator=g, dtype=torch.int8)
        B = torch.randint(-128, 128, b_shape, generator=g, dtype=torch.int8)
    C = torch.randint(-2**31, 2**31, (M, N), generator=g, dtype=torch.int64).to(torch.int32)
    bias = torch.randint(-2**31, 2**31, (N,), generator=g, dtype=torch.int64).to(torch.int32)
    return A, B, C, bias


@pytest.mark.parametrize("K", [64, 1000, 1024])
@pytest.mark.parametrize("alpha,beta,with_bias", [(1, 0, False), (-3, 2, True),
                                                   (1 << 20, 1 << 30, True)])
def test_int8_past_one_wave_exact(K, alpha, beta, with_bias):
    M, N, K = _shape(K)
    tiles = -(-M // 256) * -(-N // 256)
    assert tiles % _clusters() != 0, "the shape must leave a part-filled last wave"
    A, B, C, bias = _operands(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, seed=K + alpha)
    bias = bias if with_bias else None
    got = _run(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, A, B, C, bias, alpha, beta)
    want = oracle.gemm_i8_ex(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, alpha, A, K, B, N, beta, C,
                             N, bias)
    assert np.array_equal(got.numpy(), want)


@pytest.mark.parametrize("layouts", [(gen.ROW_MAJOR, gen.COL_MAJOR), (gen.COL_MAJOR, gen.ROW_MAJOR),
                                     (gen.COL_MAJOR, gen.COL_MAJOR)], ids=["rc", "cr", "cc"])
def test_int8_past_one_wave_layouts(layouts):
    la, lb = layouts
    M, N, K = _shape(1000)
    A, B, C, bias = _operands(la, lb, M, N, K, seed=3)
    got = _run(la, lb, M, N, K, A, B, C, bias, 5, -1)
    want = oracle.gemm_i8_ex(la, lb, M, N, K, 5, A, A.shape[1], B, B.shape[1], -1, C, N, bias)
    assert np.array_equal(got.numpy(), want)


def test_int8_past_one_wave_largest_products():
    # every product 2^14, K = 2048: each 1024-deep chunk sums to 2^24, the
    # largest exact fp32 integer, and the two chunks then meet in int32
    M, N, K = _shape(2048)
    A, B, C, _ = _operands(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, seed=0, extreme=True)
    got = _run(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, A, B, C, None, 1, 0)
    assert (got == 2048 * 16384).all()


def test_int8_past_one_wave_repeats():
    M, N, K = _shape(1024)
    A, B, C, bias = _operands(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, seed=11)
    first = _run(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, A, B, C, bias, 7, 3)
    for _ in range(4):
        assert torch.equal(_run(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, A, B, C, bias, 7, 3), first)


@pytest.mark.parametrize("K,layout_b", [(131072, gen.COL_MAJOR), (131072, gen.ROW_MAJOR),
                                         (139264, gen.COL_MAJOR)])
def test_int8_at_the_largest_k(K, layout_b):
    # K = 2^17 with every entry -128: each product is 2^14 and a full dot
    # product 2^31, one past the int32 range, so it wraps to -2^31 (the
    # 1024-deep chunks stay exact in fp32; their int32 sum wraps).  Beside
    # it, sums just inside the range: row 1 has one +127 (2^31 - 2^14 -
    # 16256), column 3 of B one +1 (2^31 - 2^14 - 128), row 2 is all +127
    # (-16256 * 2^17).  K = 139264 (136 chunks) goes further past the range.
    # Every element is checked against the oracle's int64 sum reduced mod
    # 2^32.  Two tile rows on the CTA-pair kernel (M = 260, the second
    # ragged), alpha = 1, beta = 0
    M, N = 260, 130
    A = torch.full((M, K), -128, dtype=torch.int8)
    A[1, 5] = 127
    A[2, :] = 127
    B = torch.full((N, K) if layout_b == gen.COL_MAJOR else (K, N), -128, dtype=torch.int8)
    if layout_b == gen.COL_MAJOR:
        B[3, 7] = 1
    else:
        B[7, 3] = 1
    C = torch.zeros(M, N, dtype=torch.int32)
    got = _run(gen.ROW_MAJOR, layout_b, M, N, K, A, B, C, None, 1, 0)
    ref = oracle.gemm_i8_ex(gen.ROW_MAJOR, layout_b, M, N, K, 1, A, K, B, B.shape[1], 0, C, N,
                            None)
    assert np.array_equal(got.numpy(), ref.astype(np.int32)), \
        f"K={K}: mismatch at {np.argwhere(got.numpy() != ref.astype(np.int32))[:5].tolist()}"
    if K == 131072:
        assert int(got[0, 0]) == -(2 ** 31)  # (-128)(-128) 2^17 times = 2^31, wrapped
