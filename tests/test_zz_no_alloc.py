"""dga_gemm_i8_noalloc, the INT8 entry point that allocates nothing.

Some callers cannot hand the library a workspace: a plugin that receives only
its input and output buffers from the host application, or an engine that
reserves all device memory at start-up and refuses allocations afterwards.
For them dga_gemm_i8_noalloc runs the INT8 tensor-core GEMM with a fixed
scratch area compiled into the library.  These tests call it through the C
ABI and require its output to equal, bit for bit, what dga_gemm computes with
a caller workspace -- on two different calls in a row, so the second call
also shows that leftovers of the first in the shared scratch do not matter.

This file is collected last on purpose; it must also pass on its own in a
fresh process.
"""
import ctypes

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _problem(M, N, K, layout, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (N, K) if layout == gen.COL_MAJOR else (K, N), generator=g,
                      dtype=torch.int8)
    C = torch.randint(-1000, 1000, (M, N), generator=g, dtype=torch.int32)
    return A.cuda(), B.cuda(), C.cuda()


def _lds(layout, M, N, K):
    return K, (K if layout == gen.COL_MAJOR else N), N


def _run_noalloc(layout, A, B, C, alpha, beta):
    M, K = A.shape
    N = C.shape[1]
    lda, ldb, ldc = _lds(layout, M, N, K)
    al, be = ctypes.c_int32(alpha), ctypes.c_int32(beta)
    return dga.dga_gemm_i8_noalloc(layout, M, N, K, ctypes.byref(al), A.data_ptr(), lda,
                                   B.data_ptr(), ldb, ctypes.byref(be), C.data_ptr(), ldc,
                                   torch.cuda.current_stream().cuda_stream)


def _run_regular(layout, A, B, C, alpha, beta):
    M, K = A.shape
    N = C.shape[1]
    lda, ldb, ldc = _lds(layout, M, N, K)
    ws_bytes = dga.dga_gemm_workspace_size(gen.I8, gen.I32, layout, M, N, K, lda, ldb, ldc,
                                           dga.PATH_TCGEN05)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    al, be = ctypes.c_int32(alpha), ctypes.c_int32(beta)
    return dga.dga_gemm(gen.I8, gen.I32, layout, M, N, K, ctypes.byref(al), A.data_ptr(), lda,
                        B.data_ptr(), ldb, ctypes.byref(be), C.data_ptr(), ldc, ws.data_ptr(),
                        ws_bytes, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("first,second", [
    ((1000, 777, 1500, gen.ROW_MAJOR, 1, 0), (4093, 4099, 4096, gen.ROW_MAJOR, 1, 0)),
    ((300, 2600, 2056, gen.COL_MAJOR, -3, 2), (131, 67, 520, gen.ROW_MAJOR, 5, -1)),
])
def test_noalloc_matches_dga_gemm_on_two_calls(first, second):
    for seed, (M, N, K, layout, alpha, beta) in enumerate((first, second)):
        A, B, C0 = _problem(M, N, K, layout, seed)
        C_noalloc = C0.clone()
        C_regular = C0.clone()
        assert _run_noalloc(layout, A, B, C_noalloc, alpha, beta) == dga.OK
        assert _run_regular(layout, A, B, C_regular, alpha, beta) == dga.OK
        assert dga.dga_sync_status(torch.cuda.current_stream().cuda_stream) == dga.OK
        assert torch.equal(C_noalloc, C_regular), f"call {seed + 1}: outputs differ"


def test_noalloc_refuses_sizes_beyond_its_scratch():
    # bf16-encoded operands, both K-major: A takes M * K * 2 bytes, B
    # N * K * 2 (K a multiple of 8); 5200 * 4096 * 2 + 4099 * 4096 * 2 > 72 MiB
    M, N, K = 5200, 4099, 4096
    assert M * K * 2 + N * K * 2 > dga.NOALLOC_SCRATCH_BYTES
    A, B, C = _problem(M, N, K, gen.ROW_MAJOR, 7)
    before = C.clone()
    assert _run_noalloc(gen.ROW_MAJOR, A, B, C, 1, 0) == dga.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(C, before), "a refused call must not touch C"


def test_noalloc_argument_errors_use_its_own_positions():
    A, B, C = _problem(8, 8, 8, gen.ROW_MAJOR, 1)
    one = ctypes.c_int32(1)
    s = torch.cuda.current_stream().cuda_stream
    assert dga.dga_gemm_i8_noalloc(gen.ROW_MAJOR, -1, 8, 8, ctypes.byref(one), A.data_ptr(), 8,
                                   B.data_ptr(), 8, ctypes.byref(one), C.data_ptr(), 8, s) == -2
    assert dga.dga_gemm_i8_noalloc(gen.ROW_MAJOR, 8, 8, 8, ctypes.byref(one), A.data_ptr(), 4,
                                   B.data_ptr(), 8, ctypes.byref(one), C.data_ptr(), 8, s) == -7
