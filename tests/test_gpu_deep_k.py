"""GPU parity at a very deep K, through the C ABI, on sampled elements.

K = 2^20 with 2560 x 2048 outputs: on the FP32 SIMT path that is 65536
16-deep slices per 128 x 256 tile and a stream-K remainder of 8 tiles whose
(tile, slice) units number 2^19 (the wide kernels' 32-bit slice loop and
their 64-bit unit arithmetic); on the BF16 tensor-core path 16384 k-blocks
per tile and a last wave of 4 tiles cut into 4 parts of 4096 k-blocks.  The
inputs are drawn on the device; 512 sampled elements are checked against the
oracle, which is given only the sampled rows of A and columns of B (sample s
is row s of the one and column s of the other).  The GEMM is the BLAS update
of "AI Programming: Matrix Product", section "Dense matrix multiplication".
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

M, N, K = 2560, 2048, 1 << 20
SAMPLES = 512


@pytest.mark.parametrize("in_dtype,path", [(gen.F32, dga.PATH_SIMT),
                                           (gen.BF16, dga.PATH_TCGEN05)])
def test_deep_k_sampled(in_dtype, path):
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(17)
    tdt = torch.float32 if in_dtype == gen.F32 else torch.bfloat16
    A = (torch.rand(M, K, device=dev, generator=g) * 2 - 1).to(tdt)
    # B column-major (N x K) on the tensor path, row-major (K x N) on the SIMT one
    if in_dtype == gen.F32:
        B = torch.rand(K, N, device=dev, generator=g) * 2 - 1
        layout_b, ldb = gen.ROW_MAJOR, N
    else:
        B = (torch.rand(N, K, device=dev, generator=g) * 2 - 1).to(tdt)
        layout_b, ldb = gen.COL_MAJOR, K
    C = torch.empty(M, N, device=dev)
    ws_bytes = dga.dga_gemm_workspace_size(in_dtype, gen.F32, layout_b, M, N, K, K, ldb, N, path)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = ctypes.c_float(1.0), ctypes.c_float(0.0)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_ex(in_dtype, gen.F32, layout_b, M, N, K, ctypes.byref(al), A.data_ptr(), K,
                         B.data_ptr(), ldb, ctypes.byref(be), C.data_ptr(), N,
                         ws.data_ptr() if ws_bytes else None, ws_bytes, path, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    assert dga.dga_last_path() == path
    # the stream-K remainder (3 launches) or the split last wave (2)
    assert dga.dga_last_launch_count() == (3 if path == dga.PATH_SIMT else 2)
    rng = np.random.default_rng(5)
    rows = rng.integers(0, M, SAMPLES)
    cols = rng.integers(0, N, SAMPLES)
    got = C[torch.as_tensor(rows, device=dev), torch.as_tensor(cols, device=dev)].cpu()
    a_rows = A[torch.as_tensor(rows, device=dev)].cpu()                    # SAMPLES x K
    if layout_b == gen.ROW_MAJOR:
        b_cols = B[:, torch.as_tensor(cols, device=dev)].cpu().contiguous()  # K x SAMPLES
    else:
        b_cols = B[torch.as_tensor(cols, device=dev)].cpu()                  # SAMPLES x K
    idx = np.arange(SAMPLES)
    ref, bound = oracle.gemm_fp_sampled(in_dtype, gen.F32, layout_b, K, 1.0, a_rows, K, b_cols,
                                        SAMPLES if layout_b == gen.ROW_MAJOR else K, 0.0, None,
                                        None, idx, idx)
    assert_close(got, ref, bound, gen.F32, f"deep K {in_dtype}")
