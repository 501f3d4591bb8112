"""FP16 output at the edge of its range, through the C ABI, bit for bit.

Every output is an exact fp32 sum of power-of-two fp16 products chosen so
that the one rounding to fp16 decides: 65504 (the largest finite value),
65519 (rounds down to it), 65520 (the tie between 65504 and 65536: to even,
i.e. past the range, +inf), their negatives, 2^17 (far past: inf) and
small values.  The oracle rounds the same exact sums once
(round-to-nearest-even, overflow to infinity), so the bits must agree, on
the generic kernel, the single-CTA and CTA-pair tcgen05 kernels and the
split last wave's reduce.  The output conversion is the rounding of "AI
Programming: Matrix Product", section "Dense matrix multiplication" (the
BLAS update C <- alpha A B + beta C in the output type).
"""
import ctypes

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_exact

pytestmark = pytest.mark.gpu

TARGETS = [65504, 65519, 65520, -65504, -65519, -65520, 1 << 17, -(1 << 17), 3, -5, 0, 2047]


def _powers(x):
    """x as a sum of distinct powers of two (exact in fp16 each)."""
    s = -1 if x < 0 else 1
    x = abs(x)
    return [s * (1 << b) for b in range(20) if x >> b & 1]


def _problem(M, N, K):
    """A (M x K) with row i holding the binary digits of TARGETS[i % len] in its
    first columns, B (N x K, column-major) all ones in those columns (so every
    column of row i sums to the target), the rest zero."""
    A = torch.zeros(M, K, dtype=torch.float16)
    for i in range(M):
        for k, p in enumerate(_powers(TARGETS[i % len(TARGETS)])):
            A[i, k] = p
    B = torch.zeros(N, K, dtype=torch.float16)
    B[:, :20] = 1.0
    return A, B


def _run(path, M, N, K, A, B):
    dev = torch.device("cuda")
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = torch.full((M, N), 7.0, dtype=torch.float16, device=dev)  # beta = 0: never read
    ws_bytes = dga.dga_gemm_workspace_size(gen.F16, gen.F16, gen.COL_MAJOR, M, N, K, K, K, N,
                                           path)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = ctypes.c_float(1.0), ctypes.c_float(0.0)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_ex(gen.F16, gen.F16, gen.COL_MAJOR, M, N, K, ctypes.byref(al), Ad.data_ptr(),
                         K, Bd.data_ptr(), K, ctypes.byref(be), Cd.data_ptr(), N,
                         ws.data_ptr() if ws_bytes else None, ws_bytes, path, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    assert dga.dga_last_path() == path
    return Cd.cpu(), dga.dga_last_launch_count()


@pytest.mark.parametrize("path,M,N,K", [
    (dga.PATH_GENERIC, 40, 33, 64),
    (dga.PATH_TCGEN05, 100, 300, 64),       # single-CTA kernel (M <= 128)
    (dga.PATH_TCGEN05, 300, 520, 128),      # CTA-pair kernel, ragged edges
    (dga.PATH_TCGEN05, 2560, 2048, 1024),   # CTA pairs with the split last wave (80 tiles)
])
def test_f16_output_range(path, M, N, K):
    A, B = _problem(M, N, K)
    got, launches = _run(path, M, N, K, A, B)
    if M == 2560 and torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert launches == 2  # the GEMM and the split's reduce
    ref, _ = oracle.gemm_fp(gen.F16, gen.F16, gen.COL_MAJOR, M, N, K, 1.0, A, K, B, K, 0.0)
    assert_exact(got, ref, gen.F16, f"f16 range {M}x{N}x{K}")
    g = got.float()
    assert torch.isinf(g[2]).all() and (g[2] > 0).all()        # 65520 ties up to +inf
    assert (g[1] == 65504).all() and (g[0] == 65504).all()     # 65519 rounds down
    assert torch.isinf(g[5]).all() and (g[5] < 0).all()
