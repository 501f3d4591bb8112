"""The FP32 FMA-rate probe does the work it reports.

The probe's FLOP count is what the FP32 roofline peak is cross-checked
against, so its outputs are checked bit for bit: each thread's 8 chains of
a <- fma(a, m, b) are replayed in numpy.  An fp32 fused multiply-add is the
exact a*m + b rounded once to fp32; with a near 1, m = 1 + 2^-23 and
b = 1e-7f the exact value fits in a double (a*m has 48 significant bits and
b's bits lie within them), so float32(double(a)*m + b) is that single
rounding.  The chains start at fmaf(1e-3f, t, 1) (t = thread + chain), exact
in a double for the same reason.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga

pytestmark = pytest.mark.gpu

THREADS, CTAS_PER_SM, CHAINS, FMA_PER_ITER = 256, 4, 8, 64


def _fma32(a, m, b):
    return (np.asarray(a, np.float64) * np.asarray(m, np.float64) + np.float64(b)).astype(np.float32)


def _expected(packed, iters, n_threads):
    tid = (np.arange(n_threads) % THREADS).astype(np.float32)
    m, b = np.float32(1.0000001), np.float32(1e-7)
    steps = iters * FMA_PER_ITER // (2 * CHAINS if packed else CHAINS)
    s = np.zeros(n_threads, dtype=np.float32)
    for c in range(CHAINS):
        lo = _fma32(np.float32(1e-3) * np.ones_like(tid), tid + np.float32(c), 1.0)
        chains = [lo, lo + np.float32(0.5)] if packed else [lo]
        for _ in range(steps):
            chains = [_fma32(a, m, b) for a in chains]
        s = s + (chains[0] + chains[1] if packed else chains[0])
    return s


@pytest.mark.parametrize("packed", [0, 1])
def test_probe_outputs_and_flops(packed):
    n = dga.dga_probe_fp32_fma_out_floats()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n == sms * CTAS_PER_SM * THREADS
    out = torch.full((n,), float("nan"), device="cuda")
    flops = ctypes.c_double(0.0)
    iters = 3
    s = torch.cuda.current_stream().cuda_stream
    assert dga.dga_probe_fp32_fma(packed, iters, out.data_ptr(), n, ctypes.byref(flops), s) == dga.OK
    assert dga.dga_sync_status(s) == dga.OK
    assert flops.value == 2.0 * n * iters * FMA_PER_ITER
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got, _expected(packed, iters, n))
    assert dga.dga_probe_fp32_fma(packed, iters, out.data_ptr(), n - 1, ctypes.byref(flops), s) == -4


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (67, 53, 45), (130, 257, 300)])
def test_naive_probe_matches_the_oracle(M, N, K):
    # the counter-calibration kernel computes C = A * B: exact on small
    # integers (all partial sums below 2^24), within the oracle's bound on
    # uniform inputs
    import oracle
    from dense_gemm_accelerator_gb300 import inputs as gen
    from tests.helpers import assert_close, assert_exact
    g = torch.Generator().manual_seed(M + N + K)
    s = torch.cuda.current_stream().cuda_stream
    for small in (True, False):
        if small:
            A = gen.small_int_matrix((M, K), gen.F32, g)
            B = gen.small_int_matrix((K, N), gen.F32, g)
        else:
            A = gen.random_matrix((M, K), gen.F32, g)
            B = gen.random_matrix((K, N), gen.F32, g)
        Ad, Bd = A.cuda(), B.cuda()
        C = torch.full((M, N), float("nan"), device="cuda")
        assert dga.dga_probe_naive_sgemm(M, N, K, Ad.data_ptr(), Bd.data_ptr(), C.data_ptr(), s) == dga.OK
        assert dga.dga_sync_status(s) == dga.OK
        ref, bound = oracle.gemm_fp(gen.F32, gen.F32, gen.ROW_MAJOR, M, N, K, 1.0, A, K, B, N, 0.0)
        if small:
            assert_exact(C.cpu(), ref, gen.F32, f"naive {M}x{N}x{K} small integers")
        else:
            assert_close(C.cpu(), ref, bound, gen.F32, f"naive {M}x{N}x{K}")


@pytest.mark.parametrize("iters", [1, 37])
def test_int8_mma_probe_outputs_and_ops(iters):
    # every lane of warp w holds A bytes c = w % 5 + 1 and B bytes -2: each
    # m16n8k32 step adds 32 * c * (-2) to each of a thread's 8 x 4
    # accumulators, whatever the fragment layout, so thread t ends at
    # -2048 * c * iters; the op count is 8 chains x 2*16*8*32 per warp and step
    n = dga.dga_probe_fp32_fma_out_floats()
    out = torch.full((n,), 12345, dtype=torch.int32, device="cuda")
    ops = ctypes.c_double(0.0)
    stream = torch.cuda.current_stream().cuda_stream
    assert dga.dga_probe_int8_mma(iters, out.data_ptr(), n, ctypes.byref(ops), stream) == dga.OK
    assert dga.dga_sync_status(stream) == dga.OK
    warp = np.arange(n) // 32
    want = -2048 * (warp % 5 + 1) * iters
    assert np.array_equal(out.cpu().numpy(), want.astype(np.int32))
    assert ops.value == (n // 32) * iters * 8 * (2 * 16 * 8 * 32)
