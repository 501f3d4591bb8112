"""Shared test helpers: run the GPU path through the C ABI and compare with
the CPU oracle element by element.

Acceptance (per element, computed by the oracle in fp64):
  * integer work and integer-valued floating-point cases: bit-exact;
  * otherwise |C_gpu - ref| <= 1e-4 * sum_k |alpha*a_ik*b_kj| + |beta*c_ij| * 2^-22,
    plus one output-rounding ulp of ref when the output is bf16 or fp16 (both
    ulp terms, and the roundings exact cases must match, come from the oracle).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen

TORCH = gen.TORCH_DTYPE


def run_gpu(path, in_dtype, out_dtype, layout_b, A, B, C, alpha, beta, lda=None, ldb=None,
            ldc=None, M=None, N=None, K=None, offsets=(0, 0, 0), expect=dga.OK, workspace=True):
    """Copy host buffers to the GPU, call dga_gemm_ex through the C ABI and
    return C as a host tensor (same shape as the host C buffer).

    A, B, C are host tensors holding the matrices with their leading
    dimensions (lda = A.shape[1] unless given, and so on).  `offsets` shifts
    each device pointer by that many elements (to test unaligned pointers)."""
    dev = torch.device("cuda")
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    lda = A.shape[1] if lda is None else lda
    if layout_b == gen.COL_MAJOR:
        N = B.shape[0] if N is None else N
    else:
        N = B.shape[1] if N is None else N
    ldb = B.shape[1] if ldb is None else ldb
    ldc = C.shape[1] if ldc is None else ldc

    def to_dev(t, off):
        flat = t.reshape(-1)
        buf = torch.empty(flat.numel() + off + 16, dtype=t.dtype, device=dev)
        buf[off:off + flat.numel()].copy_(flat)
        return buf, buf.data_ptr() + off * t.element_size()

    Ab, a_ptr = to_dev(A, offsets[0])
    Bb, b_ptr = to_dev(B, offsets[1])
    Cb, c_ptr = to_dev(C, offsets[2])
    ws_bytes = dga.dga_gemm_workspace_size(in_dtype, out_dtype, layout_b, M, N, K, lda, ldb, ldc,
                                           path)
    # the size query assumes aligned pointers; packing never needs more than
    # one M x K and one N x K copy of 16-bit (or, for TF32, 32-bit) elements,
    # plus alignment
    ws_bytes = max(ws_bytes, 4 * (M + N) * ((K + 7) // 8 * 8) + 1024)
    if not workspace:
        ws_bytes = 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al = dga.scalar(alpha, in_dtype)
    be = dga.scalar(beta, in_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_ex(in_dtype, out_dtype, layout_b, M, N, K, ctypes.byref(al), a_ptr, lda,
                         b_ptr, ldb, ctypes.byref(be), c_ptr, ldc,
                         ws.data_ptr() if ws_bytes else None, ws_bytes, path, stream)
    assert st == expect, f"dga_gemm_ex returned {st} ({dga.dga_status_string(st)})"
    sync = dga.dga_sync_status(stream)
    assert sync == dga.OK, dga.dga_status_string(sync)
    out = Cb[offsets[2]:offsets[2] + C.numel()].reshape(C.shape).cpu()
    return out


def oracle_ref(in_dtype, out_dtype, layout_b, A, B, C, alpha, beta, M=None, N=None, K=None,
               lda=None, ldb=None, ldc=None):
    M = A.shape[0] if M is None else M
    K = A.shape[1] if K is None else K
    N = (B.shape[0] if layout_b == gen.COL_MAJOR else B.shape[1]) if N is None else N
    lda = A.shape[1] if lda is None else lda
    ldb = B.shape[1] if ldb is None else ldb
    ldc = C.shape[1] if ldc is None else ldc
    if in_dtype == gen.I8:
        return oracle.gemm_i8(layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc), None
    return oracle.gemm_fp(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta,
                          C, ldc)


def as_f64(t):
    return t.double().numpy() if t.dtype != torch.int32 else t.numpy()


def assert_close(got, ref, bound, out_dtype, what=""):
    """Element-wise acceptance against the oracle's bound."""
    g = got.double().numpy()
    tol = bound.copy()
    if out_dtype == gen.BF16:
        tol = tol + oracle.ulp_bf16(ref)
    elif out_dtype == gen.F16:
        tol = tol + oracle.ulp_f16(ref)
    err = np.abs(g - ref)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.nanargmax(np.where(bad, err - tol, -np.inf))
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside the bound; first {idx.tolist()}; "
            f"worst excess {(err - tol).ravel()[worst]:.3e} at flat {worst} "
            f"(got {g.ravel()[worst]!r}, ref {ref.ravel()[worst]!r}, tol {tol.ravel()[worst]:.3e})")


def assert_exact(got, ref, out_dtype, what=""):
    """Bit-exact: got equals ref rounded once to the output type."""
    if out_dtype == gen.I32:
        want = ref.astype(np.int32)
        ok = np.array_equal(got.numpy(), want)
        if not ok:
            bad = np.argwhere(got.numpy() != want)[:5]
            raise AssertionError(f"{what}: int32 mismatch at {bad.tolist()}")
        return
    if out_dtype == gen.F32:
        want = ref.astype(np.float32)
        gotn = got.numpy()
    elif out_dtype == gen.BF16:
        want = oracle.round_bf16(ref)
        gotn = got.view(torch.int16).numpy().view(np.uint16)
    else:
        want = oracle.round_f16(ref)
        gotn = got.view(torch.int16).numpy().view(np.uint16)
    if not np.array_equal(gotn, want):
        bad = np.argwhere(gotn != want)[:5]
        raise AssertionError(f"{what}: not bit-exact at {bad.tolist()}")
