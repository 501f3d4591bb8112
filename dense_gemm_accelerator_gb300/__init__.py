"""Dense GEMM on one GB300 (sm_103a): a thin Python binding of libdga.so.

Every function named ``dga_*`` here is the C entry point of the same name in
``include/dga.h``; this module only marshals arguments (ctypes).  All the
work runs in the library's CUDA kernels: there is no CPU or PyTorch compute
path, and a missing library raises instead of falling back.

:func:`gemm` is the convenience form for PyTorch tensors:
``C <- alpha * A @ B + beta * C`` on the current CUDA stream, with A and C
row-major and B row- or column-major (read from its strides).
"""
from __future__ import annotations

import ctypes
import os
import threading

from .inputs import BF16, COL_MAJOR, F16, F32, I8, I32, ROW_MAJOR, TF32  # noqa: F401  (codes)

PATH_AUTO, PATH_GENERIC, PATH_SIMT, PATH_TCGEN05, PATH_SKINNY = 0, 1, 2, 3, 4
PATH_NAMES = {PATH_AUTO: "auto", PATH_GENERIC: "generic", PATH_SIMT: "simt",
              PATH_TCGEN05: "tcgen05", PATH_SKINNY: "skinny"}

OK = 0
ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_PATH, ERR_WORKSPACE, ERR_OVERLAP, ERR_DEVICE = \
    1, 2, 3, 4, 5, 6, 7
ERR_BAD_INDEX = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdga.so")

# Symbols declared in include/dga.h, with their ctypes signatures.
_I64, _VP, _SZ, _CI = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
SIGNATURES = {
    "dga_gemm": (_CI, [_CI, _CI, _CI, _I64, _I64, _I64, _VP, _VP, _I64, _VP, _I64, _VP, _VP,
                       _I64, _VP, _SZ, _VP]),
    "dga_gemm_ex": (_CI, [_CI, _CI, _CI, _I64, _I64, _I64, _VP, _VP, _I64, _VP, _I64, _VP, _VP,
                          _I64, _VP, _SZ, _CI, _VP]),
    "dga_gemm_workspace_size": (_SZ, [_CI, _CI, _CI, _I64, _I64, _I64, _I64, _I64, _I64, _CI]),
    "dga_select_path": (_CI, [_CI, _CI, _CI, _I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64]),
    "dga_last_path": (_CI, []),
    "dga_last_launch_count": (_CI, []),
    "dga_sync_status": (_CI, [_VP]),
    "dga_last_cuda_error": (_CI, []),
    "dga_status_string": (ctypes.c_char_p, [_CI]),
    "dga_version": (_CI, []),
    "dga_selftest_bounded_wait": (_CI, [_I64, _VP]),
    "dga_gemm_general": (_CI, [_CI, _CI, _CI, _CI, _I64, _I64, _I64, _VP, _VP, _I64, _VP, _I64,
                               _VP, _VP, _I64, _VP, _VP, _SZ, _CI, _VP]),
    "dga_gemm_general_workspace_size": (_SZ, [_CI, _CI, _CI, _CI, _I64, _I64, _I64, _I64, _I64,
                                              _I64, _CI]),
    "dga_sum_rows": (_CI, [_CI, _I64, _I64, _VP, _I64, _VP, _VP]),
    "dga_gemm_i8_noalloc": (_CI, [_CI, _I64, _I64, _I64, _VP, _VP, _I64, _VP, _I64, _VP, _VP,
                                  _I64, _VP]),
    "dga_spmv_csr": (_CI, [_I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "dga_spmv_csr_workspace_size": (_SZ, [_I64, _I64]),
    "dga_probe_fp32_fma": (_CI, [_CI, _I64, _VP, _I64, _VP, _VP]),
    "dga_probe_fp32_fma_out_floats": (_I64, []),
    "dga_probe_int8_mma": (_CI, [_I64, _VP, _I64, _VP, _VP]),
    "dga_probe_naive_sgemm": (_CI, [_I64, _I64, _I64, _VP, _VP, _VP, _VP]),
}

_lock = threading.Lock()
_lib_handle = None


class DgaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = f"dga status {status}: {dga_status_string(status)}"
        if status == ERR_CUDA:
            msg += f" (cudaError {dga_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


def lib() -> ctypes.CDLL:
    """The loaded libdga.so.  Raises if it has not been built."""
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib_handle = handle
        return _lib_handle


# ---- the C entry points, same names and arguments ---------------------------

def dga_gemm(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
             workspace, workspace_bytes, stream):
    return lib().dga_gemm(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta,
                          C, ldc, workspace, workspace_bytes, stream)


def dga_gemm_ex(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                workspace, workspace_bytes, path, stream):
    return lib().dga_gemm_ex(in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb,
                             beta, C, ldc, workspace, workspace_bytes, path, stream)


def dga_gemm_general(in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                     beta, C, ldc, bias, workspace, workspace_bytes, path, stream):
    return lib().dga_gemm_general(in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, A, lda,
                                  B, ldb, beta, C, ldc, bias, workspace, workspace_bytes, path,
                                  stream)


def dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N, K, lda, ldb,
                                    ldc, path):
    return lib().dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N, K,
                                                 lda, ldb, ldc, path)


def dga_sum_rows(dtype, rows, cols, G, ldg, out, stream):
    return lib().dga_sum_rows(dtype, rows, cols, G, ldg, out, stream)


def dga_gemm_workspace_size(in_dtype, out_dtype, layout_b, M, N, K, lda, ldb, ldc, path):
    return lib().dga_gemm_workspace_size(in_dtype, out_dtype, layout_b, M, N, K, lda, ldb, ldc,
                                         path)


def dga_select_path(in_dtype, out_dtype, layout_b, M, N, K, A, lda, B, ldb, C, ldc):
    return lib().dga_select_path(in_dtype, out_dtype, layout_b, M, N, K, A, lda, B, ldb, C, ldc)


def dga_last_path():
    return lib().dga_last_path()


def dga_last_launch_count():
    return lib().dga_last_launch_count()


def dga_sync_status(stream):
    return lib().dga_sync_status(stream)


def dga_last_cuda_error():
    return lib().dga_last_cuda_error()


def dga_status_string(status):
    return lib().dga_status_string(status).decode()


def dga_version():
    return lib().dga_version()


def dga_selftest_bounded_wait(limit_ns, stream):
    return lib().dga_selftest_bounded_wait(limit_ns, stream)


NOALLOC_SCRATCH_BYTES = 72 << 20


def dga_gemm_i8_noalloc(layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream):
    return lib().dga_gemm_i8_noalloc(layout_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                     stream)


def dga_spmv_csr(rows, cols, nnz, row_offsets, column_indices, values, alpha, x, beta, y,
                 workspace, workspace_bytes, stream):
    return lib().dga_spmv_csr(rows, cols, nnz, row_offsets, column_indices, values, alpha, x,
                              beta, y, workspace, workspace_bytes, stream)


def dga_spmv_csr_workspace_size(rows, nnz):
    return lib().dga_spmv_csr_workspace_size(rows, nnz)


def dga_probe_fp32_fma(packed, iters, out, out_floats, flops, stream):
    return lib().dga_probe_fp32_fma(packed, iters, out, out_floats, flops, stream)


def dga_probe_fp32_fma_out_floats():
    return lib().dga_probe_fp32_fma_out_floats()


def dga_probe_int8_mma(iters, out, out_ints, ops, stream):
    return lib().dga_probe_int8_mma(iters, out, out_ints, ops, stream)


def dga_probe_naive_sgemm(M, N, K, A, B, C, stream):
    return lib().dga_probe_naive_sgemm(M, N, K, A, B, C, stream)


# ---- tensor convenience layer ----------------------------------------------

def _dtype_code(t):
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16, torch.int8: I8,
            torch.int32: I32}[t.dtype]


def scalar(value, in_dtype):
    """ctypes scalar for alpha/beta: int32 for INT8 inputs, else float."""
    return ctypes.c_int32(int(value)) if in_dtype == I8 else ctypes.c_float(float(value))


def _layout_of(T, name):
    """(layout, ld) of a 2-D tensor viewed as rows x cols: row-major when its
    columns are contiguous, column-major when its rows are; else an error."""
    if T.stride(1) == 1 or T.size(1) <= 1:
        return ROW_MAJOR, max(T.stride(0), max(T.size(1), 1))
    if T.stride(0) == 1:
        return COL_MAJOR, max(T.stride(1), max(T.size(0), 1))
    raise ValueError(f"{name} must be row-major or column-major")


def operand_layout(A, B, C):
    """(lda, layout_b, ldb, ldc) from tensor strides for a row-major A;
    raises on layouts the ABI cannot express (no copies are made)."""
    if A.dim() != 2 or B.dim() != 2 or C.dim() != 2:
        raise ValueError("A, B and C must be 2-D")
    if A.stride(1) != 1 and A.size(1) > 1:
        raise ValueError("A must be row-major (unit stride along K)")
    if C.stride(1) != 1 and C.size(1) > 1:
        raise ValueError("C must be row-major (unit stride along N)")
    if B.stride(1) == 1 or B.size(1) <= 1:
        layout_b, ldb = ROW_MAJOR, max(B.stride(0), max(B.size(1), 1))
    elif B.stride(0) == 1:
        layout_b, ldb = COL_MAJOR, max(B.stride(1), max(B.size(0), 1))
    else:
        raise ValueError("B must be row-major or column-major")
    lda = max(A.stride(0), max(A.size(1), 1))
    ldc = max(C.stride(0), max(C.size(1), 1))
    return lda, layout_b, ldb, ldc


def gemm(A, B, C=None, alpha=1.0, beta=0.0, out_dtype=None, path=PATH_AUTO, workspace=None,
         stream=None, bias=None, tf32=False):
    """C <- alpha * A @ B + beta * C (+ bias) on the GPU; returns C.

    A: (M, K) and B: (K, N) CUDA tensors, each row- or column-major (a
    transposed view of a contiguous tensor is column-major).  C: (M, N)
    row-major, allocated when None (then beta must be 0).  bias: optional (N,)
    tensor of C's dtype added to every row.  The workspace, when the chosen
    path needs one, is allocated from PyTorch's caching allocator unless given.
    tf32=True (fp32 A and B only) asks for the lossy TF32 tensor-core product
    (DGA_TF32); fp32 inputs are otherwise multiplied exactly in fp32.
    """
    import torch
    in_dtype = _dtype_code(A)
    if _dtype_code(B) != in_dtype:
        raise TypeError("A and B must have the same dtype")
    if tf32:
        if in_dtype != F32:
            raise TypeError("tf32=True needs fp32 A and B")
        in_dtype = TF32
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    N = B.shape[1]
    if B.shape[0] != K:
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}")
    if C is None:
        if beta != 0:
            raise ValueError("beta != 0 needs C")
        if out_dtype is None:
            out_dtype = I32 if in_dtype == I8 else (F32 if in_dtype == TF32 else in_dtype)
        C = torch.empty((M, N), dtype={F32: torch.float32, BF16: torch.bfloat16,
                                       F16: torch.float16, I32: torch.int32}[out_dtype],
                        device=A.device)
    out_dtype = _dtype_code(C)
    if tuple(C.shape) != (M, N) or C.dim() != 2 or (C.stride(1) != 1 and N > 1):
        raise ValueError(f"C must be a row-major ({M}, {N}) tensor")
    layout_a, lda = _layout_of(A, "A")
    layout_b, ldb = _layout_of(B, "B")
    ldc = max(C.stride(0), max(N, 1))
    if bias is not None:
        if bias.dim() != 1 or bias.numel() != N or bias.stride(0) != 1 or _dtype_code(bias) != out_dtype:
            raise ValueError("bias must be a contiguous (N,) tensor of C's dtype")
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    ws_bytes = dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N, K,
                                               lda, ldb, ldc, path)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=A.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_have = workspace.numel() * workspace.element_size() if workspace is not None else 0
    a = scalar(alpha, in_dtype)
    b = scalar(beta, in_dtype)
    st = dga_gemm_general(in_dtype, out_dtype, layout_a, layout_b, M, N, K, ctypes.byref(a),
                          A.data_ptr(), lda, B.data_ptr(), ldb, ctypes.byref(b), C.data_ptr(), ldc,
                          bias.data_ptr() if bias is not None else None, ws_ptr, ws_have, path,
                          stream)
    if st != OK:
        raise DgaError(st, "dga_gemm_general")
    return C


def sum_rows(G, out=None, stream=None):
    """fp32 column sums of a row-major 2-D tensor G (the batch sum of an output
    gradient); returns out."""
    import torch
    rows, cols = G.shape
    if G.stride(1) != 1 and cols > 1:
        raise ValueError("G must be row-major")
    if out is None:
        out = torch.empty(cols, dtype=torch.float32, device=G.device)
    if stream is None:
        stream = torch.cuda.current_stream(G.device).cuda_stream
    st = dga_sum_rows(_dtype_code(G), rows, cols, G.data_ptr(), max(G.stride(0), max(cols, 1)),
                      out.data_ptr(), stream)
    if st != OK:
        raise DgaError(st, "dga_sum_rows")
    return out


def spmv_csr(row_offsets, column_indices, values, x, y=None, alpha=1.0, beta=0.0, cols=None,
             workspace=None, stream=None):
    """y <- alpha * A @ x + beta * y for the CSR matrix A given by int32
    row_offsets (rows + 1), int32 column_indices and fp32 values (nnz each),
    all CUDA tensors; x has cols = x.numel() entries unless `cols` is given.
    Returns y (allocated when None; then beta must be 0)."""
    import ctypes as ct

    import torch
    rows = row_offsets.numel() - 1
    nnz = values.numel()
    cols = x.numel() if cols is None else cols
    for t, name, dt in ((row_offsets, "row_offsets", torch.int32),
                        (column_indices, "column_indices", torch.int32),
                        (values, "values", torch.float32), (x, "x", torch.float32)):
        if t.dtype != dt or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous {dt} tensor")
    if column_indices.numel() != nnz:
        raise ValueError("column_indices and values must have the same length")
    if y is None:
        if beta != 0:
            raise ValueError("beta != 0 needs y")
        y = torch.empty(rows, dtype=torch.float32, device=values.device)
    if y.dtype != torch.float32 or not y.is_contiguous() or y.numel() != rows:
        raise ValueError(f"y must be a contiguous float32 tensor of {rows} entries")
    if stream is None:
        stream = torch.cuda.current_stream(values.device).cuda_stream
    ws_bytes = dga_spmv_csr_workspace_size(rows, nnz)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=values.device)
    a, b = ct.c_float(float(alpha)), ct.c_float(float(beta))
    st = dga_spmv_csr(rows, cols, nnz, row_offsets.data_ptr(), column_indices.data_ptr(),
                      values.data_ptr(), ct.byref(a), x.data_ptr(), ct.byref(b), y.data_ptr(),
                      workspace.data_ptr() if workspace is not None else None,
                      workspace.numel() if workspace is not None else 0, stream)
    if st != OK:
        raise DgaError(st, "dga_spmv_csr")
    return y


def linear_forward(X, W, bias=None, Y=None):
    """Y = X @ W^T + bias for X [batch, in], W [out, in] (PyTorch's Linear
    layout), bias [out]: one dga_gemm_general call (W^T is column-major)."""
    return gemm(X, W.t(), Y, bias=bias)


def linear_backward(X, W, G, need_bias=True):
    """Gradients of Y = X W^T + b for the output gradient G [batch, out]:
    dX = G W, dW = G^T X, db = the batch sum of G (fp32).  Two
    dga_gemm_general calls and one dga_sum_rows call."""
    dX = gemm(G, W)
    dW = gemm(G.t(), X)
    db = sum_rows(G) if need_bias else None
    return dX, dW, db
