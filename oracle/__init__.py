"""CPU oracle for dense GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
the two share no code: this package holds a plain C triple loop
(``gemm_oracle.c``) and a ctypes wrapper around it.

It computes ``ref = alpha * A @ B + beta * C`` with an fp64 accumulator
(int64 for INT8 inputs), as BLAS GEMM is defined in "AI Programming: Matrix
Product" (elainafan.one), section "Dense matrix multiplication", following
the CPU triple loop of its section "Row-major order".  Beside ``ref`` it
returns the per-element error bound

    bound = rel * sum_k |alpha * a_ik * b_kj| + |beta * c_ij| * 2**-22

with rel = 1e-4, or 2**-9 + 2**-20 + 1e-4 for TF32 inputs (fp32 operands
whose products the tensor cores form at 10 fraction bits), plus one
output-rounding ulp of ref for 16-bit output (:func:`ulp_bf16`,
:func:`ulp_f16`).  :func:`round_bf16` and :func:`round_f16` give the
nearest-even 16-bit encodings that exact cases must match.

It also holds the CSR sparse matrix-vector product of the same page
(sections "CSR" and "SpMV"): ``spmv_csr`` returns ``alpha * A @ x + beta * y``
row by row in fp64 and the bound ``1e-4 * |alpha| * sum |a_ip x_p| +
|beta * y_i| * 2**-22``.

Every function is pinned by ``tests/test_oracle.py`` against facts that do not
come from this code: identity and permutation matrices, alpha/beta semantics,
exact Python-integer and rational arithmetic on small cases, the MAC count
M*N*K, IEEE round-to-nearest-even for bf16 and fp16, and (for the sampled
entry points) Python integers and the full matrix at the sampled elements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F16, I8, I32, TF32 = 0, 1, 2, 3, 4, 5
ROW_MAJOR, COL_MAJOR = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_OUT = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT, "liboracle.so")
_LIB_COUNT = os.path.join(_OUT, "liboracle_count.so")
_lock = threading.Lock()
_libs: dict = {}


def _compile(src: str, out: str, defines=()) -> None:
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           *[f"-D{d}" for d in defines], src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)


def build(force: bool = False) -> None:
    """Compile the oracle (plain C + OpenMP) into ``oracle/_build``."""
    os.makedirs(_OUT, exist_ok=True)
    for out, defines in ((_LIB, ()), (_LIB_COUNT, ("ORACLE_COUNT_MACS",))):
        if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
            _compile(_SRC, out, defines)


def build_variant(src_path: str, out_path: str, defines=()) -> "Oracle":
    """Compile another copy of the oracle source (the tests use this to check
    that deliberately broken copies fail the pins) and load it."""
    _compile(src_path, out_path, defines)
    return Oracle(out_path)


_FP_NP = {F32: np.float32, BF16: np.uint16, F16: np.uint16, TF32: np.float32}


def _buf(arr, dtype, name):
    """Return a C-contiguous numpy buffer of the expected storage type.

    bf16/fp16 elements travel as their raw 16-bit encodings (uint16)."""
    if hasattr(arr, "detach"):  # a torch CPU tensor: hand over its storage bits
        import torch
        t = arr.detach().contiguous()
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        arr = t.numpy()
    arr = np.ascontiguousarray(arr)
    want = np.dtype(dtype)
    if arr.dtype != want:
        if arr.dtype.itemsize == want.itemsize and arr.dtype.kind in "iu" and want.kind in "iu":
            arr = arr.view(want)
        else:
            raise TypeError(f"{name}: expected storage {want}, got {arr.dtype}")
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data


def _sampled_ldc(c, ldc, beta):
    """The sampled entry points cannot infer C's leading dimension (they see
    no N), so it must be passed whenever C is read."""
    if c is None:
        if beta != 0:
            raise ValueError("beta != 0 needs C")
        return 0
    if ldc is None or ldc < 1:
        raise ValueError("C given without its leading dimension ldc")
    return ldc


class Oracle:
    """ctypes view of one compiled copy of ``gemm_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, f64, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int32
        ci = ctypes.c_int
        lib.oracle_gemm_fp.argtypes = [ci, ci, ci, i64, i64, i64, f64, vp, i64, vp, i64, f64,
                                       vp, i64, vp, vp]
        lib.oracle_gemm_fp_ex.argtypes = [ci, ci, ci, ci, i64, i64, i64, f64, vp, i64, vp, i64,
                                          f64, vp, i64, vp, vp, vp]
        lib.oracle_gemm_i8_ex.argtypes = [ci, ci, i64, i64, i64, i32, vp, i64, vp, i64, i32, vp,
                                          i64, vp, vp]
        lib.oracle_sum_rows.argtypes = [ci, i64, i64, vp, i64, vp, vp]
        lib.oracle_gemm_fp_sampled.argtypes = [ci, ci, ci, i64, f64, vp, i64, vp, i64, f64, vp,
                                               i64, i64, vp, vp, vp, vp]
        lib.oracle_gemm_i8.argtypes = [ci, i64, i64, i64, i32, vp, i64, vp, i64, i32, vp, i64, vp]
        lib.oracle_gemm_i8_sampled.argtypes = [ci, i64, i32, vp, i64, vp, i64, i32, vp, i64, i64,
                                               vp, vp, vp]
        lib.oracle_round_bf16.argtypes = [f64]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_ulp_bf16.argtypes = [f64]
        lib.oracle_ulp_bf16.restype = f64
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = f64
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_f16.restype = f64
        lib.oracle_mac_count.restype = i64
        lib.oracle_spmv_csr.argtypes = [i64, i64, vp, vp, vp, f64, vp, f64, vp, vp, vp]
        lib.oracle_round_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_ulp_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_round_f16_array.argtypes = [vp, vp, i64]
        lib.oracle_ulp_f16_array.argtypes = [vp, vp, i64]
        self.lib = lib
        self.path = path

    def gemm_fp(self, in_dtype, out_dtype, layout_b, M, N, K, alpha, A, lda, B, ldb, beta,
                C=None, ldc=None):
        """ref, bound = alpha*A@B + beta*C and its error bound, both (M, N) fp64.

        A, B, C are flat or 2-D buffers indexed with the leading dimensions
        lda, ldb, ldc exactly as the C function documents."""
        a = _buf(A, _FP_NP[in_dtype], "A")
        b = _buf(B, _FP_NP[in_dtype], "B")
        c = None if C is None else _buf(C, _FP_NP[out_dtype], "C")
        if c is None and beta != 0:
            raise ValueError("beta != 0 needs C")
        ref = np.empty((M, N), np.float64)
        bound = np.empty((M, N), np.float64)
        rc = self.lib.oracle_gemm_fp(in_dtype, out_dtype, layout_b, M, N, K, float(alpha),
                                     _ptr(a), lda, _ptr(b), ldb, float(beta), _ptr(c),
                                     ldc or N, _ptr(ref), _ptr(bound))
        if rc != 0:
            raise ValueError(f"oracle_gemm_fp: unsupported dtype pair ({in_dtype}, {out_dtype})")
        return ref, bound

    def gemm_fp_ex(self, in_dtype, out_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                   beta, C=None, ldc=None, bias=None):
        """gemm_fp with A's layout (0 row-major M x K, 1 stored K x M) and an
        optional bias row of N output-dtype elements added to every row."""
        a = _buf(A, _FP_NP[in_dtype], "A")
        b = _buf(B, _FP_NP[in_dtype], "B")
        c = None if C is None else _buf(C, _FP_NP[out_dtype], "C")
        bi = None if bias is None else _buf(bias, _FP_NP[out_dtype], "bias")
        if c is None and beta != 0:
            raise ValueError("beta != 0 needs C")
        ref = np.empty((M, N), np.float64)
        bound = np.empty((M, N), np.float64)
        rc = self.lib.oracle_gemm_fp_ex(in_dtype, out_dtype, layout_a, layout_b, M, N, K,
                                        float(alpha), _ptr(a), lda, _ptr(b), ldb, float(beta),
                                        _ptr(c), ldc or N, _ptr(bi), _ptr(ref), _ptr(bound))
        if rc != 0:
            raise ValueError(f"oracle_gemm_fp_ex: unsupported dtype pair ({in_dtype}, {out_dtype})")
        return ref, bound

    def gemm_i8_ex(self, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb, beta=0, C=None,
                   ldc=None, bias=None):
        a = _buf(A, np.int8, "A")
        b = _buf(B, np.int8, "B")
        c = None if C is None else _buf(C, np.int32, "C")
        bi = None if bias is None else _buf(bias, np.int32, "bias")
        out = np.empty((M, N), np.int32)
        self.lib.oracle_gemm_i8_ex(layout_a, layout_b, M, N, K, int(alpha), _ptr(a), lda, _ptr(b),
                                   ldb, int(beta), _ptr(c), ldc or N, _ptr(bi), _ptr(out))
        return out

    def sum_rows(self, dtype, rows, cols, G, ldg=None):
        """(sums, bound): column j summed over the rows of G, in fp64."""
        g = _buf(G, _FP_NP[dtype], "G")
        out = np.empty(cols, np.float64)
        bound = np.empty(cols, np.float64)
        if self.lib.oracle_sum_rows(dtype, rows, cols, _ptr(g), ldg or cols, _ptr(out),
                                    _ptr(bound)) != 0:
            raise ValueError("oracle_sum_rows: unsupported dtype")
        return out, bound

    def gemm_fp_sampled(self, in_dtype, out_dtype, layout_b, K, alpha, A, lda, B, ldb, beta,
                        C, ldc, rows, cols):
        """ref, bound at the elements (rows[s], cols[s]) only.

        C is indexed with ldc, which must be given whenever C is."""
        a = _buf(A, _FP_NP[in_dtype], "A")
        b = _buf(B, _FP_NP[in_dtype], "B")
        c = None if C is None else _buf(C, _FP_NP[out_dtype], "C")
        ldc = _sampled_ldc(c, ldc, beta)
        rows = np.ascontiguousarray(rows, np.int64)
        cols = np.ascontiguousarray(cols, np.int64)
        ref = np.empty(rows.shape, np.float64)
        bound = np.empty(rows.shape, np.float64)
        rc = self.lib.oracle_gemm_fp_sampled(in_dtype, out_dtype, layout_b, K, float(alpha),
                                             _ptr(a), lda, _ptr(b), ldb, float(beta), _ptr(c),
                                             ldc, rows.size, _ptr(rows), _ptr(cols),
                                             _ptr(ref), _ptr(bound))
        if rc != 0:
            raise ValueError("oracle_gemm_fp_sampled: unsupported dtype pair")
        return ref, bound

    def gemm_i8(self, layout_b, M, N, K, alpha, A, lda, B, ldb, beta=0, C=None, ldc=None):
        """alpha*A@B + beta*C for int8 A, B and int32 C, exact, reduced mod 2**32."""
        a = _buf(A, np.int8, "A")
        b = _buf(B, np.int8, "B")
        c = None if C is None else _buf(C, np.int32, "C")
        if c is None and beta != 0:
            raise ValueError("beta != 0 needs C")
        out = np.empty((M, N), np.int32)
        self.lib.oracle_gemm_i8(layout_b, M, N, K, int(alpha), _ptr(a), lda, _ptr(b), ldb,
                                int(beta), _ptr(c), ldc or N, _ptr(out))
        return out

    def gemm_i8_sampled(self, layout_b, K, alpha, A, lda, B, ldb, beta, C, ldc, rows, cols):
        """gemm_i8 at the elements (rows[s], cols[s]) only (ldc as for gemm_fp_sampled)."""
        a = _buf(A, np.int8, "A")
        b = _buf(B, np.int8, "B")
        c = None if C is None else _buf(C, np.int32, "C")
        ldc = _sampled_ldc(c, ldc, beta)
        rows = np.ascontiguousarray(rows, np.int64)
        cols = np.ascontiguousarray(cols, np.int64)
        out = np.empty(rows.shape, np.int32)
        self.lib.oracle_gemm_i8_sampled(layout_b, K, int(alpha), _ptr(a), lda, _ptr(b), ldb,
                                        int(beta), _ptr(c), ldc, rows.size, _ptr(rows),
                                        _ptr(cols), _ptr(out))
        return out

    def spmv_csr(self, rows, cols, row_offsets, column_indices, values, x, alpha=1.0, beta=0.0,
                 y=None):
        """(ref, bound): alpha * A @ x + beta * y for the CSR matrix A
        (int32 row_offsets of rows + 1 entries, int32 column_indices and fp32
        values of nnz entries), both (rows,) fp64."""
        ro = _buf(row_offsets, np.int32, "row_offsets")
        ci = _buf(column_indices, np.int32, "column_indices")
        va = _buf(values, np.float32, "values")
        xx = _buf(x, np.float32, "x")
        yy = None if y is None else _buf(y, np.float32, "y")
        if yy is None and beta != 0:
            raise ValueError("beta != 0 needs y")
        if ro.size != rows + 1:
            raise ValueError("row_offsets must have rows + 1 entries")
        ref = np.empty(rows, np.float64)
        bound = np.empty(rows, np.float64)
        rc = self.lib.oracle_spmv_csr(rows, cols, _ptr(ro), _ptr(ci), _ptr(va), float(alpha),
                                      _ptr(xx), float(beta), _ptr(yy), _ptr(ref), _ptr(bound))
        if rc != 0:
            raise ValueError("oracle_spmv_csr: not a CSR matrix of the given shape")
        return ref, bound

    def round_bf16(self, x) -> np.ndarray:
        """Nearest-even bf16 encodings (uint16) of the fp64 values x."""
        flat = np.ascontiguousarray(np.asarray(x, np.float64).ravel())
        out = np.empty(flat.size, np.uint16)
        self.lib.oracle_round_bf16_array(_ptr(flat), _ptr(out), flat.size)
        return out.reshape(np.shape(x))

    def ulp_bf16(self, x) -> np.ndarray:
        flat = np.ascontiguousarray(np.asarray(x, np.float64).ravel())
        out = np.empty(flat.size, np.float64)
        self.lib.oracle_ulp_bf16_array(_ptr(flat), _ptr(out), flat.size)
        return out.reshape(np.shape(x))

    def round_f16(self, x) -> np.ndarray:
        """Nearest-even IEEE binary16 encodings (uint16) of the fp64 values x."""
        flat = np.ascontiguousarray(np.asarray(x, np.float64).ravel())
        out = np.empty(flat.size, np.uint16)
        self.lib.oracle_round_f16_array(_ptr(flat), _ptr(out), flat.size)
        return out.reshape(np.shape(x))

    def ulp_f16(self, x) -> np.ndarray:
        flat = np.ascontiguousarray(np.asarray(x, np.float64).ravel())
        out = np.empty(flat.size, np.float64)
        self.lib.oracle_ulp_f16_array(_ptr(flat), _ptr(out), flat.size)
        return out.reshape(np.shape(x))

    def decode_bf16(self, bits) -> np.ndarray:
        flat = np.asarray(bits, np.uint16).ravel()
        out = np.fromiter((self.lib.oracle_decode_bf16(int(v)) for v in flat), np.float64,
                          flat.size)
        return out.reshape(np.shape(bits))

    def decode_f16(self, bits) -> np.ndarray:
        flat = np.asarray(bits, np.uint16).ravel()
        out = np.fromiter((self.lib.oracle_decode_f16(int(v)) for v in flat), np.float64,
                          flat.size)
        return out.reshape(np.shape(bits))

    def mac_count(self) -> int:
        """MACs executed since the last reset (instrumented build; -1 otherwise)."""
        return int(self.lib.oracle_mac_count())

    def reset_mac_count(self) -> None:
        self.lib.oracle_reset_mac_count()


def default(counting: bool = False) -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    path = _LIB_COUNT if counting else _LIB
    with _lock:
        if path not in _libs:
            build()
            _libs[path] = Oracle(path)
        return _libs[path]


def gemm_fp(*args, **kw):
    return default().gemm_fp(*args, **kw)


def gemm_fp_sampled(*args, **kw):
    return default().gemm_fp_sampled(*args, **kw)


def gemm_i8(*args, **kw):
    return default().gemm_i8(*args, **kw)


def gemm_i8_sampled(*args, **kw):
    return default().gemm_i8_sampled(*args, **kw)


def gemm_fp_ex(*args, **kw):
    return default().gemm_fp_ex(*args, **kw)


def gemm_i8_ex(*args, **kw):
    return default().gemm_i8_ex(*args, **kw)


def sum_rows(*args, **kw):
    return default().sum_rows(*args, **kw)


def spmv_csr(*args, **kw):
    return default().spmv_csr(*args, **kw)


def round_bf16(x):
    return default().round_bf16(x)


def ulp_bf16(x):
    return default().ulp_bf16(x)


def round_f16(x):
    return default().round_f16(x)


def ulp_f16(x):
    return default().ulp_f16(x)


SOURCE = _SRC
