"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers; it holds none of the GEMM arithmetic.
It is the one module that both the CUDA path's callers (tests, bench) and the
CPU oracle's callers use, so that both sides see identical inputs.

Recipe (one CPU ``torch.Generator`` per workload, ``manual_seed(seed)``,
drawing A, then B, then C):

* fp32 uniform[-1, 1):   ``torch.rand(shape) * 2 - 1``
* N(0, sigma) as bf16:   ``(torch.randn(shape) * sigma).to(torch.bfloat16)``
  (float32 draw, round-to-nearest-even to bf16)
* int8 uniform [-128, 127]: ``torch.randint(-128, 128, shape, dtype=int8)``
* CSR sparse matrices (:func:`csr_powerlaw`): row lengths from a Pareto law
  (a few rows thousands of entries long, most a few dozen, some empty),
  column indices near the row's diagonal position, values uniform[-1, 1);
  x uniform[-1, 1).  The sparse-matrix sections of "AI Programming: Matrix
  Product" give no sizes; the structure follows their remark that row lengths
  can differ a lot.

The workloads are the synthetic square and skinny shapes that the pages
measure ("Matrix multiplication: arithmetic intensity, tiling and Tensor
Core", sections 5.1-5.5; "CUDA Kernel tuning: from naive matrix
multiplication to Tensor Core", section 3) resized to this GPU's scale.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# dtype / layout codes shared with the C ABI (values fixed by include/dga.h);
# TF32 operands are fp32 in memory
F32, BF16, F16, I8, I32, TF32 = 0, 1, 2, 3, 4, 5
ROW_MAJOR, COL_MAJOR = 0, 1

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16,
               I8: torch.int8, I32: torch.int32, TF32: torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    in_dtype: int
    out_dtype: int
    layout_b: int
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist_a: tuple = ("uniform",)      # ("uniform",) | ("normal", sigma) | ("int8",)
    dist_b: tuple = ("uniform",)
    dist_c: tuple = ("uniform",)
    seed: int = 0
    note: str = field(default="", compare=False)
    # "gemm": one C <- alpha*A*B + beta*C.  "spmv": y <- alpha*A*x + beta*y
    # for a CSR matrix of M rows and N columns (csr_powerlaw).  "fc": one fully-connected layer
    # step with batch M, N outputs and K inputs -- forward Y = X W^T + b and
    # backward dX = G W, dW = G^T X, db = sum over the batch of G; dist_a
    # draws X, dist_b W and b, dist_c the output gradient G.
    kind: str = "gemm"


WORKLOADS = {
    "fp32_256": Workload("fp32_256", F32, F32, ROW_MAJOR, 256, 256, 256, 1.0, 0.0,
                         note="FP32 M=N=K=256, alpha=1, beta=0, seed 0"),
    "fp32_4096": Workload("fp32_4096", F32, F32, ROW_MAJOR, 4096, 4096, 4096, 1.5, 0.5,
                          note="FP32 SIMT M=N=K=4096, alpha=1.5, beta=0.5"),
    "bf16_8192": Workload("bf16_8192", BF16, F32, COL_MAJOR, 8192, 8192, 8192, 1.0, 0.0,
                          ("normal", 1.0), ("normal", 1.0),
                          note="BF16 in, FP32 out, M=N=K=8192, B column-major"),
    "skinny_m1": Workload("skinny_m1", BF16, BF16, COL_MAJOR, 1, 8192, 8192, 1.0, 0.0,
                          ("normal", 1.0), ("normal", 0.02),
                          note="X[1,8192] x W[8192,8192]^T, bf16 out"),
    "skinny_m8": Workload("skinny_m8", BF16, BF16, COL_MAJOR, 8, 8192, 8192, 1.0, 0.0,
                          ("normal", 1.0), ("normal", 0.02),
                          note="X[8,8192] x W[8192,8192]^T, bf16 out"),
    "skinny_m16": Workload("skinny_m16", BF16, BF16, COL_MAJOR, 16, 8192, 8192, 1.0, 0.0,
                           ("normal", 1.0), ("normal", 0.02),
                           note="X[16,8192] x W[8192,8192]^T, bf16 out"),
    "int8_ragged": Workload("int8_ragged", I8, I32, ROW_MAJOR, 4093, 4099, 4096, 1, 0,
                            ("int8",), ("int8",), ("int8",),
                            note="INT8 x INT8 -> INT32, M=4093 N=4099 K=4096"),
    "f16_8192": Workload("f16_8192", F16, F32, COL_MAJOR, 8192, 8192, 8192, 1.0, 0.0,
                         ("normal", 1.0), ("normal", 1.0),
                         note="FP16 in, FP32 out, M=N=K=8192, B column-major"),
    "bf16_8192_rowb": Workload("bf16_8192_rowb", BF16, F32, ROW_MAJOR, 8192, 8192, 8192, 1.0,
                               0.0, ("normal", 1.0), ("normal", 1.0),
                               note="BF16 in, FP32 out, M=N=K=8192, B row-major"),
    "tf32_8192": Workload("tf32_8192", TF32, F32, COL_MAJOR, 8192, 8192, 8192, 1.0, 0.0,
                          note="FP32 in memory multiplied as TF32 on the tensor cores, FP32 out, "
                               "M=N=K=8192, B column-major, A and B uniform[-1,1)"),
    "spmv_powerlaw": Workload("spmv_powerlaw", F32, F32, ROW_MAJOR, 4194304, 4194304, 0, 1.0, 0.0,
                              kind="spmv",
                              note="CSR SpMV y = A x, 4194304 x 4194304, Pareto(1.5) row lengths "
                                   "(min 8, max 16384, 5% empty rows, mean ~23), columns within "
                                   "+-4096 of the diagonal"),
    "spmv_small": Workload("spmv_small", F32, F32, ROW_MAJOR, 20000, 30000, 0, 1.0, 0.0,
                           kind="spmv", note="CSR SpMV, 20000 x 30000, same structure"),
    "fc_bf16_8192": Workload("fc_bf16_8192", BF16, BF16, COL_MAJOR, 8192, 8192, 8192, 1.0, 0.0,
                             ("normal", 1.0), ("normal", 0.02), ("normal", 1.0), kind="fc",
                             note="fully-connected layer step, bf16, batch 8192, 8192 -> 8192"),
    "fc_f32_4096": Workload("fc_f32_4096", F32, F32, COL_MAJOR, 4096, 4096, 4096, 1.0, 0.0,
                            kind="fc",
                            note="fully-connected layer step, fp32, batch 4096, 4096 -> 4096"),
}


def _draw(shape, dist, dtype_code, gen):
    kind = dist[0]
    if kind == "uniform":
        t = torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
        return t.to(TORCH_DTYPE[dtype_code])
    if kind == "normal":
        t = torch.randn(shape, generator=gen, dtype=torch.float32) * dist[1]
        return t.to(TORCH_DTYPE[dtype_code])
    if kind == "int8":
        if dtype_code == I8:
            return torch.randint(-128, 128, shape, generator=gen, dtype=torch.int8)
        return torch.randint(-128, 128, shape, generator=gen, dtype=torch.int32)
    raise ValueError(kind)


def make_inputs(w: Workload, seed: int | None = None, with_c: bool | None = None):
    """Return (A, B, C) as CPU tensors for workload ``w``.

    A is M x K row-major.  B is K x N row-major, or (column-major) stored as
    an N x K row-major tensor.  C is M x N in the output dtype, drawn only
    when beta != 0 (or ``with_c``), else None."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    A = _draw((w.M, w.K), w.dist_a, w.in_dtype, gen)
    b_shape = (w.N, w.K) if w.layout_b == COL_MAJOR else (w.K, w.N)
    B = _draw(b_shape, w.dist_b, w.in_dtype, gen)
    want_c = (w.beta != 0) if with_c is None else with_c
    C = _draw((w.M, w.N), w.dist_c, w.out_dtype, gen) if want_c else None
    return A, B, C


def random_matrix(shape, dtype_code, gen, dist=("uniform",)):
    """A single seeded matrix (for the shape sweeps of the tests)."""
    return _draw(shape, dist, dtype_code, gen)


def small_int_matrix(shape, dtype_code, gen, lo=-4, hi=4):
    """Integer-valued entries in [lo, hi], stored in ``dtype_code``."""
    t = torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int32)
    return t.to(TORCH_DTYPE[dtype_code])


# Structure of the synthetic CSR matrices.
CSR_STRUCTURE = dict(pareto_alpha=1.5, min_len=8, max_len=16384, empty_frac=0.05, window=4096)


def csr_powerlaw(rows, cols, gen, device="cpu", pareto_alpha=1.5, min_len=8, max_len=16384,
                 empty_frac=0.05, window=4096):
    """A seeded synthetic CSR matrix: (row_offsets int32 [rows + 1],
    column_indices int32 [nnz], values float32 [nnz]).

    Row lengths: floor(min_len * u^(-1/pareto_alpha)) capped at max_len, u
    uniform in (0, 1] (a Pareto law: mean about 3 * min_len for alpha 1.5),
    and a fraction empty_frac of rows set empty.  Columns: row i's entries
    sit at (i * cols // rows + offset) mod cols, offset uniform in
    [-window, window] (unsorted, repeats possible).  Values uniform[-1, 1).
    Draw order: lengths, empty flags, column offsets, values."""
    u = 1.0 - torch.rand(rows, generator=gen, device=device, dtype=torch.float64)
    lengths = torch.floor(min_len * u.pow(-1.0 / pareto_alpha)).clamp_(max=max_len).to(torch.int64)
    empty = torch.rand(rows, generator=gen, device=device) < empty_frac
    lengths[empty] = 0
    offsets = torch.zeros(rows + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(lengths, 0)
    nnz = int(offsets[-1])
    if nnz >= 2 ** 31:
        raise ValueError("too many entries for int32 offsets")
    row_of = torch.repeat_interleave(torch.arange(rows, device=device), lengths)
    off = torch.randint(-window, window + 1, (nnz,), generator=gen, device=device)
    cols_idx = torch.remainder(row_of * cols // rows + off, cols).to(torch.int32)
    del row_of, off
    values = torch.rand(nnz, generator=gen, device=device) * 2 - 1
    return offsets.to(torch.int32), cols_idx, values


def make_csr_inputs(w: Workload, seed: int | None = None, device="cpu"):
    """(row_offsets, column_indices, values, x, y) for an "spmv" workload;
    y is drawn only when beta != 0."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    offs, cols, vals = csr_powerlaw(w.M, w.N, gen, device, **CSR_STRUCTURE)
    x = torch.rand(w.N, generator=gen, device=device) * 2 - 1
    y = torch.rand(w.M, generator=gen, device=device) * 2 - 1 if w.beta != 0 else None
    return offs, cols, vals, x, y
