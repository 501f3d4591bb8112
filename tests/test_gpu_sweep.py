"""Ragged-shape sweep and repeat determinism for every kernel family.

Shapes are drawn (seeded) from the sizes around the tile and warp boundaries
{1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 127, 129, 255, 257}: each family is
forced through dga_gemm_ex and compared with the CPU oracle element by
element (bit-exact for INT8, within the oracle's bound otherwise).  A
second test runs one ragged case per family 20 times and requires the
outputs to be identical bit for bit: every reduction order in the kernels is
fixed (split-K partials are added in part order, INT8 chunks in k order).
"""
import random

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, assert_exact, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 127, 129, 255, 257]
S, T, K_, GEN = dga.PATH_SIMT, dga.PATH_TCGEN05, dga.PATH_SKINNY, dga.PATH_GENERIC

# (family, in dtype, out dtype, B layout)
FAMILIES = [
    ("simt", S, gen.F32, gen.F32, gen.ROW_MAJOR),
    ("simt_colB", S, gen.F32, gen.F32, gen.COL_MAJOR),
    ("tc_bf16", T, gen.BF16, gen.F32, gen.COL_MAJOR),
    ("tc_bf16_rowB", T, gen.BF16, gen.BF16, gen.ROW_MAJOR),
    ("tc_f16", T, gen.F16, gen.F32, gen.COL_MAJOR),
    ("tc_tf32", T, gen.TF32, gen.F32, gen.ROW_MAJOR),
    ("tc_int8", T, gen.I8, gen.I32, gen.ROW_MAJOR),
    ("skinny", K_, gen.BF16, gen.BF16, gen.COL_MAJOR),
    ("generic", GEN, gen.BF16, gen.F32, gen.ROW_MAJOR),
]


def _shapes(family, count=8):
    rng = random.Random(family)
    out = []
    while len(out) < count:
        M, N, K = (rng.choice(SIZES) for _ in range(3))
        if family == "skinny":
            M = min(M, 16)
        out.append((M, N, K))
    return out


def _operands(in_dtype, out_dtype, layout, M, N, K, seed, ld_k=None):
    """A (M x ld_k) and B (N x ld_k column-major, K x N row-major) hold the
    K-long rows in leading dimensions of ld_k >= K elements."""
    g = torch.Generator().manual_seed(seed)
    dist = ("int8",) if in_dtype == gen.I8 else ("uniform",)
    ld_k = K if ld_k is None else ld_k
    A = gen.random_matrix((M, ld_k), in_dtype, g, dist)
    B = gen.random_matrix((N, ld_k) if layout == gen.COL_MAJOR else (K, N), in_dtype, g, dist)
    C = gen.random_matrix((M, N), out_dtype, g,
                          ("int8",) if out_dtype == gen.I32 else ("uniform",))
    return A, B, C


@pytest.mark.parametrize("family,path,in_dtype,out_dtype,layout", FAMILIES,
                         ids=[f[0] for f in FAMILIES])
def test_ragged_sweep(family, path, in_dtype, out_dtype, layout):
    i8 = in_dtype == gen.I8
    alpha, beta = (3, -2) if i8 else (1.25, 0.5)
    for n, (M, N, K) in enumerate(_shapes(family)):
        # the skinny path reads through TMA: 16-byte row strides, so its
        # operands keep K in leading dimensions rounded up to 8 elements
        ld_k = (K + 7) // 8 * 8 if family == "skinny" else K
        A, B, C = _operands(in_dtype, out_dtype, layout, M, N, K, seed=n, ld_k=ld_k)
        got = run_gpu(path, in_dtype, out_dtype, layout, A, B, C, alpha, beta, M=M, N=N, K=K)
        assert dga.dga_last_path() == path
        ref, bound = oracle_ref(in_dtype, out_dtype, layout, A, B, C, alpha, beta, M=M, N=N, K=K)
        what = f"{family} {M}x{N}x{K}"
        if i8:
            assert_exact(got, ref, gen.I32, what)
        else:
            assert_close(got, ref, bound, out_dtype, what)


@pytest.mark.parametrize("family,path,in_dtype,out_dtype,layout", FAMILIES,
                         ids=[f[0] for f in FAMILIES])
def test_repeat_determinism(family, path, in_dtype, out_dtype, layout):
    # a ragged case large enough for several tiles (and, for SIMT, the split-K
    # tail: fewer tiles than resident blocks)
    M = 16 if family == "skinny" else 257
    N = 1031
    K = 1536 if family == "skinny" else 1537  # skinny: 16-byte row strides
    A, B, C = _operands(in_dtype, out_dtype, layout, M, N, K, seed=7)
    alpha, beta = (1, 1) if in_dtype == gen.I8 else (1.0, 0.75)
    first = run_gpu(path, in_dtype, out_dtype, layout, A, B, C, alpha, beta)
    for _ in range(19):
        again = run_gpu(path, in_dtype, out_dtype, layout, A, B, C, alpha, beta)
        assert torch.equal(first, again), f"{family}: repeat differs"
