"""Pins that tie the CPU oracle to facts outside itself.

Each pin takes an ``oracle.Oracle`` (the real build, or a deliberately broken
copy in the mutation test) and raises AssertionError when the oracle
disagrees with what the mathematics or the pages fix:

* identity and permutation matrices (exact results, transposition detected);
* BLAS alpha/beta semantics (beta == 0 never reads C, alpha == 0 never reads
  A and B), linearity in alpha;
* integer-valued inputs against Python integers (exact);
* tiny random shapes against exact rational arithmetic, within the fp64
  summation error bound, and the error-bound formula itself;
* INT8 against Python integers, including wrap-around mod 2**32;
* the MAC count M*N*K (2MNK FLOPs) of the instrumented build;
* bf16 decoding and IEEE round-to-nearest-even encoding, for bf16 and
  fp16, and the one-ulp output-rounding terms of both;
* the sampled entry points against Python integers and against the full
  matrix at the sampled elements, with padded leading dimensions;
* CSR SpMV: the page's worked 3 x 4 example, dense products of COO
  triplets in Python integers and exact rationals (empty rows, a long row,
  repeated columns), identity and permutation matrices, alpha/beta
  semantics, and rejection of arrays that are not a CSR matrix;
* TF32 inputs: the same exact result as FP32, and a bound that covers the
  result of operands cut to 10 fraction bits, by truncation or by rounding
  (computed here from the binary32 encoding, in exact rationals).

The GEMM definition pinned here is BLAS's C <- alpha*A*B + beta*C, "AI
Programming: Matrix Product" (elainafan.one), section "Dense matrix
multiplication"; row-major offsets row*ld + col from its section "Row-major
order".
"""
from __future__ import annotations

import json
import os
import random
from fractions import Fraction

import numpy as np
import torch

F32, BF16, F16, I8, I32, TF32 = 0, 1, 2, 3, 4, 5
ROW, COL = 0, 1


def _rng(seed):
    g = torch.Generator().manual_seed(seed)
    return g


def _f32(shape, g):
    return (torch.rand(shape, generator=g) * 2 - 1).numpy().astype(np.float32)


def _bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- identity --

def pin_identity(o):
    g = _rng(1)
    M = K = 23
    N = 17
    eye = np.eye(M, dtype=np.float32)
    B = _f32((K, N), g)
    C = _f32((M, N), g)
    alpha, beta = 1.5, -0.5
    ref, _ = o.gemm_fp(F32, F32, ROW, M, N, K, alpha, eye, K, B, N, beta, C, N)
    want = alpha * B.astype(np.float64) + beta * C.astype(np.float64)
    assert np.array_equal(ref, want), "I*B"
    # B = I: result is alpha*A + beta*C
    A = _f32((M, K), g)
    C2 = _f32((M, K), g)
    ref, _ = o.gemm_fp(F32, F32, ROW, M, K, K, alpha, A, K, np.eye(K, dtype=np.float32), K,
                       beta, C2, K)
    want = alpha * A.astype(np.float64) + beta * C2.astype(np.float64)
    assert np.array_equal(ref, want), "A*I"
    # bf16 storage: identity picks out the decoded B exactly
    Bt = torch.randn((K, N), generator=g)
    eyeb = _bf16_bits(torch.eye(M))
    ref, _ = o.gemm_fp(BF16, F32, ROW, M, N, K, 1.0, eyeb, K, _bf16_bits(Bt), N, 0.0)
    assert np.array_equal(ref, Bt.to(torch.bfloat16).double().numpy()), "bf16 I*B"


# ------------------------------------------------------------- permutation --

def pin_permutation(o):
    g = _rng(2)
    M, K, N = 9, 13, 11
    perm_rows = torch.randperm(K, generator=g).numpy()
    P = np.zeros((M, K), np.float32)
    rows_used = perm_rows[:M]
    P[np.arange(M), rows_used] = 1.0          # P @ B = B[rows_used]
    B = _f32((K, N), g)
    ref, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, P, K, B, N, 0.0)
    assert np.array_equal(ref, B[rows_used].astype(np.float64)), "P*B row-major"
    # same B stored column-major (N x K): must give the same answer
    Bt = np.ascontiguousarray(B.T)
    ref_c, _ = o.gemm_fp(F32, F32, COL, M, N, K, 1.0, P, K, Bt, K, 0.0)
    assert np.array_equal(ref_c, B[rows_used].astype(np.float64)), "P*B column-major"
    # A @ Q permutes columns: column j of the result is column cols[j] of A
    cols = torch.randperm(K, generator=g).numpy()[:N]
    Q = np.zeros((K, N), np.float32)
    Q[cols, np.arange(N)] = 1.0
    A = _f32((M, K), g)
    ref, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, A, K, Q, N, 0.0)
    assert np.array_equal(ref, A[:, cols].astype(np.float64)), "A*Q"
    # leading dimensions larger than the row length
    lda, ldb = K + 5, N + 3
    Apad = np.full((M, lda), np.nan, np.float32)
    Apad[:, :K] = A
    Qpad = np.full((K, ldb), np.nan, np.float32)
    Qpad[:, :N] = Q
    ref, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, Apad, lda, Qpad, ldb, 0.0)
    assert np.array_equal(ref, A[:, cols].astype(np.float64)), "padded lda/ldb"


# -------------------------------------------------------------- alpha/beta --

def pin_alpha_beta(o):
    g = _rng(3)
    M, N, K = 7, 6, 5
    A = _f32((M, K), g)
    B = _f32((K, N), g)
    Cnan = np.full((M, N), np.nan, np.float32)
    ref, bound = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, A, K, B, N, 0.0, Cnan, N)
    assert np.isfinite(ref).all() and np.isfinite(bound).all(), "beta=0 read C"
    Anan = np.full((M, K), np.nan, np.float32)
    C = _f32((M, N), g)
    Bnan = np.full((K, N), np.nan, np.float32)
    ref, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 0.0, Anan, K, Bnan, N, 2.0, C, N)
    assert np.array_equal(ref, 2.0 * C.astype(np.float64)), "alpha=0 read A/B"
    # beta*C with alpha=1, beta=1 on integer data is the exact sum
    Ai = torch.randint(-4, 5, (M, K), generator=g).numpy().astype(np.float32)
    Bi = torch.randint(-4, 5, (K, N), generator=g).numpy().astype(np.float32)
    Ci = torch.randint(-9, 10, (M, N), generator=g).numpy().astype(np.float32)
    r1, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, Ai, K, Bi, N, 1.0, Ci, N)
    r0, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 1.0, Ai, K, Bi, N, 0.0, Ci, N)
    assert np.array_equal(r1, r0 + Ci), "beta=1 adds C"
    # linearity in alpha
    ra, _ = o.gemm_fp(F32, F32, ROW, M, N, K, 3.0, Ai, K, Bi, N, 0.0)
    rb, _ = o.gemm_fp(F32, F32, ROW, M, N, K, -5.0, Ai, K, Bi, N, 0.0)
    rab, _ = o.gemm_fp(F32, F32, ROW, M, N, K, -2.0, Ai, K, Bi, N, 0.0)
    assert np.array_equal(ra + rb, rab), "linearity in alpha"


# ------------------------------------------------------- exact small ints --

def _py_gemm(A, B, C, alpha, beta, layout_b):
    M, K = len(A), len(A[0])
    N = len(B) if layout_b == COL else len(B[0])
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = 0
            for k in range(K):
                b = B[j][k] if layout_b == COL else B[k][j]
                s += A[i][k] * b
            row.append(alpha * s + (beta * C[i][j] if beta else 0))
        out.append(row)
    return out


def pin_small_integers(o):
    g = _rng(4)
    M, N, K = 13, 11, 17
    for in_dtype in (F32, BF16):
        for layout in (ROW, COL):
            A = torch.randint(-4, 5, (M, K), generator=g)
            Bshape = (N, K) if layout == COL else (K, N)
            B = torch.randint(-4, 5, Bshape, generator=g)
            C = torch.randint(-8, 9, (M, N), generator=g)
            want = _py_gemm(A.tolist(), B.tolist(), C.tolist(), 3, -2, layout)
            if in_dtype == F32:
                a, b = A.float().numpy(), B.float().numpy()
            else:
                a, b = _bf16_bits(A.float()), _bf16_bits(B.float())
            ldb = K if layout == COL else N
            ref, _ = o.gemm_fp(in_dtype, F32, layout, M, N, K, 3.0, a, K, b, ldb, -2.0,
                               C.float().numpy(), N)
            assert np.array_equal(ref, np.array(want, np.float64)), (in_dtype, layout)


def pin_int8(o):
    g = _rng(5)
    M, N, K = 9, 10, 37
    for layout in (ROW, COL):
        A = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
        Bshape = (N, K) if layout == COL else (K, N)
        B = torch.randint(-128, 128, Bshape, generator=g, dtype=torch.int8)
        C = torch.randint(-2**31, 2**31, (M, N), generator=g, dtype=torch.int64).to(torch.int32)
        ldb = K if layout == COL else N
        for alpha, beta in ((1, 0), (-3, 7), (1 << 20, 1 << 30), (0, -1)):
            got = o.gemm_i8(layout, M, N, K, alpha, A.numpy(), K, B.numpy(), ldb, beta,
                            C.numpy(), N)
            want = _py_gemm(A.tolist(), B.tolist(), C.tolist(), alpha, beta, layout)
            wrapped = [[((v + 2**31) % 2**32) - 2**31 for v in row] for row in want]
            assert np.array_equal(got, np.array(wrapped, np.int64)), (layout, alpha, beta)
        # leading dimensions larger than the row length, padding full of junk
        lda, ldb_p = K + 3, ldb + 5
        Ap = torch.randint(-128, 128, (M, lda), generator=g, dtype=torch.int8)
        Ap[:, :K] = A
        Bp = torch.randint(-128, 128, (Bshape[0], ldb_p), generator=g, dtype=torch.int8)
        Bp[:, :Bshape[1]] = B
        got = o.gemm_i8(layout, M, N, K, 1, Ap.numpy(), lda, Bp.numpy(), ldb_p)
        want = _py_gemm(A.tolist(), B.tolist(), C.tolist(), 1, 0, layout)
        assert np.array_equal(got, np.array(want, np.int64)), ("padded", layout)
        # all -128: the largest magnitude products
        Am = torch.full((2, 64), -128, dtype=torch.int8)
        Bm = torch.full((64, 3) if layout == ROW else (3, 64), -128, dtype=torch.int8)
        got = o.gemm_i8(layout, 2, 3, 64, 1, Am.numpy(), 64, Bm.numpy(),
                        3 if layout == ROW else 64)
        assert (got == 64 * 16384).all()


# ------------------------------------------------- rationals on tiny shapes --

def pin_tiny_rational(o):
    rnd = random.Random(6)
    u = Fraction(1, 2**53)
    for trial in range(60):
        M, N, K = rnd.randint(1, 8), rnd.randint(1, 8), rnd.randint(1, 8)
        layout = rnd.choice((ROW, COL))
        # float32 values with spread exponents, so roundings really happen
        def val():
            return np.float32(rnd.uniform(-1, 1) * 2.0 ** rnd.randint(-20, 20))
        A = np.array([[val() for _ in range(K)] for _ in range(M)], np.float32)
        Bshape = (N, K) if layout == COL else (K, N)
        B = np.array([[val() for _ in range(Bshape[1])] for _ in range(Bshape[0])], np.float32)
        C = np.array([[val() for _ in range(N)] for _ in range(M)], np.float32)
        alpha = float(np.float32(rnd.uniform(-2, 2)))
        beta = rnd.choice((0.0, float(np.float32(rnd.uniform(-2, 2)))))
        ldb = K if layout == COL else N
        ref, bound = o.gemm_fp(F32, F32, layout, M, N, K, alpha, A, K, B, ldb, beta, C, N)
        for i in range(M):
            for j in range(N):
                terms = []
                for k in range(K):
                    b = B[j, k] if layout == COL else B[k, j]
                    terms.append(Fraction(float(A[i, k])) * Fraction(float(b)))
                s = sum(terms, Fraction(0))
                fa, fb = Fraction(alpha), Fraction(beta)
                cterm = fb * Fraction(float(C[i, j])) if beta != 0 else Fraction(0)
                exact = fa * s + cterm
                abs_terms = sum((abs(t) for t in terms), Fraction(0))
                mag = abs(fa) * abs_terms + abs(cterm)
                n = K + 2
                gamma = n * u / (1 - n * u)
                err = abs(Fraction(float(ref[i, j])) - exact)
                assert err <= gamma * mag + Fraction(2) ** -1074, (trial, i, j)
                want_bound = Fraction(1, 10**4) * abs(fa) * abs_terms + abs(cterm) * Fraction(1, 2**22)
                assert abs(Fraction(float(bound[i, j])) - want_bound) <= 8 * u * want_bound + \
                    Fraction(2) ** -1074, ("bound", trial, i, j)


# --------------------------------------------------------------- MAC count --

def pin_mac_count(o_counting):
    g = _rng(7)
    for (M, N, K) in ((3, 5, 7), (16, 1, 33), (1, 9, 1)):
        A = _f32((M, K), g)
        B = _f32((K, N), g)
        o_counting.reset_mac_count()
        o_counting.gemm_fp(F32, F32, ROW, M, N, K, 1.0, A, K, B, N, 0.0)
        assert o_counting.mac_count() == M * N * K, (M, N, K)
        Ai = np.zeros((M, K), np.int8)
        Bi = np.zeros((K, N), np.int8)
        o_counting.reset_mac_count()
        o_counting.gemm_i8(ROW, M, N, K, 1, Ai, K, Bi, N)
        assert o_counting.mac_count() == M * N * K
    o_counting.reset_mac_count()
    o_counting.gemm_fp(F32, F32, ROW, 4, 4, 4, 0.0, np.zeros((4, 4), np.float32), 4,
                       np.zeros((4, 4), np.float32), 4, 0.0)
    assert o_counting.mac_count() == 0, "alpha=0 must not multiply"
    # CSR SpMV: one multiply per stored nonzero (empty rows cost nothing)
    offs = np.array([0, 3, 3, 7, 8], np.int32)
    cols = np.array([0, 1, 2, 0, 0, 3, 1, 2], np.int32)
    o_counting.reset_mac_count()
    o_counting.spmv_csr(4, 4, offs, cols, np.ones(8, np.float32), np.ones(4, np.float32))
    assert o_counting.mac_count() == 8, "SpMV MACs = nnz"


# ------------------------------------------------------------------- bf16 --

def _bf16_value(bits):
    """Value of a bf16 encoding from the IEEE definition (sign, 8-bit
    exponent with bias 127, 7 fraction bits), as an exact Fraction."""
    s = -1 if bits >> 15 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0:
        return s * Fraction(m, 2**7) * Fraction(2) ** -126
    return s * (1 + Fraction(m, 2**7)) * Fraction(2) ** (e - 127)


def pin_bf16_decode(o):
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    got = o.decode_bf16(bits)
    for b, v in zip(bits.tolist(), got.tolist()):
        e = (b >> 7) & 0xFF
        if e == 0xFF:
            if b & 0x7F:
                assert v != v
            else:
                assert v == (float("-inf") if b >> 15 else float("inf"))
        else:
            assert Fraction(v) == _bf16_value(b), hex(b)


def pin_f16_decode(o):
    bits = np.arange(0, 1 << 16, 61, dtype=np.uint16)
    got = o.decode_f16(bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def pin_bf16_round(o):
    # hand cases from round-to-nearest-even on 8 significant bits
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0**-8, 0x3F80),            # tie -> even mantissa (0)
        (1.0 + 3 * 2.0**-8, 0x3F82),        # tie -> even mantissa (2)
        (1.0 + 2.0**-8 + 2.0**-30, 0x3F81),  # just above the tie
        (-1.5, 0xBFC0),
        (2.0**-133, 0x0001),                # smallest subnormal
        (2.0**-134, 0x0000),                # tie between 0 and 2^-133 -> 0
        (3 * 2.0**-134, 0x0002),            # tie between 1 and 2 quanta -> 2
        ((2 - 2.0**-7) * 2.0**127, 0x7F7F),  # largest finite
        ((2 - 2.0**-8) * 2.0**127, 0x7F80),  # tie with 2^128 -> overflow to inf
        (0.0, 0x0000),
        (-0.0, 0x8000),
    ]
    got = o.round_bf16(np.array([x for x, _ in cases], np.float64))
    for (x, want), g in zip(cases, got.tolist()):
        assert g == want, (x, hex(g), hex(want))
    # agreement with torch's float32 -> bf16 round-to-nearest-even on many values
    g = _rng(8)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-140, 128, (20000,),
                                                                  generator=g).float())
    x = x[torch.isfinite(x)]
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.round_bf16(x.double().numpy())
    assert np.array_equal(got, want)


def pin_ulp_bf16(o):
    cases = {1.0: 2.0**-7, 1.5: 2.0**-7, -3.0: 2.0**-6, 2.0**-126: 2.0**-133,
             3 * 2.0**-130: 2.0**-133, 2.0**127: 2.0**120, 0.0: 2.0**-133}
    got = o.ulp_bf16(np.array(list(cases.keys())))
    assert np.array_equal(got, np.array(list(cases.values())))


def pin_f16_round(o):
    # hand cases from round-to-nearest-even on 11 significant bits
    cases = [
        (1.0, 0x3C00),
        (1.0 + 2.0**-11, 0x3C00),            # tie -> even mantissa (0)
        (1.0 + 3 * 2.0**-11, 0x3C02),        # tie -> even mantissa (2)
        (1.0 + 2.0**-11 + 2.0**-30, 0x3C01),  # just above the tie
        (-1.5, 0xBE00),
        (2049.0, 0x6800),                    # quantum 2 at 2^11: tie -> 2048
        (2051.0, 0x6802),                    # tie -> 2052
        (2.0**-14, 0x0400),                  # smallest normal
        (2.0**-14 - 2.0**-25, 0x0400),       # tie between 1023 and 1024 quanta -> normal
        (2.0**-24, 0x0001),                  # smallest subnormal
        (2.0**-25, 0x0000),                  # tie between 0 and 2^-24 -> 0
        (3 * 2.0**-25, 0x0002),              # tie between 1 and 2 quanta -> 2
        (65504.0, 0x7BFF),                   # largest finite
        (65519.0, 0x7BFF),
        (65520.0, 0x7C00),                   # tie with 2^16 -> overflow to inf
        (1e5, 0x7C00),                       # far above the largest finite
        (-70000.0, 0xFC00),
        (-1e9, 0xFC00),
        (0.0, 0x0000),
        (-0.0, 0x8000),
    ]
    got = o.round_f16(np.array([x for x, _ in cases], np.float64))
    for (x, want), g in zip(cases, got.tolist()):
        assert g == want, (x, hex(g), hex(want))
    # agreement with torch's float32 -> float16 round-to-nearest-even
    g = _rng(18)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-30, 18, (20000,),
                                                                  generator=g).float())
    want = x.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = o.round_f16(x.double().numpy())
    assert np.array_equal(got, want)


def pin_ulp_f16(o):
    cases = {1.0: 2.0**-10, 1.5: 2.0**-10, -3.0: 2.0**-9, 1024.0: 1.0, 65504.0: 32.0,
             2.0**-14: 2.0**-24, 3 * 2.0**-20: 2.0**-24, 0.0: 2.0**-24}
    got = o.ulp_f16(np.array(list(cases.keys())))
    assert np.array_equal(got, np.array(list(cases.values())))


# ------------------------------------------------------ sampled entries --

def _padded(g, rows, cols, ld, make):
    """A rows x ld buffer whose first cols columns hold make((rows, cols)) and
    whose padding holds other values of the same kind, so that an element read
    with the wrong leading dimension or index differs."""
    full = make((rows, ld))
    full[:, :cols] = make((rows, cols))
    return full


def pin_sampled(o):
    """The sampled entry points (the checkers of full-size parity tests)
    compute the same elements as the full oracle and as Python integers, with
    padded leading dimensions for A, B and C: a swapped row/column index or a
    wrong leading dimension fails."""
    g = _rng(19)
    rnd = np.random.default_rng(19)
    M, N, K = 37, 53, 29
    n_s = 240
    rows = np.concatenate([[0, M - 1, 0, M - 1], rnd.integers(0, M, n_s)]).astype(np.int64)
    cols = np.concatenate([[0, N - 1, N - 1, 0], rnd.integers(0, N, n_s)]).astype(np.int64)

    def small_ints(shape):
        return torch.randint(-4, 5, shape, generator=g).numpy()

    for layout in (ROW, COL):
        Bshape = (N, K) if layout == COL else (K, N)
        lda, ldb, ldc = K + 3, Bshape[1] + 5, N + 7
        A = _padded(g, M, K, lda, small_ints)
        B = _padded(g, Bshape[0], Bshape[1], ldb, small_ints)
        C = _padded(g, M, N, ldc, small_ints)
        Ap, Bp, Cp = A[:, :K].tolist(), B[:, :Bshape[1]].tolist(), C[:, :N].tolist()
        want = np.array(_py_gemm(Ap, Bp, Cp, 3, -2, layout), np.float64)[rows, cols]
        for in_dtype, out_dtype in ((F32, F32), (BF16, BF16), (F16, F32), (BF16, F32)):
            def enc(x, dt):
                t = torch.from_numpy(x.astype(np.float32))
                if dt == BF16:
                    return _bf16_bits(t)
                if dt == F16:
                    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
                return t.numpy()
            a, b, c = enc(A, in_dtype), enc(B, in_dtype), enc(C, out_dtype)
            ref_s, bound_s = o.gemm_fp_sampled(in_dtype, out_dtype, layout, K, 3.0, a, lda, b,
                                               ldb, -2.0, c, ldc, rows, cols)
            ref_f, bound_f = o.gemm_fp(in_dtype, out_dtype, layout, M, N, K, 3.0, a, lda, b, ldb,
                                       -2.0, c, ldc)
            what = (in_dtype, out_dtype, layout)
            assert np.array_equal(ref_s, ref_f[rows, cols]), ("ref vs full", what)
            assert np.array_equal(bound_s, bound_f[rows, cols]), ("bound vs full", what)
            assert np.array_equal(ref_s, want), ("ref vs Python integers", what)
        # INT8: full range, wrap mod 2^32 with large alpha and beta
        def i8(shape):
            return torch.randint(-128, 128, shape, generator=g, dtype=torch.int8).numpy()

        def i32(shape):
            return torch.randint(-2**31, 2**31, shape, generator=g,
                                 dtype=torch.int64).to(torch.int32).numpy()
        A8 = _padded(g, M, K, lda, i8)
        B8 = _padded(g, Bshape[0], Bshape[1], ldb, i8)
        C32 = _padded(g, M, N, ldc, i32)
        for alpha, beta in ((1, 0), (-7, 3), (1 << 20, 1 << 30)):
            got_s = o.gemm_i8_sampled(layout, K, alpha, A8, lda, B8, ldb, beta, C32, ldc,
                                      rows, cols)
            got_f = o.gemm_i8(layout, M, N, K, alpha, A8, lda, B8, ldb, beta, C32, ldc)
            py = _py_gemm(A8[:, :K].tolist(), B8[:, :Bshape[1]].tolist(), C32[:, :N].tolist(),
                          alpha, beta, layout)
            wrapped = np.array([[((v + 2**31) % 2**32) - 2**31 for v in r] for r in py], np.int64)
            assert np.array_equal(got_s, got_f[rows, cols]), ("i8 vs full", layout, alpha)
            assert np.array_equal(got_s, wrapped[rows, cols]), ("i8 vs Python", layout, alpha)
    # C without its leading dimension is refused, not indexed with a guess
    for call in (lambda: o.gemm_fp_sampled(F32, F32, ROW, 2, 1.0, np.ones(4, np.float32), 2,
                                           np.ones(4, np.float32), 2, 1.0,
                                           np.ones(4, np.float32), None, [1], [1]),
                 lambda: o.gemm_i8_sampled(ROW, 2, 1, np.ones(4, np.int8), 2, np.ones(4, np.int8),
                                           2, 1, np.ones(4, np.int32), None, [1], [1])):
        try:
            call()
        except ValueError:
            continue
        raise AssertionError("sampled call without ldc accepted")


# ---------------------------------------------- A layout, bias, row sums --

def pin_transposed_a(o):
    """A stored K x M (column-major A) must give the same result as the same
    matrix stored M x K; a permutation A detects a transposition."""
    g = _rng(9)
    M, K, N = 7, 11, 5
    A = _f32((M, K), g)
    B = _f32((K, N), g)
    At = np.ascontiguousarray(A.T)
    r_row, _ = o.gemm_fp_ex(F32, F32, ROW, ROW, M, N, K, 1.0, A, K, B, N, 0.0)
    r_col, _ = o.gemm_fp_ex(F32, F32, COL, ROW, M, N, K, 1.0, At, M, B, N, 0.0)
    assert np.array_equal(r_row, r_col), "column-major A"
    rows = torch.randperm(K, generator=g).numpy()[:M]
    P = np.zeros((M, K), np.float32)
    P[np.arange(M), rows] = 1.0
    ref, _ = o.gemm_fp_ex(F32, F32, COL, ROW, M, N, K, 1.0, np.ascontiguousarray(P.T), M, B, N, 0.0)
    assert np.array_equal(ref, B[rows].astype(np.float64)), "P^T stored column-major"
    # INT8 too, with padded leading dimension
    Ai = torch.randint(-128, 128, (K, M + 3), generator=g, dtype=torch.int8)
    Bi = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8)
    got = o.gemm_i8_ex(COL, ROW, M, N, K, 1, Ai.numpy(), M + 3, Bi.numpy(), N)
    want = _py_gemm(Ai[:, :M].t().tolist(), Bi.tolist(), None, 1, 0, ROW)
    assert np.array_equal(got, np.array(want, np.int64)), "int8 column-major A"


def pin_bias(o):
    """The bias row is added once to every row; with alpha = beta = 0 the
    result is the bias itself (the Linear layer's Y = X W^T + b)."""
    g = _rng(10)
    M, K, N = 6, 9, 8
    A = torch.randint(-4, 5, (M, K), generator=g).float().numpy()
    W = torch.randint(-4, 5, (N, K), generator=g).float().numpy()    # [out, in]
    bias = torch.randint(-50, 51, (N,), generator=g).float().numpy()
    ref, _ = o.gemm_fp_ex(F32, F32, ROW, COL, M, N, K, 1.0, A, K, W, K, 0.0, bias=bias)
    want = _py_gemm(A.astype(int).tolist(), W.astype(int).tolist(), None, 1, 0, COL)
    want = np.array(want, np.float64) + bias[None, :]
    assert np.array_equal(ref, want), "X W^T + b"
    ref, _ = o.gemm_fp_ex(F32, F32, ROW, COL, M, N, K, 0.0, A, K, W, K, 0.0, bias=bias)
    assert np.array_equal(ref, np.broadcast_to(bias, (M, N))), "bias alone"
    Ai = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int8)
    Bi = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int8)
    bi = torch.randint(-1000, 1000, (N,), generator=g, dtype=torch.int32)
    got = o.gemm_i8_ex(ROW, ROW, M, N, K, 1, Ai.numpy(), K, Bi.numpy(), N, bias=bi.numpy())
    want = np.array(_py_gemm(Ai.tolist(), Bi.tolist(), None, 1, 0, ROW), np.int64) + bi.numpy()[None, :]
    assert np.array_equal(got, want), "int8 bias"


def pin_sum_rows(o):
    """Column sums against Python integers (the bias gradient)."""
    g = _rng(11)
    R, Cc = 37, 13
    G = torch.randint(-20, 21, (R, Cc + 2), generator=g).float()
    got, bound = o.sum_rows(F32, R, Cc, G.numpy(), Cc + 2)
    want = [sum(int(G[i, j]) for i in range(R)) for j in range(Cc)]
    assert np.array_equal(got, np.array(want, np.float64))
    assert np.allclose(bound, 1e-4 * G[:, :Cc].abs().sum(0).double().numpy())
    got_b, _ = o.sum_rows(BF16, R, Cc, _bf16_bits(G), Cc + 2)
    assert np.array_equal(got_b, got)


# -------------------------------------------------------------------- TF32 --
#
# "Matrix multiplication: arithmetic intensity, tiling and Tensor Core",
# sections 5.5 and 5.7: TF32 keeps the fp32 exponent but only 10 mantissa
# bits, so it is lossy.  How an fp32 value becomes TF32 is not stated; the
# two plain readings, truncation and round-to-nearest-even, are both built
# here from the binary32 encoding (sign, 8-bit exponent, 23-bit fraction).

def _tf32_value(x, mode):
    """Exact value of the fp32 number x with its fraction cut to 10 bits."""
    bits = int(np.array([x], np.float32).view(np.uint32)[0])
    sign = -1 if bits >> 31 else 1
    e = (bits >> 23) & 0xFF
    frac = bits & 0x7FFFFF
    assert 0 < e < 0xFF, "normal numbers only"
    keep, rem = frac >> 13, frac & 0x1FFF
    if mode == "nearest" and (rem > 0x1000 or (rem == 0x1000 and keep & 1)):
        keep += 1   # may carry into the exponent: (1 + 1024/1024) = 2, still exact
    return sign * (1 + Fraction(keep, 1024)) * Fraction(2) ** (e - 127)


def pin_tf32(o):
    g = _rng(12)
    # (a) the reference is the exact product of the stored fp32 operands:
    #     the same as for FP32 inputs, for both layouts, with beta and a bias
    M, N, K = 9, 7, 21
    A = _f32((M, K), g)
    for layout in (ROW, COL):
        B = _f32((N, K) if layout == COL else (K, N), g)
        C = _f32((M, N), g)
        bias = _f32((N,), g)
        ldb = K if layout == COL else N
        r32, b32 = o.gemm_fp_ex(F32, F32, ROW, layout, M, N, K, 1.25, A, K, B, ldb, -0.5, C, N,
                                bias=bias)
        rtf, btf = o.gemm_fp_ex(TF32, F32, ROW, layout, M, N, K, 1.25, A, K, B, ldb, -0.5, C, N,
                                bias=bias)
        assert np.array_equal(r32, rtf), ("tf32 ref", layout)
        assert (btf > b32).all(), "tf32 bound wider than fp32"
    # (b) the bound covers both readings of the TF32 reduction
    rnd = random.Random(13)
    for trial in range(40):
        M, N, K = rnd.randint(1, 6), rnd.randint(1, 6), rnd.randint(1, 9)
        def val():
            return np.float32(rnd.uniform(0.5, 1.0) * rnd.choice((-1, 1)) * 2.0 ** rnd.randint(-30, 30))
        A = np.array([[val() for _ in range(K)] for _ in range(M)], np.float32)
        B = np.array([[val() for _ in range(N)] for _ in range(K)], np.float32)
        C = np.array([[val() for _ in range(N)] for _ in range(M)], np.float32)
        alpha = float(np.float32(rnd.uniform(-2, 2)))
        beta = rnd.choice((0.0, float(np.float32(rnd.uniform(-2, 2)))))
        ref, bound = o.gemm_fp(TF32, F32, ROW, M, N, K, alpha, A, K, B, N, beta, C, N)
        for mode in ("trunc", "nearest"):
            for i in range(M):
                for j in range(N):
                    s = sum((_tf32_value(A[i, k], mode) * _tf32_value(B[k, j], mode)
                             for k in range(K)), Fraction(0))
                    cterm = Fraction(beta) * Fraction(float(C[i, j])) if beta != 0 else 0
                    exact = Fraction(alpha) * s + cterm
                    assert abs(exact - Fraction(float(ref[i, j]))) <= Fraction(float(bound[i, j])), \
                        (trial, mode, i, j)
    # (c) the widening is needed, and not much more than needed: with both
    #     operands just below 1 + 2^-10, truncation loses almost 2^-9 of the
    #     product
    a = np.float32(1.0 + 2.0**-10 - 2.0**-23)
    Ak = np.array([[a]], np.float32)
    ref, bound = o.gemm_fp(TF32, F32, ROW, 1, 1, 1, 1.0, Ak, 1, Ak, 1, 0.0)
    lost = Fraction(float(ref[0, 0])) - _tf32_value(a, "trunc") ** 2
    assert lost > Fraction(2) ** -9 * Fraction(99, 100)
    assert lost <= Fraction(float(bound[0, 0])) < 2 * lost


# --------------------------------------------------------------- CSR SpMV --
#
# "AI Programming: Matrix Product", sections "COO", "CSR" and "SpMV": a CSR
# matrix keeps values and column indices of the nonzeros row after row, and
# row_offsets[i] .. row_offsets[i+1] is row i's half-open range; SpMV
# multiplies every nonzero by the vector element of its column and sums the
# products of each row.  The checks build the same matrix independently, as
# COO triplets (row, column, value), and compute the dense product from them.

def _csr_from_triplets(n_rows, triplets):
    """CSR arrays from (row, col, value) triplets by the page's recipe: a
    histogram of row indices, a prefix sum into row_offsets, then a scatter
    (keeping the triplets' order within a row)."""
    counts = [0] * n_rows
    for r, _, _ in triplets:
        counts[r] += 1
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    fill = offs[:-1].copy()
    cols = [0] * len(triplets)
    vals = [0.0] * len(triplets)
    for r, c, v in triplets:
        cols[fill[r]] = c
        vals[fill[r]] = v
        fill[r] += 1
    return (np.array(offs, np.int32), np.array(cols, np.int32), np.array(vals, np.float32))


def _dense_spmv(n_rows, triplets, x, alpha, beta, y):
    """alpha * A x + beta * y, exactly, with A summed from the triplets."""
    out = []
    for i in range(n_rows):
        s = sum((Fraction(float(np.float32(v))) * Fraction(float(x[c]))
                 for r, c, v in triplets if r == i), Fraction(0))
        t = Fraction(alpha) * s
        if beta != 0:
            t += Fraction(beta) * Fraction(float(y[i]))
        out.append(t)
    return out


def pin_spmv(o):
    # (a) the page's example, its COO and CSR forms taken from the golden file
    here = os.path.dirname(os.path.abspath(__file__))
    with open(os.path.join(here, "golden", "csr_example.json")) as f:
        ex = json.load(f)
    m, n = ex["shape"]
    coo = ex["coo"]
    trip = list(zip(coo["rows"], coo["cols"], coo["values"]))
    csr = ex["csr"]
    for x in ([1, 2, 3, 4], [-1, 0.5, 2, -3]):
        xs = np.array(x, np.float32)
        ref, _ = o.spmv_csr(m, n, np.array(csr["row_offsets"], np.int32),
                            np.array(csr["column_indices"], np.int32),
                            np.array(csr["values"], np.float32), xs)
        assert [Fraction(float(v)) for v in ref] == _dense_spmv(m, trip, xs, 1, 0, None), x
    # (b) integer values: exact, with empty rows, one long row and a column
    #     repeated within a row (the repeats add up, as in the dense matrix)
    rnd = random.Random(14)
    for trial in range(6):
        n_rows, n_cols = rnd.randint(1, 40), rnd.randint(1, 30)
        trip = []
        for i in range(n_rows):
            length = rnd.choice((0, 0, 1, 2, 3, 5, 8))
            if i == n_rows // 2:
                length = 300
            for _ in range(length):
                trip.append((i, rnd.randrange(n_cols), float(rnd.randint(-9, 9))))
        if trip:
            r, c, _ = trip[0]
            trip.append((r, c, 4.0))          # a repeated (row, column) pair
        trip.sort(key=lambda t: t[0])
        offs, cols, vals = _csr_from_triplets(n_rows, trip)
        x = np.array([rnd.randint(-7, 7) for _ in range(n_cols)], np.float32)
        y = np.array([rnd.randint(-5, 5) for _ in range(n_rows)], np.float32)
        for alpha, beta in ((1.0, 0.0), (3.0, -2.0), (0.0, 1.5)):
            ref, _ = o.spmv_csr(n_rows, n_cols, offs, cols, vals, x, alpha, beta, y)
            want = _dense_spmv(n_rows, trip, x, alpha, beta, y)
            assert [Fraction(float(v)) for v in ref] == want, (trial, alpha, beta)
    # (c) fp32 values with spread exponents: within the fp64 summation bound,
    #     and the returned bound is the documented one
    u = Fraction(1, 2**53)
    for trial in range(10):
        n_rows, n_cols = rnd.randint(1, 12), rnd.randint(1, 12)
        trip = [(rnd.randrange(n_rows), rnd.randrange(n_cols),
                 float(np.float32(rnd.uniform(-1, 1) * 2.0 ** rnd.randint(-20, 20))))
                for _ in range(rnd.randint(0, 40))]
        trip.sort(key=lambda t: t[0])
        offs, cols, vals = _csr_from_triplets(n_rows, trip)
        x = np.array([rnd.uniform(-1, 1) * 2.0 ** rnd.randint(-10, 10) for _ in range(n_cols)],
                     np.float32)
        y = np.array([rnd.uniform(-1, 1) for _ in range(n_rows)], np.float32)
        ref, bound = o.spmv_csr(n_rows, n_cols, offs, cols, vals, x, 0.75, 0.5, y)
        want = _dense_spmv(n_rows, trip, x, 0.75, 0.5, y)
        for i in range(n_rows):
            terms = [Fraction(float(np.float32(v))) * Fraction(float(x[c])) for r, c, v in trip if r == i]
            mag = Fraction(3, 4) * sum((abs(t) for t in terms), Fraction(0)) + \
                abs(Fraction(1, 2) * Fraction(float(y[i])))
            k = len(terms) + 2
            assert abs(Fraction(float(ref[i])) - want[i]) <= k * u / (1 - k * u) * mag + \
                Fraction(2) ** -1074, (trial, i)
            want_bound = Fraction(1, 10**4) * Fraction(3, 4) * sum((abs(t) for t in terms), Fraction(0)) + \
                abs(Fraction(1, 2) * Fraction(float(y[i]))) * Fraction(1, 2**22)
            assert abs(Fraction(float(bound[i])) - want_bound) <= 8 * u * want_bound + Fraction(2) ** -1074
    # (d) identity and permutation matrices: exact copies of x
    n_ = 17
    x = np.array([rnd.uniform(-1, 1) for _ in range(n_)], np.float32)
    offs, cols, vals = _csr_from_triplets(n_, [(i, i, 1.0) for i in range(n_)])
    ref, _ = o.spmv_csr(n_, n_, offs, cols, vals, x)
    assert np.array_equal(ref, x.astype(np.float64)), "identity"
    perm = list(range(n_))
    rnd.shuffle(perm)
    offs, cols, vals = _csr_from_triplets(n_, [(i, perm[i], 1.0) for i in range(n_)])
    ref, _ = o.spmv_csr(n_, n_, offs, cols, vals, x)
    assert np.array_equal(ref, x[perm].astype(np.float64)), "permutation"
    # (e) BLAS semantics: beta == 0 never reads y, alpha == 0 never reads A or x
    offs, cols, vals = _csr_from_triplets(3, [(0, 1, 2.0), (2, 0, -1.0)])
    ynan = np.full(3, np.nan, np.float32)
    ref, bound = o.spmv_csr(3, 2, offs, cols, vals, np.array([1, 2], np.float32), 1.0, 0.0, ynan)
    assert np.isfinite(ref).all() and np.isfinite(bound).all(), "beta=0 read y"
    y = np.array([1, -2, 4], np.float32)
    ref, _ = o.spmv_csr(3, 2, offs, cols, np.full(2, np.nan, np.float32),
                        np.full(2, np.nan, np.float32), 0.0, -0.5, y)
    assert np.array_equal(ref, -0.5 * y.astype(np.float64)), "alpha=0 read A/x"
    # (f) arrays that are not a CSR matrix of the shape are rejected
    bad = [(np.array([0, 2, 1, 2], np.int32), np.array([0, 1], np.int32)),   # decreasing
           (np.array([1, 1, 2, 2], np.int32), np.array([0, 1], np.int32)),   # first offset != 0
           (np.array([0, 1, 2, 2], np.int32), np.array([0, 2], np.int32))]   # column 2 of 2
    for offs, cols in bad:
        try:
            o.spmv_csr(3, 2, offs, cols, np.ones(2, np.float32), np.ones(2, np.float32))
        except ValueError:
            continue
        raise AssertionError(("accepted", offs.tolist(), cols.tolist()))


ALL_PINS = [pin_identity, pin_permutation, pin_alpha_beta, pin_small_integers, pin_int8,
            pin_tiny_rational, pin_bf16_decode, pin_f16_decode, pin_bf16_round, pin_ulp_bf16,
            pin_f16_round, pin_ulp_f16, pin_sampled, pin_transposed_a, pin_bias, pin_sum_rows,
            pin_tf32, pin_spmv]
