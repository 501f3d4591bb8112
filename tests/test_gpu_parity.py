"""GPU parity: every kernel family against the CPU oracle, through the C ABI.

Sizes span several tiles and a ragged tail at sizes the oracle finishes in
seconds; the full-size workloads are checked on sampled elements (every
element of the first and last rows and columns, plus random ones).
"""
import numpy as np
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, assert_exact, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

S, T, K_, GEN = dga.PATH_SIMT, dga.PATH_TCGEN05, dga.PATH_SKINNY, dga.PATH_GENERIC


def _mats(in_dtype, out_dtype, layout_b, M, N, K, seed, dist=("uniform",), lda=None, ldb=None,
          ldc=None):
    g = torch.Generator().manual_seed(seed)
    lda = lda or K
    ldc = ldc or N
    if layout_b == gen.COL_MAJOR:
        ldb = ldb or K
        Bshape = (N, ldb)
    else:
        ldb = ldb or N
        Bshape = (K, ldb)
    if in_dtype == gen.I8:
        dist = ("int8",)
    A = gen.random_matrix((M, lda), in_dtype, g, dist)
    B = gen.random_matrix(Bshape, in_dtype, g, dist)
    C = gen.random_matrix((M, ldc), out_dtype, g, ("int8",) if out_dtype == gen.I32 else ("uniform",))
    return A, B, C


def check(path, in_dtype, out_dtype, layout_b, M, N, K, alpha=1.0, beta=0.0, seed=0, lda=None,
          ldb=None, ldc=None, offsets=(0, 0, 0), dist=("uniform",)):
    A, B, C = _mats(in_dtype, out_dtype, layout_b, M, N, K, seed, dist, lda, ldb, ldc)
    got = run_gpu(path, in_dtype, out_dtype, layout_b, A, B, C, alpha, beta, M=M, N=N, K=K,
                  offsets=offsets)
    assert dga.dga_last_path() == path
    ref, bound = oracle_ref(in_dtype, out_dtype, layout_b, A, B, C, alpha, beta, M=M, N=N, K=K)
    gm = got[:, :N]
    what = f"path={dga.PATH_NAMES[path]} in={in_dtype} out={out_dtype} B={layout_b} {M}x{N}x{K}"
    if in_dtype == gen.I8:
        assert_exact(gm, ref, gen.I32, what)
    else:
        assert_close(gm, ref, bound, out_dtype, what)
    # padding columns of C (ldc > N) must be untouched
    if C.shape[1] > N:
        assert torch.equal(got[:, N:], C[:, N:]), "wrote outside C"


# ------------------------------------------------------------------- SIMT --

SIMT_SHAPES = [(1, 1, 1), (7, 9, 3), (128, 128, 8), (129, 257, 33), (255, 129, 17),
               (256, 256, 256), (300, 200, 1001), (64, 520, 96)]


@pytest.mark.parametrize("M,N,K", SIMT_SHAPES)
def test_simt_shapes(M, N, K):
    check(S, gen.F32, gen.F32, gen.ROW_MAJOR, M, N, K, 1.5, 0.5, seed=M + N + K)


def test_simt_config_256():
    # FP32 M=N=K=256, alpha=1, beta=0, inputs uniform[-1,1) from seed 0
    w = gen.WORKLOADS["fp32_256"]
    A, B, _ = gen.make_inputs(w)
    C = torch.zeros(w.M, w.N)
    got = run_gpu(S, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, w.alpha, w.beta)
    ref, bound = oracle_ref(gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, w.alpha, w.beta)
    assert_close(got, ref, bound, gen.F32, "fp32_256")


@pytest.mark.parametrize("M,N,K", [(1152, 1152, 1024), (1000, 1100, 1500), (300, 300, 3000),
                                   (1408, 1408, 2048)])
def test_simt_split_tail(M, N, K):
    # fewer tiles than resident blocks: every tile is split along K into
    # workspace partials that a second kernel reduces
    A, B, C = _mats(gen.F32, gen.F32, gen.ROW_MAJOR, M, N, K, 21)
    got = run_gpu(S, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.5, 0.5)
    assert dga.dga_last_launch_count() == 2, "expected the split tail"
    ref, bound = oracle_ref(gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.5, 0.5)
    assert_close(got, ref, bound, gen.F32, f"split tail {M}x{N}x{K}")
    # without workspace the same call runs whole tiles, one launch
    got2 = run_gpu(S, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.5, 0.5, workspace=False)
    assert dga.dga_last_launch_count() == 1
    assert_close(got2, ref, bound, gen.F32, f"whole tiles {M}x{N}x{K}")


@pytest.mark.parametrize("layout", [gen.ROW_MAJOR, gen.COL_MAJOR])
def test_simt_split_last_wave(layout):
    """2560 x 2432 x 768 (N not a multiple of 256, so not the wide kernel's
    shape): 380 tiles of 128 x 128 on 304 two-per-SM slots, a last wave
    under a third full.  The top 2048 rows (16 tile rows, 304 tiles) run on
    the interior kernel; the bottom 512 rows (76 tiles) are cut into three K
    parts by the general kernel and reduced by a third launch.  Checked
    against the oracle on the rows around the band boundary and the last
    rows."""
    import oracle
    M, N = 2560, 2432
    K = 768
    A, B, C = _mats(gen.F32, gen.F32, layout, M, N, K, seed=21)
    got = run_gpu(S, gen.F32, gen.F32, layout, A, B, C, 1.5, 0.5, M=M, N=N, K=K)
    assert dga.dga_last_launch_count() == 3
    for r0, r1 in ((1920, 2176), (2432, 2560)):
        ref, bound = oracle.gemm_fp(gen.F32, gen.F32, layout, r1 - r0, N, K, 1.5,
                                    A[r0:r1].contiguous(), K, B, B.shape[1], 0.5,
                                    C[r0:r1].contiguous(), N)
        assert_close(got[r0:r1], ref, bound, gen.F32, f"rows {r0}-{r1}")


def test_simt_padded_ld():
    check(S, gen.F32, gen.F32, gen.ROW_MAJOR, 130, 70, 50, 1.0, 1.0, lda=52, ldb=76, ldc=73)


# ---------------------------------------------------------------- tcgen05 --

TC_SHAPES = [(128, 256, 64), (1, 1, 1), (129, 257, 65), (300, 520, 1000), (256, 512, 4096),
             (1000, 300, 136), (128, 16, 8)]


@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_tc_bf16_f32(M, N, K):
    check(T, gen.BF16, gen.F32, gen.COL_MAJOR, M, N, K, 1.0, 0.0, seed=M * 7 + K)


@pytest.mark.parametrize("M,N,K", [(200, 300, 264), (129, 40, 72)])
def test_tc_bf16_bf16_beta(M, N, K):
    check(T, gen.BF16, gen.BF16, gen.COL_MAJOR, M, N, K, 0.75, -1.25, seed=K)


@pytest.mark.parametrize("M,N,K", [(200, 300, 264), (64, 1000, 520)])
def test_tc_row_major_b(M, N, K):
    check(T, gen.BF16, gen.F32, gen.ROW_MAJOR, M, N, K, 1.0, 0.5, seed=N)


def test_tc_f16():
    check(T, gen.F16, gen.F32, gen.COL_MAJOR, 257, 300, 200, 1.0, 0.0)
    check(T, gen.F16, gen.F16, gen.COL_MAJOR, 140, 260, 96, 1.0, 0.0)


def test_tc_unaligned_lda_and_pointers():
    check(T, gen.BF16, gen.F32, gen.COL_MAJOR, 150, 270, 99, 1.0, 0.0, lda=101, ldb=99)
    check(T, gen.BF16, gen.F32, gen.COL_MAJOR, 150, 270, 128, 1.0, 0.0, offsets=(1, 3, 1))


@pytest.mark.parametrize("M,N,K", [(77, 91, 600), (259, 515, 1100), (128, 256, 512),
                                   (130, 300, 1537), (1, 1, 1)])
def test_tc_int8(M, N, K):
    check(T, gen.I8, gen.I32, gen.ROW_MAJOR, M, N, K, 1, 0, seed=K)


def test_tc_int8_col_major_alpha_beta():
    check(T, gen.I8, gen.I32, gen.COL_MAJOR, 140, 270, 700, -3, 7, seed=3)


def test_tc_int8_one_repack_launch():
    # both operands are repacked (A by rows, the row-major B transposed to
    # K-major) in one launch, and the GEMM follows it as a programmatic
    # dependent: two launches, the result still bit-exact (ragged sizes, ldb
    # not a multiple of 16)
    check(T, gen.I8, gen.I32, gen.ROW_MAJOR, 300, 259, 1030, 1, 0, seed=4, ldb=263)
    assert dga.dga_last_launch_count() == 2
    # bf16 with leading dimensions TMA cannot express (lda = 99, ldb = 101):
    # both repacked, again in one launch
    check(T, gen.BF16, gen.F32, gen.COL_MAJOR, 260, 140, 99, 1.0, 0.0, seed=5, ldb=101)
    assert dga.dga_last_launch_count() == 2


def test_tc_int8_extreme_magnitudes():
    # all -128: every product is +2^14, the largest partial sums there are
    M, N, K = 130, 260, 2048
    A = torch.full((M, K), -128, dtype=torch.int8)
    B = torch.full((K, N), -128, dtype=torch.int8)
    C = torch.zeros(M, N, dtype=torch.int32)
    got = run_gpu(T, gen.I8, gen.I32, gen.ROW_MAJOR, A, B, C, 1, 0)
    assert (got == K * 16384).all()
    # alternating signs with the largest magnitudes
    A = torch.where(torch.arange(K) % 2 == 0, -128, 127).to(torch.int8).repeat(M, 1)
    got = run_gpu(T, gen.I8, gen.I32, gen.ROW_MAJOR, A, B, C, 1, 0)
    ref, _ = oracle_ref(gen.I8, gen.I32, gen.ROW_MAJOR, A, B, C, 1, 0)
    assert_exact(got, ref, gen.I32, "alternating")


# ------------------------------------------------------------------- TF32 --
#
# fp32 operands multiplied as TF32 on the tensor cores (opt-in, lossy): the
# oracle's reference is the exact fp32 product and its bound is widened for
# operands kept to 10 fraction bits.

TF32_SHAPES = [(128, 256, 32), (1, 1, 1), (129, 257, 65), (300, 520, 1000), (256, 512, 4096),
               (1000, 300, 136), (128, 16, 4), (77, 91, 600)]


@pytest.mark.parametrize("M,N,K", TF32_SHAPES)
def test_tc_tf32(M, N, K):
    check(T, gen.TF32, gen.F32, gen.COL_MAJOR, M, N, K, 1.0, 0.0, seed=M * 3 + K)


@pytest.mark.parametrize("M,N,K", [(200, 300, 264), (64, 1000, 520)])
def test_tc_tf32_row_major_b_beta(M, N, K):
    # a row-major B is transposed into the workspace (TF32 reads K-major only)
    check(T, gen.TF32, gen.F32, gen.ROW_MAJOR, M, N, K, 1.5, 0.5, seed=N)


def test_tc_tf32_unaligned():
    check(T, gen.TF32, gen.F32, gen.COL_MAJOR, 150, 270, 99, 1.0, 0.0, lda=101, ldb=99)
    check(T, gen.TF32, gen.F32, gen.COL_MAJOR, 150, 270, 128, 1.0, 0.0, offsets=(1, 3, 1))


def test_tf32_is_opt_in():
    # fp32 inputs never take the TF32 path; TF32 inputs go to the tensor cores
    A, B, C = _mats(gen.F32, gen.F32, gen.COL_MAJOR, 256, 256, 256, 4)
    run_gpu(dga.PATH_AUTO, gen.F32, gen.F32, gen.COL_MAJOR, A, B, C, 1, 0)
    assert dga.dga_last_path() == S
    run_gpu(dga.PATH_AUTO, gen.TF32, gen.F32, gen.COL_MAJOR, A, B, C, 1, 0)
    assert dga.dga_last_path() == T
    # the generic family accepts TF32 too (it multiplies exactly, within the bound)
    check(GEN, gen.TF32, gen.F32, gen.ROW_MAJOR, 45, 71, 37, 1.25, -0.5, offsets=(1, 1, 1))


# ----------------------------------------------------------------- skinny --

@pytest.mark.parametrize("M,N,K", [(1, 8192, 8192), (8, 1000, 1024), (16, 96, 256), (3, 33, 72),
                                   (9, 64, 8), (16, 40, 4104), (5, 15000, 200),
                                   (16, 20000, 136), (2, 152, 520), (16, 2432, 64)])
def test_skinny(M, N, K):
    # (5, 15000): 98-99 rows per CTA; (16, 20000): two waves of CTAs;
    # (2, 152): one 16-row group per CTA on 9 CTAs; K % 256 != 0 tails
    check(K_, gen.BF16, gen.BF16, gen.COL_MAJOR, M, N, K, 1.0, 0.0, seed=M + N)


def test_skinny_f32_out_beta():
    check(K_, gen.BF16, gen.F32, gen.COL_MAJOR, 12, 300, 520, 2.0, -1.0)
    check(K_, gen.F16, gen.F16, gen.COL_MAJOR, 16, 130, 264, 1.0, 0.5)


# ---------------------------------------------------------------- generic --

@pytest.mark.parametrize("pair", [(gen.F32, gen.F32), (gen.BF16, gen.F32), (gen.BF16, gen.BF16),
                                  (gen.F16, gen.F32), (gen.F16, gen.F16), (gen.I8, gen.I32)])
@pytest.mark.parametrize("layout", [gen.ROW_MAJOR, gen.COL_MAJOR])
def test_generic_all_pairs(pair, layout):
    check(GEN, pair[0], pair[1], layout, 45, 71, 37, 1 if pair[0] == gen.I8 else 1.25,
          2 if pair[0] == gen.I8 else -0.5, offsets=(1, 1, 1))


# ------------------------------------------------- exactness and semantics --

@pytest.mark.parametrize("path,in_dtype,out_dtype,layout", [
    (S, gen.F32, gen.F32, gen.ROW_MAJOR), (T, gen.BF16, gen.F32, gen.COL_MAJOR),
    (T, gen.BF16, gen.BF16, gen.ROW_MAJOR), (K_, gen.BF16, gen.BF16, gen.COL_MAJOR),
    (GEN, gen.F32, gen.F32, gen.COL_MAJOR), (T, gen.F16, gen.F32, gen.COL_MAJOR),
    (T, gen.TF32, gen.F32, gen.COL_MAJOR), (T, gen.TF32, gen.F32, gen.ROW_MAJOR),
    (K_, gen.F16, gen.F32, gen.COL_MAJOR)])
def test_small_integers_bit_exact(path, in_dtype, out_dtype, layout):
    # small integers are exact in every input format (TF32 included: 10
    # fraction bits) and every partial sum stays below 2^24
    M = 16 if path == K_ else 150
    N, K = 270, 520
    g = torch.Generator().manual_seed(11)
    A = gen.small_int_matrix((M, K), in_dtype, g)
    B = gen.small_int_matrix((N, K) if layout == gen.COL_MAJOR else (K, N), in_dtype, g)
    C = gen.small_int_matrix((M, N), out_dtype, g)
    got = run_gpu(path, in_dtype, out_dtype, layout, A, B, C, 1.0, 1.0)
    ref, _ = oracle_ref(in_dtype, out_dtype, layout, A, B, C, 1.0, 1.0)
    assert_exact(got, ref, out_dtype, f"small ints path {path}")


@pytest.mark.parametrize("path,in_dtype,layout", [
    (S, gen.F32, gen.ROW_MAJOR), (T, gen.BF16, gen.COL_MAJOR), (T, gen.BF16, gen.ROW_MAJOR),
    (GEN, gen.BF16, gen.COL_MAJOR), (K_, gen.BF16, gen.COL_MAJOR), (T, gen.TF32, gen.COL_MAJOR),
    (T, gen.TF32, gen.ROW_MAJOR)])
def test_permutation_detects_transpose(path, in_dtype, layout):
    # A = P (a row selection), so C = B[rows]: exact, and any transposition of B fails
    M = 16 if path == K_ else 140
    K, N = 200, 136
    g = torch.Generator().manual_seed(5)
    rows = torch.randperm(K, generator=g)[:M]
    A = torch.zeros(M, K).index_put_((torch.arange(M), rows), torch.ones(M)).to(gen.TORCH_DTYPE[in_dtype])
    Bkn = gen.random_matrix((K, N), in_dtype, g)
    B = Bkn.t().contiguous() if layout == gen.COL_MAJOR else Bkn
    out_dtype = gen.F32
    C = torch.zeros(M, N)
    got = run_gpu(path, in_dtype, out_dtype, layout, A, B, C, 1.0, 0.0)
    want = Bkn[rows].float()
    if in_dtype == gen.TF32:
        # one nonzero product per output: B's value as the tensor core keeps
        # it, within 2^-10 of its magnitude (truncated or rounded)
        assert (torch.abs(got - want) <= torch.abs(want) * 2.0 ** -10).all()
        assert torch.equal(got == 0, want == 0)
    else:
        assert torch.equal(got, want)


@pytest.mark.parametrize("path", [S, T, K_, GEN])
def test_beta_zero_ignores_nan_c(path):
    in_dtype = gen.F32 if path in (S, GEN) else gen.BF16
    layout = gen.ROW_MAJOR if path in (S, GEN) else gen.COL_MAJOR
    M = 8 if path == K_ else 70
    A, B, C = _mats(in_dtype, gen.F32, layout, M, 90, 64, 1)
    C = torch.full_like(C, float("nan"))
    got = run_gpu(path, in_dtype, gen.F32, layout, A, B, C, 1.0, 0.0)
    assert torch.isfinite(got).all()


def test_alpha_zero_and_k_zero():
    A, B, C = _mats(gen.F32, gen.F32, gen.ROW_MAJOR, 33, 45, 20, 2)
    Anan = torch.full_like(A, float("nan"))
    got = run_gpu(dga.PATH_AUTO, gen.F32, gen.F32, gen.ROW_MAJOR, Anan, B, C, 0.0, 2.0)
    assert torch.equal(got, 2.0 * C)
    got = run_gpu(dga.PATH_AUTO, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.0, 0.0, K=0)
    assert torch.equal(got, torch.zeros_like(C))


def test_m_or_n_zero_touches_nothing():
    A, B, C = _mats(gen.F32, gen.F32, gen.ROW_MAJOR, 4, 4, 4, 3)
    got = run_gpu(dga.PATH_AUTO, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.0, 0.0, M=0)
    assert torch.equal(got, C)


def test_auto_selection():
    cases = [
        (gen.F32, gen.F32, gen.ROW_MAJOR, 64, 64, 64, S),
        (gen.BF16, gen.F32, gen.COL_MAJOR, 256, 256, 256, T),
        (gen.BF16, gen.BF16, gen.COL_MAJOR, 8, 512, 512, K_),
        (gen.I8, gen.I32, gen.ROW_MAJOR, 64, 64, 64, T),
    ]
    for in_dtype, out_dtype, layout, M, N, K, want in cases:
        A, B, C = _mats(in_dtype, out_dtype, layout, M, N, K, 4)
        run_gpu(dga.PATH_AUTO, in_dtype, out_dtype, layout, A, B, C, 1, 0)
        assert dga.dga_last_path() == want, (in_dtype, layout, M)


def test_deterministic_repeats():
    A, B, C = _mats(gen.BF16, gen.F32, gen.COL_MAJOR, 300, 600, 777, 9)
    outs = [run_gpu(T, gen.BF16, gen.F32, gen.COL_MAJOR, A, B, C, 1.0, 0.0) for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    A, B, C = _mats(gen.F32, gen.F32, gen.ROW_MAJOR, 300, 600, 777, 9)
    outs = [run_gpu(S, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.0, 0.0) for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_overlap_rejected():
    dev = torch.device("cuda")
    buf = torch.zeros(64 * 64 * 2, device=dev)
    import ctypes
    one = ctypes.c_float(1.0)
    zero = ctypes.c_float(0.0)
    st = dga.dga_gemm_ex(gen.F32, gen.F32, gen.ROW_MAJOR, 64, 64, 64, ctypes.byref(one),
                         buf.data_ptr(), 64, buf.data_ptr() + 64 * 64 * 4, 64, ctypes.byref(zero),
                         buf.data_ptr() + 32 * 64 * 4, 64, None, 0, dga.PATH_AUTO,
                         torch.cuda.current_stream().cuda_stream)
    assert st == dga.ERR_OVERLAP


def test_forced_path_rejects_unfit_args():
    A, B, C = _mats(gen.F32, gen.F32, gen.ROW_MAJOR, 8, 8, 8, 1)
    run_gpu(T, gen.F32, gen.F32, gen.ROW_MAJOR, A, B, C, 1.0, 0.0, expect=dga.ERR_PATH)


# ------------------------------------------- full-size workloads, sampled --

def _sample(M, N, n, seed):
    g = np.random.default_rng(seed)
    rows = [g.integers(0, M, n)]
    cols = [g.integers(0, N, n)]
    for r in (0, 1, M - 2, M - 1):
        if 0 <= r < M:
            rows.append(np.full(N, r))
            cols.append(np.arange(N))
    for c in (0, 1, N - 2, N - 1):
        if 0 <= c < N:
            rows.append(np.arange(M))
            cols.append(np.full(M, c))
    return np.concatenate(rows), np.concatenate(cols)


@pytest.mark.parametrize("name", ["fp32_4096", "bf16_8192", "skinny_m1", "skinny_m8",
                                  "skinny_m16", "int8_ragged", "f16_8192", "bf16_8192_rowb",
                                  "tf32_8192"])
def test_full_size_workload(name):
    import oracle
    w = gen.WORKLOADS[name]
    A, B, C0 = gen.make_inputs(w, with_c=True)
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C0.to(dev)
    Bview = Bd.t() if w.layout_b == gen.COL_MAJOR else Bd
    dga.gemm(Ad, Bview, Cd, w.alpha, w.beta, tf32=w.in_dtype == gen.TF32)
    torch.cuda.synchronize()
    got = Cd.cpu()
    ldb = w.K if w.layout_b == gen.COL_MAJOR else w.N
    rows, cols = _sample(w.M, w.N, 65536, 1)
    if w.in_dtype == gen.I8:
        want = oracle.gemm_i8_sampled(w.layout_b, w.K, w.alpha, A, w.K, B, ldb, w.beta, C0, w.N,
                                      rows, cols)
        assert np.array_equal(got.numpy()[rows, cols], want)
        return
    ref, bound = oracle.gemm_fp_sampled(w.in_dtype, w.out_dtype, w.layout_b, w.K, w.alpha, A,
                                        w.K, B, ldb, w.beta, C0, w.N, rows, cols)
    assert_close(got[torch.from_numpy(rows), torch.from_numpy(cols)], ref, bound, w.out_dtype, name)
