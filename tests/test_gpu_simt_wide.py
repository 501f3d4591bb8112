"""GPU parity of the FP32 SIMT path's wide kernel (128 x 256 block tiles, one
block per SM) and of its stream-K schedule, through the C ABI, against the
CPU oracle element by element.

The wide kernel runs for problems of whole 128 x 256 tiles with at least one
full wave of them (152 tiles on a GB300).  A whole number of waves runs tile
by tile, one launch; otherwise the whole waves run tile by tile, a second
kernel's blocks (one per SM) each take an equal contiguous share of the
remaining (tile, 16-deep K-slice) units, and the tiles split between blocks
are summed in block order by a third kernel.  The shapes below reach: one exact wave,
stream-K with a small and a large remainder of tiles, K of one and of three
slices per tile (a share boundary can then fall only between tiles, or at a
third of one), and a deep K; without the workspace the 128 x 128 kernel (or,
for a last wave more than half full, whole wide tiles) runs instead.  Every
operand layout pair is covered, with beta and a bias row, and with
small-integer inputs the result must be exact.  The GEMM is the BLAS update
of "AI Programming: Matrix Product", section "Dense matrix multiplication".
"""
import ctypes

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, assert_exact

pytestmark = pytest.mark.gpu

S = dga.PATH_SIMT
WBM, WBN = 128, 256


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _operands(layout_a, layout_b, M, N, K, seed, small_ints):
    g = torch.Generator().manual_seed(seed)

    def draw(shape):
        if small_ints:
            return gen.small_int_matrix(shape, gen.F32, g, -64, 63)
        return gen.random_matrix(shape, gen.F32, g)
    A = draw((M, K) if layout_a == gen.ROW_MAJOR else (K, M))
    B = draw((K, N) if layout_b == gen.ROW_MAJOR else (N, K))
    C = draw((M, N))
    bias = draw((1, N)).reshape(N)
    return A, B, C, bias


def _run(layout_a, layout_b, M, N, K, A, B, C, bias, alpha, beta, workspace=True):
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    bd = bias.to(dev) if bias is not None else None
    lda, ldb, ldc = A.shape[1], B.shape[1], C.shape[1]
    ws_bytes = dga.dga_gemm_general_workspace_size(gen.F32, gen.F32, layout_a, layout_b, M, N, K,
                                                   lda, ldb, ldc, S)
    if not workspace:
        ws_bytes = 0
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = ctypes.c_float(alpha), ctypes.c_float(beta)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_general(gen.F32, gen.F32, layout_a, layout_b, M, N, K, ctypes.byref(al),
                              Ad.data_ptr(), lda, Bd.data_ptr(), ldb, ctypes.byref(be),
                              Cd.data_ptr(), ldc, bd.data_ptr() if bd is not None else None,
                              ws.data_ptr() if ws_bytes else None, ws_bytes, S, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    assert dga.dga_last_path() == S
    return Cd.cpu(), dga.dga_last_launch_count()


def _stream_k(M, N, sms):
    """Whether the wide kernel takes the stream-K schedule (the tile count is
    not a whole number of waves), from the rule rather than the library."""
    return ((M // WBM) * (N // WBN)) % sms != 0


def _case_shapes(sms):
    """(name, M, N, K) for each schedule case on a device with `sms` SMs (8
    tile columns; the tile rows make one wave, or a wave and a remainder)."""
    n = 8 * WBN
    one = sms // 8 * WBM if sms % 8 == 0 else sms * WBM
    if sms % 8 != 0:
        n = WBN
    more = one + WBM
    return [
        ("one_wave", one, n, 272),
        ("sk_small_tail", more, n, 512),
        ("sk_one_slice", more, n, 16),
        ("sk_three_slices", more, n, 48),
        ("sk_large_tail", one + (sms // 8 * 2 // 3 + 1) * WBM, n, 64),
        ("sk_deep", more, n, 1024),
    ]


LAYOUTS = [(gen.ROW_MAJOR, gen.ROW_MAJOR), (gen.ROW_MAJOR, gen.COL_MAJOR),
           (gen.COL_MAJOR, gen.ROW_MAJOR), (gen.COL_MAJOR, gen.COL_MAJOR)]


@pytest.mark.parametrize("case", range(6))
@pytest.mark.parametrize("layouts", LAYOUTS, ids=["rr", "rc", "cr", "cc"])
def test_wide_schedule_exact_small_integers(case, layouts):
    # integer inputs in [-64, 63] with K <= 1024: every partial sum is an
    # integer of magnitude at most 1024 * 64 * 64 + 2 * 64 < 2^24, so every FMA
    # order gives the exact result, bias and beta included (alpha = 1,
    # beta = -1, integer C and bias)
    sms = _sms()
    name, M, N, K = _case_shapes(sms)[case]
    la, lb = layouts
    A, B, C, bias = _operands(la, lb, M, N, K, seed=case * 7 + la * 2 + lb, small_ints=True)
    got, launches = _run(la, lb, M, N, K, A, B, C, bias, 1.0, -1.0)
    assert (M // WBM) * (N // WBN) >= sms, name
    assert launches == (3 if _stream_k(M, N, sms) else 1), (name, launches)
    ref, _ = oracle.gemm_fp_ex(gen.F32, gen.F32, la, lb, M, N, K, 1.0, A, A.shape[1], B,
                               B.shape[1], -1.0, C, N, bias)
    assert_exact(got, ref, gen.F32, f"{name} A={la} B={lb}")


@pytest.mark.parametrize("layouts", LAYOUTS, ids=["rr", "rc", "cr", "cc"])
@pytest.mark.parametrize("with_bias,beta", [(False, 0.0), (False, 0.5), (True, 0.0), (True, 0.5)])
def test_wide_schedule_uniform(layouts, with_bias, beta):
    # uniform[-1, 1) inputs within the oracle's bound; the schedule case
    # rotates with the layout and epilogue so each meets several of them
    sms = _sms()
    case = (LAYOUTS.index(layouts) + 2 * int(with_bias) + int(beta != 0)) % 6
    name, M, N, K = _case_shapes(sms)[case]
    la, lb = layouts
    A, B, C, bias = _operands(la, lb, M, N, K, seed=100 + case, small_ints=False)
    bias = bias if with_bias else None
    got, _ = _run(la, lb, M, N, K, A, B, C, bias, 1.5, beta)
    ref, bound = oracle.gemm_fp_ex(gen.F32, gen.F32, la, lb, M, N, K, 1.5, A, A.shape[1], B,
                                   B.shape[1], beta, C, N, bias)
    assert_close(got, ref, bound, gen.F32, f"{name} A={la} B={lb} bias={with_bias} beta={beta}")


def test_wide_stream_k_workspace():
    # the query reports two partial 128 x 256 tiles per SM for stream-K, none
    # for whole waves
    sms = _sms()
    for case, want in ((0, 0), (1, 2 * sms * WBM * WBN * 4)):
        _, M, N, K = _case_shapes(sms)[case]
        for la, lb in LAYOUTS:
            lda = K if la == gen.ROW_MAJOR else M
            ldb = N if lb == gen.ROW_MAJOR else K
            assert dga.dga_gemm_general_workspace_size(gen.F32, gen.F32, la, lb, M, N, K, lda,
                                                       ldb, N, S) == want
    # without it: the 128 x 128 kernel (small remainder) or whole wide tiles
    # (a last wave more than half full); exact on small integers either way
    for case in (1, 4):
        _, M, N, K = _case_shapes(sms)[case]
        A, B, C, bias = _operands(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, seed=5 + case,
                                  small_ints=True)
        got, _ = _run(gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, A, B, C, None, 1.0, 1.0,
                      workspace=False)
        ref, _ = oracle.gemm_fp_ex(gen.F32, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, 1.0,
                                   A, K, B, N, 1.0, C, N, None)
        assert_exact(got, ref, gen.F32, f"case {case} without workspace")


def test_wide_repeats_bit_for_bit():
    # fixed summation order: 10 calls of a stream-K case agree bit for bit
    sms = _sms()
    _, M, N, K = _case_shapes(sms)[2]
    A, B, C, bias = _operands(gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, seed=9, small_ints=False)
    first, _ = _run(gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, A, B, C, bias, 1.5, 0.5)
    for _ in range(9):
        again, _ = _run(gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, A, B, C, bias, 1.5, 0.5)
        assert torch.equal(again, first)
