"""GPU parity of the tensor-core CTA-pair kernel's split last wave, through
the C ABI, against the CPU oracle element by element.

A floating-point problem of more 256 x 256 tiles than there are CTA pairs
(76 on a GB300) runs its last, part-filled wave's tiles cut along K into s
parts when that shortens the wave and the workspace the size query reports
is given: s in 2..4, none shallower than 8 k-blocks, at most two rounds of
parts, chosen to make ceil(r * s / 76) / s smallest for r last-wave tiles.
The parts' raw fp32 sums go to the workspace and a second launch adds them
in part (K) order and applies alpha, beta, the bias row and the output type
(INT8 does not split).  The shapes below split 2, 3 and 4 ways, put the
remainder at half a wave and one tile past it, leave a remainder no split
shortens (52 tiles), and leave ragged edges in both directions; with
small-integer inputs every partial sum is exact, so the result must equal
the oracle's exactly rounded once to the output type.  The GEMM is the BLAS update of "AI Programming:
Matrix Product", section "Dense matrix multiplication", with the bias row of
its "Fully-connected layer" section.
"""
import ctypes

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
import oracle
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, assert_exact

pytestmark = pytest.mark.gpu

T = dga.PATH_TCGEN05


def _clusters():
    return torch.cuda.get_device_properties(0).multi_processor_count // 2


def _tiles(M, N):
    return ((M + 255) // 256) * ((N + 255) // 256)


def _splits(M, N, K, in_dtype):
    """The split the rule gives (1: none) for a device with _clusters() pairs,
    restated from the rule: the s in 2..min(4, k-blocks / 8) with r * s <= 2
    pairs-count whose ceil(r * s / pairs) / s is smallest, if below 1."""
    nc = _clusters()
    tiles = _tiles(M, N)
    if tiles <= nc or tiles % nc == 0:
        return 1
    rem = tiles % nc
    kb = (K + (31 if in_dtype == gen.TF32 else 63)) // (32 if in_dtype == gen.TF32 else 64)
    best, best_len = 1, 1.0
    for sp in range(2, min(4, kb // 8) + 1):
        if rem * sp > 2 * nc:
            break
        length = -(-rem * sp // nc) / sp
        if length < best_len:
            best, best_len = sp, length
    return best


def _operands(in_dtype, out_dtype, M, N, K, seed, small_ints):
    g = torch.Generator().manual_seed(seed)

    def draw(shape, dt):
        if small_ints:
            return gen.small_int_matrix(shape, dt, g, -8, 8)
        return gen.random_matrix(shape, dt, g)
    A = draw((M, K), in_dtype)
    B = draw((N, K), in_dtype)  # column-major B (N x K), the layout of a Linear weight
    C = draw((M, N), out_dtype)
    bias = draw((1, N), out_dtype).reshape(N)
    return A, B, C, bias


def _ru(x, m):
    return (x + m - 1) // m * m


def _run(in_dtype, out_dtype, M, N, K, A, B, C, bias, alpha, beta, workspace=True):
    """workspace=False: only the bytes the call cannot run without (none for
    these aligned floating-point operands; INT8's two bf16 copies)."""
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    bd = bias.to(dev) if bias is not None else None
    ws_bytes = dga.dga_gemm_general_workspace_size(in_dtype, out_dtype, gen.ROW_MAJOR,
                                                   gen.COL_MAJOR, M, N, K, K, K, N, T)
    if not workspace:
        ws_bytes = 0
        if in_dtype == gen.I8:
            ws_bytes = _ru(M * _ru(K, 8) * 2, 256) + _ru(N * _ru(K, 8) * 2, 256)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = dga.scalar(alpha, in_dtype), dga.scalar(beta, in_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_general(in_dtype, out_dtype, gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K,
                              ctypes.byref(al), Ad.data_ptr(), K, Bd.data_ptr(), K,
                              ctypes.byref(be), Cd.data_ptr(), N,
                              bd.data_ptr() if bd is not None else None,
                              ws.data_ptr() if ws_bytes else None, ws_bytes, T, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    assert dga.dga_last_path() == T
    return Cd.cpu(), dga.dga_last_launch_count()


def _shapes(nc):
    """(name, M, N, K): 8 tile columns, the tile rows giving one wave plus a
    remainder of 4 tiles, exactly half a wave, and one tile past half."""
    rows_one = nc // 8  # 9 full tile rows of 8 on a GB300 (72 tiles) ...
    return [
        # 80 tiles on 76 pairs: remainder 4, K = 1024 (16 k-blocks): 2 parts
        ("rem4_two_parts", 256 * 10, 256 * 8, 1024),
        # the same with K = 2048 (32 k-blocks): 4 parts
        ("rem4_four_parts", 256 * 10, 256 * 8, 2048),
        # ragged edges on the split tiles (10 x 8 tiles, the last row and column
        # short) and a partial last k-block (K = 1096: rows of 2192 or 4384
        # bytes, which TMA reads in place)
        ("ragged", 256 * 9 + 100, 256 * 7 + 70, 1096),
        # remainder exactly half a wave: 76 + 38 = 114 tiles (19 x 6), 2 parts
        ("half_wave", 256 * 19, 256 * 6, 1024),
        # one tile past half: 76 + 39 = 115 tiles (23 x 5), 3 parts (K = 1536:
        # 24 k-blocks, enough for three parts of at least 8)
        ("past_half", 256 * 23, 256 * 5, 1536),
        # 76 + 52 = 128 tiles (16 x 8): two parts would take two rounds, three
        # more than two rounds of parts: not split
        ("no_gain", 256 * 16, 256 * 8, 1024),
    ] if rows_one * 8 <= nc else []


CASES = [(gen.BF16, gen.F32), (gen.BF16, gen.BF16), (gen.F16, gen.F32), (gen.F16, gen.F16),
         (gen.TF32, gen.F32)]


@pytest.mark.parametrize("case", range(6))
@pytest.mark.parametrize("dtypes", CASES, ids=["bf16_f32", "bf16_bf16", "f16_f32", "f16_f16",
                                                "tf32_f32"])
def test_split_last_wave_exact(case, dtypes):
    # entries in [-8, 8], K <= 2048: every partial and total sum is an integer
    # below 2^24 in magnitude, exact in fp32 in any order; alpha = 1, beta =
    # -1 and an integer C and bias keep the epilogue exact before the single
    # rounding to the output type
    nc = _clusters()
    shapes = _shapes(nc)
    if not shapes:
        pytest.skip("the shapes assume a device with 8k CTA pairs")
    name, M, N, K = shapes[case]
    in_dtype, out_dtype = dtypes
    A, B, C, bias = _operands(in_dtype, out_dtype, M, N, K, seed=case * 5 + CASES.index(dtypes),
                              small_ints=True)
    got, launches = _run(in_dtype, out_dtype, M, N, K, A, B, C, bias, 1.0, -1.0)
    sp = _splits(M, N, K, in_dtype)
    assert launches == (2 if sp > 1 else 1), (name, launches, sp)
    assert (sp > 1) == (name != "no_gain"), (name, sp)
    ref, _ = oracle.gemm_fp_ex(in_dtype, out_dtype, gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, 1.0,
                               A, K, B, K, -1.0, C, N, bias)
    assert_exact(got, ref, out_dtype, f"{name} {in_dtype}->{out_dtype}")
    # without the workspace: whole tiles, one launch, the same exact result
    got0, launches0 = _run(in_dtype, out_dtype, M, N, K, A, B, C, bias, 1.0, -1.0,
                           workspace=False)
    assert launches0 == 1
    assert torch.equal(got0, got), name


@pytest.mark.parametrize("dtypes", CASES, ids=["bf16_f32", "bf16_bf16", "f16_f32", "f16_f16",
                                                "tf32_f32"])
@pytest.mark.parametrize("beta,with_bias", [(0.0, False), (0.5, True)])
def test_split_last_wave_uniform(dtypes, beta, with_bias):
    # uniform inputs within the oracle's bound (the split changes the order
    # of the fp32 additions, not the bound), beta = 0 never reading C
    nc = _clusters()
    shapes = _shapes(nc)
    if not shapes:
        pytest.skip("the shapes assume a device with 8k CTA pairs")
    name, M, N, K = shapes[2]
    in_dtype, out_dtype = dtypes
    A, B, C, bias = _operands(in_dtype, out_dtype, M, N, K, seed=40 + CASES.index(dtypes),
                              small_ints=False)
    if beta == 0.0:
        C = torch.full_like(C, float("nan"))
    bias = bias if with_bias else None
    got, launches = _run(in_dtype, out_dtype, M, N, K, A, B, C, bias, 1.5, beta)
    assert launches == 2
    ref, bound = oracle.gemm_fp_ex(in_dtype, out_dtype, gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K,
                                   1.5, A, K, B, K, beta, C, N, bias)
    assert_close(got, ref, bound, out_dtype, f"{name} {in_dtype}->{out_dtype} beta={beta}")


def test_split_last_wave_repeats_bit_for_bit():
    # the parts are added in a fixed order: repeated calls agree bit for bit
    nc = _clusters()
    shapes = _shapes(nc)
    if not shapes:
        pytest.skip("the shapes assume a device with 8k CTA pairs")
    _, M, N, K = shapes[1]
    A, B, C, bias = _operands(gen.BF16, gen.F32, M, N, K, seed=77, small_ints=False)
    first, _ = _run(gen.BF16, gen.F32, M, N, K, A, B, C, bias, 1.0, 0.25)
    for _ in range(5):
        again, _ = _run(gen.BF16, gen.F32, M, N, K, A, B, C, bias, 1.0, 0.25)
        assert torch.equal(again, first)


def test_split_workspace_query():
    # the query adds two 256 x 256 32-bit slots per CTA pair when a split is
    # possible (at most two rounds of parts); single-wave problems get none
    nc = _clusters()
    slot = 256 * 256 * 4
    q = dga.dga_gemm_general_workspace_size
    assert q(gen.BF16, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR, 2560, 2048, 1024, 1024, 1024, 2048,
             T) == 2 * nc * slot
    assert q(gen.BF16, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR, 512, 512, 1024, 1024, 1024, 512,
             T) == 0
    assert q(gen.BF16, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR, 2560, 2048, 512, 512, 512, 2048,
             T) == 0  # 8 k-blocks: too shallow for two parts


def _run_layouts(in_dtype, out_dtype, layout_a, layout_b, M, N, K, A, B, C, bias, lda, ldb):
    dev = torch.device("cuda")
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    bd = bias.to(dev)
    ws_bytes = dga.dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N,
                                                   K, lda, ldb, N, T)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    al, be = dga.scalar(1.0, in_dtype), dga.scalar(-1.0, in_dtype)
    stream = torch.cuda.current_stream().cuda_stream
    st = dga.dga_gemm_general(in_dtype, out_dtype, layout_a, layout_b, M, N, K, ctypes.byref(al),
                              Ad.data_ptr(), lda, Bd.data_ptr(), ldb, ctypes.byref(be),
                              Cd.data_ptr(), N, bd.data_ptr(), ws.data_ptr(), ws_bytes, T, stream)
    assert st == dga.OK, dga.dga_status_string(st)
    assert dga.dga_sync_status(stream) == dga.OK
    return Cd.cpu(), dga.dga_last_launch_count()


@pytest.mark.parametrize("in_dtype,out_dtype,layout_a,layout_b,pad,repacks", [
    # a row-major B read in place (MN-major): the split alone
    (gen.BF16, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, 0, 0),
    # a column-major A read in place
    (gen.F16, gen.F16, gen.COL_MAJOR, gen.COL_MAJOR, 0, 0),
    # a leading dimension TMA cannot express (B padded by 3): B copied row by
    # row into the front of the workspace, the partial sums behind it
    (gen.BF16, gen.BF16, gen.ROW_MAJOR, gen.COL_MAJOR, 3, 1),
    # TF32 with a row-major B: B transposed into the workspace, then the split
    (gen.TF32, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, 0, 1),
])
def test_split_with_other_layouts_and_repacks(in_dtype, out_dtype, layout_a, layout_b, pad,
                                              repacks):
    # 80 tiles on 76 pairs (remainder 4) with K = 1024: the last wave is split,
    # after a repack where one is needed; exact on small integers
    nc = _clusters()
    if _shapes(nc) == []:
        pytest.skip("the shapes assume a device with 8k CTA pairs")
    M, N, K = 256 * 10, 256 * 8, 1024
    g = torch.Generator().manual_seed(11 + pad)
    a_shape = (M, K + pad) if layout_a == gen.ROW_MAJOR else (K, M + pad)
    b_shape = (K, N + pad) if layout_b == gen.ROW_MAJOR else (N, K + pad)
    A = gen.small_int_matrix(a_shape, in_dtype, g, -8, 8)
    B = gen.small_int_matrix(b_shape, in_dtype, g, -8, 8)
    C = gen.small_int_matrix((M, N), out_dtype, g, -8, 8)
    bias = gen.small_int_matrix((1, N), out_dtype, g, -8, 8).reshape(N)
    got, launches = _run_layouts(in_dtype, out_dtype, layout_a, layout_b, M, N, K, A, B, C, bias,
                                 A.shape[1], B.shape[1])
    assert launches == repacks + 2, launches  # repack (if any), GEMM, reduce
    ref, _ = oracle.gemm_fp_ex(in_dtype, out_dtype, layout_a, layout_b, M, N, K, 1.0, A,
                               A.shape[1], B, B.shape[1], -1.0, C, N, bias)
    assert_exact(got, ref, out_dtype, f"{in_dtype}->{out_dtype} A={layout_a} B={layout_b}")


@pytest.mark.parametrize("case", [0, 3, 4, 5])
def test_int8_last_wave_not_split(case):
    # INT8 never splits its last wave (three parts measured slower on the
    # 4093 x 4099 x 4096 shape: each part pays a whole INT8 epilogue): the
    # repack and the GEMM, whatever workspace is given, the same exact bits
    nc = _clusters()
    shapes = _shapes(nc)
    if not shapes:
        pytest.skip("the shapes assume a device with 8k CTA pairs")
    name, M, N, K = shapes[case]
    g = torch.Generator().manual_seed(90 + case)
    A = gen.random_matrix((M, K), gen.I8, g, ("int8",))
    B = gen.random_matrix((N, K), gen.I8, g, ("int8",))
    C = gen.random_matrix((M, N), gen.I32, g, ("int8",))
    bias = gen.random_matrix((1, N), gen.I32, g, ("int8",)).reshape(N)
    got, launches = _run(gen.I8, gen.I32, M, N, K, A, B, C, bias, 3, -2)
    assert launches == 2, (name, launches)  # repack, GEMM
    ref = oracle.gemm_i8_ex(gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, 3, A, K, B, K, -2, C, N, bias)
    assert_exact(got, ref, gen.I32, f"int8 {name}")
    got0, launches0 = _run(gen.I8, gen.I32, M, N, K, A, B, C, bias, 3, -2, workspace=False)
    assert launches0 == 2
    assert torch.equal(got0, got), name
