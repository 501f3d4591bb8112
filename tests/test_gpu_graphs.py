"""The library's calls captured into CUDA graphs and replayed.

A serving loop drives fixed-shape kernels through CUDA graphs rather than
eager launches.  Every kernel family is captured here in a representative
configuration -- including the multi-launch ones whose later launches are
programmatic dependents of the earlier (the FP32 stream-K remainder and its
reduce, the tensor-core split last wave's reduce, the INT8 GEMM behind its
operand repack, the skinny kernel) -- and each replay must reproduce the eager
call bit for bit (every path sums in a fixed order), with the device status
word clear.  Outputs are filled with a sentinel before each replay, so a
replay that wrote nothing fails.
"""

import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _graph_matches_eager(run, outputs, reset=None, replays=3):
    """Runs `run` eagerly, captures it, replays it `replays` times; every
    replay must give the eager outputs.  `reset` restores inputs the call
    reads and writes (C with beta != 0) before each run."""
    stream = torch.cuda.current_stream().cuda_stream
    if reset:
        reset()
    run()
    torch.cuda.synchronize()
    assert dga.dga_sync_status(stream) == dga.OK
    want = [o.clone() for o in outputs]
    g = torch.cuda.CUDAGraph()
    if reset:
        reset()
    with torch.cuda.graph(g):
        run()
    for _ in range(replays):
        if reset:
            reset()
        else:
            for o in outputs:
                o.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert dga.dga_sync_status(torch.cuda.current_stream().cuda_stream) == dga.OK
        for o, w in zip(outputs, want):
            assert torch.equal(o, w)
    return g


def _ws(in_dtype, out_dtype, layout_a, layout_b, M, N, K, lda, ldb, ldc):
    n = dga.dga_gemm_general_workspace_size(in_dtype, out_dtype, layout_a, layout_b, M, N, K,
                                            lda, ldb, ldc, dga.PATH_AUTO)
    return torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")


def test_graph_fp32_stream_k():
    # 2560 x 2048 on 128 x 256 tiles: 160 tiles, one wave of 152 and a
    # stream-K remainder (three launches, two of them programmatic dependents)
    g = torch.Generator(device="cuda").manual_seed(1)
    M, N, K = 2560, 2048, 512
    A = torch.rand(M, K, device="cuda", generator=g) * 2 - 1
    B = torch.rand(K, N, device="cuda", generator=g) * 2 - 1
    C0 = torch.rand(M, N, device="cuda", generator=g) * 2 - 1
    C = C0.clone()
    ws = _ws(gen.F32, gen.F32, gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, K, N, N)

    def run():
        dga.gemm(A, B, C, alpha=1.5, beta=0.5, workspace=ws)
    _graph_matches_eager(run, [C], reset=lambda: C.copy_(C0))
    assert dga.dga_last_launch_count() == 3


def test_graph_tensor_core_split_last_wave():
    # 80 tiles of 256 x 256 on 76 CTA pairs: the last wave split along K, its
    # reduce a programmatic dependent of the GEMM
    g = torch.Generator(device="cuda").manual_seed(2)
    M, N, K = 2560, 2048, 1024
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    W = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    bias = torch.randn(N, device="cuda", generator=g)
    C = torch.empty(M, N, device="cuda")
    ws = _ws(gen.BF16, gen.F32, gen.ROW_MAJOR, gen.COL_MAJOR, M, N, K, K, K, N)

    def run():
        dga.gemm(A, W.t(), C, bias=bias, workspace=ws)
    _graph_matches_eager(run, [C])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert dga.dga_last_launch_count() == 2


def test_graph_int8_repack_and_gemm():
    # the operand repack and the GEMM behind it (programmatic dependent), a
    # ragged shape with a row-major B
    g = torch.Generator(device="cuda").manual_seed(3)
    M, N, K = 300, 259, 1030
    A = torch.randint(-128, 128, (M, K), device="cuda", generator=g, dtype=torch.int8)
    B = torch.randint(-128, 128, (K, N), device="cuda", generator=g, dtype=torch.int8)
    C0 = torch.randint(-1000, 1000, (M, N), device="cuda", generator=g, dtype=torch.int32)
    C = C0.clone()
    ws = _ws(gen.I8, gen.I32, gen.ROW_MAJOR, gen.ROW_MAJOR, M, N, K, K, N, N)

    def run():
        dga.gemm(A, B, C, alpha=3, beta=-2, workspace=ws)
    _graph_matches_eager(run, [C], reset=lambda: C.copy_(C0))
    assert dga.dga_last_launch_count() == 2


@pytest.mark.parametrize("m", [1, 8, 16])
def test_graph_skinny(m):
    g = torch.Generator(device="cuda").manual_seed(4 + m)
    N, K = 1024, 2048
    X = torch.randn(m, K, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    Y = torch.empty(m, N, device="cuda", dtype=torch.bfloat16)

    def run():
        dga.gemm(X, W.t(), Y)
    _graph_matches_eager(run, [Y])
    assert dga.dga_last_path() == dga.PATH_SKINNY


def test_graph_spmv_and_column_sums():
    # a CSR matrix with rows of 0 to 60 entries (merge kernel and its carry
    # fix-up), then the column sums of a bf16 matrix, in one graph
    g = torch.Generator().manual_seed(5)
    rows, cols = 20000, 30000
    lengths = torch.randint(0, 61, (rows,), generator=g)
    offsets = torch.zeros(rows + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    nnz = int(offsets[-1])
    col_idx = torch.randint(0, cols, (nnz,), generator=g, dtype=torch.int32)
    vals = torch.rand(nnz, generator=g) * 2 - 1
    x = torch.rand(cols, generator=g) * 2 - 1
    o, c, v, xd = offsets.cuda(), col_idx.cuda(), vals.cuda(), x.cuda()
    y = torch.empty(rows, device="cuda")
    ws = torch.empty(max(dga.dga_spmv_csr_workspace_size(rows, nnz), 1), dtype=torch.uint8,
                     device="cuda")
    G = torch.randn(4096, 1000, generator=g).to(torch.bfloat16).cuda()
    sums = torch.empty(1000, device="cuda")

    def run():
        dga.spmv_csr(o, c, v, xd, y, workspace=ws)
        dga.sum_rows(G, out=sums)
    _graph_matches_eager(run, [y, sums])
