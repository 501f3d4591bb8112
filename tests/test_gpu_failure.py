"""Failure detection on the GPU without faulting or hanging it.

A kernel waits on an mbarrier that nothing arrives at, through the same
bounded wait the GEMM roles use, with a 20 ms limit.  The host must then read
DGA_ERR_DEVICE_TIMEOUT from dga_sync_status, the status must clear, and the
context must still run GEMMs.
"""
import pytest
import torch

import dense_gemm_accelerator_gb300 as dga
from dense_gemm_accelerator_gb300 import inputs as gen
from tests.helpers import assert_close, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    s = torch.cuda.current_stream().cuda_stream
    assert dga.dga_sync_status(s) == dga.OK
    assert dga.dga_selftest_bounded_wait(20_000_000, s) == dga.OK
    assert dga.dga_sync_status(s) == dga.ERR_DEVICE_TIMEOUT
    assert dga.dga_sync_status(s) == dga.OK  # read and cleared
    g = torch.Generator().manual_seed(3)
    A = gen.random_matrix((130, 200), gen.BF16, g)
    B = gen.random_matrix((140, 200), gen.BF16, g)
    C = torch.zeros(130, 140)
    got = run_gpu(dga.PATH_TCGEN05, gen.BF16, gen.F32, gen.COL_MAJOR, A, B, C, 1.0, 0.0)
    ref, bound = oracle_ref(gen.BF16, gen.F32, gen.COL_MAJOR, A, B, C, 1.0, 0.0)
    assert_close(got, ref, bound, gen.F32, "after timeout")
