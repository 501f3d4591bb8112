"""Runs the naive-GEMM counter probe once at M = N = K = 2048 on the current
GPU, for an ncu capture of its load counters, which "GEMM optimisation, part
0", section 2.3, prints for this kernel (536,870,912 global load requests and
1,073,741,824 sectors).  The inputs are seeded uniform[-1, 1) fp32.

    python tests/naive_probe_run.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_accelerator_gb300 as dga
    n = 2048
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.rand(n, n, device="cuda", generator=g) * 2 - 1
    B = torch.rand(n, n, device="cuda", generator=g) * 2 - 1
    C = torch.empty(n, n, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = dga.dga_probe_naive_sgemm(n, n, n, A.data_ptr(), B.data_ptr(), C.data_ptr(), s)
    if st != dga.OK or dga.dga_sync_status(s) != dga.OK:
        raise SystemExit(f"naive probe failed: {dga.dga_status_string(st)}")
    print("naive probe ok")


if __name__ == "__main__":
    main()
