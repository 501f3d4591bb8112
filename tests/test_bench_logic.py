"""bench.py's host logic without a GPU: FLOP/byte accounting against the
figures the pages print, and the multi-rank path (max over ranks, whole-job
throughput, rank-0-only reference arm) with world_size-2 gloo process groups.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


def _page_figures():
    with open(os.path.join(HERE, "golden", "page_figures.json")) as f:
        return json.load(f)["figures"]


def test_accounting_matches_page_figures():
    fig = {f["id"]: f for f in _page_figures()}
    # 2*N^3 FLOPs of a 2048^3 GEMM
    assert bench.gemm_flops(2048, 2048, 2048) == pytest.approx(fig["naive_2048_flops"]["value"], rel=1e-3)
    # GEMV (M x N fp32 matrix times vector): 2MN / 4MN = 0.5 FLOP/B
    M = N = 8192
    gemv = bench.intensity(bench.gemm_flops(M, 1, N), bench.gemm_bytes(M, 1, N, 4, 4, False))
    assert gemv == pytest.approx(fig["gemv_intensity"]["value"], rel=1e-3)
    # square N = 1024: 2N^3 / 12N^2 ~ 170 FLOP/B
    sq = bench.intensity(bench.gemm_flops(1024, 1024, 1024), bench.gemm_bytes(1024, 1024, 1024, 4, 4, False))
    assert sq == pytest.approx(fig["square_1024_intensity"]["value"], rel=0.01)
    # block tile T: T/4 FLOP/B -> 8 at T=32, 32 at T=128
    assert bench.tile_intensity(32) == fig["tile_32_intensity"]["value"]
    assert bench.tile_intensity(128) == fig["tile_128_intensity"]["value"]
    # naive kernel: one FMA per 8 bytes read -> 0.25 FLOP/B
    assert bench.intensity(2 * 2048, 8 * 2048) == fig["naive_intensity"]["value"]
    # 8x8 register tile: 64 FMA per 16 shared-memory reads
    assert 64 / (8 + 8) == fig["register_tile_fma_per_read"]["value"]
    # RTX 5080 machine balance
    assert 56.28e12 / 960e9 == pytest.approx(fig["rtx5080_balance"]["value"])
    # global load requests of the naive kernel at 2048^3 with 16x16 blocks:
    # 2 loads per k per thread, one request per warp instruction
    assert 2048 ** 3 * 2 // 32 == fig["naive_load_requests"]["value"]


def test_peaks_from_measured_file(tmp_path, monkeypatch):
    pk = bench.load_peaks(152)
    assert pk["fp32_ffma_tflops"] == pytest.approx(152 * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12)
    assert pk["source"] in ("measured", "fallback")


def test_job_throughput_weak_scaling():
    # two ranks, 10 steps of 1e12 FLOP each, slowest rank 2 s -> 10 TFLOP/s
    assert bench.job_throughput(1e12, 2, 10, 2000.0, 1e12) == pytest.approx(10.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = 100.0 + 50.0 * rank          # rank 1 is the slow one
    m = bench.max_over_ranks(local, world)
    v = bench.job_throughput(1e9, world, 4, m, 1e12)
    out.put((rank, m, v))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 150.0                   # every rank sees the slowest rank's time
        assert v == pytest.approx(2 * 1e9 * 4 / 0.150 / 1e12)


def test_reference_arm_rank0_only_under_torchrun():
    # two CPU ranks: rank 0 prints the reference line, rank 1 exits quietly
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(28500 + os.getpid() % 1000),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "fp32_256",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT,
                         env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_code_digest_ignores_comments_only(tmp_path):
    # a traffic record stays valid across comment edits and is dropped when code changes
    import bench
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) {\n    return x + 1;  // add one\n}\n")
    b = tmp_path / "b.cu"
    b.write_text("/* another\n   header */\nint f(int x) {\n\n    return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) {\n    return x + 2;\n}\n")
    assert bench.code_digest(str(a)) == bench.code_digest(str(b))
    assert bench.code_digest(str(a)) != bench.code_digest(str(c))


def test_spec_peak_fields():
    # bf16-rate tensor rows also quote the unit-count peak: SMs x 8192 FLOP/clk
    # at the maximum and at the sampled clock; TF32 and non-tensor rows do not
    import bench
    peaks = {"sm_count": 152, "sm_max_mhz": 2070.0}
    rf = {"bound": "tensor", "achieved": 1800.0, "peak_kind": "bf16 tensor"}
    bench.add_spec_peak(rf, peaks, 1035.0)
    at_max = 152 * 8192 * 2070e6 / 1e12
    assert abs(rf["spec"]["at_max_clock"] - at_max) < 1e-9
    assert abs(rf["spec"]["frac_at_max_clock"] - 1800.0 / at_max) < 1e-12
    assert abs(rf["spec"]["at_observed_clock"] - at_max / 2) < 1e-9
    tf32 = {"bound": "tensor", "achieved": 900.0, "peak_kind": "tf32 tensor (measured bf16 x nominal 1.1/2.25)"}
    bench.add_spec_peak(tf32, peaks, 2070.0)
    assert "spec" not in tf32
    hbm = {"bound": "hbm", "achieved": 6000.0}
    bench.add_spec_peak(hbm, peaks, 2070.0)
    assert "spec" not in hbm


def test_per_dtype_rows_fit_a_short_tail():
    # The driver keeps only the end of the bench's output line (about 3000
    # characters with its own framing), so the extra keys come last and a
    # full set of per_dtype rows -- each with the fields its kind of workload
    # carries, a throttle reason on every tensor row -- must stay well within
    # that.
    peaks = bench.load_peaks(152)
    peaks["fp32_ffma_probe"] = {"ffma_tflops": 79.91234, "ffma2_tflops": 79.81234}
    peaks["int8_mma_sync_tops"] = 157.91234
    per = {}
    names = [n for n in bench.PER_DTYPE] + [n + "_sustained" for n in bench.SUSTAINED]
    for i, name in enumerate(names):
        hbm = name.startswith(("skinny", "spmv"))
        bound = "hbm" if hbm else ("alu" if name == "fc_f32_4096" else "tensor")
        rf = {"bound": bound, "achieved": 1772.123456789 + i,
              "unit": "GB/s" if hbm else "TFLOP/s", "frac": 0.93412345678,
              "peak_kind": "bf16 tensor", "ms_mean": 0.620512345,
              "traffic": None if name.startswith("fc") else 1340498400.0,
              "launches_per_call": 4.0 if name.startswith("fc") else 1.0,
              "clocks": {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "samples": 2,
                         "reasons": ["sw_power_cap"] if bound == "tensor" else []}}
        if name.startswith("spmv"):
            rf["nnz"] = 92038930.0
        if name.endswith("_sustained"):
            rf["calls"], rf["seconds"] = 6450.0, 4.00123
        bench.add_spec_peak(rf, peaks, 1965.0)
        per[name] = bench.compact_row(rf)
        if name.startswith("int8"):
            per[name]["x_probe"] = bench.sig(rf["achieved"] / peaks["int8_mma_sync_tops"], 3)
    tail = json.dumps({"peaks": bench.compact_peaks(peaks), "per_dtype": per})
    assert len(tail) < 2700, len(tail)
    assert set(per) >= {"bf16_8192", "skinny_m1", "skinny_m8", "skinny_m16", "int8_ragged"}
    row = per["bf16_8192"]
    assert row["frac"] == 0.934 and row["achieved"] == 1772.0 and row["traffic_mb"] == 1340.0
    assert row["spec_frac_obs"] == round(1772.123456789 / (152 * 8192 * 1965e-6), 3)


def test_sig_rounds_to_significant_digits():
    assert bench.sig(1772.123456, 4) == 1772.0
    assert bench.sig(0.000123456, 3) == 0.000123
    assert bench.sig(58.34934825, 6) == 58.3493
    assert bench.sig(1340498400.0, 3) == 1340000000.0
    assert bench.sig(0.0) == 0.0 and bench.sig(7) == 7 and bench.sig(None) is None
