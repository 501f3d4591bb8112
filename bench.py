"""Benchmark: dense GEMM throughput on GB300 against its roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one GEMM of the named workload (default fp32_4096: FP32 SGEMM
M=N=K=4096, alpha=1.5, beta=0.5, the SIMT path) through the library's C ABI,
with every input resident in HBM.  Input sets are rotated so that the bytes a
step touches are never in L2 from the step before (the rotation spans more
than 2x the 129 MB L2).  Rank 0 prints ONE JSON line.

Extra keys beside the contract's, last on the line: `peaks` (every roofline
denominator and where it came from) and `per_dtype`, the other hot-path
workloads -- BF16 8192^3 on tcgen05, skinny M in {1, 8, 16}, INT8
4093x4099x4096, FP16 8192^3, BF16 8192^3 with a row-major B, FP32 8192^3
multiplied as TF32 (the opt-in lossy tensor-core path), CSR SpMV, and one
fully-connected layer step (forward, both gradient GEMMs and the bias
gradient) in bf16 at 8192 and in fp32 at 4096 -- each timed as a burst the
same way, plus BF16 and FP16 8192^3 run back to back for 4 s (`*_sustained`).
A row holds `achieved` (in `unit`), `frac` (of the measured burst peak; of
the measured sustained one for `*_sustained`), `ms` per call, `traffic_mb`
(DRAM MB per launch from the committed ncu record, when it matches the
current code), `sm_mhz` (median sampled SM clock), and for the bf16-rate
tensor rows `spec_frac_max` and `spec_frac_obs` (of the unit-count peak, SMs
x 8192 FLOP/clk, at the maximum clock and at the sampled clock: the
clock-normalised figure); the INT8 row adds `x_probe`, its rate over that
of the integer mma.sync instruction as the library's probe measures it
(`peaks.int8_mma_tops`): how far the exact bf16 encoding on the tcgen05
pipe runs past what an INT8 GEMM built on that instruction could.

`--impl reference` times the CPU oracle (plain fp64 triple loop, as it
stands) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS/TOPS and % of GB300 roofline per dtype; skinny-M HBM GB/s"
L2_BYTES = 129 * 1024 * 1024

# ------------------------------------------------------------ accounting --
#
# FLOPs and algorithmic bytes.  A GEMM does K multiplies and K adds per
# output: 2*M*N*K FLOPs ("GEMM optimisation, part 0" (chongfengling.github.io),
# section "Measurement"; "Matrix multiplication: arithmetic intensity, tiling
# and Tensor Core", section 5.2).  Algorithmic bytes count each operand once:
# A and B read, C written, and C read as well when beta != 0 (section 5.1's
# "minimum bytes" column).  Intensity I = FLOPs / bytes (section 5.1).

DTYPE_BYTES = {0: 4, 1: 2, 2: 2, 3: 1, 4: 4, 5: 4}  # 5: TF32 (fp32 storage)


def gemm_flops(M, N, K):
    return 2 * M * N * K


def gemm_bytes(M, N, K, in_bytes, out_bytes, reads_c):
    return in_bytes * (M * K + K * N) + out_bytes * M * N * (2 if reads_c else 1)


def intensity(flops, nbytes):
    return flops / nbytes


def tile_intensity(T, elem_bytes=4):
    """Per K-step of a T x T block tile: 2*T^3 FLOPs over 2*T^2 elements."""
    return (2 * T ** 3) / (elem_bytes * 2 * T ** 2)


def fc_accounting(w):
    """One fully-connected layer step ("AI Programming: Matrix Product",
    section "Fully-connected layer"): batch b = M, n_in = K, n_out = N.
    Three GEMMs of 2*b*n_in*n_out FLOPs each (Y = X W^T, dX = G W,
    dW = G^T X) plus b*n_out adds for db.  Bytes: each GEMM's operands once
    (X, W, Y + the bias row; G, W, dX; G, X, dW) and G read once more for db."""
    b, n_in, n_out = w.M, w.K, w.N
    e, o = DTYPE_BYTES[w.in_dtype], DTYPE_BYTES[w.out_dtype]
    fl = 3 * gemm_flops(b, n_out, n_in) + b * n_out
    by = (gemm_bytes(b, n_out, n_in, e, o, False) + o * n_out      # forward + bias row
          + gemm_bytes(b, n_in, n_out, e, o, False)                 # dX
          + gemm_bytes(n_out, n_in, b, e, o, False)                 # dW
          + e * b * n_out + 4 * n_out)                              # db
    return fl, by


def spmv_accounting(w, nnz):
    """CSR SpMV y = alpha A x + beta y ("AI Programming: Matrix Product",
    section "SpMV"): one multiply and one add per stored entry; bytes read
    once each: row offsets (rows + 1 int32), column indices and values (nnz
    int32 + nnz fp32), x (cols fp32), y written (and read when beta != 0)."""
    fl = 2 * nnz
    by = 4 * (w.M + 1) + 8 * nnz + 4 * w.N + 4 * w.M * (2 if w.beta != 0 else 1)
    return fl, by


def workload_accounting(w, nnz=None):
    if w.kind == "spmv":
        return spmv_accounting(w, nnz)
    if w.kind == "fc":
        return fc_accounting(w)
    fl = gemm_flops(w.M, w.N, w.K)
    by = gemm_bytes(w.M, w.N, w.K, DTYPE_BYTES[w.in_dtype], DTYPE_BYTES[w.out_dtype], w.beta != 0)
    return fl, by


# ------------------------------------------------------------------ peaks --

def load_peaks(sm_count):
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM
    throughput of the GB300s (MEASURED_PEAKS.json), else the stated
    fallback; the FP32 FFMA peak from unit counts and the maximum SM clock."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "measured"
    try:
        with open(path) as f:
            pk = json.load(f)
        hbm = float(pk["hbm_gbs"])
        bf16 = float(pk["bf16_tflops"])
        bf16_sus = float(pk.get("bf16_tflops_sustained", bf16))
        sm_max = float(pk.get("sm_max_mhz", 2070.0))
    except (OSError, KeyError, ValueError):
        src = "fallback"
        hbm, bf16, bf16_sus, sm_max = 6800.0, 1900.0, 1700.0, 2070.0
    # 128 FP32 lanes per SM, one FFMA (2 FLOP) per lane per clock
    fp32 = sm_count * 128 * 2 * sm_max * 1e6 / 1e12
    # TF32 has no measured figure: the measured bf16 peak times the nominal
    # dense ratio (1.1 PFLOP/s TF32 against 2.25 PFLOP/s BF16 per GPU)
    tf32 = bf16 * 1.1 / 2.25
    return {"source": src, "hbm_gbs": hbm, "bf16_tflops": bf16, "tf32_tflops": tf32,
            "tf32_basis": "measured bf16 x nominal 1.1/2.25",
            "bf16_tflops_sustained": bf16_sus, "fp32_ffma_tflops": fp32,
            "fp32_ffma_basis": f"{sm_count} SMs x 128 lanes x 2 FLOP x {sm_max:.0f} MHz",
            "sm_max_mhz": sm_max, "sm_count": sm_count}


# the other hot-path workloads, each timed as a burst after the main one
PER_DTYPE = ("bf16_8192", "skinny_m1", "skinny_m8", "skinny_m16", "int8_ragged", "f16_8192",
             "bf16_8192_rowb", "tf32_8192", "spmv_powerlaw", "fc_bf16_8192", "fc_f32_4096")
# and run back to back for SUSTAINED_SECONDS under the power cap, where the
# clock settles lower (fractions against the sustained peak and per clock)
SUSTAINED = ("bf16_8192", "f16_8192")
SUSTAINED_SECONDS = 4.0

# dense bf16 tensor FLOPs per SM per clock (4096 MACs), the unit-count figure
# the tensor rows are also quoted against beside the measured cuBLAS peak
SPEC_BF16_FLOP_PER_CLK_PER_SM = 8192


def add_spec_peak(rf, peaks, sm_mhz):
    """For a bf16-rate tensor row (bf16, fp16, INT8 as bf16 products): the
    peak from unit counts (SMs x 8192 FLOP/clk) at the maximum SM clock and at
    the clock sampled while the row was timed, and the fractions of both."""
    if rf.get("bound") != "tensor" or "tf32" in rf.get("peak_kind", ""):
        return
    per_mhz = peaks["sm_count"] * SPEC_BF16_FLOP_PER_CLK_PER_SM * 1e6 / 1e12
    at_max = per_mhz * peaks["sm_max_mhz"]
    rf["spec"] = {"basis": f"{peaks['sm_count']} SMs x {SPEC_BF16_FLOP_PER_CLK_PER_SM} FLOP/clk",
                  "at_max_clock": at_max, "frac_at_max_clock": rf["achieved"] / at_max}
    if sm_mhz:
        at_obs = per_mhz * sm_mhz
        rf["spec"].update({"observed_mhz": sm_mhz, "at_observed_clock": at_obs,
                           "frac_at_observed_clock": rf["achieved"] / at_obs})


def sig(x, digits=4):
    """x rounded to `digits` significant digits (the JSON line stays short
    enough for a tail of a few thousand characters to hold all of it)."""
    if not isinstance(x, float) or x == 0.0 or x != x:
        return x
    from math import floor, log10
    return round(x, digits - 1 - int(floor(log10(abs(x)))))


def compact_row(rf):
    """One per_dtype row: throughput, its roofline fraction and the fields
    that explain it, with short keys (meanings in the module docstring)."""
    row = {"achieved": sig(rf["achieved"]), "unit": rf["unit"], "frac": sig(rf["frac"], 3),
           "ms": sig(rf["ms_mean"])}
    if rf.get("traffic") is not None:
        row["traffic_mb"] = sig(float(rf["traffic"]) / 1e6, 4)
    clk = rf.get("clocks", {})
    if clk.get("sm_mhz") is not None:
        row["sm_mhz"] = int(round(clk["sm_mhz"]))
    if clk.get("reasons"):
        row["reasons"] = clk["reasons"]
    spec = rf.get("spec")
    if spec:
        row["spec_frac_max"] = sig(spec["frac_at_max_clock"], 3)
        if "frac_at_observed_clock" in spec:
            row["spec_frac_obs"] = sig(spec["frac_at_observed_clock"], 3)
    if rf.get("launches_per_call", 1.0) != 1.0:
        row["launches"] = rf["launches_per_call"]
    for k in ("nnz", "calls", "seconds"):
        if k in rf:
            row[k] = sig(float(rf[k]))
    return row


def compact_peaks(peaks):
    """The roofline denominators, rounded, with where each came from."""
    out = {"source": peaks["source"], "hbm_gbs": peaks["hbm_gbs"],
           "bf16_tflops": peaks["bf16_tflops"], "bf16_sus": peaks["bf16_tflops_sustained"],
           "tf32_tflops": sig(peaks["tf32_tflops"]), "fp32_ffma_tflops": sig(peaks["fp32_ffma_tflops"]),
           "fp32_basis": peaks["fp32_ffma_basis"], "sm_count": peaks["sm_count"],
           "sm_max_mhz": peaks["sm_max_mhz"]}
    probe = peaks.get("fp32_ffma_probe") or {}
    if "error" in probe:
        out["fma_probe_error"] = probe["error"][:80]
    elif probe:
        out["fma_probe"] = [sig(probe["ffma_tflops"]), sig(probe["ffma2_tflops"])]
    if peaks.get("int8_mma_sync_tops"):
        out["int8_mma_tops"] = sig(peaks["int8_mma_sync_tops"])
    return out


def int8_mma_probe(device, iters=1024, reps=5):
    """The library's INT8 instruction-rate probe: best of `reps` event-timed
    launches of independent mma.sync m16n8k32 s8 chains, in TOP/s -- the
    ceiling of an INT8 GEMM built on that instruction, beside which the
    INT8 row (exact bf16 encoding on the tcgen05 pipe) is reported."""
    import ctypes
    import torch
    import dense_gemm_accelerator_gb300 as dga
    n = dga.dga_probe_fp32_fma_out_floats()
    out = torch.empty(n, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    ops = ctypes.c_double(0.0)
    best = 0.0
    for i in range(reps + 1):  # the first launch is a warm-up
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        st = dga.dga_probe_int8_mma(iters, out.data_ptr(), n, ctypes.byref(ops), stream.cuda_stream)
        e1.record(stream)
        if st != dga.OK:
            raise RuntimeError(f"INT8 probe: {dga.dga_status_string(st)}")
        e1.synchronize()
        if i:
            best = max(best, ops.value / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    st = dga.dga_sync_status(stream.cuda_stream)
    if st != dga.OK:
        raise RuntimeError(f"INT8 probe: {dga.dga_status_string(st)}")
    return best


def fp32_fma_probe(device, iters=12000, reps=5):
    """The library's FP32 FMA-rate probe: best of `reps` event-timed launches
    of independent fmaf chains and of fma.rn.f32x2 chains (about 3 ms each),
    in TFLOP/s.  Cross-checks the FP32 peak derived from unit counts."""
    import ctypes
    import torch
    import dense_gemm_accelerator_gb300 as dga
    n = dga.dga_probe_fp32_fma_out_floats()
    out = torch.empty(n, device=device)
    stream = torch.cuda.current_stream(device)
    res = {"iters": iters, "launch": f"{n // 256} CTAs x 256 threads, 8 chains x 64 FMA per iteration"}
    for packed, key in ((0, "ffma_tflops"), (1, "ffma2_tflops")):
        flops = ctypes.c_double(0.0)
        best = 0.0
        for i in range(reps + 1):  # the first launch is a warm-up
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st = dga.dga_probe_fp32_fma(packed, iters, out.data_ptr(), n, ctypes.byref(flops),
                                        stream.cuda_stream)
            e1.record(stream)
            if st != dga.OK:
                raise RuntimeError(f"FMA probe: {dga.dga_status_string(st)}")
            e1.synchronize()
            if i:
                best = max(best, flops.value / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        res[key] = best
    st = dga.dga_sync_status(stream.cuda_stream)
    if st != dga.OK:
        raise RuntimeError(f"FMA probe: {dga.dga_status_string(st)}")
    return res


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, line in self.lines:
            if not (t0 <= t <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- GPU workloads --

class Runner:
    """Device-resident input sets for one workload and the dga call on them."""

    def __init__(self, w, device, sets, seed=0):
        import torch

        import dense_gemm_accelerator_gb300 as dga
        from dense_gemm_accelerator_gb300 import inputs as gen
        self.w, self.dga, self.gen = w, dga, gen
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.sets = []
        tdt = gen.TORCH_DTYPE
        for _ in range(sets):
            A = self._draw((w.M, w.K), w.dist_a, w.in_dtype, g, device)
            Bs = (w.N, w.K) if w.layout_b == gen.COL_MAJOR else (w.K, w.N)
            B = self._draw(Bs, w.dist_b, w.in_dtype, g, device)
            C = self._draw((w.M, w.N), w.dist_c if w.beta != 0 else ("uniform",), w.out_dtype, g,
                           device) if w.beta != 0 else torch.empty((w.M, w.N), dtype=tdt[w.out_dtype],
                                                                   device=device)
            self.sets.append((A, B, C))
        A, B, C = self.sets[0]
        lda, layout, ldb, ldc = dga.operand_layout(A, self._bview(B), C)
        self.lda, self.ldb, self.ldc = lda, ldb, ldc
        self.ws_bytes = dga.dga_gemm_workspace_size(w.in_dtype, w.out_dtype, w.layout_b, w.M, w.N,
                                                    w.K, lda, ldb, ldc, dga.PATH_AUTO)
        self.ws = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=device)
        self.alpha = dga.scalar(w.alpha, w.in_dtype)
        self.beta = dga.scalar(w.beta, w.in_dtype)

    def _bview(self, B):
        return B.t() if self.w.layout_b == self.gen.COL_MAJOR else B

    @staticmethod
    def _draw(shape, dist, code, g, device):
        import torch

        from dense_gemm_accelerator_gb300 import inputs as gen
        if dist[0] == "uniform":
            return (torch.rand(shape, generator=g, device=device) * 2 - 1).to(gen.TORCH_DTYPE[code])
        if dist[0] == "normal":
            return (torch.randn(shape, generator=g, device=device) * dist[1]).to(gen.TORCH_DTYPE[code])
        return torch.randint(-128, 128, shape, generator=g, device=device,
                             dtype=torch.int8 if code == gen.I8 else torch.int32)

    def call(self, i, stream):
        import ctypes
        A, B, C = self.sets[i % len(self.sets)]
        w, dga = self.w, self.dga
        st = dga.dga_gemm(w.in_dtype, w.out_dtype, w.layout_b, w.M, w.N, w.K,
                          ctypes.byref(self.alpha), A.data_ptr(), self.lda, B.data_ptr(), self.ldb,
                          ctypes.byref(self.beta), C.data_ptr(), self.ldc, self.ws.data_ptr(),
                          self.ws_bytes, stream)
        if st != dga.OK:
            raise dga.DgaError(st, f"dga_gemm ({w.name})")
        return dga.dga_last_launch_count()


class FcRunner:
    """Device-resident inputs of one fully-connected layer step and the four
    library calls that make it: Y = X W^T + b (W^T is the column-major view
    of W [n_out, n_in]), dX = G W, dW = G^T X (G^T is the column-major view
    of G [batch, n_out]) and db = the batch sum of G."""

    def __init__(self, w, device, sets, seed=0):
        import torch

        import dense_gemm_accelerator_gb300 as dga
        from dense_gemm_accelerator_gb300 import inputs as gen
        self.w, self.dga, self.gen = w, dga, gen
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        b, n_in, n_out = w.M, w.K, w.N
        draw = Runner._draw
        self.sets = []
        for _ in range(sets):
            X = draw((b, n_in), w.dist_a, w.in_dtype, g, device)
            W = draw((n_out, n_in), w.dist_b, w.in_dtype, g, device)
            bias = draw((n_out,), w.dist_b, w.out_dtype, g, device)
            G = draw((b, n_out), w.dist_c, w.in_dtype, g, device)
            self.sets.append((X, W, bias, G))
        odt = gen.TORCH_DTYPE[w.out_dtype]
        self.Y = torch.empty((b, n_out), dtype=odt, device=device)
        self.dX = torch.empty((b, n_in), dtype=odt, device=device)
        self.dW = torch.empty((n_out, n_in), dtype=odt, device=device)
        self.db = torch.empty((n_out,), dtype=torch.float32, device=device)
        R, C = gen.ROW_MAJOR, gen.COL_MAJOR
        # (layout_a, layout_b, M, N, K, lda, ldb, ldc) of forward, dX, dW
        self.shapes = [(R, C, b, n_out, n_in, n_in, n_in, n_out),
                       (R, R, b, n_in, n_out, n_out, n_in, n_in),
                       (C, R, n_out, n_in, b, n_out, n_in, n_in)]
        self.ws_bytes = max(dga.dga_gemm_general_workspace_size(w.in_dtype, w.out_dtype, *sh,
                                                                dga.PATH_AUTO)
                            for sh in self.shapes)
        self.ws = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=device)
        self.one = dga.scalar(1.0, w.in_dtype)
        self.zero = dga.scalar(0.0, w.in_dtype)
        self.paths = []

    def call(self, i, stream):
        import ctypes
        X, W, bias, G = self.sets[i % len(self.sets)]
        w, dga = self.w, self.dga
        operands = [(X, W, self.Y, bias), (G, W, self.dX, None), (G, X, self.dW, None)]
        launches = 0
        self.paths = []
        for sh, (A, B, C, bv) in zip(self.shapes, operands):
            la, lb, M, N, K, lda, ldb, ldc = sh
            st = dga.dga_gemm_general(w.in_dtype, w.out_dtype, la, lb, M, N, K,
                                      ctypes.byref(self.one), A.data_ptr(), lda, B.data_ptr(), ldb,
                                      ctypes.byref(self.zero), C.data_ptr(), ldc,
                                      bv.data_ptr() if bv is not None else None,
                                      self.ws.data_ptr(), self.ws_bytes, dga.PATH_AUTO, stream)
            if st != dga.OK:
                raise dga.DgaError(st, f"dga_gemm_general ({w.name})")
            launches += dga.dga_last_launch_count()
            self.paths.append(dga.PATH_NAMES[dga.dga_last_path()])
        st = dga.dga_sum_rows(w.in_dtype, w.M, w.N, G.data_ptr(), w.N, self.db.data_ptr(), stream)
        if st != dga.OK:
            raise dga.DgaError(st, f"dga_sum_rows ({w.name})")
        return launches + 1


class SpmvRunner:
    """Device-resident synthetic CSR matrices (the power-law structure of
    inputs.csr_powerlaw, drawn with torch's CUDA generator) and the
    dga_spmv_csr call on them."""

    def __init__(self, w, device, sets, seed=0):
        import torch

        import dense_gemm_accelerator_gb300 as dga
        from dense_gemm_accelerator_gb300 import inputs as gen
        self.w, self.dga = w, dga
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.sets = []
        for _ in range(sets):
            offs, cols, vals = gen.csr_powerlaw(w.M, w.N, g, device, **gen.CSR_STRUCTURE)
            x = torch.rand(w.N, generator=g, device=device) * 2 - 1
            self.sets.append((offs, cols, vals, x))
        self.nnz = [st[2].numel() for st in self.sets]
        self.mean_nnz = sum(self.nnz) / len(self.nnz)
        self.y = torch.empty(w.M, dtype=torch.float32, device=device)
        self.ws_bytes = max(dga.dga_spmv_csr_workspace_size(w.M, n) for n in self.nnz)
        self.ws = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=device)
        self.alpha = dga.scalar(w.alpha, gen.F32)
        self.beta = dga.scalar(w.beta, gen.F32)
        self.paths = ["spmv"]

    def call(self, i, stream):
        import ctypes
        offs, cols, vals, x = self.sets[i % len(self.sets)]
        w, dga = self.w, self.dga
        st = dga.dga_spmv_csr(w.M, w.N, vals.numel(), offs.data_ptr(), cols.data_ptr(),
                              vals.data_ptr(), ctypes.byref(self.alpha), x.data_ptr(),
                              ctypes.byref(self.beta), self.y.data_ptr(), self.ws.data_ptr(),
                              self.ws_bytes, stream)
        if st != dga.OK:
            raise dga.DgaError(st, f"dga_spmv_csr ({w.name})")
        return dga.dga_last_launch_count()


def runner_for(w, device, sets, seed=0):
    return {"fc": FcRunner, "spmv": SpmvRunner}.get(w.kind, Runner)(w, device, sets, seed)


def sets_for(w, min_sets=2):
    """Enough input sets that one rotation spans > 2x L2."""
    from dense_gemm_accelerator_gb300 import inputs as gen
    if w.kind == "spmv":  # mean row length ~23: values + column indices ~184 bytes per row
        per = 8 * 23 * w.M
        return int(max(min_sets, -(-2 * L2_BYTES // per) + 1))
    if w.kind == "fc":  # X, W, G (the outputs are shared by all sets)
        per = DTYPE_BYTES[w.in_dtype] * (w.M * w.K + w.N * w.K + w.M * w.N)
    else:
        per = DTYPE_BYTES[w.in_dtype] * (w.M * w.K + w.K * w.N) + DTYPE_BYTES[w.out_dtype] * w.M * w.N
    n = max(min_sets, -(-2 * L2_BYTES // per) + 1)
    del gen
    return int(n)


def time_kernel(runner, steps, warmup):
    """Back-to-back calls on one stream; CUDA events around the whole batch, so
    host-side call overhead does not leak into a short kernel's time."""
    import torch
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    for i in range(warmup):
        runner.call(i, s)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches = 0
    e0.record(stream)
    for i in range(steps):
        launches += runner.call(warmup + i, s)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, launches


def roofline_for(w, ms_mean, peaks, sustained=False, nnz=None):
    fl, by = workload_accounting(w, nnz)
    from dense_gemm_accelerator_gb300 import inputs as gen
    if w.name.startswith("skinny") or w.kind == "spmv":
        ach = by / (ms_mean * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes": by}
    ach = fl / (ms_mean * 1e-3) / 1e12
    if w.in_dtype == gen.F32:
        return {"bound": "alu", "achieved": ach, "peak": peaks["fp32_ffma_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["fp32_ffma_tflops"],
                "algorithmic_flops": fl}
    pk = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    if w.in_dtype == gen.TF32:
        pk = peaks["tf32_tflops"] * (peaks["bf16_tflops_sustained"] / peaks["bf16_tflops"]
                                     if sustained else 1.0)
    return {"bound": "tensor", "achieved": ach, "peak": pk, "unit": "TFLOP/s" if w.in_dtype != gen.I8 else "TOP/s",
            "frac": ach / pk, "algorithmic_flops": fl,
            "peak_kind": {gen.I8: "bf16 tensor (INT8 runs as exact bf16 products)",
                          gen.F16: "bf16 tensor (fp16 has the same nominal rate)",
                          gen.TF32: "tf32 tensor (measured bf16 x nominal 1.1/2.25)"}.get(
                              w.in_dtype, "bf16 tensor")}


def code_digest(path):
    """First 16 hex digits of the SHA-256 of a CUDA source with its comments
    and blank lines removed: a traffic record stays valid across edits that
    change no code."""
    import re
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def traffic_record(kernel_src, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current code of the kernel's source (comments aside); else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry:
        return None
    src = os.path.join(ROOT, "dense_gemm_accelerator_gb300", "csrc", kernel_src)
    try:
        digest = code_digest(src)
    except OSError:
        return None
    if entry.get("code_sha256_16") != digest:
        return None
    return entry.get("bytes_per_launch")


KERNEL_SOURCE = {"fp32": "sgemm_simt.cu", "bf16": "gemm_tcgen05.cu", "skinny": "gemv_skinny.cu",
                 "int8": "gemm_tcgen05.cu", "spmv": "spmv_csr.cu"}


def source_of(w):
    if w.kind == "spmv":
        return KERNEL_SOURCE["spmv"]
    if w.name.startswith("skinny"):
        return KERNEL_SOURCE["skinny"]
    if w.name.startswith("fp32"):
        return KERNEL_SOURCE["fp32"]
    return KERNEL_SOURCE["int8" if w.name.startswith("int8") else "bf16"]


# ----------------------------------------------------------------- e2e leg --

def e2e_leg(w, steps, warmup, device):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory, runs the GEMM and reads C back to
    pinned host memory.  The copies are pipelined the way a host-fed caller
    would: device inputs are double-buffered, a copy-in stream moves step
    i+1's A, B (and C) while the GEMM of step i runs on the compute stream, and
    a copy-out stream returns step i's C; events keep every buffer's copy-in,
    GEMM and copy-out in order.  The timed region starts before the first
    copy-in and ends after the last copy-out."""
    import torch

    import dense_gemm_accelerator_gb300 as dga
    from dense_gemm_accelerator_gb300 import inputs as gen
    A, B, C = gen.make_inputs(w, with_c=w.beta != 0)
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = C.pin_memory() if C is not None else None
    odt = gen.TORCH_DTYPE[w.out_dtype]
    out = [torch.empty((w.M, w.N), dtype=odt).pin_memory() for _ in range(2)]
    dA = [torch.empty_like(hA, device=device) for _ in range(2)]
    dB = [torch.empty_like(hB, device=device) for _ in range(2)]
    dC = [torch.empty((w.M, w.N), dtype=odt, device=device) for _ in range(2)]
    compute = torch.cuda.current_stream()
    copy_in = torch.cuda.Stream(device=device)
    copy_out = torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    gemm_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(copy_in):
            if used[b]:
                copy_in.wait_event(out_done[b])  # step i-2 is done with buffer b
            dA[b].copy_(hA, non_blocking=True)
            dB[b].copy_(hB, non_blocking=True)
            if hC is not None:
                dC[b].copy_(hC, non_blocking=True)
            in_ready[b].record(copy_in)
        compute.wait_event(in_ready[b])
        dga.gemm(dA[b], dB[b].t() if w.layout_b == gen.COL_MAJOR else dB[b], dC[b], w.alpha,
                 w.beta, tf32=w.in_dtype == gen.TF32, stream=compute.cuda_stream)
        gemm_done[b].record(compute)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(gemm_done[b])
            out[b].copy_(dC[b], non_blocking=True)
            out_done[b].record(copy_out)
        used[b] = True

    def run(n, first):
        for i in range(n):
            step(first + i)
        for b in range(2):
            if used[b]:
                compute.wait_event(out_done[b])  # the region ends after the last copy-out

    run(warmup, 0)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    copy_in.wait_event(t0)  # no copy of the timed steps starts before t0
    run(steps, warmup)
    t1.record(compute)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    fl, by = workload_accounting(w)
    h2d = hA.numel() * hA.element_size() + hB.numel() * hB.element_size() + \
        (hC.numel() * hC.element_size() if hC is not None else 0)
    d2h = out[0].numel() * out[0].element_size()
    if w.name.startswith("skinny"):
        val, unit = by / (ms * 1e-3) / 1e9, "GB/s"
    else:
        val, unit = fl / (ms * 1e-3) / 1e12, ("TOPS" if w.in_dtype == gen.I8 else "TFLOPS")
    return {"value": sig(val, 5), "unit": unit, "ms_per_step": sig(ms, 5), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipeline": "double-buffered; copy-in of step i+1 and copy-out of step i-1 "
                        "overlap the GEMM of step i"}


# ------------------------------------------------------- CPU oracle timing --

def cpu_model():
    """The host CPU's model name from /proc/cpuinfo; on Arm hosts, which list
    no model name, the machine type with the first core's implementer and
    part codes."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" not in line:
                    continue
                key, val = (x.strip() for x in line.split(":", 1))
                fields.setdefault(key.lower(), val)
    except OSError:
        pass
    for key in ("model name", "cpu model"):
        if key in fields:
            return fields[key]
    if "cpu part" in fields:
        return (f"{platform.machine()} (implementer {fields.get('cpu implementer', '?')}, "
                f"part {fields['cpu part']})")
    return platform.machine()


class OracleSample:
    """Times the CPU oracle, as it stands, on the first `rows` output rows of
    the workload (all N columns, full K), on this host's cores."""

    def __init__(self, w):
        self.threads = len(os.sched_getaffinity(0))
        os.environ.setdefault("OMP_NUM_THREADS", str(self.threads))
        self.threads = int(os.environ["OMP_NUM_THREADS"])
        from dense_gemm_accelerator_gb300 import inputs as gen
        self.w, self.gen = w, gen
        self.A, self.B, self.C = gen.make_inputs(w, with_c=w.beta != 0)
        self.ldb = w.K if w.layout_b == gen.COL_MAJOR else w.N

    def run(self, rows):
        import oracle
        w, gen = self.w, self.gen
        a = self.A[:rows].contiguous()
        c = self.C[:rows].contiguous() if self.C is not None else None
        t = time.perf_counter()
        if w.in_dtype == gen.I8:
            oracle.gemm_i8(w.layout_b, rows, w.N, w.K, w.alpha, a, w.K, self.B, self.ldb, w.beta,
                           c, w.N)
        else:
            oracle.gemm_fp(w.in_dtype, w.out_dtype, w.layout_b, rows, w.N, w.K, w.alpha, a, w.K,
                           self.B, self.ldb, w.beta, c, w.N)
        return time.perf_counter() - t

    def rows_for(self, target_s):
        probe = max(1, min(self.w.M, self.threads))
        dt = self.run(probe)
        return int(min(self.w.M, max(probe, probe * target_s / max(dt, 1e-6))))


# ------------------------------------------------------------------- main --

def max_over_ranks(local_ms, world, device=None):
    """The slowest rank's timed-region length (ms): the job finishes when the
    last replica does.  Works with any process-group backend (NCCL on the
    GPUs, gloo in the CPU tests)."""
    if world <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step_per_rank, world, steps, max_ms, scale):
    """Whole-job throughput: the units every rank processed (weak scaling:
    each replica runs the full workload) over the slowest rank's time."""
    return world * units_per_step_per_rank * steps / (max_ms * 1e-3) / scale


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    if w.kind != "gemm":
        print(json.dumps({"impl": "reference", "unavailable":
                          f"the oracle arm times single GEMM workloads; {w.name} is a layer step"}))
        return 0
    # each step is a bounded sample, sized so the whole run stays within minutes
    per_step_s = max(0.5, min(4.0, 150.0 / (args.steps + args.warmup)))
    sampler = OracleSample(w)
    rows = sampler.rows_for(per_step_s)
    fl_total, dt_total = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        dt = sampler.run(rows)
        if i >= args.warmup:
            fl_total += gemm_flops(rows, w.N, w.K)
            dt_total += dt
    val = fl_total / dt_total / 1e12
    unit = "TFLOPS"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt_total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                       "beta": w.beta},
            "cpu_baseline": {"value": val, "unit": unit, "cores": sampler.threads, "kind": "oracle",
                             "cpu": cpu_model(),
                             "sample": f"first {rows} of {w.M} output rows, all {w.N} columns, "
                                       f"full K={w.K}, per step"},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="fp32_4096")
    ap.add_argument("--impl", default="dga", choices=["dga", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip per_dtype, e2e and cpu legs")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target length of the oracle's CPU-baseline sample")
    args = ap.parse_args()

    from dense_gemm_accelerator_gb300 import inputs as gen
    w = gen.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w)

    import torch
    import torch.distributed as dist

    import __graft_entry__
    rank, world, local = dist_env()
    if world == 1:
        __graft_entry__.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
        if rank == 0:
            __graft_entry__.build()
        dist.barrier()
    import dense_gemm_accelerator_gb300 as dga
    dga.lib()

    props = torch.cuda.get_device_properties(device)
    peaks = load_peaks(props.multi_processor_count)
    # the FP32 denominator is derived from unit counts; the probe checks it
    # and replaces it if the pipe is measured faster
    try:
        probe = fp32_fma_probe(device)
    except RuntimeError as e:  # the cross-check failed: keep the unit-count peak, say why
        probe = {"error": str(e)}
    peaks["fp32_ffma_probe"] = probe
    try:  # context for the INT8 row: the legacy integer instruction's rate
        peaks["int8_mma_sync_tops"] = int8_mma_probe(device)
    except RuntimeError:
        peaks["int8_mma_sync_tops"] = None
    if "error" not in probe:
        best_probe = max(probe["ffma_tflops"], probe["ffma2_tflops"])
        if best_probe > 1.01 * peaks["fp32_ffma_tflops"]:
            peaks["fp32_ffma_tflops"] = best_probe
            peaks["fp32_ffma_basis"] = "FMA probe (measured above the unit-count figure)"

    runner = runner_for(w, device, sets_for(w), seed=rank)
    stream = torch.cuda.current_stream()
    s = stream.cuda_stream
    for i in range(args.warmup):
        runner.call(i, s)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    launches = 0
    for i in range(args.steps):
        launches += runner.call(args.warmup + i, s)
    g1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_end = time.time()
    time.sleep(0.2)
    clocks.stop()
    total_ms = max_over_ranks(g0.elapsed_time(g1), world, device)
    ms_per_step = total_ms / args.steps
    # the dominant kernel's time per launch: the whole call's time per step
    # (the paths measured here launch one kernel per call; when a call
    # launches more, their sum is attributed to the call)
    kmean = g0.elapsed_time(g1) / args.steps
    nnz = getattr(runner, "mean_nnz", None)
    fl, by = workload_accounting(w, nnz)
    if w.name.startswith("skinny") or w.kind == "spmv":
        value, unit = job_throughput(by, world, args.steps, total_ms, 1e9), "GB/s"
    else:
        value = job_throughput(fl, world, args.steps, total_ms, 1e12)
        unit = "TOPS" if w.in_dtype == gen.I8 else "TFLOPS"
    roof = roofline_for(w, kmean, peaks, nnz=nnz)
    roof["traffic"] = traffic_record(source_of(w), w.name)
    roof["kernel_ms_mean"] = kmean
    roof["launches_per_step"] = launches / args.steps
    main_clocks = clocks.summary(t_begin, t_end)
    add_spec_peak(roof, peaks, main_clocks.get("sm_mhz"))
    for k in ("achieved", "peak", "frac", "kernel_ms_mean"):
        roof[k] = sig(roof[k], 6)

    line = {"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {gen.F32: "f32", gen.BF16: "bf16", gen.F16: "f16", gen.I8: "int8",
                      gen.TF32: "tf32"}[w.in_dtype],
            "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                       "beta": w.beta, "layout_b": "col" if w.layout_b else "row",
                       "path": (",".join(runner.paths) if w.kind in ("fc", "spmv")
                                else dga.PATH_NAMES[dga.dga_last_path()]),
                       "l2": f"inputs rotated over {len(runner.sets)} resident sets (> 2x L2 per rotation)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof, "gpu_launches": launches,
            "clocks": main_clocks}
    del runner
    torch.cuda.empty_cache()

    # (a fully-connected workload as the main one is for profiling: its
    # extras -- e2e, the oracle sample -- are defined for single GEMMs)
    if rank == 0 and world == 1 and not args.no_extras and w.kind == "gemm":
        line["e2e"] = e2e_leg(w, max(3, args.steps), 2, device)
        sampler = OracleSample(w)
        rows = sampler.rows_for(args.cpu_seconds)
        dt = sampler.run(rows)
        rate = gemm_flops(rows, w.N, w.K) / dt
        line["cpu_baseline"] = {"value": sig(rate / 1e12), "unit": "TFLOPS",
                                "cores": sampler.threads, "cpu": cpu_model(), "kind": "oracle",
                                "sample": f"first {rows} of {w.M} output rows (all {w.N} columns, "
                                          f"K={w.K}) in {dt:.1f} s"}
        per = {}
        legs = [(n, None) for n in PER_DTYPE if n != w.name]
        legs += [(n, SUSTAINED_SECONDS) for n in SUSTAINED]
        for name, seconds in legs:
            ow = gen.WORKLOADS[name]
            r = runner_for(ow, device, sets_for(ow, 3 if name.startswith("skinny") else 2))
            if seconds is None:
                iters = 200 if name.startswith("skinny") else (10 if ow.kind == "fc" else 30)
            else:  # back to back for `seconds`, from the burst row's time per call
                iters = max(30, int(seconds * 1e3 / per.get(name, {}).get("ms", 1.0)))
            leg_clocks = ClockSampler(local)
            leg_clocks.start()
            time.sleep(0.15)
            t0 = time.time()
            ms, nl = time_kernel(r, iters, 5 if ow.kind != "fc" else 2)
            t1 = time.time()
            leg_clocks.stop()
            rf = roofline_for(ow, ms, peaks, sustained=seconds is not None,
                              nnz=getattr(r, "mean_nnz", None))
            rf["traffic"] = traffic_record(source_of(ow), name) if ow.kind != "fc" else None
            rf["ms_mean"] = ms
            rf["launches_per_call"] = nl / iters
            rf["clocks"] = leg_clocks.summary(t0 - 0.05, t1 + 0.05)
            if ow.kind == "spmv":
                rf["nnz"] = r.mean_nnz
            if rf["bound"] == "tensor":
                rf["frac_of_sustained"] = rf["achieved"] / peaks["bf16_tflops_sustained"]
            if seconds is not None:
                rf["calls"], rf["seconds"] = float(iters), iters * ms * 1e-3
            add_spec_peak(rf, peaks, rf["clocks"].get("sm_mhz"))
            row = compact_row(rf)
            if ow.in_dtype == gen.I8 and peaks.get("int8_mma_sync_tops"):
                # against the best rate of the integer mma.sync instruction
                row["x_probe"] = sig(rf["achieved"] / peaks["int8_mma_sync_tops"], 3)
            per[name if seconds is None else name + "_sustained"] = row
            del r
            torch.cuda.empty_cache()
        line["peaks"] = compact_peaks(peaks)
        line["per_dtype"] = per
    else:
        line["peaks"] = compact_peaks(peaks)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
