"""Benchmark: fp32 GEMM C = A x B at M = N = K = 4096 on GB300 (libgemm_f32).

One step = one gemm_f32 call in `exact` mode (FP32-accurate 3xTF32 on the
tensor cores; `--mode` selects another mode) on the square 4096^3 workload: A, B i.i.d. uniform[-1, 1) from
fixed seeds, row-major, C overwritten. Inputs are resident in HBM before the
timed region; L2 is flushed (a 256 MiB write) between timed steps, outside the
per-step CUDA events. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica of the workload on its own GPU
(no collective on the data path; weak scaling); the time is the max over ranks.
`--impl reference` times the fp64 CPU oracle on the host cores instead (rank 0
only), a bounded sample of the same workload per step.
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
sys.path.insert(0, ROOT)

METRIC = "GFLOP/s (2MNK/t) for fp32 GEMM at 4096³; % of TF32/FP32 roofline"
WORKLOADS = {
    "c1": "square fp32 GEMM M=N=K=512, row-major, A and B i.i.d. uniform[-1,1) from seed, C overwritten",
    "c2": "square fp32 GEMM M=N=K=1024, row-major, A,B uniform[-1,1) from seed",
    "c3": "square fp32 GEMM M=N=K=2048, row-major, A,B uniform[-1,1) from seed",
    "c4": "square fp32 GEMM M=N=K=4096, row-major, A,B uniform[-1,1) from seed (headline size)",
    "c5a": "ragged fp32 GEMM M=1000, K=777, N=1531, row-major, A,B normal(0,1) from seed",
    "c5b": "transformer-projection fp32 GEMM M=8192, K=4096, N=11008, row-major, A,B normal(0,1) from seed",
}
WORKLOAD = WORKLOADS["c4"]
M = N = K = 4096
FLUSH_BYTES = 256 << 20
# Nominal dense tensor rates of one GB300: TF32 1.1 PFLOP/s, BF16 2.25 PFLOP/s
# (without 2:4 sparsity). Their ratio turns the measured bf16 peak into the
# TF32 denominator.
TF32_PER_BF16 = 1.1 / 2.25
FP32_LANES_PER_SM = 128
# Workloads timed in the configs leg besides the benchmark's own, and the
# steps each takes (8192 x 11008 x 4096 runs 2 ms per exact call).
CONFIG_LEG = (("c1", 50), ("c2", 50), ("c3", 50), ("c4", 50), ("c5a", 50), ("c5b", 10))


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--mode", default="exact", choices=["exact", "tf32", "exact_simt"],
                    help="accuracy mode of the timed steps (the headline is exact)")
    ap.add_argument("--no-extras", action="store_true", help="skip the other modes, e2e and CPU legs")
    ap.add_argument("--config", default="c4", choices=sorted(WORKLOADS),
                    help="workload (the benchmark is c4; the others are for the record)")
    ap.add_argument("--layout", default="nn", choices=["nn", "nt", "tn", "tt"],
                    help="operand storage (n: as is, t: transposed) through gemm_f32_general; "
                         "the benchmark is nn through gemm_f32")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(bf16=float(p["bf16_tflops"]), bf16_sustained=float(p["bf16_tflops_sustained"]),
                    hbm=float(p["hbm_gbs"]), sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(bf16=1900.0, bf16_sustained=1700.0, hbm=6800.0, sm_max_mhz=2070.0,
                    source="fallback")


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None
        self.error = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError as e:
            self.error = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return {"unavailable": self.error or "nvidia-smi not started"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(t=t, sm=float(parts[1]), sm_max=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_start - 0.06 <= r["t"] <= self.t_stop + 0.06]
        used = inside or [r for r in rows if self.t_start - 0.5 <= r["t"] <= self.t_stop + 0.5]
        if not used:
            return {"unavailable": "no nvidia-smi samples during the timed region"}
        reasons = set()
        for r in used:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in used),
                "sm_max_mhz": max(r["sm_max"] for r in used),
                "reasons": sorted(reasons), "samples": len(used),
                "window": "timed region" if inside else "timed region +-0.5 s"}


# ----------------------------------------------------------- GPU timing --

def time_steps(torch, fn, steps, warmup, flush_buf, stream, barrier=None):
    """Per-step device times (ms) of fn() with an L2 flush between steps."""
    for _ in range(warmup):
        flush_buf.zero_()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush_buf.zero_()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    wall = time.perf_counter() - t0
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], wall


def kernel_label(g, kernel, mode):
    """Name of the kernel gemm_f32 runs for this selection: the TMA-fed TF32
    pass and 3xTF32 run on CTA-pair kernels."""
    if kernel == g.KERNEL_SIMT:
        return "simt_gemm"
    if kernel == g.KERNEL_TC_TMA:
        return "tc_pair_tma_3xtf32" if mode == "exact" else "tc_pair_tma_tf32"
    if kernel == g.KERNEL_TC_LSU:
        return "tc_lsu_3xtf32" if mode == "exact" else "tc_lsu_tf32"
    return str(kernel)


def time_back_to_back(torch, fn, steps, warmup, stream):
    """Mean device time (ms) of fn() over `steps` calls enqueued back to back
    between one pair of CUDA events (for inputs larger than L2, which need no
    flush; the queue stays ahead of the GPU, so host enqueue time is hidden)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def traffic_lookup(kernel: str, workload: str, mode: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    src = hashlib.sha256()
    if kernel.startswith("simt"):
        files = ("simt_gemm.cu",)
    elif kernel.startswith("reduce"):
        files = ("reduce.cu",)
    else:
        files = ("tc_gemm.cu", "ptx.cuh")
    for f in files:
        with open(os.path.join(ROOT, "dense_fp32_gemm_major_gb300", "csrc", f), "rb") as fh:
            src.update(fh.read())
    sha = src.hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None, sha
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if (kv.get("kernel") == kernel and kv.get("workload") == workload
                    and kv.get("mode") == mode and kv.get("src_sha256") == sha):
                return int(kv["dram_bytes_per_launch"]), sha
    return None, sha


# ------------------------------------------------------- rank reduction --

def reduce_max(value: float, dist=None, device="cpu") -> float:
    """Max of `value` over all ranks (identity without a process group)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gflops(max_total_ms: float, world: int, steps: int, flops_per_step: float) -> float:
    """Aggregate throughput: every rank runs `steps` replicas of the workload;
    the job takes as long as its slowest rank."""
    return world * steps * flops_per_step / (max_total_ms / 1e3) / 1e9


# -------------------------------------------------------------- CPU legs --

def oracle_rows_gflops(a, b, budget_s: float, max_rows: int | None = None):
    """Time the fp64 oracle on whole rows of the product until ~budget_s."""
    import numpy as np
    import oracle

    threads = oracle.num_threads()
    batch = max(1, threads)
    rows_done, elapsed, start = 0, 0.0, 0
    m, k = a.shape
    n = b.shape[1]
    while elapsed < budget_s and (max_rows is None or rows_done < max_rows):
        rows = (np.arange(batch) + start) % m
        t0 = time.perf_counter()
        oracle.gemm_rows(a, b, rows)
        elapsed += time.perf_counter() - t0
        rows_done += batch
        start += batch
    flops = 2.0 * rows_done * n * k
    return flops / elapsed / 1e9, threads, rows_done, elapsed


def check_result(torch, dC, rank):
    """After the timed steps: every element of C was written (C was NaN-filled
    before the first step) and is finite. Rank 0 only; the comparison with
    the oracle is the tests' job."""
    if rank != 0:
        return None
    finite = bool(torch.isfinite(dC).all().item())
    return {"c_nan_filled_before_first_step": True, "all_finite_after_last_step": finite}


def run_reference(args, rank):
    import synth

    if rank != 0:
        return
    a, b, cfg = synth.config_operands("c4")
    import oracle

    threads = oracle.num_threads()
    rows_per_step = max(1, threads)
    # untimed warm-up steps, then exactly `steps` timed steps of rows_per_step rows each
    for w in range(args.warmup):
        oracle.gemm_rows(a, b, [(w * rows_per_step + i) % M for i in range(rows_per_step)])
    t0 = time.perf_counter()
    for s in range(args.steps):
        oracle.gemm_rows(a, b, [(s * rows_per_step + i) % M for i in range(rows_per_step)])
    wall = time.perf_counter() - t0
    flops = 2.0 * args.steps * rows_per_step * N * K
    value = flops / wall / 1e9
    sample = (f"{rows_per_step} whole rows of the 4096^3 product per step "
              f"({rows_per_step}x4096x4096 multiply-adds, fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "sample": sample},
        "cpu_baseline": {"value": round(value, 3), "unit": "GFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main --

def main():
    global M, N, K, WORKLOAD
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
        return

    import numpy as np
    import torch

    import dense_fp32_gemm_major_gb300 as g
    import synth

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier(device_ids=[local])

    a, b, cfg = synth.config_operands(args.config)
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    WORKLOAD = WORKLOADS[args.config]
    transa, transb = (1 if args.layout[0] == "t" else 0), (1 if args.layout[1] == "t" else 0)
    if args.layout != "nn":
        WORKLOAD += f"; A stored {'K x M' if transa else 'M x K'}, B stored {'N x K' if transb else 'K x N'}"
    dA = torch.from_numpy(np.ascontiguousarray(a.T) if transa else a).cuda()
    dB = torch.from_numpy(np.ascontiguousarray(b.T) if transb else b).cuda()
    lda, ldb = dA.shape[1], dB.shape[1]
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    dA_lib = dA if not transa else dA.t()
    dB_lib = dB if not transb else dB.t()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def gemm_call(mode):
        if args.layout != "nn":
            def fn():
                st = g.gemm_f32_general(g.ROW_MAJOR, transa, transb, M, N, K, 1.0, dA.data_ptr(),
                                        lda, dB.data_ptr(), ldb, 0.0, dC.data_ptr(), N, mode,
                                        g.KERNEL_AUTO, sptr)
                if st != g.OK:
                    raise g.GemmError(st, "gemm_f32_general")
            return fn

        def fn():
            st = g.gemm_f32(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N, mode, sptr)
            if st != g.OK:
                raise g.GemmError(st)
        return fn

    mode = g.MODES[args.mode]
    kernel = g.gemm_f32_select(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                               mode, g.KERNEL_AUTO)
    kernel_name = kernel_label(g, kernel, args.mode)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    fn = gemm_call(mode)
    dC.fill_(float("nan"))  # every step overwrites C; checked after the last one
    for _ in range(args.warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    times, wall = time_steps(torch, fn, args.steps, 0, flush, stream, barrier)
    if sampler:
        sampler.mark_stop()
    clocks = sampler.stop() if sampler else None
    st = g.gemm_f32_poll_device_status(sptr)
    if st != g.OK:
        raise g.GemmError(st, "device status")
    check = check_result(torch, dC, rank)
    if check is not None and not check["all_finite_after_last_step"]:
        raise RuntimeError("C holds NaN/Inf after the timed steps")

    total_ms = reduce_max(sum(times), dist, "cuda")
    flops = 2.0 * M * N * K
    value = whole_job_gflops(total_ms, world, args.steps, flops)
    ms_per_step = total_ms / args.steps

    pk = peaks()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    tf32_peak = pk["bf16"] * TF32_PER_BF16
    alu_peak = sms * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
    if args.layout != "nn" and kernel != g.KERNEL_SIMT:
        # A stored transposed reaches the TMA-fed 3xTF32 kernel through a
        # transposed copy (the TF32 pair kernel reads it as it is)
        kernel_name += "_" + args.layout + (
            "_after_transpose" if transa and kernel == g.KERNEL_TC_TMA and args.mode == "exact"
            else "")
    traffic, sha = traffic_lookup(kernel_name, args.config, args.mode)
    if args.mode == "exact_simt":
        achieved = flops / (ms_per_step / 1e3) / 1e12
        roofline = {"bound": "alu", "achieved": round(achieved, 2), "peak": round(alu_peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / alu_peak, 4), "traffic": traffic,
                    "kernel": kernel_name,
                    "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x "
                                   f"{pk['sm_max_mhz']:.0f} MHz"}
    else:
        mult = 3 if args.mode == "exact" else 1  # 3xTF32: three TF32 MMAs per fp32 multiply-add
        achieved = mult * flops / (ms_per_step / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(tf32_peak, 1),
                    "unit": "TFLOP/s", "frac": round(achieved / tf32_peak, 4), "traffic": traffic,
                    "kernel": kernel_name,
                    "peak_source": f"{pk['source']} bf16 burst {pk['bf16']} TFLOP/s x nominal "
                                   f"dense TF32/BF16 ratio 1.1/2.25 = {TF32_PER_BF16:.4f}",
                    "achieved_counts": f"{mult} x 2MNK TF32 flops"}

    extras = {}
    cpu = None
    e2e = None
    if rank == 0 and not args.no_extras:
        # the other modes, fewer steps, same protocol
        others = [("exact", g.EXACT, "tensor", tf32_peak, 3), ("tf32", g.TF32, "tensor", tf32_peak, 1),
                  ("exact_simt", g.EXACT_SIMT, "alu", alu_peak, 1)]
        for mname, mcode, bound, peak, mult in others:
            if mname == args.mode:
                continue
            steps = 30 if mname == "exact_simt" else 200
            ts, _ = time_steps(torch, gemm_call(mcode), steps, 5, flush, stream)
            ms = statistics.mean(ts)
            ach = mult * flops / (ms / 1e3) / 1e12
            mk = g.gemm_f32_select(M, N, K, dA.data_ptr(), K, dB.data_ptr(), N, dC.data_ptr(), N,
                                   mcode, g.KERNEL_AUTO)
            mkname = kernel_label(g, mk, mname)
            mtraffic, _ = traffic_lookup(mkname, args.config, mname)
            extras[mname] = {"value": round(flops / (ms / 1e3) / 1e9, 1), "unit": "GFLOP/s",
                             "ms_per_step": round(ms, 4), "steps": steps,
                             "roofline": {"bound": bound, "achieved": round(ach, 2),
                                          "peak": round(peak, 1), "unit": "TFLOP/s",
                                          "frac": round(ach / peak, 4), "traffic": mtraffic,
                                          "kernel": mkname}}
        # context, not a denominator: the vendor library on the same workload
        # (torch.matmul -> cuBLAS), one TF32 pass and full FP32
        lib_ref = {}
        tf32_flag = torch.backends.cuda.matmul.allow_tf32
        for name, allow in (("cublas_tf32", True), ("cublas_fp32", False)):
            torch.backends.cuda.matmul.allow_tf32 = allow
            ref_out = torch.empty((M, N), dtype=torch.float32, device="cuda")
            ts, _ = time_steps(torch, lambda: torch.matmul(dA_lib, dB_lib, out=ref_out), 50, 5,
                               flush, stream)
            lib_ref[name] = {"value": round(flops / (statistics.mean(ts) / 1e3) / 1e9, 1),
                             "unit": "GFLOP/s", "ms_per_step": round(statistics.mean(ts), 4)}
            del ref_out
        torch.backends.cuda.matmul.allow_tf32 = tf32_flag
        extras["library_reference"] = lib_ref
        # context, not a denominator: what the TF32 tensor pipe and the FP32
        # FMA pipe deliver to MMA-only / FFMA-only probe kernels here
        pst, ptf32, pfp32, ptf32_mhz, pfp32_mhz = g.gemm_f32_measure_peaks()
        if pst == g.OK:
            probe = {"tf32_mma_tflops": round(ptf32, 1), "tf32_sm_mhz": round(ptf32_mhz),
                     "fp32_fma_tflops": round(pfp32, 1), "fp32_sm_mhz": round(pfp32_mhz),
                     "note": "probe kernels (gemm_f32_measure_peaks): operands non-zero, SM "
                             "clock measured inside each kernel (clock64 ticks / globaltimer); "
                             "the roofline fractions stay against the measured bf16 peak x the "
                             "nominal ratio"}
            extras["probe_peaks"] = probe
            pk_ctx, pk_mhz = (pfp32, pfp32_mhz) if roofline["bound"] == "alu" else (ptf32, ptf32_mhz)
            roofline["probe_peak"] = round(pk_ctx, 1)
            roofline["probe_sm_mhz"] = round(pk_mhz)
            roofline["frac_of_probe_peak"] = round(roofline["achieved"] / pk_ctx, 4)
            if clocks and clocks.get("sm_mhz") and pk_mhz > 0:
                # flops per SM clock against the probe's flops per SM clock:
                # the kernel at the median clock sampled over its timed steps
                roofline["frac_of_probe_peak_per_clock"] = round(
                    (roofline["achieved"] / clocks["sm_mhz"]) / (pk_ctx / pk_mhz), 4)
        else:
            ptf32 = None
        # every workload of the benchmark table in both tensor-core modes:
        # fewer steps, same protocol (L2 flushed between steps), through gemm_f32
        configs = {}
        for cname, csteps in CONFIG_LEG:
            ca, cb, ccfg = synth.config_operands(cname)
            cm, cn, ck = ccfg["M"], ccfg["N"], ccfg["K"]
            xa, xb = torch.from_numpy(ca).cuda(), torch.from_numpy(cb).cuda()
            xc = torch.empty((cm, cn), dtype=torch.float32, device="cuda")
            cflops = 2.0 * cm * cn * ck
            entry = {"workload": WORKLOADS[cname], "M": cm, "N": cn, "K": ck}
            for mname, mcode, mult in (("exact", g.EXACT, 3), ("tf32", g.TF32, 1)):
                def cfn(mcode=mcode):
                    st = g.gemm_f32(cm, cn, ck, xa.data_ptr(), ck, xb.data_ptr(), cn, xc.data_ptr(),
                                    cn, mcode, sptr)
                    if st != g.OK:
                        raise g.GemmError(st)
                xc.fill_(float("nan"))
                ts, _ = time_steps(torch, cfn, csteps, 5, flush, stream)
                ms = statistics.mean(ts)
                ach = mult * cflops / (ms / 1e3) / 1e12
                mk = g.gemm_f32_select(cm, cn, ck, xa.data_ptr(), ck, xb.data_ptr(), cn,
                                       xc.data_ptr(), cn, mcode, g.KERNEL_AUTO)
                entry[mname] = {
                    "value": round(cflops / (ms / 1e3) / 1e9, 1), "unit": "GFLOP/s",
                    "us_per_call": round(ms * 1e3, 2),
                    "us_per_call_median": round(statistics.median(ts) * 1e3, 2),
                    "steps": csteps, "kernel": kernel_label(g, mk, mname),
                    "achieved_tflops": round(ach, 2), "achieved_counts": f"{mult} x 2MNK TF32 flops",
                    "frac": round(ach / tf32_peak, 4),
                    "frac_of_probe_peak": round(ach / ptf32, 4) if ptf32 else None,
                    "all_finite": bool(torch.isfinite(xc).all().item())}
            configs[cname] = entry
            del xa, xb, xc
        extras["configs"] = configs
        # the pages' second workload: the per-group tree reduction of 2^26 fp32
        # values (two dispatches), HBM-bound; the vector (256 MiB) exceeds L2,
        # so steps run back to back without a flush
        rn = 1 << 26
        xr = torch.from_numpy(synth.uniform_pm1((rn,), 1026).reshape(-1)).cuda()
        rout = torch.empty(1, dtype=torch.float32, device="cuda")

        def reduce_fn():
            st = g.reduce_f32_sum(rn, xr.data_ptr(), rout.data_ptr(), 0, sptr)
            if st != g.OK:
                raise g.GemmError(st, "reduce_f32_sum")

        rms = time_back_to_back(torch, reduce_fn, 500, 20, stream)
        rgbs = 4.0 * rn / (rms / 1e3) / 1e9
        rtraffic, _ = traffic_lookup("reduce_partials_kernel", "2p26", "sum")
        extras["reduce_sum"] = {
            "workload": "sum of 2^26 fp32 values, uniform[-1,1) from seed (reduce_f32_sum: "
                        "per-group partials, then a second dispatch)",
            "value": round(rgbs, 1), "unit": "GB/s", "ms_per_step": round(rms, 4), "steps": 500,
            "gpu_launches_per_step": 2,
            "l2": "input (256 MiB) larger than L2; steps back to back, no flush",
            "roofline": {"bound": "hbm", "achieved": round(rgbs, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(rgbs / pk["hbm"], 4),
                         "algorithmic_bytes": 4 * rn, "traffic": rtraffic,
                         "kernel": "reduce_partials_kernel (+ reduce_final_kernel, 1 CTA)"}}
        del xr
        # end to end through the host-buffer entry point (pinned host memory)
        ha = torch.from_numpy(a).pin_memory().numpy()
        hb = torch.from_numpy(b).pin_memory().numpy()
        hc = torch.empty((M, N), dtype=torch.float32).pin_memory().numpy()
        e2e_steps = max(3, min(args.steps, 30))
        for _ in range(3):
            g.matmul_host(ha, hb, "exact", out=hc)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            g.matmul_host(ha, hb, "exact", out=hc)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e = {"value": round(flops / e2e_s / 1e9, 1), "unit": "GFLOP/s",
               "h2d_bytes_per_step": 4 * (M * K + K * N), "d2h_bytes_per_step": 4 * M * N,
               "api": "gemm_f32_host (blocking; pinned host buffers)", "steps": e2e_steps}
        # the oracle on the host cores, a bounded sample of the same workload
        gf, threads, rows, secs = oracle_rows_gflops(a, b, budget_s=12.0)
        cpu = {"value": round(gf, 3), "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} whole rows of the {M}x{N}x{K} product ({rows}x{N}x{K} "
                         f"multiply-adds in fp64), {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "mode": args.mode,
                       "layout": args.layout, "kernel": kernel_name, "l2": "flushed (256 MiB write) between timed steps",
                       "replicas": world, "parallelism": "replicas" if world > 1 else "single"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "check": check,
            "clocks": clocks,
            "modes": extras,
            "timing": {"per_step_ms_median": round(statistics.median(times), 4),
                       "per_step_ms_min": round(min(times), 4),
                       "per_step_ms_max": round(max(times), 4), "wall_s": round(wall, 3),
                       "kernel_src_sha256": sha},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
