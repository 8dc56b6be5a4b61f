"""Benchmark: emulated FP64 GEMM (Ozaki scheme II on GB300 tensor cores).

One step = one whole ozk_dgemm call (exponent scan, residue quantisation, one
residue GEMM per modulus with fused mod reduction, CRT combine with unscale)
on the 4096^3 workload, N(0,1) inputs, 14 moduli, inputs resident in HBM.
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs as one process per GPU (torchrun); every rank computes its own
replica of the workload (the path has no exchange step), so scaling is weak
and `value` sums the work of all ranks over the slowest rank's time.
`--impl reference` times the CPU oracle (plain C, OpenMP) on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from fp64_gemm_emulation_exponent_gb300 import workloads  # noqa: E402

METRIC = "emulated-DGEMM effective FP64 TFLOP/s at 4096^3 (53-bit) and % INT8 tensor peak"
WORKLOAD = "square4096_normal"
N_MODULI = 14
STAGES = ["scan", "quantize", "residue_gemm", "crt_combine"]


def rows_fused(M: int, kpad: int) -> bool:
    """Whether ozk_dgemm scans the rows of A inside their quantisation (the
    library's rule: a row fits one block, kpad <= 4096, and M * kpad >= 2^22)."""
    return kpad <= 4096 and M * kpad >= 1 << 22


def kernels_per_step(M: int, kpad: int) -> int:
    """Our kernels per ozk_dgemm call: scan, quantize (which derives the scales
    from the scanned maxima), residue_gemm, crt, and the fused scan-and-quantize
    of A's rows when that is used (the maxima's memset is a runtime call)."""
    return 5 if rows_fused(M, kpad) else 4


PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "residue_gemm_traffic.json")


# ---------------------------------------------------------------------------
# distributed plumbing (host-side only: barrier and max/sum over ranks)
# ---------------------------------------------------------------------------
class Ranks:
    def __init__(self, world: int):
        self.world = world
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if world > 1:
            import torch.distributed as dist

            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return reduce_over_ranks(self.pg, x, "max")

    def sum(self, x: float) -> float:
        return reduce_over_ranks(self.pg, x, "sum")

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def reduce_over_ranks(dist, x: float, op: str) -> float:
    """max or sum of a host float over all ranks (identity without a group)."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def replica_throughput(flops_per_step: float, steps: int, ranks_times_s: list) -> float:
    """Whole-job TFLOP/s: all ranks' work over the slowest rank's time."""
    return len(ranks_times_s) * flops_per_step * steps / max(ranks_times_s) / 1e12


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir: str):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(log_dir, f"clocks_rank{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# measured peaks and the committed ncu traffic figure
# ---------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("residue_gemm.cu", "ozk_internal.h"):
        h.update(open(os.path.join(ROOT, "fp64_gemm_emulation_exponent_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload_key: str):
    """DRAM bytes per residue-GEMM launch from the committed ncu summary, or
    None when the kernel source changed since those counters were taken."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    d = json.load(open(PROFILE_TRAFFIC))
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    entry = d.get("workloads", {}).get(workload_key)
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (rows x columns block of C, full K)
# ---------------------------------------------------------------------------
def oracle_block_rate(A, B, n, rows, cols):
    import oracle

    t0 = time.perf_counter()
    oracle.dgemm(A[:rows], B[:, :cols].copy(), n)
    dt = time.perf_counter() - t0
    return 2.0 * rows * cols * A.shape[1] / dt / 1e12, dt


def cpu_baseline(A, B, n, target_s=12.0):
    import oracle

    # calibrate the row count of the sample so that it takes about target_s
    rows, cols = 4, 256
    _, dt = oracle_block_rate(A, B, n, rows, cols)
    while dt < target_s / 4 and rows < A.shape[0]:
        rows = int(min(A.shape[0], max(rows * 2, rows * target_s / max(dt, 1e-3) / 2)))
        _, dt = oracle_block_rate(A, B, n, rows, cols)
    if dt < target_s / 2 and rows < A.shape[0]:
        rows = int(min(A.shape[0], rows * target_s / max(dt, 1e-3)))
    rate, dt = oracle_block_rate(A, B, n, rows, cols)
    return {"value": rate, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"C[0:{rows}, 0:{cols}] of the {A.shape[0]}x{B.shape[1]}x{A.shape[1]} workload "
                      f"(full K, {n} moduli, every stage incl. CRT-vs-direct check), {dt:.1f} s wall"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args, ranks: Ranks):
    if ranks.rank != 0:
        return None
    import oracle

    w = workloads.WORKLOADS[args.workload]
    n = args.moduli
    A, B = workloads.workload_operands(w)
    # per step: a rows x cols block of C over the full K.  The oracle spreads
    # rows over its threads and prepares the block's columns once per call,
    # so the block holds at least 16 whole rounds of rows for every thread
    # (the per-call column work then costs what about one round does); it is
    # sized (once, untimed) so that warm-up and timed steps together take
    # about two minutes, narrowing the columns first where a step would
    # otherwise take longer than its share
    threads = max(1, oracle.threads())
    per_step = min(6.0, 120.0 / max(1, args.steps + args.warmup))
    cols = min(256, w.N)
    rows = min(w.M, 16 * threads)
    _, dt = oracle_block_rate(A, B, n, rows, cols)
    while dt > per_step and cols > 8:
        cols //= 2
        dt /= 2
    if dt < per_step / 2:
        rounds = max(1, int(per_step / max(dt, 1e-3)))
        rows = min(w.M, rows * rounds)
    for _ in range(args.warmup):
        oracle_block_rate(A, B, n, rows, cols)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_block_rate(A, B, n, rows, cols)
    dt = time.perf_counter() - t0
    value = 2.0 * rows * cols * w.K * args.steps / dt / 1e12
    sample = (f"per step C[0:{rows}, 0:{cols}] of {w.M}x{w.N}x{w.K} (full K, {n} moduli, "
              f"{threads} oracle threads)")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config(w, n),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config(w, n):
    from fp64_gemm_emulation_exponent_gb300 import ozk

    ab = 8 * (w.M * w.K + w.K * w.N)
    sl = 2 * n * (w.M + w.N) * ozk.ozk_kpad(w.K)
    return {"workload": f"{w.name}: M={w.M} N={w.N} K={w.K}, A,B i.i.d. {w.dist} seeded "
                        f"{1000 + w.seed}/{2000 + w.seed}, {n} moduli "
                        f"(beta={ozk.ozk_beta(w.K, n)} bits per operand)",
            "M": w.M, "N": w.N, "K": w.K, "n_moduli": n,
            "l2": f"inputs larger than L2 (A+B = {ab / 1e6:.0f} MB fp64; residue slices {sl / 1e6:.0f} MB per step)",
            "parallelism": "replicas (one independent GEMM per GPU)"}


def run_gpu(args, ranks: Ranks):
    import torch

    from fp64_gemm_emulation_exponent_gb300 import ozk

    torch.cuda.set_device(ranks.local)
    w = workloads.WORKLOADS[args.workload]
    M, N, K, n = w.M, w.N, w.K, args.moduli
    A, B = workloads.workload_operands(w)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), dtype=torch.float64, device="cuda")
    need = ozk.ozk_workspace_size(M, N, K, n)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flops = 2.0 * M * N * K

    def step(ev=None):
        ozk.ozk_dgemm_ws_timed(M, N, K, dA, K, dB, N, dC, N, n, ws, need, ev, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if ozk.ozk_stream_status() != 0:
        raise RuntimeError("device status after warm-up")

    events = [[ozk.Event() for _ in range(5)] for _ in range(args.steps)]
    t_start, t_stop = ozk.Event(), ozk.Event()
    sampler = ClockSampler(ranks.local, args.clock_log)
    sampler.start()
    time.sleep(0.3)
    ranks.barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        step(events[k])
    t_stop.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    clocks = sampler.stop()
    status = ozk.ozk_stream_status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    elapsed_ms = t_start.elapsed_ms(t_stop)
    stage_ms = {s: 0.0 for s in STAGES}
    for ev in events:
        for i, s in enumerate(STAGES):
            stage_ms[s] += ev[i].elapsed_ms(ev[i + 1])
    stage_ms = {s: v / args.steps for s, v in stage_ms.items()}
    my_time = elapsed_ms / 1e3
    times = [my_time]
    if ranks.world > 1:
        slowest = ranks.max(my_time)
        times = [slowest] * ranks.world  # replica_throughput uses world x work / slowest
    value = replica_throughput(flops, args.steps, times)

    # the same calls without the stage events (ozk_dgemm_ws, what a caller
    # runs): the events between stages hold each kernel's launch until the
    # previous one has ended, which the library's dependent launches otherwise
    # overlap; reported beside the timed line, not as its value
    c0, c1 = ozk.Event(), ozk.Event()
    ranks.barrier()
    torch.cuda.synchronize()
    c0.record(stream)
    for _ in range(args.steps):
        ozk.ozk_dgemm_ws(M, N, K, dA, K, dB, N, dC, N, n, ws, need, stream)
    c1.record(stream)
    torch.cuda.synchronize()
    if ozk.ozk_stream_status() != 0:
        raise RuntimeError("device status in the calls without stage events")
    call_ms = ranks.max(c0.elapsed_ms(c1) / args.steps)
    call_only = {"value": ranks.world * flops / (call_ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": call_ms,
                 "mode": "ozk_dgemm_ws back to back on the same inputs, no stage events"}

    # end to end: host (pinned) buffers through the C-ABI, copies in the timed region
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float64).pin_memory()
    e2e_steps = max(3, min(args.steps, 100))
    for _ in range(3):
        ozk.ozk_dgemm_host(M, N, K, hA, K, hB, N, hC, N, n, stream)
    ranks.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ozk.ozk_dgemm_host(M, N, K, hA, K, hB, N, hC, N, n, stream)
    e2e_s = time.perf_counter() - t0
    e2e_s = ranks.max(e2e_s)
    e2e_value = ranks.world * flops * e2e_steps / e2e_s / 1e12
    ok_e2e = bool(np.array_equal(hC.numpy().view(np.uint64), dC.cpu().numpy().view(np.uint64)))
    # the same, calls pipelined: ozk_dgemm_host_async returns once enqueued, so
    # the next call's copies in overlap this call's stages (every call still
    # copies its A and B in and its C out); one synchronisation at the end
    hC.zero_()
    for _ in range(3):
        ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, n, stream)
    stream.synchronize()
    ranks.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ozk.ozk_dgemm_host_async(M, N, K, hA, K, hB, N, hC, N, n, stream)
    stream.synchronize()
    pipe_s = ranks.max(time.perf_counter() - t0)
    pipe_value = ranks.world * flops * e2e_steps / pipe_s / 1e12
    ok_pipe = bool(np.array_equal(hC.numpy().view(np.uint64), dC.cpu().numpy().view(np.uint64)))
    if ozk.ozk_stream_status(stream) != 0:
        raise RuntimeError("device status after the end-to-end runs")

    # the same workload with the sharper (norm) scaling rule at the moduli count
    # it needs for the same contract: at 4096^3 N(0,1), 13 moduli keep
    # eta <= 1e-14 (tests/test_precision_contract.py asserts it)
    norm_rule = None
    if not args.no_norm_rule and ozk.ozk_gamma(K, args.norm_moduli) > 0:
        nn = args.norm_moduli
        need_n = ozk.ozk_workspace_size(M, N, K, nn)
        ws_n = torch.empty(need_n, dtype=torch.uint8, device="cuda")

        def step_norm(ev=None):
            ozk.ozk_dgemm_norm_ws_timed(M, N, K, dA, K, dB, N, dC, N, nn, ws_n, need_n, ev, stream)

        for _ in range(max(args.warmup, 3)):
            step_norm()
        torch.cuda.synchronize()
        ev_n = [[ozk.Event() for _ in range(5)] for _ in range(args.steps)]
        n0, n1 = ozk.Event(), ozk.Event()
        ranks.barrier()
        torch.cuda.synchronize()
        n0.record(stream)
        for k in range(args.steps):
            step_norm(ev_n[k])
        n1.record(stream)
        torch.cuda.synchronize()
        if ozk.ozk_stream_status() != 0:
            raise RuntimeError("device status in the norm-rule run")
        nms = n0.elapsed_ms(n1) / args.steps
        nst = {st: sum(e[i].elapsed_ms(e[i + 1]) for e in ev_n) / args.steps for i, st in enumerate(STAGES)}
        norm_rule = {"n_moduli": nn, "scaling": "norm (2-norm bound per row/column)",
                     "gamma": ozk.ozk_gamma(K, nn), "ms_per_step": nms,
                     "value": ranks.world * flops / (ranks.max(nms / 1e3)) / 1e12, "unit": "TFLOP/s",
                     "stages_ms": nst, "contract": "eta <= 1e-14 asserted by the precision-contract tests"}
        del ws_n

    pk = peaks()
    gemm_s = stage_ms["residue_gemm"] / 1e3
    algo_flops = 2.0 * M * N * K * n  # one M x N x K residue GEMM per modulus
    achieved = algo_flops / gemm_s / 1e12
    # the GEMM is timed launch by launch (about a millisecond each, between
    # memory-bound stages), not over a seconds-long loop: the burst figure
    peak = pk["bf16_tflops"]
    roofline = {
        "bound": "tensor", "kernel": "residue_gemm (tcgen05 kind::f16, fp16-exact residues)",
        "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
        # fp16 operands: the measured bf16 peak times the nominal fp16:bf16 dense ratio of 1
        "peak_source": f"bf16_tflops (burst) x 1 (fp16 dense rate = bf16 dense rate), {pk['source']}",
        "traffic": committed_traffic(f"{w.name}/n{n}"),
        "algorithmic": f"2*M*N*K*n = {algo_flops:.4g} flop per launch",
    }
    hbm = pk["hbm_gbs"]
    # with the fused row kernel A is read once, in the quantize stage, and the
    # scan stage reads B alone
    fused = rows_fused(M, ozk.ozk_kpad(K))
    mem_stages = {
        "scan": 8.0 * (K * N if fused else M * K + K * N),
        "quantize": 8.0 * (M * K + K * N) + 2.0 * n * (M + N) * ozk.ozk_kpad(K),
        "crt_combine": (n + 8.0) * M * N,
    }
    stage_roofline = {s: {"achieved_gbs": b / (stage_ms[s] / 1e3) / 1e9,
                          "frac_of_hbm": b / (stage_ms[s] / 1e3) / 1e9 / hbm} for s, b in mem_stages.items()}

    line = None
    if ranks.rank == 0:
        cpu = cpu_baseline(A, B, n) if (ranks.world == 1 and not args.no_cpu_baseline) else None
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ranks.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config(w, n),
            "tensor_path": "residues in [-128,127] as fp16 on tcgen05 kind::f16 (sm_103a has no kind::i8); "
                           "fp32 TMEM sums exact per 1024-term chunk, reduced mod p on the packed fp32 "
                           "pipe and stored by TMA; CTA-pair tcgen05.mma.cta_group::2 for K >= 2048",
            "fp16_tensor_tflops_issued": 2.0 * M * N * ozk.ozk_kpad(K) * n / gemm_s / 1e12,
            "int8_tensor_peak": "none on sm_103a: ptxas rejects tcgen05.mma kind::i8 for sm_103a, so the "
                                "residue GEMMs run on the fp16 tensor path (same dense rate as bf16)",
            "stages_ms": stage_ms, "stage_hbm_roofline": stage_roofline,
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 8 * (M * K + K * N),
                    "d2h_bytes_per_step": 8 * M * N, "steps": e2e_steps, "matches_device_result": ok_e2e,
                    "mode": "ozk_dgemm_host, one synchronous call per step"},
            "norm_rule": norm_rule,
            "call_only": call_only,
            "e2e_pipelined": {"value": pipe_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 8 * (M * K + K * N),
                              "d2h_bytes_per_step": 8 * M * N, "steps": e2e_steps, "matches_device_result": ok_pipe,
                              "mode": "ozk_dgemm_host_async, calls back to back on one stream, one final sync"},
            "gpu_launches": kernels_per_step(M, ozk.ozk_kpad(K)) * args.steps,
            "clocks": clocks,
            "context": {"pages_rtx4060_laptop_4096_custom_partial_crt_ms": 123.54,
                        "pages_rtx4060_laptop_4096_native_dgemm_ms": 669.75},
        }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ozk", choices=["ozk", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS),
                    help="GEMM shape to time (the headline line uses the default)")
    ap.add_argument("--moduli", type=int, default=N_MODULI)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--norm-moduli", type=int, default=13,
                    help="moduli count of the extra norm-rule measurement")
    ap.add_argument("--no-norm-rule", action="store_true", help="skip the norm-rule measurement")
    ap.add_argument("--clock-log", default=tempfile.gettempdir(),
                    help="folder for the nvidia-smi clock samples taken during the timed region")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    ranks = Ranks(world)
    try:
        if args.impl == "reference":
            line = run_reference(args, ranks)
        else:
            line = run_gpu(args, ranks)
    finally:
        ranks.close()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
