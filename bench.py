"""Benchmark: ragged MXFP8 weight-gradient grouped GEMM on GB300.

One step = one full call of the hot path (plan + scale re-layout kernel and
the main tcgen05 contraction kernel) over one batch of synthetic input that is
already resident in HBM; the L2 is flushed (a 256 MiB write, then a 256 MiB
read) before every timed step, outside the timed interval. Quantisation builds the inputs and is
not timed ("Ragged MXFP8 Weight Gradients", section 7: operator time on
pre-quantised operands).

Metric: TFLOP/s = 2 N K sum_g len_g / time. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 16B] [--impl reference]

--impl reference times the CPU oracle (the plain fp64 definition) on the
host's cores on a bounded sample of the same workload.

Default workload: the 671B down-projection expert shape (E=32, N=7168,
K=2048, M=524288 tokens), the largest of the named workloads in tokens and
bytes that runs on one GPU; the others run with --config.

Besides the mean over the K timed steps (the reported value), the line
carries the spread of those steps and of three passes of at least one second
of back-to-back calls (no L2 flush, no synchronisation between calls), as
median, minimum and maximum.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from moe_ragged_contraction_gb300 import inputs as I  # noqa: E402

DEFAULT_CONFIG = "671Bd"
METRIC = "TFLOP/s (2*N*K*sum(M_g)) ragged MXFP8 wgrad, % of GB300 MXFP8 tensor peak"
FP8_OVER_BF16 = 2.0  # nominal dense ratio: 4.5 PF fp8 / 2.25 PF bf16
L2_FLUSH_BYTES = 256 << 20
MAIN_KERNEL_SRC = os.path.join(ROOT, "moe_ragged_contraction_gb300", "csrc", "wgrad_kernels.cu")


class L2Flush:
    """Evicts the L2 between timed steps (outside the timed interval): a
    256 MiB write (larger than the 129 MB L2), then a 256 MiB read of another
    buffer, which leaves the L2 holding only clean lines of that buffer. The
    timed step then starts with none of its inputs in L2 and without the
    write's dirty lines still draining to HBM underneath it (measured: they
    cost the 16B step about 3 us)."""

    DESCRIPTION = "flushed before every timed step (256 MiB write, then 256 MiB read)"

    def __init__(self, device):
        import torch

        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        # float32: the sum is one reduction kernel that only reads (an integer
        # sum would first widen the buffer into a temporary, i.e. write again)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def kernel_source_hash() -> str:
    """Hash of the sources that define the main kernel, its prep kernels and
    their host-side setup (the quantisers are not part of it)."""
    h = hashlib.sha256()
    d = os.path.dirname(MAIN_KERNEL_SRC)
    for f in ("abi.cu", "mxw_internal.h", "mxw_ptx.cuh", "wgrad_kernels.cu"):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


HBM_FALLBACK_GBS = 6800.0


def mxfp8_peak():
    """Dense MXFP8 peak in TFLOP/s: the measured bf16 burst peak x the nominal
    fp8/bf16 ratio (measured file), else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        return FP8_OVER_BF16 * float(mp["bf16_tflops"]), "measured bf16 burst x2 (nominal fp8/bf16)", mp
    except (OSError, KeyError, ValueError):
        return FP8_OVER_BF16 * 1900.0, "fallback 1.9 PF bf16 x2 (nominal fp8/bf16)", None


def measured_traffic(config: str):
    """DRAM bytes per launch of the main kernel from the committed ncu summary,
    or None if the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    ent = t.get(config)
    if not ent or ent.get("kernel_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), p[5], p[6], p[7], p[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for nm, v in zip(names, r[2:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------ multi-rank aggregation

def max_over_ranks(x: float, dist=None, device=None) -> float:
    """Largest value over all ranks (the job is as slow as its slowest rank)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank: float, world: int, ms_per_step: float) -> float:
    """Replicas only: every rank processes the same workload, so the job does
    world x the work in the slowest rank's time."""
    return world * flop_per_rank / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm

def make_device_inputs(name: str, device):
    """Seeded fp32 operands generated on the GPU, quantised by the library's
    tokenwise quantiser (input building; not timed)."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    w = I.WORKLOADS[name]
    ops = []
    for stream, rows in ((0, w.N), (1, w.K)):
        q = torch.empty((rows, w.M), dtype=torch.uint8, device=device)
        s = torch.empty((rows, w.M // 32), dtype=torch.uint8, device=device)
        step = max(1, (1 << 30) // (4 * w.M))  # <= 1 GiB of fp32 at a time
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            x = I.device_operand(r1 - r0, w.M, w.seed * 7919 + r0, stream, w.dist, device=device)
            mx.quantize_tokenwise(x, q[r0:r1], s[r0:r1])
            del x
        ops += [q, s]
    offs = torch.from_numpy(I.offsets(I.group_sizes(name))).to(device)
    torch.cuda.synchronize()
    return ops[0], ops[1], ops[2], ops[3], offs


# ------------------------------------------------------------------ CPU oracle sample (baseline)

POOL_BLOCKS = 8      # 16-row blocks of A and of B whose rows the oracle sample draws from
POOL_BLOCK_ROWS = 16


def pool_rows(w, seed: int = 0):
    """Rows of A (output rows n) and of B (output columns k) that the CPU
    sample draws its output elements from: POOL_BLOCKS random 16-row blocks of
    each (whole blocks, so that the host-side generator, seeded per 16-row
    block, can produce exactly these rows)."""
    rng = np.random.default_rng(7000 + seed)

    def pick(rows):
        nblk = (rows + POOL_BLOCK_ROWS - 1) // POOL_BLOCK_ROWS
        blks = np.sort(rng.choice(nblk, size=min(POOL_BLOCKS, nblk), replace=False))
        r = (blks[:, None] * POOL_BLOCK_ROWS + np.arange(POOL_BLOCK_ROWS)[None, :]).ravel()
        return r[r < rows]

    return pick(w.N), pick(w.K)


def oracle_sample_rate(Ap, sAp, Bp, sBp, offs, w, target_s: float, threads: int, seed: int = 0):
    """Time the oracle on a bounded sample of the workload's output: for every
    non-empty expert, a number of output rows n drawn at random from the
    pooled rows Ap = A[pool_n], each with every pooled column k of
    Bp = B[pool_k], in the order the oracle walks the full output (expert,
    then row, then column); as many rows as fit about target_s seconds.
    Returns (TFLOP/s, seconds, description)."""
    import oracle

    offs = np.asarray(offs)
    sizes = np.diff(np.concatenate([[0], offs]))
    live = np.nonzero(sizes > 0)[0]
    rng = np.random.default_rng(seed)
    pn, pk = Ap.shape[0], Bp.shape[0]

    def run(rows):
        gs, ns = [], []
        for g in live:
            for n in np.sort(rng.integers(0, pn, rows)):
                gs.append(np.full(pk, g)); ns.append(np.full(pk, n))
        g = np.concatenate(gs).astype(np.int32)
        n = np.concatenate(ns).astype(np.int32)
        k = np.tile(np.arange(pk, dtype=np.int32), rows * len(live))
        flop = 2.0 * float(np.sum(sizes[g]))
        t0 = time.perf_counter()
        oracle.wgrad_points(Ap, sAp, Bp, sBp, offs, w.E, pn, pk, w.M, g, n, k, nthreads=threads)
        return flop, time.perf_counter() - t0

    rows = 2
    flop, dt = run(rows)  # calibration
    rows = int(max(1, round(rows * target_s / max(dt, 1e-6))))
    flop, dt = run(rows)
    desc = (f"{rows} output rows x {pk} columns of each of the {len(live)} non-empty experts "
            f"(rows drawn from {pn} rows of A, columns the {pk} rows of B of {POOL_BLOCKS} random "
            f"16-row blocks of each), {flop / 2:.3g} MACs, rate extrapolated to the whole workload")
    return flop / dt / 1e12, dt, desc


def bench_config(name: str, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    w = I.WORKLOADS[name]
    return {"workload": name, "E": w.E, "N": w.N, "K": w.K, "M": w.M, "routing": w.description,
            "l2": L2Flush.DESCRIPTION, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def spread(values) -> dict:
    v = np.asarray(values, dtype=np.float64)
    return {"median": float(np.median(v)), "min": float(v.min()), "max": float(v.max()), "n": int(v.size)}


def hold_gpu(steps: int) -> None:
    """Keep the current stream busy for about 0.2 ms per step that follows
    (a spin kernel), long enough for the host to enqueue them."""
    import torch

    torch.cuda._sleep(int(4e5 * steps))


def bench_gpu(args):
    import torch

    import moe_ragged_contraction_gb300 as mx

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    mx.build()
    mx.load()

    w = I.WORKLOADS[args.config]
    A, sA, B, sB, offs = make_device_inputs(args.config, device)
    out = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=device)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)

    def step(main_pair=None):
        if main_pair is not None:
            mx.set_timing_events(*main_pair)
        mx.wgrad_grouped(A, sA, B, sB, offs, out=out)

    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_id = str(torch.cuda.current_device())
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    # warm-up: W steps, then ~0.5 s of back-to-back calls so clocks settle
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + (0.0 if args.quick else 0.5)
    while time.perf_counter() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize()

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    evm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in evm:  # torch creates the CUDA event on first record; the library needs real handles
        a.record(stream)
        b.record(stream)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # the timed steps run the plain product call (its main kernel is launched
    # as a programmatic dependent of the prep kernel and overlaps its tail).
    # A device-side sleep first keeps the GPU busy while the host enqueues all
    # K steps, so each step's events bracket device time only, not the host's
    # per-call enqueue latency (the end-to-end figure below includes that).
    hold_gpu(K)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(np.sum(step_ms)), dist, device)
    # the main kernel's own duration: the same steps again with events recorded
    # right before and after its launch (which serialises it behind the prep
    # kernel, so this is its full launch-to-end time)
    hold_gpu(K)
    for i in range(K):
        flush()
        step(main_pair=evm[i])
    torch.cuda.synchronize()
    main_ms = [a.elapsed_time(b) for a, b in evm]
    # spread: three passes of at least one second of back-to-back calls each
    # (no L2 flush, no synchronisation between calls), bracketed by events
    calls = int(max(10, np.ceil(1.0 / max(1e-6, float(np.mean(step_ms)) * 1e-3))))
    b2b = []
    for _ in range(0 if args.quick else 3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_gpu(min(calls, 200))
        e0.record(stream)
        for _ in range(calls):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        b2b.append(float(w.flop) / (e0.elapsed_time(e1) / calls * 1e-3) / 1e12)
    assert mx.device_status(clear=True) == 0, "device flagged an error during the benchmark"

    e2e = None
    if not args.quick and not args.no_e2e:
        # end to end through the public API with host buffers: every step copies its
        # inputs host -> device (pinned host memory) and its result device -> host
        # inside the timed interval. Consecutive steps overlap like a streaming
        # pipeline: the copy-in of step i+1, the call of step i and the copy-out of
        # step i-1 run on three streams over two device buffer sets, ordered by
        # events (a set's inputs are overwritten only after its call finished, its
        # output only after it was copied out).
        hA, hsA, hB, hsB, hoffs = (t.cpu().pin_memory() for t in (A, sA, B, sB, offs))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hA, hsA, hB, hsB, hoffs))
        d2h = hout.numel() * hout.element_size()
        sets = [tuple(torch.empty_like(t) for t in (A, sA, B, sB, offs, out)) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in range(2)]    # the set's inputs have landed
        ev_used = [torch.cuda.Event() for _ in range(2)]  # the set's call has finished
        ev_out = [torch.cuda.Event() for _ in range(2)]   # the set's output has been copied out

        def e2e_step(i):
            b = i % 2
            dA, dsA, dB, dsB, doffs, dout = sets[b]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_used[b])
                for d, h in ((dA, hA), (dsA, hsA), (dB, hB), (dsB, hsB), (doffs, hoffs)):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])
            mx.wgrad_grouped(dA, dsA, dB, dsB, doffs, out=dout, stream=stream)
            ev_used[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_used[b])
                hout.copy_(dout, non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(max(3, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i in range(K):
            e2e_step(i)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / K
        e2e = {"value": float(w.flop) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelining": "copy-in, call and copy-out of consecutive steps overlap (three streams, "
                             "two device buffer sets)"}
    clocks = sampler.stop()

    flop = float(w.flop)
    ms_per_step = total_ms / K
    value = whole_job_tflops(flop, world, ms_per_step)
    peak, peak_src, peaks = mxfp8_peak()
    main_avg = float(np.mean(main_ms))
    achieved = flop / (main_avg * 1e-3) / 1e12
    traffic = measured_traffic(args.config)
    # the bound of the dominant kernel: the tensor cores, unless the
    # workload's FLOP per algorithmic byte (operands, scales, output) is below
    # the ridge of the measured peaks (many experts with few tokens each are
    # bound by writing their output)
    alg_bytes = float(w.N + w.K) * w.M * (1 + 1 / 32) + 2.0 * w.E * w.N * w.K + 4.0 * w.E
    hbm_peak = float(peaks["hbm_gbs"]) if peaks else HBM_FALLBACK_GBS
    if flop / alg_bytes < peak * 1e12 / (hbm_peak * 1e9):
        roof = {"bound": "hbm", "achieved": alg_bytes / (main_avg * 1e-3) / 1e9, "peak": hbm_peak,
                "unit": "GB/s", "frac": alg_bytes / (main_avg * 1e-3) / 1e9 / hbm_peak,
                "algorithmic_bytes_per_launch": alg_bytes,
                "peak_source": "measured copy bandwidth" if peaks else "fallback 6.8 TB/s"}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": peak_src, "algorithmic_flop_per_launch": flop}
        if peaks and "bf16_tflops_sustained" in peaks:
            # context: the timed steps follow 0.5 s of back-to-back calls, so the
            # large shapes run at the clock the 1.4 kW cap allows; the measured
            # sustained bf16 figure (4 s back to back) x 2 is that regime's peak
            ps = FP8_OVER_BF16 * float(peaks["bf16_tflops_sustained"])
            roof.update({"peak_sustained": ps, "frac_sustained": achieved / ps})
    roof.update({"traffic": traffic, "kernel": "wgrad_main", "avg_launch_ms": main_avg})

    result = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and not args.quick and world == 1:
            threads = len(os.sched_getaffinity(0))
            rn, rk = pool_rows(w)
            rn_t, rk_t = torch.from_numpy(rn).to(device), torch.from_numpy(rk).to(device)
            Ap, sAp, Bp, sBp = (t.index_select(0, r).cpu().numpy()
                                for t, r in ((A, rn_t), (sA, rn_t), (B, rk_t), (sB, rk_t)))
            rate, secs, desc = oracle_sample_rate(Ap, sAp, Bp, sBp, offs.cpu().numpy(), w, args.cpu_seconds, threads)
            cpu = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"{desc}; {secs:.1f} s on the host (fp64 plain loops)"}
        result = {
            "metric": METRIC,
            "value": value,
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "mxfp8_e4m3 (e8m0 block-32 scales), fp32 accumulate, bf16 out",
            "data": "synthetic (seeded routing and N(0,1)/Student-t operands, quantised on the GPU)",
            "config": bench_config(args.config, world),
            "pct_of_mxfp8_peak": 100.0 * value / world / peak,
            "spread": {"unit": "TFLOP/s",
                       "timed_steps": spread([flop / (t * 1e-3) / 1e12 for t in step_ms]),
                       "back_to_back": dict(spread(b2b), calls_per_pass=calls,
                                            how="3 passes of >= 1 s of back-to-back calls, no L2 flush")
                       if b2b else None},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": 2 * K,
            "clocks": clocks,
        }
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------------ vendor comparators

def bench_comparators(args):
    """Opt-in context line: the same grouped wgrad in BF16 through the vendor
    library (one cuBLAS GEMM per expert on its token slice; the pages compare
    against a BF16 grouped GEMM, "Ragged MXFP8 Weight Gradients" section 7),
    and a dense 8192^3 MXFP8 GEMM through this library (one expert) and
    through cuBLASLt (torch._scaled_mm with e8m0 block scales; its scales are
    not in the vendor's swizzled layout, so only its timing is meaningful).
    Each is timed two ways in the same process: "burst" (steps after three
    warm-ups, L2 flushed before each) and "sustained" (three passes of at
    least one second of back-to-back calls each, the regime in which the
    1.4 kW power cap sets the clock; median, minimum, maximum)."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    device = torch.device("cuda")
    mx.build()
    mx.load()
    w = I.WORKLOADS[args.config]
    flush = L2Flush(device)

    def timed(fn, steps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        return tot / steps

    def sustained(fn, flop_per_call, seconds=1.0, passes=3):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            fn()
        b.record()
        torch.cuda.synchronize()
        calls = int(max(5, np.ceil(seconds / max(1e-6, a.elapsed_time(b) / 3 * 1e-3))))
        vals = []
        for _ in range(passes):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(calls):
                fn()
            b.record()
            torch.cuda.synchronize()
            vals.append(flop_per_call / (a.elapsed_time(b) / calls * 1e-3) / 1e12)
        return dict(spread(vals), calls_per_pass=calls)

    sampler = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(device).uuid))
    sampler.start()
    res = {"comparators": True, "config": {"workload": args.config}, "unit": "TFLOP/s", "sustained": {}}
    A, sA, B, sB, offs = make_device_inputs(args.config, device)
    out = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=device)
    ours = lambda: mx.wgrad_grouped(A, sA, B, sB, offs, out=out)  # noqa: E731
    ms = timed(ours, args.steps)
    res["mxfp8_wgrad_this_library"] = w.flop / (ms * 1e-3) / 1e12
    res["sustained"]["mxfp8_wgrad_this_library"] = sustained(ours, w.flop)
    # BF16 vendor baseline: one cuBLAS bf16 GEMM per expert on the token slice
    # (torch._grouped_mm is not used: it raised a GPU fault in one run on
    # this hardware)
    a16 = torch.randn(w.N, w.M, device=device, dtype=torch.bfloat16)
    b16 = torch.randn(w.K, w.M, device=device, dtype=torch.bfloat16)
    ends = I.offsets(I.group_sizes(args.config)).tolist()
    out16 = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=device)

    def bf16_loop():
        lo = 0
        for g, hi in enumerate(ends):
            if hi > lo:
                torch.matmul(a16[:, lo:hi], b16[:, lo:hi].t(), out=out16[g])
            else:
                out16[g].zero_()
            lo = hi

    ms = timed(bf16_loop, args.steps)
    res["bf16_per_expert_cublas"] = w.flop / (ms * 1e-3) / 1e12
    res["sustained"]["bf16_per_expert_cublas"] = sustained(bf16_loop, w.flop)
    res["mxfp8_over_bf16"] = res["mxfp8_wgrad_this_library"] / res["bf16_per_expert_cublas"]
    res["mxfp8_over_bf16_sustained"] = (res["sustained"]["mxfp8_wgrad_this_library"]["median"]
                                        / res["sustained"]["bf16_per_expert_cublas"]["median"])
    del a16, b16, out16
    n = 8192
    g = torch.Generator(device=device)
    g.manual_seed(0)
    qa, qsa = mx.quantize_tokenwise(torch.randn(n, n, device=device, generator=g))
    qb, qsb = mx.quantize_tokenwise(torch.randn(n, n, device=device, generator=g))
    one = torch.tensor([n], dtype=torch.int32, device=device)
    dout = torch.empty((1, n, n), dtype=torch.bfloat16, device=device)
    dense_ours = lambda: mx.wgrad_grouped(qa, qsa, qb, qsb, one, out=dout)  # noqa: E731
    ms = timed(dense_ours, args.steps)
    res["dense8192_mxfp8_this_library"] = 2 * n ** 3 / (ms * 1e-3) / 1e12
    res["sustained"]["dense8192_mxfp8_this_library"] = sustained(dense_ours, 2.0 * n ** 3)
    try:
        a8, b8 = qa.view(torch.float8_e4m3fn), qb.view(torch.float8_e4m3fn).t()
        s_a, s_b = qsa.view(torch.float8_e8m0fnu), qsb.view(torch.float8_e8m0fnu)
        vendor = lambda: torch._scaled_mm(a8, b8, scale_a=s_a, scale_b=s_b, out_dtype=torch.bfloat16)  # noqa: E731
        ms = timed(vendor, args.steps)
        res["dense8192_mxfp8_vendor"] = 2 * n ** 3 / (ms * 1e-3) / 1e12
        res["sustained"]["dense8192_mxfp8_vendor"] = sustained(vendor, 2.0 * n ** 3)
    except Exception as e:
        res["dense8192_mxfp8_vendor"] = None
        res["dense8192_vendor_error"] = str(e).splitlines()[0][:200]
    res["clocks"] = sampler.stop()
    res["gpu_launches_note"] = "context line, not a bench line"
    return res


# ------------------------------------------------------------------ fused quantiser

def bench_quantizer(args):
    """Opt-in line: the fused bf16 quantise-and-transpose that builds this
    workload's operands (dY [M, N] and X [M, K], token-major bf16, to
    A [N, M] and B [K, M] E4M3 plus scales), HBM-bound: GB/s over the
    algorithmic bytes (2 read + 1 + 1/32 written per element)."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    mx.build()
    mx.load()
    w = I.WORKLOADS[args.config]
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    dy = torch.randn(w.M, w.N, device=device, generator=g).to(torch.bfloat16)
    x = torch.randn(w.M, w.K, device=device, generator=g).to(torch.bfloat16)
    qa = torch.empty((w.N, w.M), dtype=torch.uint8, device=device)
    sa = torch.empty((w.N, w.M // 32), dtype=torch.uint8, device=device)
    qb = torch.empty((w.K, w.M), dtype=torch.uint8, device=device)
    sb = torch.empty((w.K, w.M // 32), dtype=torch.uint8, device=device)
    flush = L2Flush(device)

    def step():
        mx.quantize_transpose_bf16(dy, qa, sa)
        mx.quantize_transpose_bf16(x, qb, sb)

    sampler = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(device).uuid))
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    hold_gpu(K)
    for i in range(K):
        flush()
        ev[i][0].record()
        step()
        ev[i][1].record()
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    clocks = sampler.stop()
    elems = float(w.M) * (w.N + w.K)
    alg = elems * (2 + 1 + 1 / 32)
    _, _, peaks = mxfp8_peak()
    hbm = float(peaks["hbm_gbs"]) if peaks else HBM_FALLBACK_GBS
    gbs = alg / (ms * 1e-3) / 1e9
    return {"metric": "GB/s fused bf16 quantise-and-transpose (operands of the wgrad)", "value": gbs,
            "unit": "GB/s", "ms_per_step": ms, "steps": K, "warmup": args.warmup,
            "config": {"workload": args.config, "M": w.M, "N": w.N, "K": w.K,
                       "l2": L2Flush.DESCRIPTION},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                         "algorithmic_bytes_per_step": alg, "kernel": "quantize_transpose_bf16_kernel"},
            "gpu_launches": 2 * K, "clocks": clocks}


# ------------------------------------------------------------------ scale-factor blocks from the quantiser

def bench_sf(args):
    """Opt-in line: the operands quantised from token-major bf16 by the fused
    quantiser that writes the scales straight into the tensor core's block
    layout, then the weight gradient over those blocks (no scale re-layout
    inside the timed call). Same metric, workload, flush and step protocol as
    the default line; the quantiser is timed separately (GB/s)."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    mx.build()
    mx.load()
    w = I.WORKLOADS[args.config]
    cfg = mx.tile_config(w.E, w.N, w.K, w.M)
    kn, tn = cfg["kn"], cfg["tn"]
    rows_a, rows_b = (tn, 256) if kn else (256, tn)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    dy = torch.randn(w.M, w.N, device=device, generator=g).to(torch.bfloat16)
    x = torch.randn(w.M, w.K, device=device, generator=g).to(torch.bfloat16)
    A = torch.empty((w.N, w.M), dtype=torch.uint8, device=device)
    B = torch.empty((w.K, w.M), dtype=torch.uint8, device=device)
    sfA = torch.empty((mx.sf_blocks_bytes(w.N, w.M, rows_a),), dtype=torch.uint8, device=device)
    sfB = torch.empty((mx.sf_blocks_bytes(w.K, w.M, rows_b),), dtype=torch.uint8, device=device)
    offs = torch.from_numpy(I.offsets(I.group_sizes(args.config))).to(device)
    out = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device=device)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)

    def quant():
        mx.quantize_transpose_bf16_sf(dy, rows_a, q=A, sf=sfA)
        mx.quantize_transpose_bf16_sf(x, rows_b, q=B, sf=sfB)

    def step(pair=None):
        if pair is not None:
            mx.set_timing_events(*pair)
        mx.wgrad_grouped_sf(A, sfA, B, sfB, offs, kn, tn, out=out)

    sampler = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(device).uuid))
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush()
        quant()
    torch.cuda.synchronize()
    K = args.steps
    evq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    hold_gpu(K)
    for i in range(K):
        flush()
        evq[i][0].record(stream)
        quant()
        evq[i][1].record(stream)
    torch.cuda.synchronize()
    q_ms = float(np.mean([a.elapsed_time(b) for a, b in evq]))
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + 0.5
    while time.perf_counter() < t_end:
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    evm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in evm:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    hold_gpu(K)
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    hold_gpu(K)
    for i in range(K):
        flush()
        step(pair=evm[i])
    torch.cuda.synchronize()
    main_ms = float(np.mean([a.elapsed_time(b) for a, b in evm]))
    calls = int(max(10, np.ceil(1.0 / max(1e-6, float(np.mean(step_ms)) * 1e-3))))
    b2b = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_gpu(min(calls, 200))
        e0.record(stream)
        for _ in range(calls):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        b2b.append(float(w.flop) / (e0.elapsed_time(e1) / calls * 1e-3) / 1e12)
    clocks = sampler.stop()
    assert mx.device_status(clear=True) == 0, "device flagged an error during the benchmark"
    flop = float(w.flop)
    peak, peak_src, peaks = mxfp8_peak()
    ms = float(np.mean(step_ms))
    elems = float(w.M) * (w.N + w.K)
    q_bytes = elems * (2 + 1) + float(sfA.numel() + sfB.numel())
    hbm = float(peaks["hbm_gbs"]) if peaks else HBM_FALLBACK_GBS
    return {"metric": METRIC + ", scales laid out by the quantiser", "value": flop / (ms * 1e-3) / 1e12,
            "unit": "TFLOP/s", "ms_per_step": ms, "steps": K, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "mxfp8_e4m3 (e8m0 block-32 scales), fp32 accumulate, bf16 out",
            "data": "synthetic (seeded routing, N(0,1) bf16 operands quantised on the GPU)",
            "config": dict(bench_config(args.config, 1), tiling={"kn": kn, "tn": tn}),
            "spread": {"unit": "TFLOP/s", "timed_steps": spread([flop / (t * 1e-3) / 1e12 for t in step_ms]),
                       "back_to_back": dict(spread(b2b), calls_per_pass=calls)},
            "roofline": {"bound": "tensor", "achieved": flop / (main_ms * 1e-3) / 1e12, "peak": peak,
                         "unit": "TFLOP/s", "frac": flop / (main_ms * 1e-3) / 1e12 / peak, "peak_source": peak_src,
                         "kernel": "wgrad_main (grid K-steps, caller's scale blocks)", "avg_launch_ms": main_ms},
            "quantizer": {"ms_per_step": q_ms, "unit": "GB/s", "value": q_bytes / (q_ms * 1e-3) / 1e9,
                          "frac_of_hbm": q_bytes / (q_ms * 1e-3) / 1e9 / hbm,
                          "what": "both operands, bf16 [M, R] -> E4M3 [R, M] + scale blocks, L2 flushed"},
            "gpu_launches": 2 * K, "clocks": clocks}


# ------------------------------------------------------------------ grouped GEMM (forward / data gradient)

def _rowwise_mxfp8(rows: int, cols: int, seed: int, stream: int, dist: str, device):
    """Seeded fp32 [rows, cols] generated and quantised on the GPU in row
    chunks, 32-element blocks along the last axis (input building; not timed)."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=device)
    step = max(1, (1 << 30) // (4 * cols))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = I.device_operand(r1 - r0, cols, seed * 7919 + r0, stream, dist, device=device)
        mx.quantize_tokenwise(x, q[r0:r1], s[r0:r1])
        del x
    return q, s


def bench_gemm(args):
    """Opt-in line: the same expert layer's other two products, as grouped
    GEMMs with ragged rows on the workload's routing: forward Y = X W[g]^T
    (X [M, K], W [E, N, K], contracting K) and data gradient dX = dY W[g]
    (dY [M, N], W stored [E, K, N], contracting N). One step = both calls."""
    import torch

    import moe_ragged_contraction_gb300 as mx

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    mx.build()
    mx.load()
    w = I.WORKLOADS[args.config]
    E, N, K, M = w.E, w.N, w.K, w.M
    X, sX = _rowwise_mxfp8(M, K, w.seed, 20, w.dist, device)
    dY, sdY = _rowwise_mxfp8(M, N, w.seed, 21, w.dist, device)
    W, sW = _rowwise_mxfp8(E * N, K, w.seed, 22, "normal", device)
    Wt, sWt = _rowwise_mxfp8(E * K, N, w.seed, 23, "normal", device)
    W, sW = W.view(E, N, K), sW.view(E, N, K // 32)
    Wt, sWt = Wt.view(E, K, N), sWt.view(E, K, N // 32)
    offs = torch.from_numpy(I.offsets(I.group_sizes(args.config))).to(device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=device)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)

    def step(pairs=None):
        if pairs is not None:
            mx.set_timing_events(*pairs[0])
        mx.grouped_gemm(X, sX, W, sW, offs, out=y)
        if pairs is not None:
            mx.set_timing_events(*pairs[1])
        mx.grouped_gemm(dY, sdY, Wt, sWt, offs, out=dx)

    sampler = ClockSampler("GPU-" + str(torch.cuda.get_device_properties(device).uuid))
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    S = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(S)]
    evm = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2)]
           for _ in range(S)]
    for pr in evm:
        for a, b in pr:
            a.record(stream)
            b.record(stream)
    torch.cuda.synchronize()
    hold_gpu(2 * S)
    for i in range(S):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    hold_gpu(2 * S)
    for i in range(S):
        flush()
        step(pairs=evm[i])
    torch.cuda.synchronize()
    fwd_ms = float(np.mean([p[0][0].elapsed_time(p[0][1]) for p in evm]))
    dgr_ms = float(np.mean([p[1][0].elapsed_time(p[1][1]) for p in evm]))
    clocks = sampler.stop()
    assert mx.device_status(clear=True) == 0, "device flagged an error during the benchmark"
    routed = int(offs[-1].item()) if E else 0
    flop_call = 2.0 * routed * N * K
    peak, peak_src, _ = mxfp8_peak()
    achieved = 2 * flop_call / ((fwd_ms + dgr_ms) * 1e-3) / 1e12
    value = 2 * flop_call / (ms * 1e-3) / 1e12
    return {"metric": "TFLOP/s (2*N*K*sum(M_g) per call) MXFP8 grouped GEMM with ragged rows, forward + data gradient",
            "value": value, "unit": "TFLOP/s", "ms_per_step": ms, "steps": S, "warmup": args.warmup,
            "higher_is_better": True,
            "dtype": "mxfp8_e4m3 (e8m0 block-32 scales), fp32 accumulate, bf16 out",
            "data": "synthetic (seeded routing, operands quantised on the GPU)",
            "config": {"workload": args.config, "E": E, "N": N, "K": K, "M": M, "routing": w.description,
                       "forward": f"[{M},{K}] x [{E},{N},{K}]^T -> [{M},{N}]",
                       "dgrad": f"[{M},{N}] x [{E},{K},{N}]^T -> [{M},{K}]",
                       "l2": L2Flush.DESCRIPTION},
            "pct_of_mxfp8_peak": 100.0 * value / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": peak_src, "kernel": "wgrad_main (row-tile mode)",
                         "algorithmic_flop_per_launch": flop_call, "traffic": measured_traffic("gemm:" + args.config),
                         "forward_main_ms": fwd_ms, "dgrad_main_ms": dgr_ms,
                         "forward_tflops": flop_call / (fwd_ms * 1e-3) / 1e12,
                         "dgrad_tflops": flop_call / (dgr_ms * 1e-3) / 1e12},
            "gpu_launches": 4 * S,
            "clocks": clocks}


# ------------------------------------------------------------------ reference arm (CPU oracle)

def _host_pool(name: str):
    """Host operands for the reference arm, only the pooled rows the oracle
    sample draws from (pool_rows): seeded fp32 rows quantised by the oracle's
    CPU quantiser (no GPU involved)."""
    import oracle

    w = I.WORKLOADS[name]
    rn, rk = pool_rows(w)
    out = []
    for stream, rows in ((0, rn), (1, rk)):
        q = np.empty((rows.size, w.M), np.uint8)
        s = np.empty((rows.size, w.M // 32), np.uint8)
        for i in range(0, rows.size, POOL_BLOCK_ROWS):
            r0 = int(rows[i])
            nr = min(POOL_BLOCK_ROWS, rows.size - i)
            x = I.host_operand(nr, w.M, w.seed, stream, w.dist, row0=r0)
            q[i:i + nr], s[i:i + nr] = oracle.quantize_tokenwise(x)
        out += [q, s]
    return out[0], out[1], out[2], out[3], I.offsets(I.group_sizes(name))


def bench_reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = I.WORKLOADS[args.config]
    Ap, sAp, Bp, sBp, offs = _host_pool(args.config)
    threads = len(os.sched_getaffinity(0))
    per_step = max(0.5, args.ref_step_seconds)
    for i in range(args.warmup):
        oracle_sample_rate(Ap, sAp, Bp, sBp, offs, w, per_step / 4, threads, seed=i)
    rates, secs, desc = [], 0.0, ""
    for i in range(args.steps):
        r, dt, desc = oracle_sample_rate(Ap, sAp, Bp, sBp, offs, w, per_step, threads, seed=1000 + i)
        rates.append(r)
        secs += dt
    value = float(np.mean(rates))
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (exact E4M3/E8M0 decode, fp64 accumulate, bf16 out)",
        "data": "synthetic (seeded routing and N(0,1)/Student-t operands, quantised on the host)",
        "config": bench_config(args.config, world),
        "spread": {"unit": "TFLOP/s", "timed_steps": spread(rates)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"each step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=list(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--comparators", action="store_true",
                    help="print a context line with vendor BF16 grouped / dense MXFP8 GEMM timings instead")
    ap.add_argument("--quantizer", action="store_true",
                    help="print a line for the fused bf16 quantise-and-transpose of the workload's operands instead")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload's expert shapes and routing recipe with this many tokens instead "
                         "(profiler captures on a small case)")
    ap.add_argument("--experts", type=int, default=0,
                    help="run the workload's expert shapes with this many experts, each with the workload's mean "
                         "token run (balanced routing; profiler captures on a small case)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) leg")
    ap.add_argument("--quick", action="store_true",
                    help="warm-up and timed steps only: no settle loop, spread passes, end-to-end leg or CPU "
                         "baseline (profiler runs)")
    ap.add_argument("--sf", action="store_true",
                    help="print a line for the weight gradient over scale blocks written by the quantiser instead")
    ap.add_argument("--gemm", action="store_true",
                    help="print a line for the layer's forward and data-gradient grouped GEMMs (ragged rows) instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.tokens:
        args.config = I.with_tokens(args.config, args.tokens)
    if args.experts:
        args.config = I.with_experts(args.config, args.experts)
    if args.comparators:
        res = bench_comparators(args)
    elif args.quantizer:
        res = bench_quantizer(args)
    elif args.gemm:
        res = bench_gemm(args)
    elif args.sf:
        res = bench_sf(args)
    else:
        res = bench_reference_arm(args) if args.impl == "reference" else bench_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
