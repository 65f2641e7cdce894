"""Benchmark of the Q4_0 prefill GEMM (+ residual) on GB300.

One step = one pass of the hot path over one batch: ``apr_qgemm`` on the
Q4_0 4096 x 4096 weight with T = 512 token rows and a residual, i.e. the
fp32 -> fp16 activation pass, then the tcgen05 GEMM whose warps stream the raw
blocks, decode them in registers, run the MMA and add the residual in the
epilogue. Inputs are seeded synthetic data (numpy PCG64, seed 0; W ~ N(0,0.02)
quantized to Q4_0, X and R ~ N(0,1)), resident in HBM. Eight input sets
(W, X, R, Y: 277 MB, more than twice the 129 MB L2) rotate between steps.

Printed (one JSON line, rank 0): the step throughput in TFLOP/s (2 T n k per
step), the roofline of the dominant kernel (the GEMM, timed alone with CUDA
events through ``apr_qgemm_f16_in``), the end-to-end throughput through the
same public call with host buffers (pinned X and R copied in, Y copied out,
every step), the CPU oracle's throughput on the host cores, and the SM clocks
sampled during the timed region. Beside them, for the rest of the path: the
T = 1 GEMV (GB/s), the FFN sublayer, the GEMM at 2048 rows, and the causal
prefill attention of the 9B layer at 512 and 2048 rows (TFLOP/s).

``--impl reference`` times the CPU oracle (there is no other implementation
of this path to run) on the same workload, a bounded sample of W rows per
step.

Multi-GPU: under torchrun every rank runs its own replica (the projections
shard over independent problems; no collective is on the data path); the
timed region is bracketed by barriers, the slowest rank's time is used and
``value`` counts the work of all ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# the CPU oracle uses every host core this process may run on
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import numpy as np  # noqa: E402

METRIC = "Q4_0/Q8_0 prefill GEMM TFLOP/s at T=512 (% tensor peak); GEMV GB/s (% HBM)"
REPEATS = 5  # timed regions of --steps steps; the headline is their median
WORKLOAD = "q4_0_gemm_residual_n4096_k4096_t512"
QTYPE, N, K, T = 2, 4096, 4096, 512
SETS = 8
FLOP = 2.0 * T * N * K


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["hbm_gbs"], "measured"
    return 1900.0, 6800.0, "fallback"


# ------------------------------------------------------------------ ranks
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_over_ranks(elapsed_s: float, units: float, world: int):
    """(max elapsed over ranks, sum of units over ranks); needs an initialised
    process group when world > 1."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ clocks
CLOCKS_DIR = tempfile.gettempdir()


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to --clocks-dir (default: the system's temporary
        # directory); the JSON line carries their summary
        self.path = os.path.join(CLOCKS_DIR, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "25"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
            self.t0 = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.window_s = time.time() - self.t0 if self.proc else None
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]) if parts[3] not in ("", "[N/A]") else 0.0,
                             parts[4], parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in loaded])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded), "window_s": round(self.window_s, 3)}


# ------------------------------------------------------------------ CPU oracle
_CASE = {}


def bench_case():
    """The seeded inputs of the benchmarked workload (made once per process)."""
    if "c" not in _CASE:
        import synth

        _CASE["c"] = synth.make_case(QTYPE, N, K, T, residual=True, seed=0)
    return _CASE["c"]


def oracle_sample(rows: int):
    """Times the oracle on the first `rows` weight rows with all T tokens."""
    import oracle
    import synth

    case = bench_case()
    bb = synth.block_bytes(QTYPE)
    Wr = case["W"][:rows]
    Rr = np.ascontiguousarray(case["R"][:, :rows])
    t0 = time.perf_counter()
    oracle.qgemm(QTYPE, Wr, rows, K, case["X"], Rr)
    dt = time.perf_counter() - t0
    return dt, 2.0 * T * rows * K, bb


def cpu_baseline(budget_s: float = 10.0):
    rows = 256
    dt, flop, _ = oracle_sample(rows)
    # grow the sample to about `budget_s` of CPU work (bounded by the full weight)
    rows = int(min(N, max(rows, rows * budget_s / max(dt, 1e-3))))
    dt, flop, _ = oracle_sample(rows)
    return {"value": flop / dt / 1e12, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"float64 oracle (numpy/OpenBLAS) on {rows} of the {N} weight rows, all {T} tokens, k={K}, "
                      f"with residual: {dt:.2f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    # each step: the oracle on a bounded sample of rows, sized so that the
    # whole run stays within about two minutes
    total = args.steps + args.warmup
    probe_dt, _, _ = oracle_sample(64)
    per_row = probe_dt / 64
    rows = int(max(8, min(N, (100.0 / max(total, 1)) / max(per_row, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(rows)
    t = 0.0
    flop = 0.0
    for _ in range(args.steps):
        dt, f, _ = oracle_sample(rows)
        t += dt
        flop += f
    value = flop / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "qtype": "Q4_0", "n": N, "k": K, "T": T, "residual": True},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
                         "sample": f"{rows} of the {N} weight rows per step, all {T} tokens"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def kernel_hash() -> str:
    """sha256 (16 hex) of the GEMM kernel's sources (the file and the headers
    its device code includes), to tie ncu counters to a kernel version."""
    import hashlib

    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "dev_common.cuh", "apr_internal.h", "iq4.cuh", "q4k.cuh"):
        with open(os.path.join(ROOT, "quantized_weight_prefill_q4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_label(n, T, sms):
    """The tile plan the library picks for this shape (the rule documented with
    plan_gemm_tc: 256-token tiles when they keep most SMs busy (192-token ones
    when those need no more waves), else split over k in two when the tiles
    fit one wave twice, else 128-token tiles)."""
    rt = (n + 127) // 128
    tiles256, tiles192 = rt * ((T + 255) // 256), rt * ((T + 191) // 192)
    if 10 * tiles256 >= 6 * sms:
        w256, w192 = -(-tiles256 // sms), -(-tiles192 // sms)
        plan = "192-token tiles" if T > 128 and w192 <= w256 else "256-token tiles"
    elif 2 * tiles256 <= sms:
        plan = "256-token tiles split over k by 2-CTA clusters"
    else:
        plan = "128-token tiles"
    return f"gemm_tc_kernel<Q4_0, residual>, {plan}"


def measured_traffic():
    """DRAM bytes per launch from the committed ncu summary, or None once the
    kernel has changed since the counters were taken."""
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tp):
        return None
    with open(tp) as f:
        rec = json.load(f).get(WORKLOAD)
    if not rec or rec.get("kernel_hash") != kernel_hash():
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------------ GPU arm
def capture_graph(calls):
    """One CUDA graph replaying `calls` (each enqueues its work on the current
    stream) back to back: the timed loops replay graphs so that the Python
    binding's per-call host time does not starve the GPU."""
    import torch

    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        for c in calls:
            c()
    torch.cuda.current_stream().wait_stream(side)
    return g


def timed_calls(calls, count, stream):
    """Seconds for `count` calls cycling through `calls`, replayed from graphs,
    measured with CUDA events on `stream` (the caller synchronises around it)."""
    import torch

    full, rest = divmod(count, len(calls))
    g = capture_graph(calls)
    g_rest = capture_graph(calls[:rest]) if rest else None
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(full):
        g.replay()
    if g_rest is not None:
        g_rest.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3


def run_ours(args):
    import torch

    import quantized_weight_prefill_q4_gb300 as q
    import synth

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    # seeded inputs: set 0 is the seed-0 case; the other sets are copies
    case = bench_case()
    sets = []
    for i in range(SETS):
        sets.append(dict(W=torch.from_numpy(case["W"]).to(dev), X=torch.from_numpy(case["X"]).to(dev),
                         R=torch.from_numpy(case["R"]).to(dev), Y=torch.empty((T, N), device=dev),
                         X16=torch.empty((T, K), dtype=torch.float16, device=dev)))
    torch.cuda.synchronize()

    def step_call(s):
        return lambda: q.apr_qgemm(QTYPE, s["W"], N, K, s["X"], T, s["Y"], s["R"])

    def step(i):
        step_call(sets[i % SETS])()

    if args.only == "gemv":
        n, k, tg = args.gemv_rows, 4096, args.gemv_tokens
        qg = args.kernel_qtype
        c = synth.make_case(qg, n, k, tg, seed=0)
        Ws = [torch.from_numpy(c["W"]).to(dev) for _ in range(16)]
        X1 = torch.from_numpy(c["X"]).to(dev)
        Y1 = torch.empty((tg, n), device=dev)
        for i in range(args.warmup + args.steps):
            q.apr_qgemv(qg, Ws[i % 16], n, k, X1, tg, Y1, stream=stream)
        q.apr_stream_status(stream)
        print(json.dumps({"only": "gemv", "launches": args.warmup + args.steps}), flush=True)
        return

    if args.only == "attention":
        Ta = args.attn_tokens
        c = synth.attention_case(Ta, 0, 16, 4, seed=80)
        x = {key: torch.from_numpy(c[key]).to(dev) for key in ("Q", "K", "V")}
        Oa = torch.empty((Ta, 16 * 256), device=dev)
        for i in range(args.warmup + args.steps):
            q.apr_prefill_attention(x["Q"], x["K"], x["V"], Oa, Ta, 0, 16, 4, 256, stream=stream)
        q.apr_stream_status(stream)
        print(json.dumps({"only": "attention", "launches": args.warmup + args.steps}), flush=True)
        return

    if args.only == "kernel":
        qt = args.kernel_qtype
        Wk = [s["W"] for s in sets]
        if qt != QTYPE:
            w = synth.quantize(qt, synth.weight_f32(N, K, 0))
            Wk = [torch.from_numpy(w).to(dev) for _ in sets]
        for s in sets:
            q.apr_convert_f32_to_f16(s["X"], T * K, s["X16"], stream=stream)
        for i in range(args.warmup + args.steps):
            s = sets[i % SETS]
            q.apr_qgemm_f16_in(qt, Wk[i % SETS], N, K, s["X16"], T, s["Y"], s["R"], stream=stream)
        q.apr_stream_status(stream)
        print(json.dumps({"only": "kernel", "qtype": qt, "launches": args.warmup + args.steps}), flush=True)
        return

    if args.only == "exact":
        for i in range(args.warmup + args.steps):
            s = sets[i % SETS]
            q.apr_qgemm_ex(QTYPE, s["W"], N, K, s["X"], T, s["Y"], residual=s["R"], leg=q.APR_LEG_EXACT_F32,
                           path=q.APR_PATH_GEMM, stream=stream)
        q.apr_stream_status(stream)
        print(json.dumps({"only": "exact", "launches": args.warmup + args.steps}), flush=True)
        return

    for i in range(max(args.warmup, 3)):
        step(i)
    q.apr_stream_status(stream)

    # ---- timed region: K steps (graph replays of the rotating sets), events
    # on the launching stream, barrier + synchronize on both sides
    barrier(ws)
    torch.cuda.synchronize()
    timing = "CUDA graph replay"
    region_s = []
    with ClockSampler(dev.index) as clk:
        try:
            # the same K-step region timed REPEATS times; value = the median
            for _ in range(REPEATS):
                region_s.append(timed_calls([step_call(s) for s in sets], args.steps, stream))
            elapsed = float(np.median(region_s))
        except RuntimeError as exc:  # a driver that cannot capture the pooled scratch
            timing = f"direct launches (graph capture failed: {str(exc)[:80]})"
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(args.steps):
                step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            elapsed = e0.elapsed_time(e1) / 1e3
    barrier(ws)
    q.apr_stream_status(stream)
    t_max, flop_all = reduce_over_ranks(elapsed, FLOP * args.steps, ws)
    value = flop_all / t_max / 1e12
    if args.only == "step":
        if rank == 0:
            print(json.dumps({"only": "step", "value": value, "unit": "TFLOP/s", "steps": args.steps,
                              "ms_per_step": 1e3 * t_max / args.steps}), flush=True)
        return

    # ---- dominant kernel alone: the tcgen05 GEMM on fp16 activations
    for s in sets:
        q.apr_convert_f32_to_f16(s["X"], T * K, s["X16"], stream=stream)
    reps = max(200, min(args.steps, 2000))
    gemm_calls = [(lambda s=s: q.apr_qgemm_f16_in(QTYPE, s["W"], N, K, s["X16"], T, s["Y"], s["R"])) for s in sets]
    gemm_s = timed_calls(gemm_calls, reps, stream) / reps
    q.apr_stream_status(stream)
    peak_tf, peak_gbs, peak_kind = _peaks()
    achieved = FLOP / gemm_s / 1e12
    traffic = measured_traffic()

    # ---- small-T GEMV (T = 1), the other half of the metric
    gemv = gemv_big = None
    if rank == 0:
        gemv = gemv_rate(q, synth, dev, stream, peak_gbs)
        gemv_big = gemv_rate(q, synth, dev, stream, peak_gbs, n=12288, k=4096)
        ffn = ffn_rate(q, synth, dev, stream)
        big = gemm_kernel_rate(q, synth, dev, stream, peak_tf, T=2048)
        attn = {f"t{t}": attention_rate(q, synth, dev, stream, peak_tf, peak_gbs, T=t) for t in (512, 2048)}
        workloads = {} if args.no_configs else every_workload(q, dev, stream, peak_tf, peak_gbs)
        layer = {f"t{t}": layer_rate(q, dev, stream, peak_tf, T=t, chunk=min(t, 2048)) for t in (512, 2048)}

    # ---- end to end: host buffers, copies inside the timed region
    e2e_steps = max(20, min(args.steps, 200))
    hX = torch.from_numpy(case["X"]).pin_memory()
    hR = torch.from_numpy(case["R"]).pin_memory()
    hY = torch.empty((T, N), dtype=torch.float32).pin_memory()
    s0 = sets[0]
    for _ in range(3):
        s0["X"].copy_(hX, non_blocking=True)
        s0["R"].copy_(hR, non_blocking=True)
        q.apr_qgemm(QTYPE, s0["W"], N, K, s0["X"], T, s0["Y"], s0["R"], stream=stream)
        hY.copy_(s0["Y"], non_blocking=True)
    torch.cuda.synchronize()
    barrier(ws)
    # Each step copies its X and R in from pinned host memory, runs apr_qgemm
    # and copies its Y out. The copies in run on one stream, the calls on the
    # compute stream and the copies out on a third, so that the copy engines
    # work on other steps while the GPU computes (the copies in, bound by the
    # host-to-device link, set the pace; splitting them over two streams gains
    # nothing); events keep every device set's uses in order (its inputs are
    # not overwritten before the call that reads them has finished, its Y not
    # before it has been copied out).
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(SETS)]
    ev_done = [torch.cuda.Event() for _ in range(SETS)]
    ev_out = [torch.cuda.Event() for _ in range(SETS)]
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    for i in range(e2e_steps):
        j = i % SETS
        s = sets[j]
        with torch.cuda.stream(s_in):
            if i >= SETS:
                s_in.wait_event(ev_done[j])
            s["X"].copy_(hX, non_blocking=True)
            s["R"].copy_(hR, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if i >= SETS:
            stream.wait_event(ev_out[j])
        q.apr_qgemm(QTYPE, s["W"], N, K, s["X"], T, s["Y"], s["R"], stream=stream)
        ev_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            hY.copy_(s["Y"], non_blocking=True)
            ev_out[j].record(s_out)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    x1.record(stream)
    torch.cuda.synchronize()
    q.apr_stream_status(stream)
    e2e_t, e2e_flop = reduce_over_ranks(x0.elapsed_time(x1) / 1e3, FLOP * e2e_steps, ws)
    assert np.isfinite(hY.numpy()).all()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "qtype": "Q4_0", "n": N, "k": K, "T": T, "residual": True,
                       "leg": "f16 inputs, f32 accumulate", "l2": f"{SETS} rotating input sets (277 MB > 2x L2)",
                       "timing": timing,
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": achieved / peak_tf, "traffic": traffic,
                         "kernel": gemm_label(N, T, torch.cuda.get_device_properties(dev).multi_processor_count),
                         "peak_kind": f"{peak_kind} bf16 dense burst (fp16 has the same nominal rate)",
                         "kernel_ms": gemm_s * 1e3},
            "e2e": {"value": e2e_flop / e2e_t / 1e12, "unit": "TFLOP/s",
                    "overlap": "copies in, apr_qgemm and copies out on three streams, 8 device sets",
                    "h2d_bytes_per_step": 2 * T * N * 4, "d2h_bytes_per_step": T * N * 4},
            "gpu_launches": 2 * args.steps,
            "repeats": {"regions": len(region_s) or 1, "steps_each": args.steps,
                        "TFLOP/s": [FLOP * args.steps / t / 1e12 for t in region_s],
                        "note": "value is the median region; gpu_launches counts one region"},
            "clocks": clk.summary(),
            "gemv": gemv,
            "gemv_12288": gemv_big,
            "ffn_sublayer": ffn,
            "gemm_t2048": big,
            "attention": attn,
            "workloads": workloads,
            "prefill_layer": layer,
        }
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ------------------------------------------------------------------ every workload
_HOST = {}


def host_weight(qtype, n, k, seed):
    """Seeded GGUF bytes of an n x k weight (the f32 draw shared by both formats).
    Past 16384 rows the first 16384 rows repeat (timing only: such a weight
    is far larger than L2, so the repeat gives no cache hits)."""
    import numpy as np
    import synth

    if n > 16384:
        base = host_weight(qtype, 16384, k, seed)
        return np.ascontiguousarray(np.tile(base, (-(-n // 16384), 1))[:n])
    key = ("w", qtype, n, k, seed)
    if key not in _HOST:
        fk = ("f", n, k, seed)
        if fk not in _HOST:
            _HOST[fk] = synth.weight_f32(n, k, seed)
        _HOST[key] = synth.quantize(qtype, _HOST[fk])
    return _HOST[key]


def host_acts(rows, cols, seed):
    import synth

    key = ("x", rows, cols, seed)
    if key not in _HOST:
        _HOST[key] = synth.activations(rows, cols, seed)
    return _HOST[key]


L2_BYTES = 129 * 2**20


def time_per_call(calls, stream, budget_s=0.04, max_reps=2000):
    """Seconds per call: one graph replay of the rotating calls to estimate,
    then enough replays for about budget_s of device time."""
    import torch

    for c in calls:
        c()
    torch.cuda.synchronize()
    est = timed_calls(calls, len(calls), stream) / len(calls)
    reps = int(min(max_reps, max(2 * len(calls), budget_s / max(est, 1e-7))))
    return timed_calls(calls, reps, stream) / reps


def projection_rate(q, dev, stream, peak_tf, peak_gbs, *, qtype, n, k, T, residual=False, gate_up=False,
                    leg=0, path=0, seed=0):
    """One projection through apr_qgemm_ex, timed over rotating input sets whose
    bytes exceed 2.5x L2 (copies of one seeded set). Algorithmic work: flops
    2 T n k (x2 for gate/up), bytes = the quantized weight(s) + X + Y (+ R)."""
    import torch

    # bytes per 256 weights (F16, Q4_0, Q8_0, Q4_K, Q5_K, Q6_K, IQ4_XS); every k here is a multiple of 256
    b256 = {1: 512, 2: 144, 8: 272, 12: 144, 13: 176, 14: 210, 23: 136}[qtype]
    wbytes = n * (k // 256) * b256 * (2 if gate_up else 1)
    byts = wbytes + 4 * T * k + 4 * T * n * (2 if residual else 1)
    nsets = int(min(16, max(2, -(-2.5 * L2_BYTES // byts))))
    W0 = torch.from_numpy(host_weight(qtype, n, k, seed)).to(dev)
    Wu0 = torch.from_numpy(host_weight(qtype, n, k, seed + 3)).to(dev) if gate_up else None
    X0 = torch.from_numpy(host_acts(T, k, seed + 1)).to(dev)
    R0 = torch.from_numpy(host_acts(T, n, seed + 2)).to(dev) if residual else None
    sets = []
    for j in range(nsets):
        sets.append(dict(W=W0 if j == 0 else W0.clone(), Wu=None if Wu0 is None else (Wu0 if j == 0 else Wu0.clone()),
                         X=X0 if j == 0 else X0.clone(), R=None if R0 is None else (R0 if j == 0 else R0.clone()),
                         Y=torch.empty((T, n), device=dev)))

    def call(st):
        return lambda: q.apr_qgemm_ex(qtype, st["W"], n, k, st["X"], T, st["Y"], residual=st["R"], Wu=st["Wu"],
                                      leg=leg, path=path)

    dt = time_per_call([call(st) for st in sets], stream)
    q.apr_stream_status(stream)
    assert bool(torch.isfinite(sets[0]["Y"]).all())
    flop = 2.0 * T * n * k * (2 if gate_up else 1)
    t_flop, t_byte = flop / (peak_tf * 1e12), byts / (peak_gbs * 1e9)
    del sets
    out = {"us": dt * 1e6, "TFLOP/s": flop / dt / 1e12, "GB/s": byts / dt / 1e9,
           "frac_tensor": t_flop / dt, "frac_hbm": t_byte / dt,
           "bound": "tensor" if t_flop >= t_byte else "hbm", "frac_roofline": max(t_flop, t_byte) / dt}
    if leg == 1:
        # the exact leg against a TF32 tensor path's peak: the measured bf16
        # peak times the nominal dense ratio 1.1 / 2.25 PFLOP/s
        out["frac_tf32_peak"] = flop / dt / (peak_tf * 1e12 * 1.1 / 2.25)
    return out


def every_workload(q, dev, stream, peak_tf, peak_gbs):
    """Every seeded workload of the path, each through the public entry point
    (input sets rotating past L2, CUDA graph replay, CUDA events):
    * the Q8_0 256 x 512 problem with 16 tokens (by the T rule and forced onto
      the tensor-core GEMM);
    * fused gate/up SwiGLU 12288 x 4096 then down 4096 x 12288 + residual, 512
      tokens, Q4_0 and Q8_0;
    * the small-T GEMV sweep: T in {1, 2, 4, 8, 16} over 4096 x 4096 and
      12288 x 4096, Q4_0 and Q8_0 (GB/s against the HBM rate), and a
      151936 x 4096 output head at T = 1 (Q4_0, Q4_K);
    * the T rule: the GEMV (exact) against the forced tensor-core GEMM on the
      fp16 leg and on the exact leg at T = 4..16 (Q4_0, both weights), and the
      GEMMs at 24 and 32;
    * a 9B-class layer's projections (qkv 6144 x 4096, out 4096 x 4096 + R,
      gate/up 12288 x 4096, down 4096 x 12288 + R, Q4_0) at 512 and 2048 rows
      on the fp16 leg and the exact-fp32 leg;
    * F16 weights: 4096 x 4096 + R at 512 tokens on both legs, gate/up 12288 x
      4096 at 512 tokens, and the GEMV at T = 1 and 4;
    * Q4_K, Q5_K, Q6_K and IQ4_XS weights: the same five workloads."""
    import torch

    F16, Q4, Q8, Q4K, Q5K, Q6K, IQ4 = 1, 2, 8, 12, 13, 14, 23
    P = lambda **kw: projection_rate(q, dev, stream, peak_tf, peak_gbs, **kw)  # noqa: E731
    out = {}
    out["q8_0_n256_k512_t16"] = {"auto (T rule: the GEMM)": P(qtype=Q8, n=256, k=512, T=16),
                                 "forced GEMM": P(qtype=Q8, n=256, k=512, T=16, path=2)}
    for qt, name in ((Q4, "q4_0"), (Q8, "q8_0")):
        out[f"swiglu_{name}_n12288_k4096_t512"] = P(qtype=qt, n=12288, k=4096, T=512, gate_up=True)
        out[f"down_{name}_n4096_k12288_t512_res"] = P(qtype=qt, n=4096, k=12288, T=512, residual=True, seed=4)
    sweep = {}
    for qt, name in ((Q4, "q4_0"), (Q8, "q8_0")):
        for n, k in ((4096, 4096), (12288, 4096)):
            for T in (1, 2, 4, 8, 16):
                r = P(qtype=qt, n=n, k=k, T=T)
                sweep[f"{name}_n{n}_k{k}_t{T}"] = {key: r[key] for key in ("us", "GB/s", "frac_hbm", "TFLOP/s")}
    out["gemv_sweep"] = sweep
    # a vocabulary-sized output head at one token (the last-token projection)
    out["gemv_head"] = {f"{name}_n151936_k4096_t1": {key: r[key] for key in ("us", "GB/s", "frac_hbm")}
                        for qt, name in ((Q4, "q4_0"), (Q4K, "q4_k"))
                        for r in [P(qtype=qt, n=151936, k=4096, T=1)]}
    rule = {}
    for n in (4096, 12288):
        for T in (4, 8, 12, 16, 24, 32):
            row = {"gemm_us": P(qtype=Q4, n=n, k=4096, T=T, path=2)["us"],
                   "exact_gemm_us": P(qtype=Q4, n=n, k=4096, T=T, path=2, leg=1)["us"]}
            if T <= 16:
                row["gemv_us"] = P(qtype=Q4, n=n, k=4096, T=T, path=1)["us"]
            rule[f"q4_0_n{n}_k4096_t{T}"] = row
    out["t_rule"] = rule
    layer = {}
    for T in (512, 2048):
        for leg, lname in ((0, "f16"), (1, "exact_f32")):
            layer[f"t{T}_{lname}"] = {
                "qkv_n6144_k4096": P(qtype=Q4, n=6144, k=4096, T=T, leg=leg, seed=10),
                "out_n4096_k4096_res": P(qtype=Q4, n=4096, k=4096, T=T, residual=True, leg=leg, seed=11),
                "gate_up_n12288_k4096": P(qtype=Q4, n=12288, k=4096, T=T, gate_up=True, leg=leg, seed=12),
                "down_n4096_k12288_res": P(qtype=Q4, n=4096, k=12288, T=T, residual=True, leg=leg, seed=13),
            }
    out["layer_9b_q4_0"] = layer
    for qt, name in ((F16, "f16"), (Q4K, "q4_k"), (Q5K, "q5_k"), (Q6K, "q6_k"), (IQ4, "iq4_xs")):
        out[name] = {
            "n4096_k4096_t512_res": P(qtype=qt, n=4096, k=4096, T=512, residual=True),
            "n4096_k4096_t512_res_exact": P(qtype=qt, n=4096, k=4096, T=512, residual=True, leg=1),
            "swiglu_n12288_k4096_t512": P(qtype=qt, n=12288, k=4096, T=512, gate_up=True),
            "gemv_n4096_k4096_t1": P(qtype=qt, n=4096, k=4096, T=1),
            "gemv_n4096_k4096_t4": P(qtype=qt, n=4096, k=4096, T=4),
        }
    torch.cuda.empty_cache()
    return out


def layer_rate(q, dev, stream, peak_tf, T=512, chunk=512, hidden=4096, inter=12288, nh=16, nkv=4):
    """apr_prefill_layer on a 9B-class layer (Q4_0, fp16 leg, 16 query heads
    over 4 KV heads, head_dim 256) over T rows at position 0 in chunks of
    `chunk` rows, three rotating weight sets (325 MB, more than L2). TFLOP/s
    counts the projections (2 T n k each, gate/up twice) and the attention's
    two products over the visible (row, key) pairs."""
    import torch

    d = 256
    qd, kvd = nh * d, nkv * d
    shapes = (((qd + 2 * kvd), hidden), (hidden, qd), (inter, hidden), (inter, hidden), (hidden, inter))
    sets = []
    for j in range(3):
        W = [torch.from_numpy(host_weight(2, r, c, 20 + i)).to(dev) for i, (r, c) in enumerate(shapes)]
        X = torch.from_numpy(host_acts(T, hidden, 30)).to(dev)
        K = torch.zeros((T, kvd), device=dev)
        V = torch.zeros((T, kvd), device=dev)
        sets.append((W, X, K, V))
    an = torch.ones(hidden, device=dev)

    def call(st):
        W, X, K, V = st
        return lambda: q.apr_prefill_layer(2, *W, hidden, inter, nh, nkv, T, 0, an, an, 1e-6, X, K, V, chunk=chunk)

    dt = time_per_call([call(st) for st in sets], stream, budget_s=0.05)
    q.apr_stream_status(stream)
    flop = 2.0 * T * hidden * (qd + 2 * kvd + qd + 3 * inter)
    aflop, _ = attention_work(T, 0, nh, nkv, d)
    tf = (flop + aflop) / dt / 1e12
    return {"workload": f"layer_q4_0_hidden{hidden}_inter{inter}_h{nh}_kv{nkv}_t{T}_chunk{chunk}", "us": dt * 1e6,
            "TFLOP/s": tf, "frac_tensor": tf / peak_tf}


def gemm_kernel_rate(q, synth, dev, stream, peak_tf, n=4096, k=4096, T=2048):
    """The GEMM kernel alone (fp16 X in, + residual) at a larger chunk of
    tokens, four rotating input sets (more than L2)."""
    import torch

    sets = []
    for j in range(4):
        c = synth.make_case(QTYPE, n, k, T, residual=True, seed=70 + j)
        d = {key: torch.from_numpy(c[key]).to(dev) for key in ("W", "R")}
        d["X16"] = torch.from_numpy(c["X"]).to(dev).half()
        d["Y"] = torch.empty((T, n), device=dev)
        sets.append(d)

    def call(s):
        return lambda: q.apr_qgemm_f16_in(QTYPE, s["W"], n, k, s["X16"], T, s["Y"], s["R"])

    for s in sets:
        call(s)()
    torch.cuda.synchronize()
    reps = 200
    dt = timed_calls([call(s) for s in sets], reps, stream) / reps
    q.apr_stream_status(stream)
    tf = 2.0 * n * k * T / dt / 1e12
    return {"workload": f"q4_0_gemm_residual_n{n}_k{k}_t{T}", "TFLOP/s": tf, "frac": tf / peak_tf, "us": dt * 1e6}


def ffn_rate(q, synth, dev, stream, hidden=4096, inter=12288, T=512):
    """The FFN sublayer of a 9B-class layer (RMSNorm, fused gate/up SwiGLU,
    down + residual, Q4_0, fp16 leg) on T rows, two rotating weight sets
    (170 MB, more than L2); TFLOP/s counts the three projections."""
    import torch

    sets = []
    for j in range(2):
        W = [torch.from_numpy(synth.quantize(QTYPE, synth.weight_f32(r, c, 50 + 3 * j + i))).to(dev)
             for i, (r, c) in enumerate(((inter, hidden), (inter, hidden), (hidden, inter)))]
        sets.append((W, torch.from_numpy(synth.activations(T, hidden, 60 + j)).to(dev)))
    w = torch.ones(hidden, device=dev)

    def call(s):
        W, X = s
        return lambda: q.apr_ffn_sublayer(QTYPE, W[0], W[1], W[2], hidden, inter, T, w, 1e-6, X)

    for s in sets:
        call(s)()
    torch.cuda.synchronize()
    reps = 200
    dt = timed_calls([call(s) for s in sets], reps, stream) / reps
    q.apr_stream_status(stream)
    flop = 2.0 * T * 3 * hidden * inter
    return {"workload": f"q4_0_ffn_hidden{hidden}_inter{inter}_t{T}", "TFLOP/s": flop / dt / 1e12, "us": dt * 1e6,
            "launches_per_call": 4}


def attention_work(T, pos0, nh, nkv, d=256):
    """Algorithmic work of one prefill-attention call: the two products over
    the visible (row, key) pairs, 4 * d * heads * sum_t (pos0 + t + 1) flops,
    and the bytes the method must move, Q in and O out ([T][heads * d] f32)
    and the K and V cache rows 0 .. pos0 + T - 1 ([.][kv_heads * d] f32)."""
    flop = 4.0 * d * nh * (T * (T + 1) / 2 + pos0 * T)
    byts = 4 * (2 * T * nh * d + 2 * (pos0 + T) * nkv * d)
    return flop, byts


def attention_rate(q, synth, dev, stream, peak_tf, peak_gbs, T=2048, pos0=0, nh=16, nkv=4):
    """Causal prefill attention of a 9B-class layer (16 query heads over 4 KV
    heads, head_dim 256) on a chunk of T rows at pos0, rotating input sets
    (more than L2 in all). TFLOP/s counts the two products over the visible
    (row, key) pairs only; frac_roofline = the larger of the flop time at the
    tensor peak and the byte time at the HBM rate, over the measured time."""
    import torch

    d = 256
    per_set = 4 * (T * nh * d + 2 * (pos0 + T) * nkv * d)
    nsets = max(2, -(-160 * 2**20 // per_set))
    sets = []
    for j in range(nsets):
        c = synth.attention_case(T, pos0, nh, nkv, d, seed=80 + j)
        x = {key: torch.from_numpy(c[key]).to(dev) for key in ("Q", "K", "V")}
        x["O"] = torch.empty((T, nh * d), device=dev)
        sets.append(x)

    def call(x):
        return lambda: q.apr_prefill_attention(x["Q"], x["K"], x["V"], x["O"], T, pos0, nh, nkv, d)

    for x in sets:
        call(x)()
    torch.cuda.synchronize()
    reps = 200
    dt = timed_calls([call(x) for x in sets], reps, stream) / reps
    q.apr_stream_status(stream)
    flop, byts = attention_work(T, pos0, nh, nkv, d)
    tf = flop / dt / 1e12
    t_flop, t_byte = flop / (peak_tf * 1e12), byts / (peak_gbs * 1e9)
    return {"workload": f"attention_h{nh}_kv{nkv}_d{d}_t{T}_pos{pos0}", "TFLOP/s": tf, "frac": tf / peak_tf,
            "bound": "tensor" if t_flop >= t_byte else "hbm", "frac_roofline": max(t_flop, t_byte) / dt,
            "us": dt * 1e6}


def gemv_rate(q, synth, dev, stream, peak_gbs, n=4096, k=4096):
    """T = 1 GEMV over a Q4_0 n x k weight, 16 rotating weights (151 MB at
    4096 x 4096, more than L2)."""
    import torch

    nsets = 16
    c = synth.make_case(QTYPE, n, k, 1, seed=0)
    Ws = [torch.from_numpy(c["W"]).to(dev) for _ in range(nsets)]
    X = torch.from_numpy(c["X"]).to(dev)
    Y = torch.empty((1, n), device=dev)
    for i in range(20):
        q.apr_qgemv(QTYPE, Ws[i % nsets], n, k, X, 1, Y, stream=stream)
    torch.cuda.synchronize()
    reps = 2000
    dt = timed_calls([(lambda w=w: q.apr_qgemv(QTYPE, w, n, k, X, 1, Y)) for w in Ws], reps, stream) / reps
    q.apr_stream_status(stream)
    byts = n * (k // 32) * 18 + k * 4 + n * 4
    gbs = byts / dt / 1e9
    # the same weights only streamed (the GEMV's data movement, no compute):
    # what a launch of this size can reach on this GPU
    wb = n * (k // 32) * 18
    fl = timed_calls([(lambda w=w: q.apr_read_stream(w, wb)) for w in Ws], reps, stream) / reps
    q.apr_stream_status(stream)
    return {"workload": f"q4_0_gemv_n{n}_k{k}_t1", "GB/s": gbs, "frac_hbm": gbs / peak_gbs, "us": dt * 1e6,
            "stream_floor_us": fl * 1e6, "frac_stream_floor": fl / dt}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload fields (every configuration)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", choices=["all", "step", "kernel", "exact", "gemv", "attention"], default="all",
                    help="step: only the timed apr_qgemm steps; kernel: only the GEMM kernel on fp16 activations "
                         "(--kernel-qtype weights); exact: only the exact-fp32 leg's GEMM call on the same problem; "
                         "gemv: only the T = 1 GEMV; attention: only the prefill attention (16 query heads, 4 KV "
                         "heads, --attn-tokens rows at position 0) (small, bounded runs for profilers)")
    ap.add_argument("--kernel-qtype", type=int, default=2, choices=[1, 2, 8, 12, 13, 14, 23],
                    help="weight type of the --only kernel and --only gemv runs (GGUF id: 1 F16, 2 Q4_0, 8 Q8_0, 12 Q4_K, "
                         "13 Q5_K, 14 Q6_K, 23 IQ4_XS)")
    ap.add_argument("--attn-tokens", type=int, default=2048, help="query rows of the --only attention run")
    ap.add_argument("--gemv-tokens", type=int, default=1, help="tokens of the --only gemv run (1..16)")
    ap.add_argument("--clocks-dir", default=None, help="where the raw nvidia-smi clock samples are written")
    ap.add_argument("--gemv-rows", type=int, default=4096, help="weight rows of the --only gemv run (k = 4096)")
    args = ap.parse_args(argv)
    if args.clocks_dir:
        global CLOCKS_DIR
        CLOCKS_DIR = args.clocks_dir
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
