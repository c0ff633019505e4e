"""Benchmark of MXFP8 grouped-matmul-finalize-routing on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--deterministic] [--impl ours|reference]

One step = one call of gmmfr_grouped_matmul_finalize_routing (prologue, grouped
GEMM with the fused logit / scatter / shared epilogue, and in deterministic
mode the row-ordered combine) on the chosen workload, weights prepared once
beforehand (the preparation is timed separately).  `value` is the effective
HBM bandwidth: algorithmic bytes (x2 and scales of experts holding tokens, x1,
token scales, logit, row_index, group_list, shared_input, out read + written)
over the device time of the call.  L2 is flushed between steps (256 MB written,
then 256 MB read), outside the timed events.  Multi-GPU runs are independent replicas.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/call and achieved HBM GB/s vs roofline, MXFP8 grouped-matmul-finalize-routing"
DEFAULT_CONFIG = 5  # the large-E workload (M 4096, K 7168, N 4096, E 256): the largest that fits one GPU
FMT_NAMES = {0: "E4M3", 1: "E5M2", 2: "E2M1"}
# GPU sleep placed before each timed call, outside its events (about 0.5 ms at 2 GHz): the
# device stays busy while the host enqueues the call, so the events time device work only
SLEEP_CYCLES = 1_000_000


def _quantiles(xs, qs):
    """Nearest-rank quantiles of a list."""
    v = sorted(xs)
    return [v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))] for q in qs]


def reduce_step_time(ms: float, world: int) -> float:
    """Slowest rank's mean step time (the job's step time).  Replicas share no
    data: the only cross-rank operation is this max."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: int, ms: float, world: int) -> float:
    """Whole-job GB/s: every rank processes one call's bytes per step."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def _config_dict(spec, counts, deterministic):
    return {"workload": spec.name, "M": spec.M, "K": spec.K, "N": spec.N, "E": spec.E, "batch": spec.batch,
            "x1": FMT_NAMES[spec.x1_dtype], "x2": FMT_NAMES[spec.x2_dtype],
            "transpose_x2": spec.transpose_x2, "group_list_type": spec.group_list_type,
            "nonempty_experts": int((counts > 0).sum()), "max_tokens_per_expert": int(counts.max()),
            "mode": "deterministic" if deterministic else "atomic",
            "l2": "flushed between steps (256 MB write, then 256 MB read: no inputs and no dirty lines in L2), weights also larger than L2",
            "parallelism": "replicas"}


class L2Flush:
    """Evicts L2 between timed steps: writes a 256 MB buffer (twice the L2), then reads
    another 256 MB buffer, so the next step starts with none of its inputs in L2 and
    with no dirty lines left to write back (a write-only flush leaves ~129 MB of dirty
    lines that the next timed kernel would pay for in HBM write-back)."""

    def __init__(self):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")

    def __call__(self):
        import torch
        self.w.zero_()
        torch.amax(self.r)


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.index = index
        self.enabled = enabled
        self.proc = None
        self.path = os.path.join("/tmp", f"gmmfr_clocks_{os.getpid()}.csv")

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        try:
            rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
        except OSError:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.strip() == "Active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def _oracle_problem(spec, inp, ncols):
    import oracle
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W
    x2 = inp["x2"].cpu()
    sc = inp["scale"].cpu()
    if spec.transpose_x2:
        x2s = x2[:, :ncols, :].contiguous()
        scs = sc[..., :ncols, :, :].contiguous()
    else:  # [E, K, N]; E2M1 holds two columns per byte along N (ncols is even)
        x2s = x2[:, :, :(ncols // 2 if spec.x2_dtype == W.E2M1 else ncols)].contiguous()
        scs = sc[..., :ncols, :].contiguous()
    shared = inp["shared_input"][:, :ncols].contiguous() if inp["shared_input"] is not None else None
    bias = inp["bias"][:, :ncols].contiguous() if inp.get("bias") is not None else None
    return oracle.Problem(M=spec.M, K=spec.K, N=ncols, E=spec.E, batch=spec.batch, x1=inp["x1"].cpu(), x2=x2s,
                          scale=scs, pertoken_scale=inp["pertoken_scale"].cpu(), group_list=inp["group_list"].cpu(),
                          row_index=inp["row_index"].cpu(), out=inp["out"].cpu()[:, :ncols].contiguous(),
                          x1_dtype=spec.x1_dtype, x2_dtype=spec.x2_dtype, transpose_x2=spec.transpose_x2,
                          scale_per_expert=spec.scale_per_expert, group_list_type=spec.group_list_type,
                          logit=inp["logit"].cpu() if inp["logit"] is not None else None, shared_input=shared,
                          shared_offset=spec.shared_offset, shared_weight=spec.shared_weight, bias=bias)


def _oracle_columns(spec, inp, seconds, probe=None):
    """Output columns [0, ncols) that the oracle finishes in about `seconds` on this host
    (multiples of 64; all N when the whole workload fits).  `probe` = (columns, seconds) of
    an earlier run, else one is made here.  Returns (ncols, est. seconds for all N, probe)."""
    import oracle
    if probe is None:
        cols = min(spec.N, 64 * max(1, oracle.num_threads()))
        t0 = time.perf_counter()
        oracle.run(_oracle_problem(spec, inp, cols))
        probe = (cols, time.perf_counter() - t0)
    est_full = probe[1] * spec.N / probe[0]
    if est_full <= seconds:
        return spec.N, est_full, probe
    ncols = int(spec.N * seconds / max(est_full, 1e-9)) // 64 * 64
    return min(spec.N, max(64, ncols)), est_full, probe


def _cpu_baseline(spec, inp, min_s=10.0, max_s=30.0):
    """The oracle, as it stands, on all host cores: the whole workload (repeated
    until about min_s of work) when a probe predicts it takes at most max_s,
    otherwise a slice of output columns sized for about min_s, scaled by N/cols.
    Returns (GB/s for the whole workload, seconds, sample text, cores)."""
    import oracle
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    threads = oracle.num_threads()
    ncols, est_full, _ = _oracle_columns(spec, inp, max_s)
    if ncols == spec.N:
        reps = max(1, int(min_s / max(est_full, 1e-3)))
    else:
        ncols, _, _ = _oracle_columns(spec, inp, min_s, (spec.N, est_full))
        reps = 1
    p = _oracle_problem(spec, inp, ncols)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.run(p)
    dt = time.perf_counter() - t0
    per_call = dt / reps * spec.N / ncols
    gbs = W.algorithmic_bytes(spec) / per_call / 1e9
    what = "the whole workload" if ncols == spec.N else f"output columns [0,{ncols}) of {spec.N}, scaled by N/{ncols}"
    return gbs, dt, f"oracle on {what}, {reps} run(s), {dt:.1f} s", threads


PROFILE_RECORD = os.path.join(ROOT, "profiles", "gemm_kernel_traffic.json")
KERNEL_SOURCES = ("kernels_gemm.cu", "ptx.cuh", "common.cuh", "pipeline.cuh")


def kernel_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the grouped GEMM kernel's sources."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, "moe_grouped_gemm_mxfp8_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profile_record(workload):
    """The committed ncu record (profiles/gemm_kernel_traffic.json) of this workload: DRAM
    bytes per gemm_kernel launch and the counters behind them, or None."""
    try:
        with open(PROFILE_RECORD) as f:
            rec = json.load(f)
    except OSError:
        return None
    return rec.get("workloads", {}).get(workload.split()[0])


def _profiled_traffic(workload, as_captured=True):
    """DRAM bytes per gemm_kernel launch from the committed ncu record of this workload, if
    the kernel sources are unchanged since that capture and the run is set up as it was
    (atomic mode, no bias, no tiling hint: `as_captured`); else None."""
    if not as_captured:
        return None
    r = profile_record(workload)
    if r is None or r.get("source_sha256_16") != kernel_source_hash():
        return None
    return int(r["traffic_bytes_per_launch"])


def _time_route(args, flush):
    """Device time of the routing step (gmmfr_moe_route) for this workload's batch,
    topk, K and E, with its own algorithmic bytes."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    rs = W.route_config(args.config)
    ri = {k: v.cuda() for k, v in W.make_route_inputs(rs).items()}
    out, ws = B.route(ri["topk_ids"], ri["topk_weights"], ri["x"], ri["x_scale"], rs.E)
    rp = B.RouteProblem(batch=rs.batch, topk=rs.topk, K=rs.K, E=rs.E, ids_type=B.INDEX_I64, group_list_type=1)
    sptr = torch.cuda.current_stream().cuda_stream

    def call():
        B.gmmfr_moe_route(rp, ri["topk_ids"].data_ptr(), ri["topk_weights"].data_ptr(), ri["x"].data_ptr(),
                          ri["x_scale"].data_ptr(), out["x1"].data_ptr(), out["pertoken_scale"].data_ptr(),
                          out["group_list"].data_ptr(), out["row_index"].data_ptr(), out["logit"].data_ptr(),
                          out["perm"].data_ptr(), ws.data_ptr(), ws.numel(), sptr)

    for _ in range(args.warmup):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    nbytes = W.route_algorithmic_bytes(rs)
    return {"workload": rs.name, "us_per_call": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "algorithmic_bytes": nbytes, "launches": 1 if rs.M <= 8192 else 3}


def _time_layer(args, flush, prob, d, prep, ws, call_us, route_us):
    """Routing step and operator back to back on one stream, as in a MoE layer: the
    operator is launched as a programmatic dependent of the routing kernel, so its
    launch overlaps the routing tail.  Reported beside the two timed separately."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    rs = W.route_config(args.config)
    ri = {k: v.cuda() for k, v in W.make_route_inputs(rs).items()}
    ro, rws = B.route(ri["topk_ids"], ri["topk_weights"], ri["x"], ri["x_scale"], rs.E)
    rp = B.RouteProblem(batch=rs.batch, topk=rs.topk, K=rs.K, E=rs.E, ids_type=B.INDEX_I64, group_list_type=1)
    sptr = torch.cuda.current_stream().cuda_stream
    dd = dict(d)
    dd.update({k: ro[k] for k in ("x1", "pertoken_scale", "group_list", "row_index", "logit")})
    out = d["out"].clone()

    def layer():
        B.gmmfr_moe_route(rp, ri["topk_ids"].data_ptr(), ri["topk_weights"].data_ptr(), ri["x"].data_ptr(),
                          ri["x_scale"].data_ptr(), ro["x1"].data_ptr(), ro["pertoken_scale"].data_ptr(),
                          ro["group_list"].data_ptr(), ro["row_index"].data_ptr(), ro["logit"].data_ptr(),
                          ro["perm"].data_ptr(), rws.data_ptr(), rws.numel(), sptr)
        B.run(prob, dd, out, prepared=prep, ws=ws)

    for _ in range(args.warmup):
        layer()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        a.record()
        layer()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    return {"workload": rs.name + " + " + prob_name(args), "us_per_layer": ms * 1e3,
            "route_us_alone": route_us, "call_us_alone": call_us,
            "saved_us": route_us + call_us - ms * 1e3, "launches": 2}


def prob_name(args):
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W
    return W.config(args.config).name


def _time_ffn(args, flush):
    """Device time of the grouped SwiGLU FFN (gmmfr_llada2_moe_grouped_gemm) on the
    LLaDA2.0-mini shape (H 2048, I 512, E 256, 4096 routed tokens)."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    fs = W.ffn_config("model")
    d = {k: v.cuda() for k, v in W.make_ffn_inputs(fs, weights_device="cuda").items()}
    prep = B.ffn_prepare(fs.H, fs.I, fs.E, d["w13_flat"], d["w2_flat"])
    res, ws = B.ffn(d["sorted_tokens"], prep, d["expert_cumsum"], fs.H, fs.I, fs.E)
    def call():
        B.ffn(d["sorted_tokens"], prep, d["expert_cumsum"], fs.H, fs.I, fs.E, result=res, ws=ws)

    for _ in range(args.warmup):
        call()
    # timed: one event pair around each call (the per-kernel events of a profiled pass would sit
    # between the two GEMMs and keep GEMM2 from starting before GEMM1 ends)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    B.gmmfr_profile_begin(args.steps)
    for _ in range(args.steps):
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        call()
    k = B.gmmfr_profile_end(args.steps)
    nbytes = W.ffn_algorithmic_bytes(fs)
    peaks, _ = _peaks()
    return {"workload": fs.name, "us_per_call": ms * 1e3, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
            "gemm1_us": statistics.mean(x[2] for x in k) * 1e3, "gemm2_us": statistics.mean(x[3] for x in k) * 1e3,
            "tflops": W.ffn_flops(fs) / (ms * 1e-3) / 1e12, "algorithmic_bytes": nbytes, "launches": 2}


def _timed_calls(call, flush, steps, reset=None, clocks_index=None, world=1):
    """`steps` steps of: L2 flush, reset() (restores out), a GPU sleep (so the host has
    enqueued the call before the device reaches it), then call() between two CUDA events on
    the current stream.  Returns (per-call ms, clock summary or None, wall seconds)."""
    import torch
    import torch.distributed as dist
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(clocks_index if clocks_index is not None else 0, enabled=clocks_index is not None) as clk:
        t_wall = time.perf_counter()
        for i in range(steps):
            flush()
            if reset is not None:
                reset()
            torch.cuda._sleep(SLEEP_CYCLES)
            starts[i].record()
            call()
            ends[i].record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], (clk.summary() if clocks_index is not None else None), t_wall


def _kernel_breakdown(call, flush, steps, reset=None):
    """The same steps again with the library's per-kernel events (which add a few
    microseconds inside a call, so they stay out of the timed steps): per call, the ms of
    each profile slot (-1 where the slot's kernel did not run)."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    B.gmmfr_profile_begin(steps)
    for _ in range(steps):
        flush()
        if reset is not None:
            reset()
        torch.cuda._sleep(SLEEP_CYCLES)
        call()
    return B.gmmfr_profile_end(steps)


def _device_inputs(spec):
    """Inputs of a workload on the device (the weights drawn there by a seeded CUDA generator)."""
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W
    inp = W.make_inputs(spec, device="cpu", weights_device="cuda")
    return inp, {k: (v.cuda() if v is not None else None) for k, v in inp.items()}


def _measure(spec, deterministic, flush, steps, warmup, d=None, prep=None):
    """Device time of one call on a workload (atomic or deterministic mode), with the GEMM
    kernel's share from a profiled pass; algorithmic bytes over the time as GB/s and as a
    fraction of the measured copy bandwidth."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    if d is None:
        _, d = _device_inputs(spec)
    prob = B.problem_from_spec(spec, deterministic)
    if prep is None:
        prep = B.prepare_weights(prob, d["x2"], d["scale"])
    ws = B.workspace(prob, True, "cuda")
    out = d["out"].clone()

    def call():
        B.run(prob, d, out, prepared=prep, ws=ws)

    def reset():
        out.copy_(d["out"])

    for _ in range(warmup):
        call()
    call_ms, _, _ = _timed_calls(call, flush, steps, reset)
    k = _kernel_breakdown(call, flush, steps, reset)
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    nbytes = W.algorithmic_bytes(spec)
    hbm = float(_peaks()[0]["hbm_gbs"])
    ms = statistics.mean(call_ms)
    gemm_ms = statistics.mean(x[2] for x in k)
    comb = [x[3] for x in k if x[3] >= 0]
    return {"workload": spec.name, "mode": "deterministic" if deterministic else "atomic",
            "us_per_call": ms * 1e3, "us_per_call_p10_p50_p90": [round(float(x) * 1e3, 2) for x in _quantiles(call_ms, (0.1, 0.5, 0.9))],
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
            "gemm_us": gemm_ms * 1e3, "gemm_frac_hbm": nbytes / (gemm_ms * 1e-3) / 1e9 / hbm,
            "combine_us": statistics.mean(comb) * 1e3 if comb else None,
            "tflops": W.flops(spec) / (ms * 1e-3) / 1e12, "algorithmic_bytes": nbytes,
            "launches_per_call": sum(1 for s in (0, 1, 2, 3) if k[0][s] >= 0), "device_error_bits": bits}


def _time_mxfp4(args, flush):
    """Device time of the operator on MXFP4 inputs (E2M1 tokens and weights, E8M0 per
    32) at the large shape (M 4096, K 7168, N 4096, E 256), against the algorithmic
    bytes of the packed FP4 inputs.  Tokens and prepared weights stay packed (one GEMM
    launch of kind::mxf4 MMAs)."""
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W
    return _measure(W.mxfp4_config(), False, flush, args.steps, args.warmup)


def _sub_workloads(args, flush, main_spec, d, prep):
    """Every other benchmark workload, one line each: the four smaller configs in atomic
    mode, and the deterministic mode on the second, fourth and largest (the largest reusing
    the timed call's inputs and prepared weights)."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import workloads as W
    res = {}
    for i in (1, 2, 3, 4):
        spec = W.config(i)
        if spec.name == main_spec.name:
            continue
        _, di = _device_inputs(spec)
        res[spec.name.split()[0]] = _measure(spec, False, flush, args.steps, args.warmup, d=di)
        if i in (2, 4):
            res[spec.name.split()[0] + " deterministic"] = _measure(spec, True, flush, args.steps, args.warmup, d=di)
        del di
        torch.cuda.empty_cache()
    if main_spec.name == W.config(5).name:
        res["C5 deterministic"] = _measure(main_spec, True, flush, args.steps, args.warmup, d=d, prep=prep)
    return res


def run_reference(args):
    """The oracle (CPU) as the reference arm, on the same workload and input bytes as the
    GPU arm (the weights drawn by the same seeded CUDA generator, then copied to the host).
    Each step runs the oracle on a bounded sample, output columns [0, ncols) of the workload,
    sized so that all warm-up and timed steps take about two and a half minutes; its rate is
    scaled to the whole workload by N / ncols."""
    import torch

    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    spec = _main_spec(args)
    inp = W.make_inputs(spec, device="cpu", weights_device="cuda" if torch.cuda.is_available() else "cpu")
    inp["x2"] = inp["x2"].cpu()
    torch.cuda.empty_cache() if torch.cuda.is_available() else None
    counts = W.expert_counts(spec)
    per_step = min(10.0, max(1.0, 150.0 / max(1, args.warmup + args.steps)))
    ncols, est_full, _ = _oracle_columns(spec, inp, per_step)
    p = _oracle_problem(spec, inp, ncols)
    nbytes = W.algorithmic_bytes(spec)
    vals = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.run(p)
        dt = (time.perf_counter() - t0) * spec.N / ncols
        if i >= args.warmup:
            vals.append(nbytes / dt / 1e9)
    v = statistics.median(vals)
    full_ms = nbytes / (v * 1e9) * 1e3
    sample = (f"oracle on output columns [0,{ncols}) of {spec.N} per step (whole workload ~{est_full:.1f} s on "
              f"{oracle.num_threads()} threads), rate scaled by N/{ncols}")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config_dict(spec, counts, args.deterministic),
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _main_spec(args):
    """The workload of the timed call: --config N (with --e32 the 32-expert copy of the large
    workload, for full profiler captures), or with --fp4 the MXFP4 operator at the large
    shape (c5) or its reduced copy (e32); --bias adds the per-expert bf16 bias."""
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    if args.fp4 == "c5":
        spec = W.mxfp4_config()
    elif args.fp4 == "e32":
        spec = W.mxfp4_small_config()
    elif args.e32:
        spec = W.large_small_config()
    else:
        spec = W.config(args.config)
    if args.bias:
        spec = dataclasses.replace(spec, name=spec.name + " bias", bias=True)
    return spec


def run_ours(args):
    import torch
    import torch.distributed as dist

    from moe_grouped_gemm_mxfp8_gb300 import binding as B
    from moe_grouped_gemm_mxfp8_gb300 import build as build_mod
    from moe_grouped_gemm_mxfp8_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    build_mod.build()
    B.load()

    spec = _main_spec(args)
    counts = W.expert_counts(spec)
    alg_bytes = W.algorithmic_bytes(spec, counts)
    flops = W.flops(spec, counts)
    inp, d = _device_inputs(spec)
    prob = B.problem_from_spec(spec, args.deterministic)
    prob.expected_tokens_per_expert = args.tokens_hint  # the tuning hint (0: chosen on the device)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    # one-time weight preparation, timed on its own
    n_prep = B.gmmfr_prepared_weights_size(prob)
    prep = torch.empty(n_prep, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        e0.record()
        B.gmmfr_prepare_weights(prob, B.view(d["x2"]), B.view(d["scale"]), prep.data_ptr(), n_prep, sptr)
        e1.record()
    torch.cuda.synchronize()
    prep_ms = e0.elapsed_time(e1)
    ws = B.workspace(prob, True, "cuda")
    out0 = d["out"].clone()
    out = d["out"].clone()
    flush = L2Flush()

    def call():
        B.run(prob, d, out, prepared=prep, ws=ws)

    def reset():
        out.copy_(out0)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    bits = B.gmmfr_check_device_errors(ws.data_ptr(), sptr)

    # the timed steps: nothing but the call between the events
    call_ms, clocks, t_wall = _timed_calls(call, flush, args.steps, reset, clocks_index=local, world=world)
    ms = reduce_step_time(statistics.mean(call_ms), world)
    kernel_ms = _kernel_breakdown(call, flush, args.steps, reset)
    gemm_ms = statistics.mean(k[2] for k in kernel_ms)
    # kernels of one call, from the slots the profiled pass saw run (input preparation, GEMM,
    # deterministic combine)
    launches_per_call = sum(1 for slot in (0, 1, 2, 3) if kernel_ms[0][slot] >= 0)
    comb = [k[3] for k in kernel_ms if k[3] >= 0]
    comb_ms = statistics.mean(comb) if comb else None

    # end to end through the public call with host buffers: H2D of the step's
    # inputs from pinned memory, the call, D2H of the result.  The inputs sit in one
    # pinned staging buffer (256-byte aligned slices) so a step makes one H2D copy.
    per_step = ["x1", "pertoken_scale", "group_list", "logit", "row_index", "shared_input", "out"]
    names = [k for k in per_step if inp[k] is not None]
    offs, off = {}, 0
    for k in names:
        offs[k] = off
        off = (off + inp[k].numel() * inp[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    for k in names:
        n = inp[k].numel() * inp[k].element_size()
        host_buf[offs[k]:offs[k] + n].copy_(inp[k].contiguous().view(-1).view(torch.uint8))
    h2d = off
    out_host = torch.empty_like(inp["out"]).pin_memory()
    d2h = out_host.numel() * out_host.element_size()

    def device_set():
        buf = torch.empty(off, dtype=torch.uint8, device="cuda")
        views = dict(d)
        for k in names:
            n = inp[k].numel() * inp[k].element_size()
            views[k] = buf[offs[k]:offs[k] + n].view(inp[k].dtype).view(inp[k].shape)
        return buf, views

    # (1) serial: each step's copy in, call and copy out one after another, after an L2 flush
    dev_buf, dd = device_set()
    ee0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ee1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        if i >= args.warmup:
            flush()
            ee0[i - args.warmup].record()
        dev_buf.copy_(host_buf, non_blocking=True)
        B.run(prob, dd, dd["out"], prepared=prep, ws=ws)
        out_host.copy_(dd["out"], non_blocking=True)
        if i >= args.warmup:
            ee1[i - args.warmup].record()
    torch.cuda.synchronize()
    e2e_serial_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ee0, ee1))

    # (2) pipelined, as a serving loop runs: two device input sets; step i's copy in (copy
    # stream) overlaps step i-1's call (compute stream), and its copy out (return stream)
    # overlaps step i+1.  Every step still copies all its inputs in and its result out.  No
    # flush between steps (the weights are larger than L2).
    sets = [(dev_buf, dd), device_set()]
    s_in, s_main, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n_all = args.warmup + args.steps
    ev_in = [torch.cuda.Event() for _ in range(n_all)]
    ev_call = [torch.cuda.Event() for _ in range(n_all)]
    ev_out = [torch.cuda.Event() for _ in range(n_all)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(n_all):
        buf, views = sets[i % 2]
        if i == args.warmup:  # the timed steps start with the warm-up steps drained
            if i > 0:
                s_in.wait_event(ev_out[i - 1])
            t_start.record(s_in)
        if i >= 2:
            s_in.wait_event(ev_out[i - 2])  # the set's previous result has been read back
        with torch.cuda.stream(s_in):
            buf.copy_(host_buf, non_blocking=True)
        ev_in[i].record(s_in)
        s_main.wait_event(ev_in[i])
        B.run(prob, views, views["out"], prepared=prep, ws=ws, stream=s_main)
        ev_call[i].record(s_main)
        s_out.wait_event(ev_call[i])
        with torch.cuda.stream(s_out):
            out_host.copy_(views["out"], non_blocking=True)
        ev_out[i].record(s_out)
    t_end.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = t_start.elapsed_time(t_end) / args.steps
    del sets, dev_buf, dd

    peaks, peak_kind = _peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    gbs = job_throughput(alg_bytes, ms, world)
    gemm_gbs = alg_bytes / (gemm_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("mxfp4 (e2m1 x e2m1, e8m0 per 32) -> f32" if spec.x1_dtype == W.E2M1 and spec.x2_dtype == W.E2M1
                  else "mxfp8 (fp8 x fp8, e8m0 per 32) -> f32"), "data": "synthetic",
        "config": _config_dict(spec, counts, args.deterministic),
        "us_per_call": ms * 1e3, "us_per_call_min": min(call_ms) * 1e3,
        "us_per_call_p10_p50_p90": [round(float(x) * 1e3, 2) for x in _quantiles(call_ms, (0.1, 0.5, 0.9))],
        "us_per_call_profiled": statistics.mean(k[4] for k in kernel_ms) * 1e3, "tflops": flops / (ms * 1e-3) / 1e12,
        "roofline_fraction_call": gbs / world / hbm_peak,
        "kernels_ms": {"gemm": gemm_ms, "combine": comb_ms},
        "weight_prep_ms": prep_ms,
        "weight_prep_gbs": 2 * n_prep / (prep_ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": gemm_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gemm_gbs / hbm_peak, "traffic": _profiled_traffic(
                         spec.name, not (args.deterministic or spec.bias or args.tokens_hint)),
                     "kernel": "gemm_kernel (grouped GEMM + fused epilogue)",
                     "achieved_how": "algorithmic bytes / mean gemm_kernel duration (CUDA events on the call's stream, profiled pass)",
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)"},
        "e2e": {"value": alg_bytes / (e2e_serial_ms * 1e-3) / 1e9 * world, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_serial_ms,
                "mode": "serial: each step's copy in, call and copy out back to back, L2 flushed before",
                "pipelined_value": alg_bytes / (e2e_ms * 1e-3) / 1e9 * world, "pipelined_ms_per_step": e2e_ms,
                "pipelined_mode": "copy in, call and copy out of consecutive steps overlap on three streams"},
        "gpu_launches": args.steps * launches_per_call,
        "device_error_bits": bits,
        "clocks": clocks,
        "wall_s_timed": t_wall,
    }
    extras = set() if args.no_extras else set(args.extras.split(","))
    if "configs" in extras:
        line["configs"] = _sub_workloads(args, flush, spec, d, prep)
    if "route" in extras:
        line["route"] = _time_route(args, flush)
        if W.route_config(args.config).M == spec.M:
            line["layer"] = _time_layer(args, flush, prob, d, prep, ws, ms * 1e3, line["route"]["us_per_call"])
    if "ffn" in extras:
        line["ffn"] = _time_ffn(args, flush)
    if "mxfp4" in extras and spec.x1_dtype != W.E2M1:
        del prep
        torch.cuda.empty_cache()
        line["mxfp4"] = _time_mxfp4(args, flush)
    if rank == 0 and not args.no_cpu_baseline:
        cgbs, cdt, sample, cores = _cpu_baseline(spec, inp)
        line["cpu_baseline"] = {"value": cgbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--fp4", default="off", choices=["off", "c5", "e32"],
                    help="time the MXFP4 (E2M1) operator instead: the large shape, or its 32-expert copy")
    ap.add_argument("--e32", action="store_true",
                    help="time the 32-expert copy of the large workload (for full profiler captures)")
    ap.add_argument("--bias", action="store_true", help="add the per-expert bf16 bias input")
    ap.add_argument("--tokens-hint", type=int, default=0,
                    help="expected_tokens_per_expert tuning hint (fixes the token group width)")
    ap.add_argument("--deterministic", action="store_true")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (the other workloads, routing step, SwiGLU FFN, MXFP4 operator)")
    ap.add_argument("--extras", default="configs,route,ffn,mxfp4",
                    help="which side measurements to run (comma list of configs, route, ffn, mxfp4; route adds the "
                         "routing + operator layer when the workload has a routing shape)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
