"""Benchmark: selective-SSM prefill tokens/s on one GB300 (plus decode steps/s and the q8 reduction).

One step = one ssm_prefill over the Zamba-7B-like long-context layer (batch 1, 65536
tokens, d_inner 7168, d_state 16, conv 4; bf16 x/z/dt/B/C, fp32 A/D/states, fp32
out), the largest single-GPU workload, inputs resident in HBM, L2 flushed (a 2x-L2
buffer write) before every timed step, each step timed with CUDA events on the
launching stream.  ``--workload`` selects another prefill workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun, one rank per GPU) every rank runs its own replica of the
workload (the mixer shards by channel and by batch row with no exchange), the
ranks meet only at the timing barriers, and value = all ranks' tokens / the
slowest rank's time ("weak" scaling).  ``--impl reference`` times the fp64 CPU
oracle on this host's cores on the same workload instead.
Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

# The timed step's workload (--workload); the default is the Zamba-7B-like long-context layer.
WORKLOADS = {
    "mamba130m_like_prefill": dict(batch=4, seqlen=2048, d_inner=1536, dtype="bf16"),
    "tiny_mixer_fp32": dict(batch=1, seqlen=256, d_inner=64, dtype="fp32"),
    "falcon_mamba7b_like_slice_prefill": dict(batch=1, seqlen=16384, d_inner=2048, dtype="bf16"),
    "zamba7b_like_long_context_prefill": dict(batch=1, seqlen=65536, d_inner=7168, dtype="bf16"),
}
DEFAULT_WORKLOAD = "zamba7b_like_long_context_prefill"
WORKLOAD = dict(name=DEFAULT_WORKLOAD, d_state=16, d_conv=4, **WORKLOADS[DEFAULT_WORKLOAD])


def _set_workload(name):
    global WORKLOAD
    WORKLOAD = dict(name=name, d_state=16, d_conv=4, **WORKLOADS[name])


def _wdtype(w):
    import torch
    return torch.bfloat16 if w["dtype"] == "bf16" else torch.float32


def _config(w, world):
    """The workload as both arms report it."""
    return {"workload": w["name"], "batch": w["batch"], "seq_len": w["seqlen"], "d_inner": w["d_inner"],
            "d_state": 16, "d_conv": 4, "inputs": f"{w['dtype']} x/z/dt/B/C, fp32 params and states",
            "out": "fp32", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed before every timed step (write of a 2x-L2 buffer)"}


# Channels of the workload the oracle runs per timed sample (channels are independent, so the
# whole layer's rate is the sample's rate scaled by d_inner / channels): about 0.5 s per sample
# on 16 host cores for the long-context layer.
ORACLE_SAMPLE_CHANNELS = 1024


def _oracle_sample(inp, w):
    """CPU copies of the first ORACLE_SAMPLE_CHANNELS channels of (device) inputs, all tokens."""
    from selective_state_space_prefill_gb300.inputs import MixerInputs
    ds = min(w["d_inner"], ORACLE_SAMPLE_CHANNELS)
    kw = {k: getattr(inp, k)[:, :, :ds].contiguous().cpu() for k in ("x", "z", "dt")}
    kw.update({k: getattr(inp, k).cpu() for k in ("B", "C")})
    kw.update({k: getattr(inp, k)[:ds].contiguous().cpu() for k in ("A", "D", "dt_bias", "conv_w", "conv_b")})
    return MixerInputs(**kw), ds
METRIC = "prefill tokens/s and decode steps/s per layer; achieved HBM GB/s vs 8 TB/s"
UNIT = "tokens/s"


# ---------------------------------------------------------------- algorithmic cost model
def prefill_bytes(batch, L, D, in_es=2, out_es=4):
    """Bytes the prefill must move: x, z, dt in + out per (t, d); B, C per token; params per
    channel (A 64 + D, dt_bias, conv_b 12 + conv_w 16 = 92 B); final states per (b, d) (64 + 12 B)."""
    return (batch * L * D * (3 * in_es + out_es) + batch * L * 2 * 16 * in_es + D * 92 + batch * D * 76)


def prefill_fp32_ops(batch, L, D):
    """FP32-pipe operations the plain sequential recurrence needs: per (t, d, n) delta*A, (delta u)*B,
    the state FMA and the C readout FMA (4 x 16 = 64); per (t, d) ~20 for conv, SiLU, softplus, skip
    and gate arithmetic."""
    return batch * L * D * (4 * 16 + 20)


def decode_bytes(batch, D, in_es=2, out_es=4):
    """ssm state 64 B read + 64 B write, conv state 12 + 12 B, x/z/dt, out per (r, d); params per
    channel; B, C per request."""
    return batch * D * (128 + 24 + 3 * in_es + out_es) + D * 92 + batch * 2 * 16 * in_es


def q8_bytes(P, n, in_es=2, out_es=2):
    return P * n * in_es + n * out_es + n * 4 + ((n + 127) // 128) * 4


def max_over_ranks(seconds: float, device=None) -> float:
    """The slowest rank's time (all ranks call it; without a process group it is the identity)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_s: float) -> float:
    """Units processed by all ranks over the slowest rank's time (weak scaling: replicas)."""
    return world * units_per_rank / slowest_s


# DRAM bytes (read + write) of one k_prefill launch, from an ncu capture summarised under
# profiles/, valid only for the workload it was taken on and the prefill source it was taken
# with (first 16 hex digits of its sha256); anything else reports null.
PREFILL_NCU_TRAFFIC = {"workload": "zamba7b_like_long_context_prefill", "bytes": 3.02e9 + 1.85e9,
                       "prefill_cu_sha256_16": "b8bfb22367bf380d"}


def _prefill_traffic(workload):
    import hashlib
    src = ROOT / "selective_state_space_prefill_gb300" / "csrc" / "prefill.cu"
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    ok = workload == PREFILL_NCU_TRAFFIC["workload"] and digest == PREFILL_NCU_TRAFFIC["prefill_cu_sha256_16"]
    return PREFILL_NCU_TRAFFIC["bytes"] if ok else None


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tc_peak():
    """Measured dense bf16 tensor TFLOP/s (burst) from MEASURED_PEAKS.json, else the fallback 1900."""
    try:
        return float(json.loads((ROOT / "MEASURED_PEAKS.json").read_text())["bf16_tflops"])
    except Exception:
        return 1900.0


def _cpu_oracle_run(inp, budget_s, threads):
    """Run the fp64 oracle over the whole workload until `budget_s` has elapsed (at least once)."""
    import oracle
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                       inp.conv_b, n_threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return reps, el


# ---------------------------------------------------------------- reference arm (the oracle)
def run_reference(args):
    import torch
    rank, _, world = _dist()
    if rank != 0:
        return
    from selective_state_space_prefill_gb300.inputs import make_mixer_inputs
    import oracle
    w = WORKLOAD
    # the same seeded draws as the timed arm (its generator runs on the device when there is one)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_mixer_inputs(w["batch"], w["seqlen"], w["d_inner"], dtype=_wdtype(w), seed=0, device=gen_dev)
    smp, ds = _oracle_sample(inp, w)
    del inp
    threads = _host_cores()
    oracle.build()
    for _ in range(args.warmup):
        _cpu_oracle_run(smp, 0.0, threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _cpu_oracle_run(smp, 0.0, threads)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    tokens = w["batch"] * w["seqlen"] * args.steps * ds / w["d_inner"]
    value = tokens / total
    sample = (f"{ds} of {w['d_inner']} channels x {w['batch']} x {w['seqlen']} tokens per step (channels are "
              f"independent; tokens/s scaled by {w['d_inner']}/{ds})" if ds < w["d_inner"] else
              f"the whole workload (all {w['d_inner']} channels x {w['batch']} x {w['seqlen']} tokens) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) tokens; A=-(n+1), D=1, log-uniform dt_bias, U(-.5,.5) conv)",
        "config": _config(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, local, world = _dist()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libssm has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from selective_state_space_prefill_gb300 import build as ssm_build
    if not ssm_build.up_to_date():
        if world > 1:
            raise SystemExit("libssm.so is not built: run __graft_entry__.build() before torchrun")
        ssm_build.build()
    from selective_state_space_prefill_gb300 import binding as ssm
    from selective_state_space_prefill_gb300.inputs import make_mixer_inputs, make_partials, make_states, \
        make_decode_inputs, make_mixer_params

    w = WORKLOAD
    B, L, D = w["batch"], w["seqlen"], w["d_inner"]
    in_es = 2 if w["dtype"] == "bf16" else 4
    inp = make_mixer_inputs(B, L, D, dtype=_wdtype(w), seed=0, device=dev)
    out = torch.empty(B, L, D, device=dev, dtype=torch.float32)
    cso = torch.empty(B, 3, D, device=dev)
    sso = torch.empty(B, D, 16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)

    def step():
        ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                    out=out, conv_state_out=cso, ssm_state_out=sso, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush.fill_(float(k))          # evict the inputs from L2 between timed steps
            evs[k][0].record(stream)
            step()
            evs[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        time.sleep(0.25)
    step_ms = [a.elapsed_time(b) for a, b in evs]
    dev_s = sum(step_ms) / 1e3
    if world > 1:
        dist.barrier()
    dev_s = max_over_ranks(dev_s, dev)
    value = whole_job_rate(B * L * args.steps, world, dev_s)
    ms_per_step = 1e3 * dev_s / args.steps
    status = ssm.device_status(clear=True)

    # ---- roofline of the prefill kernel (the only kernel of the step)
    hbm_peak, peak_kind = _peaks()
    abytes = prefill_bytes(B, L, D, in_es=in_es)
    avg_s = statistics.mean(step_ms) / 1e3
    achieved_gbs = abytes / avg_s / 1e9
    props = torch.cuda.get_device_properties(dev)
    n_sm = props.multi_processor_count
    cs = clocks.summary()
    sm_max = cs["sm_max_mhz"] or 2070.0
    fp32_peak = n_sm * 128 * sm_max * 1e6 / 1e12           # TFLOP/s-equivalent: FP32-pipe lane-ops/s
    fp32_ach = prefill_fp32_ops(B, L, D) / avg_s / 1e12
    roofline = {"bound": "alu", "achieved": fp32_ach, "peak": fp32_peak, "unit": "T fp32-ops/s",
                "frac": fp32_ach / fp32_peak, "traffic": _prefill_traffic(w["name"]),
                "traffic_unit": "DRAM bytes per launch (ncu)",
                "kernel": "k_prefill", "peak_source": f"{n_sm} SMs x 128 FP32 lanes x {sm_max:.0f} MHz",
                "hbm": {"achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                        "frac": achieved_gbs / hbm_peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                        "algorithmic_bytes_per_launch": abytes}}

    # ---- end to end through the public call with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = bench_e2e(ssm, inp, dev, args.steps, world, B, L, D)

    # ---- decode steps/s (batch 1/8/64/256 x d_inner 8192, CUDA graph of 64 steps) and the q8 reduction
    extras = {}
    if not args.no_extras:
        extras["decode"] = bench_decode(ssm, dev, stream, hbm_peak)
        extras["q8"] = bench_q8(ssm, dev, stream, hbm_peak, flush)
        extras["q8_split"] = bench_q8_split(ssm, dev, stream, hbm_peak, flush)
        extras["prefill_other_workloads"] = bench_prefill_other(ssm, dev, stream, hbm_peak, flush)
        extras["decode_block"] = bench_decode_block(ssm, dev, stream, hbm_peak, flush)
        extras["out_proj"] = bench_out_proj(ssm, dev, stream, flush, _tc_peak())
        extras["decode_configs"] = bench_decode_configs(ssm, dev, stream, hbm_peak)
        extras["ssd"] = bench_ssd(ssm, dev, stream, hbm_peak, flush, _tc_peak())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        oracle.build()
        smp, ds = _oracle_sample(inp, w)
        threads = _host_cores()
        reps, el = _cpu_oracle_run(smp, args.cpu_seconds, threads)
        cpu = {"value": reps * B * L * ds / D / el, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": (f"{ds} of {D} channels x {B} x {L} tokens (tokens/s scaled by {D}/{ds}: channels are "
                          f"independent), {reps} run(s) in {el:.1f} s" if ds < D else
                          f"the whole workload (all {D} channels x {B} x {L} tokens), {reps} run(s) in {el:.1f} s")}
        cpu_inp = smp
        # one host thread on a channel sample (channels are independent, so the rate scales)
        import oracle as _orc
        n1 = min(16 if L > 8192 else 96, ds)
        t1 = time.perf_counter()
        _orc.prefill(cpu_inp.x, cpu_inp.z, cpu_inp.dt, cpu_inp.B, cpu_inp.C, cpu_inp.A, cpu_inp.D, cpu_inp.dt_bias,
                     cpu_inp.conv_w, cpu_inp.conv_b, channels=list(range(n1)), n_threads=1)
        t1 = time.perf_counter() - t1
        cpu["one_thread_value"] = B * L * n1 / D / t1
        cpu["one_thread_sample"] = f"{n1} of {D} channels x {B} x {L} tokens on 1 thread in {t1:.2f} s"
        # the other configurations on the same cores, on channel samples (channels are independent,
        # so a layer's rate is the sample's rate scaled by the channel ratio)
        from selective_state_space_prefill_gb300.inputs import make_decode_inputs, make_mixer_params, make_states
        other = {}
        for name, (Bo, Lo, Do, ds) in {"falcon_mamba7b_like_slice_L16384_d2048": (1, 16384, 2048, 512),
                                       "mamba130m_like_b4_L2048_d1536": (4, 2048, 1536, 1536)}.items():
            smp = make_mixer_inputs(Bo, Lo, ds, dtype=torch.bfloat16, seed=0)
            t2 = time.perf_counter()
            _orc.prefill(smp.x, smp.z, smp.dt, smp.B, smp.C, smp.A, smp.D, smp.dt_bias, smp.conv_w, smp.conv_b,
                         n_threads=threads)
            t2 = time.perf_counter() - t2
            other[name] = {"tokens_per_s": Bo * Lo * ds / Do / t2, "sample": f"{ds} of {Do} channels, {t2:.2f} s"}
        Bd, Dd = 256, 8192
        tok = make_decode_inputs(Bd, Dd, seed=Bd)
        par = make_mixer_params(Dd, seed=1)
        cs0, ss0 = make_states(Bd, Dd, seed=Bd)
        t3 = time.perf_counter()
        _orc.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                         par["conv_w"], par["conv_b"], cs0, ss0)
        t3 = time.perf_counter() - t3
        other["decode_batch256_d8192"] = {"steps_per_s": 1.0 / t3, "sample": f"one whole step, {t3:.3f} s"}
        cpu["other_workloads"] = other

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) tokens; A=-(n+1), D=1, log-uniform dt_bias, U(-.5,.5) conv)",
            "config": _config(w, world),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps, "clocks": {k: cs[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "wall_s_timed_region": t_wall, "device_status": status,
        }
        line.update(extras)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_e2e(ssm, inp, dev, steps, world, B, L, D):
    """The same prefill through the public call with host buffers: every step copies x/z/dt/B/C
    from pinned host memory and out plus both states back.  Copies of step k+1 and k-1 overlap
    the prefill of step k (three streams, two device buffer sets)."""
    import torch
    host = {k: getattr(inp, k).cpu().pin_memory() for k in ("x", "z", "dt", "B", "C")}
    dbuf = [{k: torch.empty_like(getattr(inp, k)) for k in host} for _ in range(2)]
    outs = [torch.empty(B, L, D, device=dev) for _ in range(2)]
    css = [torch.empty(B, 3, D, device=dev) for _ in range(2)]
    sss = [torch.empty(B, D, 16, device=dev) for _ in range(2)]
    hout = [torch.empty(B, L, D).pin_memory() for _ in range(2)]
    hcs = [torch.empty(B, 3, D).pin_memory() for _ in range(2)]
    hss = [torch.empty(B, D, 16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = (hout[0].numel() + hcs[0].numel() + hss[0].numel()) * 4
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    for e in comp_done + out_done:
        e.record(torch.cuda.current_stream(dev))

    def step(k):
        j = k % 2
        s_in.wait_event(comp_done[j])                 # input buffers j free again
        with torch.cuda.stream(s_in):
            for name in host:
                dbuf[j][name].copy_(host[name], non_blocking=True)
        in_done = ev()
        in_done.record(s_in)
        s_cmp.wait_event(in_done)
        s_cmp.wait_event(out_done[j])                 # output buffers j read back already
        d = dbuf[j]
        ssm.prefill(d["x"], d["z"], d["dt"], d["B"], d["C"], inp.A, inp.D, inp.dt_bias, inp.conv_w,
                    inp.conv_b, out=outs[j], conv_state_out=css[j], ssm_state_out=sss[j], stream=s_cmp)
        comp_done[j].record(s_cmp)
        s_out.wait_event(comp_done[j])
        with torch.cuda.stream(s_out):
            hout[j].copy_(outs[j], non_blocking=True)
            hcs[j].copy_(css[j], non_blocking=True)
            hss[j].copy_(sss[j], non_blocking=True)
        out_done[j].record(s_out)

    for k in range(3):
        step(k)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(steps):
        step(k)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    es = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
    return {"value": whole_job_rate(B * L * steps, world, es), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "note": "pinned host buffers; copies of neighbouring steps overlap the prefill (3 streams)"}


def bench_prefill_other(ssm, dev, stream, hbm_peak, flush):
    """Prefill tokens/s on the other prefill workloads: the batch-4 Mamba-130M-like layer, the
    unsplit 8192-channel Falcon-Mamba-like layer and one 2048-channel slice of it, and a batch-1
    Mamba-130M-like layer (5 timed launches each, L2 flushed before each).  Batch-1 rows
    are also timed with the sequence cut into parallel segments (ssm_prefill_segmented,
    seg_len from binding.suggest_seg_len) when they leave SMs idle."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_mixer_inputs
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    for name, (Bt, L, D) in {"mamba130m_like_b4_L2048_d1536": (4, 2048, 1536),
                             "falcon_mamba7b_like_unsplit_L16384_d8192": (1, 16384, 8192),
                             "falcon_mamba7b_like_slice_L16384_d2048": (1, 16384, 2048),
                             "mamba130m_like_batch1_L2048_d1536": (1, 2048, 1536)}.items():
        inp = make_mixer_inputs(Bt, L, D, dtype=torch.bfloat16, seed=0, device=dev)
        out = torch.empty(Bt, L, D, device=dev)
        cs, ss = torch.empty(Bt, 3, D, device=dev), torch.empty(Bt, D, 16, device=dev)
        seg = ssm.suggest_seg_len(Bt, L, D, n_sm)
        ws = None
        if seg is not None:
            ws = torch.empty(max(1, ssm.prefill_workspace_bytes(Bt, L, D, seg)), device=dev, dtype=torch.uint8)
        for seg_len in ([None] + ([seg] if seg is not None else [])):
            f = lambda: ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                                    inp.conv_b, out=out, conv_state_out=cs, ssm_state_out=ss, stream=stream,
                                    seg_len=seg_len, workspace=ws if seg_len else None)
            for _ in range(3):
                f()
            ts = []
            for k in range(5):
                flush.fill_(float(k))
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                f()
                b_.record(stream)
                ts.append((a, b_))
            torch.cuda.synchronize(dev)
            t = statistics.median(a.elapsed_time(b_) for a, b_ in ts) / 1e3
            gbs = prefill_bytes(Bt, L, D) / t / 1e9
            key = name if seg_len is None else f"{name}_segmented"
            res[key] = {"ms": 1e3 * t, "tokens_per_s": Bt * L / t, "GB_s": gbs, "frac_hbm": gbs / hbm_peak}
            if seg_len is not None:
                res[key].update({"seg_len": seg_len, "segments": -(-L // seg_len),
                                 "kernels": "k_prefill_agg + k_prefill_carry + k_prefill"})
        del inp, out, ws
        torch.cuda.empty_cache()
    return res


def bench_out_proj(ssm, dev, stream, flush, tc_peak):
    """One rank's out_proj partial on the tensor cores (bf16 in, fp32 accumulate, bf16 out plus
    per-128-block maxima): TFLOP/s against the measured bf16 tensor peak, L2 flushed before each
    of 10 timed launches.  cuBLAS (torch.matmul, bf16) on the same operands is timed as context."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_out_proj_inputs
    res = {}
    for name, (M, N, K) in {"falcon_mamba7b_like_rank_M16384_N4096_K2048": (16384, 4096, 2048),
                            "mamba130m_like_layer_M8192_N768_K1536": (8192, 768, 1536)}.items():
        y, W = make_out_proj_inputs(M, K, N, seed=0, device=dev)
        out = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        amax = torch.empty(M * N // 128, device=dev)
        times = {}
        for impl in ("ours", "cublas"):
            if impl == "ours":
                f = lambda: ssm.out_proj_partial(y, W, out=out, block_amax=amax, stream=stream)
            else:
                f = lambda: torch.matmul(y, W.t(), out=out)
            for _ in range(3):
                f()
            ts = []
            for k in range(10):
                flush.fill_(float(k))
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                f()
                b_.record(stream)
                ts.append((a, b_))
            torch.cuda.synchronize(dev)
            times[impl] = statistics.median(a.elapsed_time(b_) for a, b_ in ts) / 1e3
        flops = 2.0 * M * N * K
        t = times["ours"]
        res[name] = {"us": 1e6 * t, "TFLOP_s": flops / t / 1e12, "frac_tensor": flops / t / 1e12 / tc_peak,
                     "cublas_us": 1e6 * times["cublas"], "cublas_TFLOP_s": flops / times["cublas"] / 1e12}
        del y, W, out, amax
        torch.cuda.empty_cache()
    res["note"] = ("k_out_proj: tcgen05.mma kind::f16, 128x256 tiles, 4-stage TMA ring, TMEM accumulator; "
                   "frac_tensor against MEASURED_PEAKS.json bf16_tflops (burst); cuBLAS is context, not used")
    return res


def ssd_prefill_bytes(B, L, H, G, P=64, N=64, out_es=4):
    """Algorithmic bytes of one SSD prefill: bf16 xBC, z, dt read once, out written once, fp32
    params read once, final conv and SSM states written once."""
    Cx = H * P + 2 * G * N
    per_token = Cx * 2 + H * P * 2 + H * 2 + H * P * out_es
    params = Cx * 4 * 5 + H * 4 * 3
    states = B * (3 * Cx * 4 + H * P * N * 4)
    return B * L * per_token + params + states


def ssd_prefill_mma_flops(B, L, H, P=64, N=64, Q=128):
    """Tensor-core work of the chunked SSD form as the kernel runs it, per 128-token chunk and head:
    G = C B^T (128 x 128 x N) and Y_intra = M X (128 x 64 x 128), Y_inter = C S^T (128 x 64 x N),
    each three hi/lo products, and the state update (128 x N x 128) as four."""
    chunks = B * H * ((L + Q - 1) // Q)
    per_chunk = 2 * (3 * Q * Q * N + 3 * Q * P * Q + 3 * Q * P * N + 2 * 2 * P * N * Q)
    return chunks * per_chunk


def bench_ssd(ssm, dev, stream, hbm_peak, flush, tc_peak):
    """The SSD (Mamba-2-style) mixer: ssd_prefill on the Zamba2-2.7B-like layer (4 x 2048 tokens,
    80 heads of 64, d_state 64, one group) and on a Zamba2-7B-like batch-1 prompt (16384 tokens,
    112 heads), L2 flushed before each of 10 timed launches; ssd_decode_step at batch 64 and 256
    of the 80-head layer (CUDA graph of back-to-back steps, state [64 x 64] per request and head)."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_ssd_inputs, make_ssd_states
    res = {}
    for name, (B, L, H, G) in {"zamba2_2p7b_like_layer_b4_l2048_h80": (4, 2048, 80, 1),
                               "zamba2_7b_like_prompt_b1_l16384_h112": (1, 16384, 112, 1)}.items():
        inp = make_ssd_inputs(B, L, H, n_groups=G, seed=0, device=dev)
        out = torch.empty(B, L, 64 * H, device=dev)
        cso = torch.empty(B, 3, inp.channels, device=dev)
        sso = torch.empty(B, H, 64, 64, device=dev)
        ws = torch.empty(ssm.ssd_prefill_workspace_bytes(B, L, H, G), device=dev, dtype=torch.uint8)
        f = lambda: ssm.ssd_prefill(inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H,
                                    G, out=out, conv_state_out=cso, ssm_state_out=sso, workspace=ws, stream=stream)
        for _ in range(3):
            f()
        ts = []
        for k in range(10):
            flush.fill_(float(k))
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            f()
            b_.record(stream)
            ts.append((a, b_))
        torch.cuda.synchronize(dev)
        t = statistics.median(a.elapsed_time(b_) for a, b_ in ts) / 1e3
        byts = ssd_prefill_bytes(B, L, H, G)
        fl = ssd_prefill_mma_flops(B, L, H)
        res[name] = {"us": 1e6 * t, "tokens_per_s": B * L / t, "GB_s": byts / t / 1e9,
                     "frac_hbm": byts / t / 1e9 / hbm_peak, "mma_TFLOP_s": fl / t / 1e12,
                     "frac_tensor": fl / t / 1e12 / tc_peak}
        del inp, out, cso, sso, ws
        torch.cuda.empty_cache()
    H, G = 80, 1
    for batch in (64, 256):
        inp = make_ssd_inputs(batch, 1, H, n_groups=G, seed=batch, device=dev)
        cs, ss = (t.to(dev) for t in make_ssd_states(batch, H, 64, 64, inp.channels, seed=batch))
        xb, z, dt = inp.xBC[:, 0].contiguous(), inp.z[:, 0].contiguous(), inp.dt[:, 0].contiguous()
        out = torch.empty(batch, 64 * H, device=dev)
        steps = 32

        def one():
            ssm.ssd_decode_step(xb, z, dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G, cs, ss, out=out,
                                stream=torch.cuda.current_stream(dev))

        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            for _ in range(3):
                one()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(steps):
                one()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize(dev)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b_.record(stream)
        torch.cuda.synchronize(dev)
        t = a.elapsed_time(b_) / 1e3 / (reps * steps)
        Cx = inp.channels
        byts = batch * (H * 64 * 64 * 4 * 2 + 3 * Cx * 4 * 2 + Cx * 2 + 64 * H * 2 + H * 2 + 64 * H * 4)
        res[f"decode_b{batch}_h80"] = {"us_per_step": 1e6 * t, "steps_per_s": 1 / t, "GB_s": byts / t / 1e9,
                                       "frac_hbm": byts / t / 1e9 / hbm_peak}
        del g
    res["note"] = ("k_ssd_pre (B, C conv + hi/lo planes, delta and decay sums) + k_ssd_chunk (tcgen05: G = C B^T, M X, C S^T and the "
                   "state update on bf16 hi/lo operand pairs, fp32 TMEM accumulators; a producer warp issues "
                   "TMA and MMA, 16 worker warps the arithmetic; more rows than resident CTAs: one CTA per SM "
                   "on an equal span of all rows' chunks, state handed on where a row is cut).  frac_hbm is "
                   "against algorithmic bytes; "
                   "mma_TFLOP_s counts the hi/lo products the kernel issues (frac_tensor of the measured bf16 "
                   "peak); decode: k_ssd_decode + k_ssd_decode_shift per step, L2-resident state at batch 64")
    return res


def bench_decode_block(ssm, dev, stream, hbm_peak, flush, batch=64, T=8, D=8192):
    """ssm_decode_tokens: a T-token block per request (speculative / verification tokens)."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_mixer_inputs, make_states
    inp = make_mixer_inputs(batch, T, D, dtype=torch.bfloat16, seed=T, device=dev)
    cs, ss = (t.to(dev) for t in make_states(batch, D, seed=T))
    out = torch.empty(batch, T, D, device=dev)
    f = lambda: ssm.decode_tokens(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w,
                                  inp.conv_b, cs, ss, out=out, stream=stream)
    for _ in range(3):
        f()
    ts = []
    for k in range(10):
        flush.fill_(float(k))
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        f()
        b_.record(stream)
        ts.append((a, b_))
    torch.cuda.synchronize(dev)
    t = statistics.median(a.elapsed_time(b_) for a, b_ in ts) / 1e3
    nbytes = batch * D * (128 + 24) + batch * T * D * (3 * 2 + 4) + D * 92 + batch * T * 64
    return {"batch": batch, "tokens_per_request": T, "d_inner": D, "us": 1e6 * t,
            "tokens_per_s": batch * T / t, "GB_s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / hbm_peak}


def bench_decode(ssm, dev, stream, hbm_peak, steps=64, D=8192):
    import torch
    from selective_state_space_prefill_gb300.inputs import make_decode_inputs, make_mixer_params, make_states
    res = {}
    par = {k: v.to(dev) for k, v in make_mixer_params(D, seed=1).items()}
    for batch in (1, 8, 64, 256):
        tok = {k: v.to(dev) for k, v in make_decode_inputs(batch, D, seed=batch).items()}
        cs, ss = (t.to(dev) for t in make_states(batch, D, seed=batch))
        out = torch.empty(batch, D, device=dev)

        def one():
            ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                            par["conv_w"], par["conv_b"], cs, ss, out=out, stream=torch.cuda.current_stream(dev))

        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)
        with torch.cuda.stream(s):
            for _ in range(3):
                one()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(steps):
                one()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t = e0.elapsed_time(e1) / 1e3 / (reps * steps)
        gbs = decode_bytes(batch, D) / t / 1e9
        res[f"batch{batch}"] = {"steps_per_s": 1.0 / t, "us_per_step": 1e6 * t, "GB_s": gbs,
                                "frac_hbm": gbs / hbm_peak}
    # extended sweep (the bandwidth regime): single launches, L2 flushed before each
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, device=dev)
    for batch in (1024, 4096):
        tok = {k: v.to(dev) for k, v in make_decode_inputs(batch, D, seed=batch).items()}
        cs, ss = (t.to(dev) for t in make_states(batch, D, seed=batch))
        out = torch.empty(batch, D, device=dev)
        f = lambda: ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"],
                                    par["dt_bias"], par["conv_w"], par["conv_b"], cs, ss, out=out, stream=stream)
        for _ in range(3):
            f()
        ts = []
        for k in range(5):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        t = statistics.median(a.elapsed_time(b) for a, b in ts) / 1e3
        gbs = decode_bytes(batch, D) / t / 1e9
        res[f"batch{batch}"] = {"steps_per_s": 1.0 / t, "us_per_step": 1e6 * t, "GB_s": gbs, "frac_hbm": gbs / hbm_peak,
                                "timing": "extended size: single launch, L2 flushed before it"}
        del tok, cs, ss, out
    del flush
    torch.cuda.empty_cache()
    res["note"] = ("d_inner 8192, bf16 tokens, fp32 states in place; batch <= 256: CUDA graph of 64 back-to-back "
                   "steps, states of batch <= 64 stay L2-resident between steps; batch 1024/4096: extended sizes")
    return res


def bench_decode_configs(ssm, dev, stream, hbm_peak):
    """Decode steps/s at the long-context configurations' own shapes, batch 1: the Falcon-Mamba-
    like slice (d_inner 2048, 512 steps after its prefill) and the Zamba-like layer (d_inner 7168,
    16384 steps), each as one CUDA graph of that many back-to-back steps."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_decode_inputs, make_mixer_params, make_states
    res = {}
    for name, (D, steps) in {"falcon_mamba7b_like_slice_d2048_512_steps": (2048, 512),
                             "zamba7b_like_d7168_16384_steps": (7168, 16384)}.items():
        par = {k: v.to(dev) for k, v in make_mixer_params(D, seed=1).items()}
        tok = {k: v.to(dev) for k, v in make_decode_inputs(1, D, seed=2).items()}
        cs, ss = (t.to(dev) for t in make_states(1, D, seed=3))
        out = torch.empty(1, D, device=dev)
        s = torch.cuda.Stream(dev)
        s.wait_stream(stream)

        def one():
            ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"], par["dt_bias"],
                            par["conv_w"], par["conv_b"], cs, ss, out=out, stream=s)

        with torch.cuda.stream(s):
            for _ in range(3):
                one()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(steps):
                one()
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t = e0.elapsed_time(e1) / 1e3 / steps
        res[name] = {"steps_per_s": 1.0 / t, "us_per_step": 1e6 * t, "GB_s": decode_bytes(1, D) / t / 1e9}
        del g
    res["note"] = "batch 1, bf16 tokens, fp32 states in place; launch-bound (one 1 x d_inner step per kernel)"
    return res


def bench_q8(ssm, dev, stream, hbm_peak, flush, P=4, graph_calls=64):
    import torch
    from selective_state_space_prefill_gb300.inputs import make_partials
    res = {}
    for batch in (1, 8, 64, 256, 4096, 16384):
        n = batch * 4096
        parts = [p.to(dev) for p in make_partials(P, (batch, 1, 4096), dtype=torch.bfloat16, seed=batch)]
        out = torch.empty(batch, 1, 4096, device=dev, dtype=torch.bfloat16)
        sums = torch.empty(n, device=dev, dtype=torch.int32)
        scales = torch.empty((n + 127) // 128, device=dev)
        for _ in range(3):
            ssm.q8_reduce(parts, out=out, sums=sums, scales=scales, stream=stream)
        if batch <= 256:
            # a few microseconds per call: one launch is dominated by launch latency, so time a
            # CUDA graph of back-to-back calls; the operands (<= 10 MB) stay in L2 between calls
            s = torch.cuda.Stream(dev)
            s.wait_stream(stream)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(graph_calls):
                    ssm.q8_reduce(parts, out=out, sums=sums, scales=scales, stream=s)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 5
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            t = e0.elapsed_time(e1) / 1e3 / (reps * graph_calls)
            res[f"batch{batch}"] = {"us": 1e6 * t, "GB_s": q8_bytes(P, n) / t / 1e9,
                                    "timing": f"graph of {graph_calls} calls, L2-resident"}
            continue
        times = []
        for k in range(10):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ssm.q8_reduce(parts, out=out, sums=sums, scales=scales, stream=stream)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
        t = statistics.median(a.elapsed_time(b) for a, b in times) / 1e3
        gbs = q8_bytes(P, n) / t / 1e9
        res[f"batch{batch}"] = {"us": 1e6 * t, "GB_s": gbs, "frac_hbm": gbs / hbm_peak,
                                "timing": "single launch, L2 flushed before it"}
    res["note"] = ("P=4 bf16 partials [batch,1,4096], block 128, bf16 out + int32 sums + scales; "
                   "batch <= 256: CUDA graph of back-to-back calls with L2-resident operands, so GB_s there "
                   "is not an HBM figure; batch 4096 and 16384 (2^26 elements) are extended sizes showing the "
                   "bandwidth regime")
    return res


def bench_q8_split(ssm, dev, stream, hbm_peak, flush, P=4, batch=16384):
    """The rank-local halves of the 8-bit all-reduce on one rank's partial of the extended
    reduction size (bf16 [16384, 1, 4096], 2^26 elements): block maxima, shared-scale codes,
    and the sum of P = 4 ranks' codes with bf16 output and int32 sums.  Each kernel is timed
    alone (10 launches, L2 flushed before each) against the bytes it must move."""
    import torch
    from selective_state_space_prefill_gb300.inputs import make_partials
    n = batch * 4096
    nblk = n // 128
    parts = [p.to(dev) for p in make_partials(P, (batch, 1, 4096), dtype=torch.bfloat16, seed=batch)]
    amax = torch.empty(nblk, device=dev)
    codes = [torch.empty(batch, 1, 4096, device=dev, dtype=torch.int8) for _ in range(P)]
    scales = torch.empty(nblk, device=dev)
    out = torch.empty(batch, 1, 4096, device=dev, dtype=torch.bfloat16)
    sums = torch.empty(n, device=dev, dtype=torch.int32)
    ssm.q8_block_absmax(parts[0], out=amax, stream=stream)
    for p, c in zip(parts, codes):
        ssm.q8_quantize_shared(p, amax, codes=c, scales=scales, stream=stream)
    steps = {
        "block_absmax": (lambda: ssm.q8_block_absmax(parts[0], out=amax, stream=stream), 2 * n + 4 * nblk),
        "quantize_shared": (lambda: ssm.q8_quantize_shared(parts[0], amax, codes=codes[0], scales=scales,
                                                           stream=stream), 2 * n + n + 8 * nblk),
        "sum_dequant_P4": (lambda: ssm.q8_sum_dequant(codes, scales, out=out, sums=sums, stream=stream),
                           P * n + 2 * n + 4 * n + 4 * nblk),
    }
    res = {}
    for name, (f, nbytes) in steps.items():
        for _ in range(3):
            f()
        times = []
        for k in range(10):
            flush.fill_(float(k))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            f()
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize(dev)
        t = statistics.median(a.elapsed_time(b) for a, b in times) / 1e3
        gbs = nbytes / t / 1e9
        res[name] = {"us": 1e6 * t, "GB_s": gbs, "frac_hbm": gbs / hbm_peak}
    res["note"] = ("one rank's share of the quantized all-reduce across GPUs (q8_block_absmax, "
                   "q8_quantize_shared, q8_sum_dequant); the MAX all-reduce of the maxima and the "
                   "all-gather of the codes are the collectives between them")
    return res


def run_profile_target(which: str):
    """Launch one kernel 4 times (3 warm-up + 1 to capture) for ncu: the prefill on the bench
    workload, the segmented prefill of a batch-1 row, the decode step at batch 256 x d_inner
    8192, q8 over P=4 bf16 [4096, 1, 4096], the out_proj partial of the Falcon-Mamba-like
    rank (16384 x 4096 x 2048), the SSD prefill of the Zamba2-2.7B-like layer (4 x 2048
    tokens, 80 heads of 64, d_state 64, one group), or its decode step at batch 256."""
    import torch
    from selective_state_space_prefill_gb300 import build as ssm_build
    if not ssm_build.up_to_date():
        ssm_build.build()
    from selective_state_space_prefill_gb300 import binding as ssm
    from selective_state_space_prefill_gb300.inputs import (make_decode_inputs, make_mixer_inputs,
                                                            make_mixer_params, make_partials, make_states)
    dev = torch.device("cuda", 0)
    if which == "prefill":
        w = WORKLOAD
        inp = make_mixer_inputs(w["batch"], w["seqlen"], w["d_inner"], dtype=_wdtype(w), seed=0, device=dev)
        for _ in range(4):
            ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b)
    elif which == "prefill_seg":
        # batch-1 Falcon-Mamba-like slice (1 x 16384 x 2048) in 3 segments of 5504 tokens
        L, D, seg = 16384, 2048, 5504
        inp = make_mixer_inputs(1, L, D, dtype=torch.bfloat16, seed=0, device=dev)
        ws = torch.empty(ssm.prefill_workspace_bytes(1, L, D, seg), device=dev, dtype=torch.uint8)
        for _ in range(4):
            ssm.prefill(inp.x, inp.z, inp.dt, inp.B, inp.C, inp.A, inp.D, inp.dt_bias, inp.conv_w, inp.conv_b,
                        seg_len=seg, workspace=ws)
    elif which == "decode":
        D, B = 8192, 256
        par = {k: v.to(dev) for k, v in make_mixer_params(D, seed=1).items()}
        tok = {k: v.to(dev) for k, v in make_decode_inputs(B, D, seed=B).items()}
        cs, ss = (t.to(dev) for t in make_states(B, D, seed=B))
        out = torch.empty(B, D, device=dev)
        for _ in range(4):
            ssm.decode_step(tok["x"], tok["z"], tok["dt"], tok["B"], tok["C"], par["A"], par["D"],
                            par["dt_bias"], par["conv_w"], par["conv_b"], cs, ss, out=out)
    elif which == "ssd":
        from selective_state_space_prefill_gb300.inputs import make_ssd_inputs
        B, L, H, G = 4, 2048, 80, 1
        inp = make_ssd_inputs(B, L, H, n_groups=G, seed=0, device=dev)
        ws = torch.empty(ssm.ssd_prefill_workspace_bytes(B, L, H, G), device=dev, dtype=torch.uint8)
        for _ in range(4):
            ssm.ssd_prefill(inp.xBC, inp.z, inp.dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G,
                            workspace=ws)
    elif which == "ssd_decode":
        from selective_state_space_prefill_gb300.inputs import make_ssd_inputs, make_ssd_states
        B, H, G = 256, 80, 1
        inp = make_ssd_inputs(B, 1, H, n_groups=G, seed=B, device=dev)
        cs, ss = (t.to(dev) for t in make_ssd_states(B, H, 64, 64, inp.channels, seed=B))
        xb, z, dt = inp.xBC[:, 0].contiguous(), inp.z[:, 0].contiguous(), inp.dt[:, 0].contiguous()
        for _ in range(4):
            ssm.ssd_decode_step(xb, z, dt, inp.conv_w, inp.conv_b, inp.A, inp.D, inp.dt_bias, H, G, cs, ss)
    elif which == "out_proj":
        from selective_state_space_prefill_gb300.inputs import make_out_proj_inputs
        y, W = make_out_proj_inputs(16384, 2048, 4096, seed=0, device=dev)
        for _ in range(4):
            ssm.out_proj_partial(y, W)
    else:
        parts = [q.to(dev) for q in make_partials(4, (4096, 1, 4096), dtype=torch.bfloat16, seed=4096)]
        for _ in range(4):
            ssm.q8_reduce(parts)
    torch.cuda.synchronize()
    print(json.dumps({"profile_target": which, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD,
                    help="the prefill workload of the timed step (default: the Zamba-7B-like long-context layer)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--profile", choices=["prefill", "prefill_seg", "decode", "q8", "out_proj", "ssd", "ssd_decode"],
                    default=None,
                    help="only launch one kernel 4 times (for an ncu capture) and exit")
    args = ap.parse_args()
    _set_workload(args.workload)
    if args.profile:
        run_profile_target(args.profile)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
