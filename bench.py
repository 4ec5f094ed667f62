#!/usr/bin/env python3
"""Benchmark: batched draft-token verification on GB300.

One step = one spec_verify call (every row of the hot path: row staging,
softmax statistics, ratio test, first-rejection reduction, residual mass,
final draw, outputs) over one batch of synthetic logits already resident in
HBM.  Default workload: B=1024 sequences, K_b ~ U{1..8}, V=128256, bf16
logits ~N(0, 2^2), draft = target + N(0, 1), half the sequences at T=1 and
half greedy.  `--workload N` selects another of the benchmark workloads.

Prints one JSON line (rank 0).  Under torchrun every rank verifies its own
batch of the same shape (weak scaling, no collective on the data path); the
timing is the max over ranks.

`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "verified draft positions/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "positions/s"
KERNEL_SOURCES = ["speculative_decoding_verification_04_gb300/csrc/spec_verify.cu",
                  "speculative_decoding_verification_04_gb300/csrc/sv_sweep.cuh",
                  "speculative_decoding_verification_04_gb300/csrc/sv_common.cuh",
                  "speculative_decoding_verification_04_gb300/csrc/sv_ptx.cuh"]
WORKLOAD_TEXT = {
    0: "B=64 K=4 V=5 fp32 N(0,1) draft+N(0,1) T=1",
    1: "B=1 K=4 V=32000 bf16 N(0,2^2) draft+N(0,1) T=1",
    2: "B=64 K=5 V=128256 bf16 N(0,3^2) draft+N(0,0.5^2) T=1",
    3: "B=256 K=8 V=151936 fp32 N(0,2^2) draft+N(0,1.5^2) T=0.7",
    4: "B=1024 K_b~U{1..8} V=128256 bf16 N(0,2^2) draft+N(0,1^2) half T=1 half greedy",
}


def _source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def _peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(hbm_gbs=6800.0, source="fallback")


def _profile_traffic(widx: int):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel source; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = _source_hash()
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f)).read()
        m_w = re.search(r"^bench_workload:\s*(\d+)\s*$", text, re.M)
        m_h = re.search(r"^kernel_source_sha256_16:\s*([0-9a-f]+)\s*$", text, re.M)
        m_b = re.search(r"^dram_bytes_per_launch:\s*([0-9]+)\s*$", text, re.M)
        if m_w and m_h and m_b and int(m_w.group(1)) == widx and m_h.group(1) == want:
            return int(m_b.group(1))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=max(smax), samples=len(sm),
                    reasons=sorted(reasons))


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(dist, value: float, device) -> float:
    """The largest of every rank's value (the job takes as long as its slowest
    rank); the value itself on a single rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _whole_job_rate(world: int, units_per_rank_step: int, steps: int, seconds: float) -> float:
    """Units all ranks processed per second: every rank verifies its own batch
    of the same shape (replicas, weak scaling), timed by the slowest rank."""
    return world * units_per_rank_step * steps / seconds


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(widx: int, step_s: float, host=None):
    """Pick n (first n sequences of the workload) so one oracle pass over them
    takes about `step_s` seconds; returns the host inputs."""
    import oracle
    B = W.SPECS[widx].B
    n = min(B, 4)
    while True:
        inp = host(n) if host else W.make_spec_host(widx, B=n)
        t0 = time.perf_counter()
        oracle.verify_inputs(inp)
        dt = time.perf_counter() - t0
        if dt >= 0.25 * step_s or n >= B:
            break
        n = min(B, max(n + 1, int(n * min(16.0, 0.3 * step_s / max(dt, 1e-4)))))
    if dt < step_s and n < B:
        n = min(B, max(n, int(n * step_s / max(dt, 1e-4))))
        inp = host(n) if host else W.make_spec_host(widx, B=n)
    return inp, n


def oracle_rate(inp):
    """Single-thread oracle throughput on host inputs: (positions/s, seconds)."""
    import oracle
    t0 = time.perf_counter()
    oracle.verify_inputs(inp)
    dt = time.perf_counter() - t0
    return float(np.sum(inp["K"])) / dt, dt


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline lines."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                vendor = next((ln.split(":", 1)[1].strip() for ln in out.splitlines()
                               if ln.split(":")[0].strip() == "Vendor ID"), "")
                return f"{vendor} {line.split(':', 1)[1].strip()}".strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            return fields["model name"]
        if "CPU part" in fields:
            return f"CPU implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rate_cores(inp, threads: int, results: list | None = None):
    """Oracle throughput with the batch cut into `threads` contiguous shards of
    sequences run at once (the oracle's C loop runs outside the GIL; the
    oracle itself is unchanged): (positions/s, seconds).  The shards' results
    are appended to `results` when given."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    B = int(len(inp["K"]))
    cuts = np.linspace(0, B, max(1, min(threads, B)) + 1).astype(int)
    keys = ("target", "draft", "tokens", "uniforms", "temperature", "K")
    shards = [dict({k: inp[k][a:b] for k in keys}, dtype=inp["dtype"])
              for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=len(shards)) as ex:
        list(ex.map(lambda _: None, range(len(shards))))
        t0 = time.perf_counter()
        parts = list(ex.map(oracle.verify_inputs, shards))
        dt = time.perf_counter() - t0
    if results is not None:
        results.extend(parts)
    return float(np.sum(inp["K"])) / dt, dt


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    widx = args.workload
    inp, n, how = None, 0, "host-generated with the same recipe"
    try:   # the whole batch of our arm, generated as it generates it (seeded, on the device), to host
        import torch
        if torch.cuda.is_available():
            dev = torch.device("cuda", 0)
            d = W.make_device(widx, dev)
            n = d["B"]
            inp = _rows_to_host(d, np.arange(n))
            del d
            torch.cuda.empty_cache()
            how = "generated on the device by the benchmark's own seeded recipe, copied to the host"
    except (ImportError, RuntimeError):
        inp = None
    if inp is None:
        inp, n = oracle_sample(widx, step_s=0.5)
    cores = host_cores()
    rates, secs = [], []
    for step in range(args.warmup + args.steps):
        rate, dt = oracle_rate_cores(inp, cores)
        if step >= args.warmup:
            rates.append(rate)
            secs.append(dt)
    value = float(statistics.median(rates))
    line = dict(
        impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus,
        steps=args.steps, warmup=args.warmup, ms_per_step=round(1e3 * statistics.median(secs), 3),
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
        config=dict(workload=WORKLOAD_TEXT[widx], bench_workload=widx, sample_sequences=n,
                    same_batch=bool(n == W.SPECS[widx].B)),
        cpu_baseline=dict(value=value, unit=UNIT, cores=cores, kind="oracle", cpu_model=cpu_model(),
                          sample=f"first {n} of {W.SPECS[widx].B} sequences of the workload "
                                 f"({int(np.sum(inp['K']))} positions) per step, {how}, cut into "
                                 f"{cores} shards of sequences run at once on {cores} threads "
                                 f"({platform.machine()})"),
        e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import speculative_decoding_verification_04_gb300 as sv

    world, rank, local = _dist()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    widx = args.workload

    d = W.make_device(widx, dev, B=args.sequences)
    B, Kmax, V = d["B"], d["Kmax"], d["V"]
    K = np.asarray(d["K"], np.int32)
    ldtype = d["dtype"]
    dcode = sv.SV_DTYPE_BF16 if ldtype == "bf16" else sv.SV_DTYPE_F32
    ws = sv.Workspace(B, Kmax, V, dcode, dev)
    out_t = torch.empty((B, Kmax + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    call_args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    stream = torch.cuda.current_stream()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # The per-step flush also keeps the host ahead of the device: writing 1 GiB
    # takes longer than one step's host-side enqueue, so no host gap lands
    # between the step's events.
    flush = torch.empty(max(2 * l2, 1 << 30), dtype=torch.uint8, device=dev)

    # the host copy of the temperatures a serving loop holds anyway: with it the
    # launch gives the greedy sequences to split clusters (same outputs)
    hint = None if args.no_temperature_hint else np.asarray(d["temperature_host"], np.float32)

    def step(verify_all=False, use_hint=True):
        if verify_all:
            sv.spec_verify_ex(*call_args, ws, verify_all=True, out_tokens=out_t,
                              out_num_accepted=out_n)
        elif hint is not None and use_hint:
            sv.spec_verify_ex(*call_args, ws, out_tokens=out_t, out_num_accepted=out_n,
                              temperature_host=hint)
        else:
            sv.spec_verify_ws(*call_args, ws, out_tokens=out_t, out_num_accepted=out_n)

    def timed(nsteps, verify_all=False, use_hint=True):
        evs = []
        for _ in range(nsteps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step(verify_all, use_hint)
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    nacc = out_n.cpu().numpy()
    pos_per_step = int(K.sum())
    bytes_need = W.bytes_needed(K, d["temperature_host"], nacc, V, d["dtype"], Kmax)
    bytes_all = W.bytes_all_rows(K, d["temperature_host"], V, d["dtype"], Kmax)

    def load_for(seconds):
        """The same flushed step back to back for `seconds` (untimed)."""
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(25):
                flush.fill_(1)
                step()
            torch.cuda.synchronize()

    # ---- timed region ----
    # nvidia-smi samples every 200 ms while the timed steps take a few ms: the
    # same step runs back to back for ~1.5 s before and ~0.5 s after them, so
    # the clock samples see the load the timed steps run under
    clocks = ClockSampler(local) if rank == 0 and not args.no_clock_window else None
    if clocks:
        load_for(1.5)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("sv_timed")
    times = timed(args.steps)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    if clocks:
        load_for(0.5)
    clk = clocks.stop() if clocks else None
    if clk:
        clk["window"] = ("sampled every 200 ms while the timed step ran back to back for ~2 s "
                         "around the timed steps")
    total_ms = _max_over_ranks(dist, float(sum(times)), dev)
    ms_per_step = total_ms / args.steps
    value = _whole_job_rate(world, pos_per_step, args.steps, total_ms / 1e3)
    errs = sv.sv_workspace_errors(ws)

    # verify-every-row variant of the same step (same outputs, all bytes read)
    times_all = timed(max(3, args.steps // 2), verify_all=True)
    ms_all = statistics.median(times_all)
    # the same step without the temperature hint (spec_verify_ws: no split)
    nacc_hinted = out_n.cpu().numpy()
    times_plain = timed(max(3, args.steps // 2), use_hint=False) if hint is not None else times
    ms_plain = statistics.median(times_plain)
    torch.cuda.synchronize()
    plain_same = bool(np.array_equal(out_n.cpu().numpy(), nacc_hinted))
    geometry = sv.sv_geometry(B, Kmax, V, dcode)

    peaks = _peaks()
    med_ms = statistics.median(times)
    achieved = bytes_need / (med_ms / 1e3) / 1e9
    traffic = _profile_traffic(widx) if args.sequences is None else None
    roofline = dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(achieved / peaks["hbm_gbs"], 4), traffic=traffic,
                    bytes_algorithmic=bytes_need, peak_source=peaks["source"],
                    traffic_ratio=round(traffic / bytes_need, 4) if traffic else None,
                    frac_of_nominal_8000_gbs=round(achieved / 8000.0, 4),
                    kernel="sv_sweep_kernel",
                    duration=("CUDA events around each spec_verify_ex call with the host "
                              "temperature copy: " if hint is not None else
                              "CUDA events around each spec_verify_ws call: ") +
                             "the 1-kernel step plus its 16-byte counter reset")

    # ---- end to end through the host entry point (pinned buffers) ----
    e2e = None
    if rank == 0 or world > 1:
        def pinned(t):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            return h
        h_t, h_d = pinned(d["target"]), pinned(d["draft"])
        h_tok, h_uni, h_tmp = pinned(d["tokens"]), pinned(d["uniforms"]), pinned(d["temperature"])
        staging = torch.empty(sv.sv_host_staging_size(B, Kmax, V, dcode), dtype=torch.uint8,
                              device=dev)
        h_ot = torch.empty((B, Kmax + 1), dtype=torch.int32, pin_memory=True)
        h_on = torch.empty((B,), dtype=torch.int32, pin_memory=True)
        host_args = (h_t, h_d, h_tok, h_uni, h_tmp, K, staging)
        sv.spec_verify_host(*host_args, out_tokens=h_ot, out_num_accepted=h_on)
        n_e2e = max(3, min(args.steps, 8))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            sv.spec_verify_host(*host_args, out_tokens=h_ot, out_num_accepted=h_on)
        e2e_s = _max_over_ranks(dist, (time.perf_counter() - t0) / n_e2e, dev)
        same = bool(np.array_equal(h_on.numpy(), nacc))
        # page-locked logits are read in place by the kernel over the host
        # link: the logit rows the method reaches (bytes_need) cross it; the
        # tokens, uniforms and temperatures are copied
        h2d = bytes_need + sum(x.numel() * x.element_size() for x in (h_tok, h_uni, h_tmp))
        d2h = h_ot.numel() * 4 + h_on.numel() * 4
        # the host link's rate for a plain copy of the same pinned logits (copy
        # engine, timed in this run): what the e2e step's transfers are bound by
        src = h_t.view(torch.uint8).reshape(-1)
        dst = staging[:src.numel()]
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        dst.copy_(src, non_blocking=True)
        c1.record()
        torch.cuda.synchronize()
        link_peak = src.numel() / (c0.elapsed_time(c1) * 1e-3) / 1e9
        link_ach = h2d / e2e_s / 1e9
        e2e = dict(value=_whole_job_rate(world, pos_per_step, 1, e2e_s), unit=UNIT, h2d_bytes_per_step=h2d,
                   d2h_bytes_per_step=d2h, ms_per_step=round(e2e_s * 1e3, 3),
                   matches_device_run=same, api="spec_verify_host",
                   logits="page-locked host memory, read in place by the kernel (the rows the method "
                          "reaches); the other inputs copied, outputs copied back, every step",
                   link=dict(achieved_gbs=round(link_ach, 1), peak_gbs=round(link_peak, 1),
                             frac=round(link_ach / link_peak, 3),
                             peak_source=f"a plain {src.numel() / 1e9:.2f} GB host-to-device copy of "
                                         f"the same pinned target logits, timed in this run"))
        del h_t, h_d, staging

    # ---- CPU oracle baseline on a bounded sample (rank 0, N=1 only) ----
    cpu = None
    parity = None
    if world == 1 and not args.no_cpu_baseline:
        def host_rows(n):
            return _rows_to_host(d, np.arange(n))
        inp, n = oracle_sample(widx, step_s=12.0, host=host_rows)
        rate1, dt1 = oracle_rate(inp)
        cores = host_cores()
        parts = []
        rate, dt = oracle_rate_cores(inp, cores, parts)
        cpu = dict(value=rate, unit=UNIT, cores=cores, kind="oracle", cpu_model=cpu_model(),
                   sample=f"first {n} of {B} sequences of this workload "
                          f"({int(np.sum(inp['K']))} positions) cut into {cores} shards of "
                          f"sequences run at once on {cores} threads ({platform.machine()}), "
                          f"{dt:.2f} s",
                   single_thread=dict(value=rate1, seconds=round(dt1, 2)))
        parity = _parity(parts, out_t.cpu().numpy()[:n], nacc[:n])

    # ---- the other workloads of the set, timed the same way (rank 0, N=1) ----
    others = None
    if world == 1 and widx == 4 and args.sequences is None and not args.no_other_workloads:
        del d, call_args, ws, out_t, out_n
        torch.cuda.empty_cache()
        others = {}
        for key in ("0", "0-toy", "1", "2", "3"):
            if key == "0-toy":
                dw = _host_to_device(W.make_toy(200_000, seed=1000), dev)
            elif key == "0":
                dw = _host_to_device(W.make_spec_host(0), dev)
            else:
                dw = W.make_device(int(key), dev)
            name = ("the p/q toy pair x200000 K=1 V=5 fp32 T=1" if key == "0-toy"
                    else WORKLOAD_TEXT[int(key)])
            others[key] = _time_workload(sv, dw, name, max(5, args.steps // 2), flush, stream, peaks)
            del dw
            torch.cuda.empty_cache()

    if rank == 0:
        line = dict(
            metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
            warmup=args.warmup, ms_per_step=round(ms_per_step, 5), higher_is_better=True,
            scaling="weak", vs_baseline=None, dtype="f32", data="synthetic",
            config=dict(workload=WORKLOAD_TEXT[widx] if args.sequences is None
                        else f"first {B} sequences of: {WORKLOAD_TEXT[widx]}",
                        bench_workload=widx, logits=ldtype,
                        B=B, Kmax=Kmax, V=V, positions_per_step=pos_per_step,
                        temperature_hint=hint is not None,
                        l2="flushed before every step (1 GiB write, > 2x L2)", parallelism=f"dp{world}"),
            roofline=roofline, cpu_baseline=cpu, e2e=e2e, gpu_launches=args.steps,
            clocks=clk,
            detail=dict(
                mean_accepted=float(np.mean(nacc)), bytes_needed=bytes_need,
                rows_per_s=round(bytes_need / (V * (2 if ldtype == "bf16" else 4)) / (med_ms / 1e3), 1),
                bytes_all_rows=bytes_all, ms_median=round(med_ms, 5),
                ms_min=round(min(times), 5),
                without_temperature_hint=dict(ms_median=round(ms_plain, 5),
                                              frac=round(bytes_need / (ms_plain / 1e3) / 1e9 /
                                                         peaks["hbm_gbs"], 4),
                                              same_outputs=plain_same),
                verify_all=dict(ms_median=round(ms_all, 5),
                                gbs=round(bytes_all / (ms_all / 1e3) / 1e9, 1),
                                frac=round(bytes_all / (ms_all / 1e3) / 1e9 / peaks["hbm_gbs"], 4)),
                device_errors=errs, kernel_source_sha256_16=_source_hash(),
                geometry=geometry, parity=parity, workloads=others))
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_sample(args):
    """The draft-side sampler (spec_sample): one token per row of the
    workload's row-0 target logits [B, V], L2 flushed before every step.  An
    auxiliary measurement beside the verification headline."""
    import torch

    import speculative_decoding_verification_04_gb300 as sv

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d = W.make_device(args.workload, dev, B=args.sequences)
    B, V = d["B"], d["V"]
    code = sv.SV_DTYPE_BF16 if d["dtype"] == "bf16" else sv.SV_DTYPE_F32
    logits = d["target"][:, 0, :].contiguous()
    uni = d["uniforms"][:, 0].contiguous()
    temp = d["temperature"]
    ws = torch.empty(sv.sv_sample_workspace_size(B, V, code), dtype=torch.uint8, device=dev)
    out = torch.empty(B, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 1 << 30), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        sv.spec_sample(logits, uni, temp, workspace=ws, out_tokens=out)
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sv.spec_sample(logits, uni, temp, workspace=ws, out_tokens=out)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(times)
    s_el = 2 if d["dtype"] == "bf16" else 4
    nbytes = B * V * s_el
    peaks = _peaks()
    achieved = nbytes / (med / 1e3) / 1e9
    line = dict(metric="sampled rows/sec (spec_sample, one draw per row)", value=B / (med / 1e3),
                unit="rows/s", n_gpus=1, steps=args.steps, warmup=args.warmup, ms_per_step=med,
                higher_is_better=True, dtype=d["dtype"], data="synthetic",
                config=dict(workload=f"row 0 of each sequence of: {WORKLOAD_TEXT[args.workload]}",
                            B=B, V=V, l2="flushed before every step"),
                roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                              unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                              bytes_algorithmic=nbytes, kernel="sv_sweep_kernel"),
                gpu_launches=args.steps)
    print(json.dumps(line))
    return 0


def run_tree(args):
    """Token-tree verification (spec_verify_tree): B = 256 full binary trees
    of 15 nodes (3 levels of proposals), V = 128256 bf16 target logits
    N(0, 2^2), draft = target + N(0, 1), T = 1, the proposals drawn from the
    draft by Gumbel-max on the device; L2 flushed before every step."""
    import torch

    import speculative_decoding_verification_04_gb300 as sv

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B = args.sequences or 256
    V, N = 128256, 15
    parent = torch.from_numpy(W.full_tree(2, 3)).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1005)
    tgt = (torch.randn((B, N, V), generator=g, device=dev) * 2.0).to(torch.bfloat16)
    drf = (tgt.float() + torch.randn((B, N, V), generator=g, device=dev)).to(torch.bfloat16)
    tok = torch.zeros((B, N), dtype=torch.int32, device=dev)
    for n in range(1, N):
        gum = -torch.log(-torch.log(torch.rand((B, V), generator=g, device=dev).clamp_(1e-30, 1.0)))
        tok[:, n] = torch.argmax(drf[:, int(parent[n])].float() + gum, dim=-1).to(torch.int32)
        del gum
    uni = torch.rand((B, N), generator=g, device=dev)
    temp = torch.ones(B, device=dev)
    par = parent.to(torch.int32).repeat(B, 1).contiguous()
    nn = torch.full((B,), N, dtype=torch.int32, device=dev)
    ws = torch.empty(int(sv.library().sv_tree_workspace_size()), dtype=torch.uint8, device=dev)
    ot = torch.empty((B, N), dtype=torch.int32, device=dev)
    op = torch.empty((B, N), dtype=torch.int32, device=dev)
    ol = torch.empty((B,), dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 1 << 30), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        sv.spec_verify_tree(tgt, drf, tok, par, uni, temp, nn, workspace=ws, out_tokens=ot,
                            out_path=op, out_len=ol)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    med = statistics.median([a.elapsed_time(b) for a, b in evs])
    # algorithmic bytes: every node the walk visits reads its target row, and
    # its draft row when it has children (all nodes are sampling nodes)
    path = op.cpu().numpy()
    lens = ol.cpu().numpy()
    par_h = W.full_tree(2, 3)
    has_kids = np.array([np.any(par_h == v) for v in range(N)])
    rows = 0
    for b in range(B):
        visited = [0] + [int(x) for x in path[b, :max(int(lens[b]), 0)]]
        rows += sum(2 if has_kids[v] else 1 for v in visited)
    nbytes = rows * V * 2
    peaks = _peaks()
    achieved = nbytes / (med / 1e3) / 1e9
    line = dict(metric="tree proposals/sec (spec_verify_tree)", value=B * (N - 1) / (med / 1e3),
                unit="proposals/s", n_gpus=1, steps=args.steps, warmup=args.warmup, ms_per_step=med,
                higher_is_better=True, dtype="bf16", data="synthetic",
                config=dict(workload=f"B={B} full binary trees of {N} nodes, V={V} bf16 N(0,2^2) "
                                     f"draft+N(0,1^2) T=1", l2="flushed before every step",
                            mean_kept=float(np.mean(lens))),
                roofline=dict(bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                              unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                              bytes_algorithmic=int(nbytes), kernel="sv_tree_kernel"),
                gpu_launches=args.steps)
    print(json.dumps(line))
    return 0


def _parity(parts, got_t, got_n) -> dict:
    """The GPU's outputs on the oracle's sample against the oracle's: hard
    mismatches (outside the oracle's tie flag, must be 0), the oracle's ties
    (a uniform within 1e-6 of a threshold or CDF boundary) and the ties on
    which the two differ."""
    ref_t = np.concatenate([p["out_tokens"] for p in parts])
    ref_n = np.concatenate([p["num_accepted"] for p in parts])
    tie = np.concatenate([p["tie"] for p in parts])
    bad = (ref_n != got_n) | np.any(ref_t != got_t, axis=1)
    return dict(sequences_checked=int(len(tie)), hard_mismatch=int((bad & ~tie).sum()),
                ties=int(tie.sum()), tie_mismatch=int((bad & tie).sum()))


def _host_to_device(inp, dev) -> dict:
    """A host-generated workload (numpy) on the device, in the layout
    make_device returns."""
    import torch
    out = dict(inp)
    for k in ("target", "draft"):
        a = np.ascontiguousarray(inp[k])
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if inp["dtype"] == "bf16" \
            else torch.from_numpy(a.astype(np.float32))
        out[k] = t.to(dev)
    out["tokens"] = torch.from_numpy(np.ascontiguousarray(inp["tokens"], np.int32)).to(dev)
    out["uniforms"] = torch.from_numpy(np.ascontiguousarray(inp["uniforms"], np.float32)).to(dev)
    out["temperature"] = torch.from_numpy(np.ascontiguousarray(inp["temperature"], np.float32)).to(dev)
    out["temperature_host"] = np.asarray(inp["temperature"], np.float32)
    return out


def _time_workload(sv, d, name, steps, flush, stream, peaks) -> dict:
    """One workload of the set through spec_verify_ws, timed as the headline
    (L2 flushed before every step, CUDA events on the launching stream)."""
    import torch
    B, Kmax, V = d["B"], d["Kmax"], d["V"]
    K = np.asarray(d["K"], np.int32)
    dcode = sv.SV_DTYPE_BF16 if d["dtype"] == "bf16" else sv.SV_DTYPE_F32
    ws = sv.Workspace(B, Kmax, V, dcode, d["target"].device)
    out_t = torch.empty((B, Kmax + 1), dtype=torch.int32, device=d["target"].device)
    out_n = torch.empty((B,), dtype=torch.int32, device=d["target"].device)
    args = (d["target"], d["draft"], d["tokens"], d["uniforms"], d["temperature"], K)
    for _ in range(3):
        flush.fill_(1)
        sv.spec_verify_ws(*args, ws, out_tokens=out_t, out_num_accepted=out_n)
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        sv.spec_verify_ws(*args, ws, out_tokens=out_t, out_num_accepted=out_n)
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    med = statistics.median(times)
    nacc = out_n.cpu().numpy()
    need = W.bytes_needed(K, d["temperature_host"], nacc, V, d["dtype"], Kmax)
    gbs = need / (med / 1e3) / 1e9
    return dict(workload=name, B=B, Kmax=Kmax, V=V, logits=d["dtype"], steps=steps, ms_median=round(med, 5),
                ms_min=round(min(times), 5), positions_per_s=float(K.sum()) / (med / 1e3),
                bytes_needed=int(need), gbs=round(gbs, 1), frac=round(gbs / peaks["hbm_gbs"], 4),
                mean_accepted=float(np.mean(nacc)), device_errors=sv.sv_workspace_errors(ws),
                geometry=sv.sv_geometry(B, Kmax, V, dcode))


def _rows_to_host(d, seqs):
    import torch
    idx = torch.as_tensor(np.asarray(seqs), device=d["target"].device, dtype=torch.long)

    def host(t):
        t = t.index_select(0, idx).cpu()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    return dict(target=host(d["target"]), draft=host(d["draft"]), dtype=d["dtype"],
                tokens=host(d["tokens"]), uniforms=host(d["uniforms"]),
                temperature=host(d["temperature"]), K=np.asarray(d["K"])[np.asarray(seqs)])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clock-window", action="store_true",
                    help="skip the ~2 s of back-to-back steps that let the clock samples see the "
                         "load (profiling captures)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only the selected workload (the default run also times "
                         "workloads 0-3 and the 200k toy pair into detail.workloads)")
    ap.add_argument("--no-temperature-hint", action="store_true",
                    help="time spec_verify_ws (no host copy of the temperatures, so no split "
                         "clusters) instead of spec_verify_ex with temperature_host")
    ap.add_argument("--sequences", type=int, default=None,
                    help="the workload's first N sequences only (profiling captures)")
    ap.add_argument("--op", choices=["verify", "sample", "tree"], default="verify",
                    help="sample: time the draft-side sampler (spec_sample); tree: token-tree "
                         "verification (spec_verify_tree)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "sample":
        return run_sample(args)
    if args.op == "tree":
        return run_tree(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
