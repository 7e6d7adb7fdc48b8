#!/usr/bin/env python
"""Verify-round benchmark on GB300: verified logit rows/s and achieved HBM GB/s.

A step is one verify round over one batch of synthetic input: the row budget
(host), the fused verify-accept kernel and, for workloads with recurrent
state, the state commit.  Steps run from a captured CUDA graph (the kernels
take microseconds, so launching them one by one from Python would measure the
launcher); consecutive steps rotate over enough input sets that a set's logits
have left the 129 MB L2 before it comes round again.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle on the same workload

Under torchrun (N > 1) every rank verifies its own batch (lanes are
independent, so there is no collective on the data path); the time is the
maximum over ranks and ``value`` counts the rows of all ranks.
"""

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verified logit rows/sec and achieved HBM GB/s (% of GB300 peak) per verify round"
UNIT = "rows/s"
L2_BYTES = 129 * 2 ** 20
DEFAULT_WORKLOAD = workloads.RAGGED_MIXED_B128  # the largest single-GPU workload
GRAPH_STEPS = 500          # steps per captured graph
SOAK_SECONDS = 1.0         # untimed replays before the timed region (clocks settle, samples exist)
FALLBACK_HBM_GBS = 6800.0  # used only if MEASURED_PEAKS.json is absent


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The files the verify and commit kernels are built from (the profiled kernels).
KERNEL_SOURCES = ["commit_kernel.cuh", "device_ptx.cuh", "philox.cuh", "spec_verify.cu", "verify_kernel.cuh",
                  "verify_variants.h", "verify_w20.cu", "verify_w20p5.cu"]


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verify_bf16_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "spec_verify.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        # A capture of a smaller case of the workload states the factor that
        # scales its per-launch traffic to the full launch.
        return int(float(fields["dram_bytes_per_launch"]) * float(fields.get("traffic_scale", "1")))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device_index)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


def round_bytes(r):
    """Algorithmic bytes of one verify launch: logits rows read, metadata, outputs."""
    lens = r.draft_lens.cpu().numpy().astype(np.int64)
    temps = r.temperatures.cpu().numpy()
    esize = r.target.element_size()
    target_rows = int((lens + 1).sum())
    draft_rows = int(lens[temps > 0].sum())
    logits = (target_rows + draft_rows) * r.vocab * esize
    meta = 4 * (r.rows + r.lanes + (r.lanes + 1) + r.lanes)   # tokens, lens, offsets, temps
    out = 4 * (r.lanes + r.rows + r.lanes)                     # committed, out_tokens, status
    return logits + meta + out, target_rows


def commit_bytes(r):
    per_lane = r.live[0].numel() * r.live.element_size()
    return 2 * per_lane * r.lanes + 8 * r.lanes


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Bench:
    def __init__(self, name, seed, device, rank):
        import speculative_decoding_verify_bf16_gb300 as sv
        self.sv = sv
        self.name = name
        self.device = device
        first = workloads.make_round(name, seed=seed + 1000 * rank, device=device)
        set_bytes = first.logits_bytes()
        n_sets = max(2, math.ceil(1.5 * L2_BYTES / set_bytes) + 1)
        n_sets = min(n_sets, 16)
        self.sets = [first] + [workloads.make_round(name, seed=seed + 1000 * rank + i, device=device,
                                                    with_state=False)
                               for i in range(1, n_sets)]
        if first.staged is not None:
            for s in self.sets[1:]:  # one recurrent state, shared: its reads dwarf L2 anyway
                s.staged, s.live = first.staged, first.live
        self.set_bytes = set_bytes
        self.outs = []
        for s in self.sets:
            self.outs.append(dict(
                committed=torch.zeros(s.lanes, dtype=torch.int32, device=device),
                out_tokens=torch.zeros(s.rows, dtype=torch.int32, device=device),
                status=torch.zeros(s.lanes, dtype=torch.int32, device=device)))
        # Ranks verify disjoint lane ranges of one notional batch: lane_base keys
        # their uniforms by global lane index.  Every set's metadata is written
        # once, before the timed launches, so no kernel on the stream writes it.
        self.args = [sv.make_args(s.target, s.draft, s.draft_tokens, s.draft_lens, s.row_offsets,
                                  s.temperatures, s.seed, o["committed"], o["out_tokens"], o["status"],
                                  rows=s.rows, lane_base=rank * s.lanes, meta_before_wait=True)
                     for s, o in zip(self.sets, self.outs)]
        # Ragged workloads draw their draft lengths per seed, so the sets differ
        # in rows and bytes: K steps count the sets they actually ran.
        per_set = [round_bytes(s) for s in self.sets]
        self.set_verify_bytes = [b for b, _ in per_set]
        self.set_rows = [r.rows for r in self.sets]
        self.verify_bytes, self.rows_per_step = per_set[0]
        self.has_state = first.staged is not None
        self.commit_bytes = commit_bytes(first) if self.has_state else 0
        self.launches_per_step = 1 + (1 if self.has_state else 0)

    def l2_note(self):
        """What the rotation of input sets does to L2, as it is."""
        between = (len(self.sets) - 1) * self.set_bytes
        head = f"inputs rotate over {len(self.sets)} sets of {self.set_bytes / 2**20:.3g} MiB logits"
        if between > L2_BYTES:
            return head + f" ({between / 1e6:.0f} MB between reuses of a set: more than the 129 MB L2)"
        return head + (f" ({between / 1e3:.0f} KB between reuses: L2-resident; the round is bound by launch "
                       f"and memory latency, not by HBM)")

    def rows_in(self, steps):
        """Verified rows over `steps` consecutive steps from step 0."""
        n = len(self.sets)
        return sum(self.set_rows[i % n] for i in range(steps))

    def mean_verify_bytes(self, steps):
        """Algorithmic bytes of one verify launch, averaged over `steps` steps from step 0."""
        n = len(self.sets)
        return sum(self.set_verify_bytes[i % n] for i in range(steps)) / steps

    def check_budget(self):
        r = self.sets[0]
        if self.name == workloads.RAGGED_MIXED_B128:
            k = self.sv.spec_row_budget(workloads.RAGGED_DRAFT_TOKENS, workloads.RAGGED_ROW_BUDGET, r.lanes)
            assert k == workloads.RAGGED_DRAFT_TOKENS and r.rows <= workloads.RAGGED_ROW_BUDGET
        else:
            k = int(r.draft_lens.max())
            assert self.sv.spec_row_budget(k, r.rows, r.lanes) == k

    def step(self, i, stream, verify=True, commit=True):
        j = i % len(self.sets)
        s = self.sets[j]
        h = stream.cuda_stream
        import ctypes
        if verify:
            code = self.sv.spec_verify_accept_raw(self.args[j], ctypes.c_void_p(h))
            if code != 0:
                raise RuntimeError(f"spec_verify_accept: {code}")
        if commit and self.has_state:
            self.sv.spec_commit_state(s.staged, s.live, self.outs[j]["committed"], self.outs[j]["status"],
                                      stream=stream)

    def capture(self, steps, stream, **kw):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(steps):
                    self.step(i, torch.cuda.current_stream(), **kw)
        return g


def timed_graph_run(bench, K, stream, world, **kw):
    """Replay graphs for exactly K steps; returns elapsed ms (events on `stream`)."""
    g_full = bench.capture(min(K, GRAPH_STEPS), stream, **kw)
    rem = K % GRAPH_STEPS if K > GRAPH_STEPS else 0
    g_rem = bench.capture(rem, stream, **kw) if rem else None
    reps = K // GRAPH_STEPS if K > GRAPH_STEPS else 1
    g_full.replay()  # upload
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    return start.elapsed_time(end), (g_full, g_rem, reps)


def soak(graphs, stream, seconds):
    g_full = graphs[0]
    t0 = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t0 < seconds:
            g_full.replay()
            torch.cuda.synchronize()


def e2e_run(bench, steps, stream):
    """Public API end to end: pinned host inputs -> H2D -> verify -> D2H of the result.

    Every step copies its whole input set from pinned host memory (the logits
    and one packed buffer of draft tokens, draft lengths, row offsets and
    temperatures) and reads back one packed buffer of committed counts and
    tokens.  Two input sets alternate, each with its own device buffers: a
    copy stream uploads step i + 1 while step i verifies, so the step is bound
    by the upload.  Returns (ms, rows verified, mean H2D bytes a step, mean D2H
    bytes a step)."""
    sv = bench.sv
    sets = bench.sets[:2] if len(bench.sets) >= 2 else bench.sets[:1] * 2

    def pack_meta(s):
        return torch.cat([s.draft_tokens.cpu(), s.draft_lens.cpu(), s.row_offsets.cpu(),
                          s.temperatures.cpu().view(torch.int32)])

    hosts, devs, shapes = [], [], []
    for s in sets:
        h = {"target": s.target.cpu().pin_memory(), "meta": pack_meta(s).pin_memory()}
        if s.draft is not None:
            h["draft"] = s.draft.cpu().pin_memory()
        hosts.append(h)
        devs.append({k: torch.empty_like(v, device=bench.device) for k, v in h.items()})
        shapes.append((s.lanes, s.rows, s.seed))

    def views(i):
        lanes, rows, _ = shapes[i]
        m = devs[i]["meta"]
        return (m[:rows], m[rows:rows + lanes], m[rows + lanes:rows + 2 * lanes + 1],
                m[rows + 2 * lanes + 1:].view(torch.float32))

    res_dev = [torch.empty(sh[0] + sh[1], dtype=torch.int32, device=bench.device) for sh in shapes]
    res_host = [torch.empty(sh[0] + sh[1], dtype=torch.int32).pin_memory() for sh in shapes]
    h2d = [sum(v.numel() * v.element_size() for v in h.values()) for h in hosts]
    d2h = [r.numel() * 4 for r in res_host]
    copy_stream = torch.cuda.Stream(device=bench.device)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        d, h = devs[i % 2], hosts[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[i % 2])  # the verify of step i - 2 has read this buffer
            for k, v in h.items():
                d[k].copy_(v, non_blocking=True)
            uploaded[i % 2].record(copy_stream)

    def verify(i):
        j = i % 2
        d = devs[j]
        lanes, rows, seed = shapes[j]
        stream.wait_event(uploaded[j])
        dt, dl, ro, te = views(j)
        r = res_dev[j]
        # the metadata comes from the copy stream (behind the event), not from a kernel
        sv.spec_verify_accept(d["target"], d.get("draft"), dt, dl, ro, te, seed + i, r[:lanes], r[lanes:],
                              stream=stream, meta_before_wait=True)
        consumed[j].record(stream)
        res_host[j].copy_(r, non_blocking=True)

    with torch.cuda.stream(stream):
        for e in consumed:
            e.record(stream)
        for i in range(3):
            upload(i)
            verify(i)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        begun = torch.cuda.Event()
        begun.record(stream)
        copy_stream.wait_event(begun)  # the timed uploads start after the start event
        upload(0)
        for i in range(steps):
            if i + 1 < steps:
                upload(i + 1)
            verify(i)
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    # the packed results of the last step equal what the binding wrote
    last = (steps - 1) % 2
    assert torch.equal(res_host[last].to(bench.device), res_dev[last])
    rows = sum(shapes[i % 2][1] for i in range(steps))
    return ms, rows, sum(h2d[i % 2] for i in range(steps)) / steps, sum(d2h[i % 2] for i in range(steps)) / steps


def cpu_oracle_parity(gpu_round, gpu_out, exempt_tol=1e-5):
    """The oracle (the C++ statement, on every host thread) on the very inputs
    the GPU verified (every lane), against the GPU's committed counts and
    tokens.  A lane counts as equal when both agree; a sampled lane that
    differs counts as exempt when one of its random decisions lay within 1e-5
    of flipping in the oracle's float64 arithmetic (|u - p/q|, or u' within
    1e-5 of a CDF boundary in normalised units), and as a mismatch otherwise."""
    from oracle import native
    r = dataclasses.replace(gpu_round, staged=None, live=None).to("cpu")
    tgt, dft, tok, lens, off, temps = cpu_oracle_inputs(r)
    res = native.verify_round(tgt, dft, tok, lens, off, temps, seed=r.seed, threads=cpu_threads())
    c_gpu = gpu_out["committed"].cpu().numpy()
    t_gpu = gpu_out["out_tokens"].cpu().numpy()
    out = {"lanes": r.lanes, "greedy_lanes": int((temps <= 0).sum()), "sampled_lanes": int((temps > 0).sum()),
           "greedy_equal": 0, "sampled_equal": 0, "sampled_exempt": 0, "mismatch": 0,
           "rows": int(off[-1]), "tokens_equal": int((t_gpu[:off[-1]] == res.out_tokens[:off[-1]]).sum())}
    for b in range(r.lanes):
        lo, hi = int(off[b]), int(off[b + 1])
        same = c_gpu[b] == res.committed[b] and np.array_equal(t_gpu[lo:hi], res.out_tokens[lo:hi])
        if same:
            out["sampled_equal" if temps[b] > 0 else "greedy_equal"] += 1
        elif temps[b] > 0 and any(m < exempt_tol for _, _, m in res.margins[b]):
            out["sampled_exempt"] += 1
        else:
            out["mismatch"] += 1
    return out


def cpu_oracle_inputs(r):
    """The arguments of the C++ oracle for round r (on the host): logits as
    stored (bfloat16 bit patterns or float32, widened exactly by the oracle)."""
    def raw(t):
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    return (raw(r.target), None if r.draft is None else raw(r.draft), r.draft_tokens.numpy(),
            r.draft_lens.numpy(), r.row_offsets.numpy(), r.temperatures.numpy())


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_time_oracle(r, budget_s, threads):
    """Whole rounds of the C++ oracle (oracle/verify_ref.cpp) on `threads` host
    threads until `budget_s` is spent; if one round would take more than a
    third of it, the first lanes only.  Returns (rows/s, threads used, sample)."""
    from oracle import native
    tgt, dft, tok, lens, off, temps = cpu_oracle_inputs(r)
    lanes = r.lanes
    take = lanes
    rows_done, t_total, reps, used = 0, 0.0, 0, threads
    while t_total < budget_s:
        t0 = time.perf_counter()
        res, used = native.verify_round(tgt, dft, tok[:off[take]], lens[:take], off[:take + 1], temps[:take],
                                        seed=r.seed, threads=threads, return_threads=True)
        dt = time.perf_counter() - t0
        assert (res.lane_status == 0).all()
        t_total += dt
        rows_done += int(off[take])
        reps += 1
        if reps == 1 and dt > budget_s / 3 and take > 1:
            take = max(1, int(take * budget_s / 3 / dt))
    sample = (f"{reps} round(s) over {'all ' if take == lanes else 'the first '}{take} of {lanes} lanes "
              f"({rows_done} rows)")
    return rows_done / t_total, used, sample


def cpu_baseline(name, seed, budget_s=12.0, gpu_round=None):
    """The oracle as it stands -- the plain C++ statement, oracle/verify_ref.cpp,
    with one std::thread worker per host thread taking lanes one at a time --
    timed on a bounded sample of the workload on this host's cores, plus the
    same on one thread (rank 0 only).  With ``gpu_round`` (an input set the GPU
    verified) it is timed on those same inputs."""
    r = dataclasses.replace(gpu_round if gpu_round is not None else workloads.make_round(
        name, seed=seed, device="cpu", with_state=False), staged=None, live=None).to("cpu")
    cores = cpu_threads()
    value, used, sample = cpu_time_oracle(r, budget_s * 0.5, cores)
    one, _, one_sample = cpu_time_oracle(r, budget_s * 0.5, 1)
    return {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
            "impl": "C++ float64 (oracle/verify_ref.cpp), std::thread workers over lanes",
            "sample": f"{sample} on {used} host threads",
            "single_thread": {"value": one, "unit": UNIT, "cores": 1, "sample": one_sample}}


def run_ours(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    import speculative_decoding_verify_bf16_gb300 as sv
    sv.build_library()
    sv.load_library()

    bench = Bench(args.workload, args.seed, device, rank)
    bench.check_budget()
    stream = torch.cuda.Stream(device=device)
    K, W = args.steps, args.warmup

    # warm-up: W eager steps
    with torch.cuda.stream(stream):
        for i in range(W):
            bench.step(i, stream)
    torch.cuda.synchronize()
    st = bench.outs[0]["status"].cpu().numpy()
    assert (st == 0).all(), st

    sampler = ClockSampler(local)
    sampler.start()
    ms_total, graphs = timed_graph_run(bench, K, stream, world)
    soak(graphs, stream, SOAK_SECONDS)
    # per-kernel timing: the same K steps with one kernel kind only
    ms_verify, _ = timed_graph_run(bench, K, stream, world, commit=False)
    ms_commit = None
    if bench.has_state:
        ms_commit, _ = timed_graph_run(bench, K, stream, world, verify=False)
    clocks = sampler.stop()

    t = torch.tensor([ms_total, ms_verify, ms_commit or 0.0], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_total, ms_verify, ms_commit = t.tolist()

    e2e_steps = max(5, min(K, 50))
    e2e_ms, e2e_rows, h2d, d2h = e2e_run(bench, e2e_steps, stream)
    e2e_t = torch.tensor([e2e_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(e2e_t, op=torch.distributed.ReduceOp.MAX)

    peak, peak_kind = measured_hbm_peak()
    verify_us = ms_verify * 1e3 / K
    verify_bytes = bench.mean_verify_bytes(K)
    verify_gbs = verify_bytes / (verify_us * 1e-6) / 1e9
    kernels = {"verify_accept": {"us_per_launch": verify_us, "algorithmic_bytes": verify_bytes,
                                 "gbs": verify_gbs, "frac_of_peak": verify_gbs / peak}}
    dominant = "verify_accept"
    if bench.has_state:
        commit_us = ms_commit * 1e3 / K
        commit_gbs = bench.commit_bytes / (commit_us * 1e-6) / 1e9
        kernels["commit_state"] = {"us_per_launch": commit_us, "algorithmic_bytes": bench.commit_bytes,
                                   "gbs": commit_gbs, "frac_of_peak": commit_gbs / peak}
        if commit_us > verify_us:
            dominant = "commit_state"
    dk = kernels[dominant]
    traffic = profiled_traffic(dominant, args.workload)
    rows_total = bench.rows_in(K) * world
    value = rows_total / (ms_total * 1e-3)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_total / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if bench.sets[0].dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {
            "workload": args.workload,
            "lanes": bench.sets[0].lanes,
            "vocab": bench.sets[0].vocab,
            "rows_per_step": bench.rows_in(K) / K,
            "logits_dtype": bench.sets[0].dtype,
            "recurrent_state": bench.has_state,
            "l2": bench.l2_note(),
            "timing": f"CUDA-graph replays of {min(K, GRAPH_STEPS)} steps, events on the launch stream",
            "parallelism": f"lanes sharded over {world} GPU(s)" if world > 1 else "1 GPU",
        },
        "hbm_gbs": {"achieved": dk["gbs"], "peak": peak, "peak_source": peak_kind},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": dk["gbs"], "peak": peak,
                     "unit": "GB/s", "frac": dk["gbs"] / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": dk["algorithmic_bytes"],
                     "us_per_launch": dk["us_per_launch"], "peak_source": peak_kind},
        "kernels": kernels,
        "e2e": {"value": e2e_rows * world / (e2e_t.item() * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "path": ("pinned host inputs -> H2D (logits + one packed metadata buffer, double-buffered on a copy "
                         "stream) -> spec_verify_accept (python binding) -> D2H of one packed result buffer; "
                         "two input sets alternate")},
        "gpu_launches": K * bench.launches_per_step,
        "clocks": clocks,
    }
    try:
        committed = bench.outs[0]["committed"].float()
        line["acceptance"] = {"mean_committed": float(committed.mean()),
                              "mean_drafts": float(bench.sets[0].draft_lens.float().mean()),
                              "of": "input set 0, every lane"}
    except Exception as e:  # a report, never a reason to lose the measurement
        line["acceptance"] = {"error": repr(e)[:200]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.seed, gpu_round=bench.sets[0])
        try:
            line["cpu_baseline"]["parity"] = cpu_oracle_parity(bench.sets[0], bench.outs[0])
        except Exception as e:  # a report, never a reason to lose the measurement
            line["cpu_baseline"]["parity"] = {"error": repr(e)[:200]}
    if rank == 0 and args.all_workloads:
        line["workloads"] = other_workloads(args, device, stream, peak)
        line["round_control"] = round_control_timing(device, stream)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def round_control_timing(device, stream, reps=500):
    """Per-round cost of the acceptance counts and the miss back-off (two tiny
    kernels a serving loop runs after each verify round), replayed in graphs.
    Both read ~12 bytes per lane, so they are bound by launch latency, not HBM."""
    import speculative_decoding_verify_bf16_gb300 as sv
    out = {}
    for lanes in (128, 4096):
        g = torch.Generator(device="cpu").manual_seed(lanes)
        k = torch.randint(0, 8, (lanes,), generator=g, dtype=torch.int32)
        committed = (torch.rand(lanes, generator=g) * (k + 1).float()).to(torch.int32) + 1
        k, committed = k.to(device), committed.to(device)
        status = torch.zeros(lanes, dtype=torch.int32, device=device)
        counts = sv.new_accept_counts(1, device)
        states = sv.new_backoff_states(lanes, device)
        nxt = torch.empty(lanes, dtype=torch.int32, device=device)
        entry = {}
        for name, fn in (("accept_counts_us", lambda: sv.spec_accept_counts_update(committed, k, status, counts,
                                                                                   stream=stream)),
                         ("backoff_step_us", lambda: sv.spec_backoff_step(states, k, committed, status, 7, nxt,
                                                                          stream=stream))):
            with torch.cuda.stream(stream):
                fn()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    for _ in range(reps):
                        fn()
            graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            entry[name] = e0.elapsed_time(e1) * 1e3 / reps
        # n-gram drafter over 2048-token histories of this many lanes
        hist = 2048
        toks = torch.randint(0, 512, (lanes * hist,), generator=g, dtype=torch.int32).to(device)
        offs = (torch.arange(lanes + 1, dtype=torch.int64) * hist).to(device)
        drafts = torch.empty(lanes, 7, dtype=torch.int32, device=device)
        lens = torch.empty(lanes, dtype=torch.int32, device=device)
        fn = lambda: sv.spec_ngram_draft(toks, offs, 7, drafts, lens, stream=stream)
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(reps):
                    fn()
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        entry["ngram_draft_us"] = e0.elapsed_time(e1) * 1e3 / reps
        entry["ngram_history_tokens"] = hist
        # per-row penalties: 8 rows a lane, 200 penalised history tokens a lane
        V = 151936 if lanes <= 128 else 8192
        kk = torch.full((lanes,), 7, dtype=torch.int32, device=device)
        offs_r = (torch.arange(lanes + 1, dtype=torch.int32) * 8).to(device)
        logits = torch.zeros(lanes * 8, V, dtype=torch.bfloat16, device=device)
        dtok = torch.randint(0, V, (lanes * 8,), generator=g, dtype=torch.int32).to(device)
        ptok = torch.sort(torch.randperm(V, generator=g)[:200].to(torch.int32)).values.repeat(lanes).to(device)
        pcnt = torch.ones(lanes * 200, dtype=torch.int32, device=device)
        poff = (torch.arange(lanes + 1, dtype=torch.int64) * 200).to(device)
        pres = torch.full((lanes,), 0.5, dtype=torch.float32, device=device)
        fn = lambda: sv.spec_apply_penalties(logits, offs_r, dtok, kk, ptok, pcnt, poff, pres, pres, stream=stream)
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(reps):
                    fn()
        graph.replay()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        entry["penalties_us"] = e0.elapsed_time(e1) * 1e3 / reps
        entry["penalties_shape"] = {"rows_per_lane": 8, "history_tokens": 200, "vocab": V}
        del logits
        entry["bound"] = ("launch latency at 128 lanes; the drafter reads 4 B per history token once (repeats hit L1),"
                          " so large batches are bound by memory latency")
        out[f"lanes_{lanes}"] = entry
    return out


def other_workloads(args, device, stream, peak):
    out = {}
    for name in workloads.WORKLOADS:
        if name == args.workload:
            continue
        b = Bench(name, args.seed, device, 0)
        b.check_budget()
        with torch.cuda.stream(stream):
            for i in range(3):
                b.step(i, stream)
        torch.cuda.synchronize()
        K = 200 if not b.has_state else 40
        ms, _ = timed_graph_run(b, K, stream, 1)
        ms_v, _ = timed_graph_run(b, K, stream, 1, commit=False)
        v_us = ms_v * 1e3 / K
        vb = b.mean_verify_bytes(K)
        entry = {"rows_per_s": b.rows_in(K) / (ms * 1e-3), "ms_per_step": ms / K,
                 "verify_us": v_us, "verify_gbs": vb / (v_us * 1e-6) / 1e9,
                 "verify_frac": vb / (v_us * 1e-6) / 1e9 / peak,
                 "verify_algorithmic_bytes": vb, "rows_per_step": b.rows_in(K) / K, "l2": b.l2_note()}
        if b.has_state:
            ms_c, _ = timed_graph_run(b, K, stream, 1, verify=False)
            c_us = ms_c * 1e3 / K
            entry.update({"commit_us": c_us, "commit_gbs": b.commit_bytes / (c_us * 1e-6) / 1e9,
                          "commit_frac": b.commit_bytes / (c_us * 1e-6) / 1e9 / peak,
                          "commit_algorithmic_bytes": b.commit_bytes})
        if not args.no_cpu_baseline:
            entry["cpu_baseline"] = cpu_baseline(name, args.seed, budget_s=3.0, gpu_round=b.sets[0])
            try:
                entry["cpu_baseline"]["parity"] = cpu_oracle_parity(b.sets[0], b.outs[0])
            except Exception as e:
                entry["cpu_baseline"]["parity"] = {"error": repr(e)[:200]}
        out[name] = entry
        del b
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def run_reference(args):
    """The reference arm: the CPU oracle (the plain C++ statement, on every
    host thread) timed as it stands on the same workload, metric and unit."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import native
    native.build()
    r = workloads.make_round(args.workload, seed=args.seed, device="cpu", with_state=False)
    tgt, dft, tok, lens, off, temps = cpu_oracle_inputs(r)
    threads = cpu_threads()
    # Each step: a bounded sample of the round (its first lanes), sized to
    # ~0.5 s and so that warm-up plus timed steps take about 150 s at most
    # (one lane a step at least).
    budget = min(0.5, 150.0 / max(1, args.steps + args.warmup))
    t0 = time.perf_counter()
    _, used = native.verify_round(tgt, dft, tok, lens, off, temps, seed=r.seed, threads=threads,
                                  return_threads=True)
    per_round = max(time.perf_counter() - t0, 1e-6)
    take = int(max(1, min(r.lanes, r.lanes * budget / per_round)))
    rows_per_step = int(off[take])

    def step():
        return native.verify_round(tgt, dft, tok[:off[take]], lens[:take], off[:take + 1], temps[:take],
                                   seed=r.seed, threads=threads, return_threads=True)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, used = step()
    dt = time.perf_counter() - t0
    value = rows_per_step * args.steps / dt
    sample = f"the first {take} of {r.lanes} lanes ({rows_per_step} rows) per step, on {used} host threads"
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "lanes": r.lanes, "vocab": r.vocab,
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample,
                         "impl": "C++ float64 (oracle/verify_ref.cpp), std::thread workers over lanes"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_launch_only(args):
    """Profiler driver: build the workload, run N eager steps, no timing."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import speculative_decoding_verify_bf16_gb300 as sv
    sv.build_library()
    sv.load_library()
    r = workloads.make_round(args.workload, seed=args.seed, device=device, commit_lanes=args.commit_lanes)
    committed = torch.zeros(r.lanes, dtype=torch.int32, device=device)
    out = torch.zeros(r.rows, dtype=torch.int32, device=device)
    status = torch.zeros(r.lanes, dtype=torch.int32, device=device)
    for i in range(args.launch_only):
        # Profilers replay a launch after restoring memory with work of their
        # own, so the metadata is read only after the wait here.
        sv.spec_verify_accept(r.target, r.draft, r.draft_tokens, r.draft_lens, r.row_offsets,
                              r.temperatures, r.seed, committed, out, status)
        if r.staged is not None:
            sv.spec_commit_state(r.staged, r.live, committed, status)
    torch.cuda.synchronize()
    assert (status.cpu() == 0).all()
    print(json.dumps({"launch_only": args.launch_only, "workload": args.workload, "lanes": r.lanes}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=workloads.WORKLOADS, default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--only", dest="all_workloads", action="store_false",
                    help="measure only --workload (by default the other workloads are measured "
                         "too and reported under 'workloads')")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch-only", type=int, default=0, metavar="N",
                    help="profiler driver: run N eager steps of --workload and exit (no timing)")
    ap.add_argument("--commit-lanes", type=int, default=None,
                    help="with --launch-only: lanes of the commit workload (smaller captures)")
    args = ap.parse_args()
    if args.launch_only:
        run_launch_only(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
