#!/usr/bin/env python3
"""Benchmark of the GB300 speculative-sampling verifier.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--impl ours|reference]

One step = one verification call (target-row pass, accept scan, race) over
one batch of the chosen workload, inputs resident in HBM. Prints one JSON
line with the metric "verified draft positions/sec and achieved HBM GB/s":
``value`` is sum(gamma_r) per second over all ranks; ``e2e`` is the same
metric through the public API with the inputs copied from pinned host memory
and the outputs copied back inside the timed region; ``roofline`` is the
dominant kernel (the target-row pass) timed live with the library's phase
events, set against the measured HBM copy bandwidth; ``cpu_baseline`` is the
CPU oracle (single thread, as written) on a bounded sample of the same
workload, and ``cpu_baseline_all_cores`` the same unchanged oracle on every
host core (disjoint request sets, one thread each). ``--impl reference``
times the single-threaded oracle alone.

Multi-GPU: one process per GPU (torchrun); every rank verifies its own batch
of the workload (requests numbered rank * B + r), no collective on the data
path; timing is the max over ranks (weak scaling).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 2 ** 20
METRIC = "verified draft positions/sec and achieved HBM GB/s (fraction of GB300 peak)"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal
WORKLOADS = {
    "c2": "B=8 gamma=3 V=32000 fp32 logits N(0,2^2)+3 boosted tokens, probabilistic draft, T=1",
    "c3": ("B=64 gamma=5 V=128256 bf16 logits N(0,3^2)+Zipf(1.1), probabilistic draft, "
           "T in {0,0.7,1}, top_k=50 / top_p=0.9 / none by thirds"),
    "c4": ("B=256 gamma=4 V=151936 bf16 logits N(0,2.5^2)+Zipf(1.0), one-hot greedy draft "
           "(no draft_probs), T=1, top_p=0.95"),
    "c5": ("B=1024 ragged gamma U{1..7} V=256000 bf16 logits N(0,2^2)+Zipf(1.2), half T=0 "
           "(argmax path), half T=0.8 with probabilistic draft"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="c5", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--accept", default="rejection", choices=["rejection", "sampler-match"],
                    help="acceptance rule: the rejection rule, or sampler-match (the "
                         "target's sampler draws every position; drafts must equal it)")
    ap.add_argument("--early-exit", action="store_true",
                    help="stop reading a request's rows at its first rejection")
    ap.add_argument("--resident", action="store_true",
                    help="with --early-exit: hold each judged row in a thread-block cluster")
    ap.add_argument("--B", type=int, default=None,
                    help="resize the workload to B requests (profiling of small cases)")
    ap.add_argument("--V", type=int, default=None,
                    help="resize the workload's vocabulary (profiling of other row lengths)")
    ap.add_argument("--top-p", type=float, default=None,
                    help="set every request's top_p (profiling of the filtered-row paths)")
    ap.add_argument("--top-k", type=int, default=None,
                    help="set every request's top_k (profiling of the filtered-row paths)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=4,
                    help="end to end: verify the batch as this many request ranges, each "
                         "range's copies overlapping the previous range's verification")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the c2/c3/c4 and early-exit timings beside the headline")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_request_base(rank: int, B: int) -> int:
    """Global index of this rank's first request (weak scaling: each rank
    verifies its own B requests)."""
    return rank * B


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(batch, num_accepted) -> dict:
    """Bytes the method must move for one call, from the call's outcome: every
    target row once, the draft_probs row of each rejected probabilistic
    request, the per-position gathers and the outputs."""
    B, V = batch["B"], batch["V"]
    cu = batch["cu_num_draft"]
    gam = np.diff(cu)
    N = int(cu[-1])
    R = N + B
    esize = 2 if batch["logits_dtype"] == "bf16" else 4
    T = batch["temperature"]
    rows = R * V * esize
    q_rows = 0
    judged_q = 0
    if batch["draft_probs"] is not None and not (int(batch.get("flags", 0)) & 2):
        hot = (T > 0)
        rejected = hot & (num_accepted < gam)
        q_rows = int(rejected.sum()) * V * 4
        judged_q = int(np.minimum(num_accepted + 1, gam)[hot].sum()) * 4
    small = (B + 1) * 4 + N * 4 + B * 4 * 3 + judged_q + (N + B) * 4 + B * 4
    # The rows up to each request's first rejection: all that early exit reads.
    needed = int(np.minimum(num_accepted + 1, gam + 1).sum()) * V * esize
    if int(batch.get("flags", 0)) & 4:
        rows = needed
    return dict(row_pass=rows, race_q=q_rows, q_gathers=judged_q, small=small,
                total=rows + q_rows + small, rows_to_first_rejection=needed,
                all_rows=R * V * esize)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = None
        self.device = device_index
        self.path = None

    def _gpu_id(self):
        try:
            import torch
            u = torch.cuda.get_device_properties(self.device).uuid
            return "GPU-" + str(u)
        except Exception:
            return str(self.device)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="spec_verify_clocks_", suffix=".csv")
            self.out = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._gpu_id(), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        try:
            os.remove(self.path)
        except OSError:
            pass
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def timed_calls(ver, db, stream, dev, K, flush):
    """K calls on `stream`, each bracketed by CUDA events on that stream (the
    L2 flush buffer, if any, rewritten before each call), then K more with the
    library's phase events (row pass, accept scan, race) recorded between its
    kernels. The per-call times come from the first loop: events between the
    kernels of a call would stop them from overlapping their launches.
    Returns the first loop's per-call milliseconds and the second loop's
    phase averages."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        ver.run(db, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ph = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ver.set_phase_events(ph[i])
        ver.run(db, stream)
    torch.cuda.synchronize(dev)
    ver.set_phase_events(None)
    phases = {"rows": sum(p[0].elapsed_time(p[1]) for p in ph) / K,
              "accept": sum(p[1].elapsed_time(p[2]) for p in ph) / K,
              "race": sum(p[2].elapsed_time(p[3]) for p in ph) / K,
              "call_with_phase_events": sum(p[0].elapsed_time(p[3]) for p in ph) / K}
    return step_ms, phases


def flush_buffer(batch, dev):
    """An L2-sized write between timed calls when the logits would fit in L2."""
    import torch
    if batch["target_logits"].nbytes < 2 * L2_BYTES:
        return torch.empty(4 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    return None


def fractions(bytes_, ms_per_step, rows_ms, peak):
    """Achieved GB/s of the row pass and of the whole call, against the
    measured copy bandwidth and against the nominal HBM3e figure."""
    rows_gbs = bytes_["row_pass"] / (rows_ms * 1e-3) / 1e9
    call_gbs = bytes_["total"] / (ms_per_step * 1e-3) / 1e9
    return {"rows_gbs": rows_gbs, "rows_frac": rows_gbs / peak,
            "rows_frac_nominal": rows_gbs / NOMINAL_HBM_GBS,
            "call_gbs": call_gbs, "call_frac": call_gbs / peak,
            "call_frac_nominal": call_gbs / NOMINAL_HBM_GBS}


def per_config_timings(sv, dev, stream, peak, main_batch, steps=30, warmup=5):
    """The other target workloads timed on the same GPU and clocks as the
    headline line: c2, c3 and c4 with the rejection rule, and the headline
    batch with early exit. Device-timed like the headline (inputs resident)."""
    import torch
    out = {}
    cases = [("c2", None, 0, 0), ("c3", None, 0, 0), ("c4", None, 0, 0)]
    if main_batch is not None:
        cases.append((main_batch["name"] + " early-exit", main_batch, sv.FLAG_EARLY_EXIT, 0))
        cases.append((main_batch["name"] + " early-exit resident", main_batch, sv.FLAG_EARLY_EXIT,
                      sv.CONFIG_EARLY_RESIDENT))
    for label, batch, flags, cfg_flags in cases:
        b = dict(batch) if batch is not None else synth.make(label)
        b["flags"] = flags
        R = b["target_logits"].shape[0]
        ver = sv.Verifier(max_batch=b["B"], max_rows=R, max_vocab=b["V"], device=dev.index,
                          config_flags=cfg_flags)
        db = sv.upload(b, dev, with_p=False)
        flush = flush_buffer(b, dev)
        for _ in range(warmup):
            ver.run(db, stream)
        torch.cuda.synchronize(dev)
        assert ver.status() == 0, f"device status bits set ({label})"
        n_acc = db.num_accepted.cpu().numpy()
        bytes_ = algorithmic_bytes(b, n_acc)
        step_ms, phases = timed_calls(ver, db, stream, dev, steps, flush)
        ms = sum(step_ms) / steps
        N = int(b["cu_num_draft"][-1])
        out[label] = {"workload": WORKLOADS.get(b["name"], b["name"]), "steps": steps,
                      "ms_per_step": ms, "value": N / (ms * 1e-3), "unit": "draft_positions/s",
                      "phases_ms": phases, "algorithmic_bytes_per_step": bytes_,
                      "l2": ("inputs larger than L2" if flush is None
                             else "L2 flushed between timed calls (512 MB write)"),
                      **fractions(bytes_, ms, phases["rows"], peak)}
        ver.close()
        del db, flush
        torch.cuda.empty_cache()
    return out


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback (an earlier GB300 copy measurement)"


# The sources the target-row pass (the dominant kernel) is built from.
ROW_PASS_SOURCES = ("common.cuh", "pipe.cuh", "rows.cuh", "hist.cuh", "rows_tma.cuh")


def kernel_source_sha() -> str:
    """Hash of the row pass's sources: the key of its committed ncu traffic."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_rejection_02_gb300", "csrc")
    for fn in ROW_PASS_SOURCES:
        with open(os.path.join(d, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(config: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when there is none for this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(config)
        if e and e.get("source_sha") == kernel_source_sha():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# The race's instruction count per raced entry, from ncu on c5 resized to
# B = 256 (profiles/k_race_c5.md: smsp__inst_executed.sum 42.25 M warp
# instructions for 128 races of 256000 entries), valid while the race's
# sources hash to the recorded value.
RACE_SOURCES = ("common.cuh", "pipe.cuh", "philox.cuh", "race.cuh")
RACE_SOURCES_SHA = "3112193ef603ac92"
RACE_INSTR_PER_ENTRY = 42.25e6 * 32 / (128 * 256000)
ISSUE_PER_SM_CLOCK = 4  # warp instructions: one per scheduler per clock, four schedulers


def race_source_sha() -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_rejection_02_gb300", "csrc")
    for fn in RACE_SOURCES:
        with open(os.path.join(d, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def race_issue(batch, num_accepted, race_ms, args, clock_info, dev):
    """The race against its instruction-issue bound: warp instructions per
    second (ncu's instructions per raced entry x the entries this call
    raced, over the race phase) against SMs x four schedulers x the SM
    clock sampled during the run. Only for the workload the count was
    measured on (c5 with the rejection rule), and null once the race's
    sources differ from the measured ones."""
    import torch
    if (args.config != "c5" or args.accept != "rejection" or args.resident or
            args.V is not None or args.top_p is not None or args.top_k is not None or
            race_source_sha() != RACE_SOURCES_SHA or not (clock_info or {}).get("sm_mhz")):
        return None
    races = int((batch["temperature"] > 0).sum())  # one race per request with T > 0
    entries = races * batch["V"]
    warp_instr = RACE_INSTR_PER_ENTRY * entries / 32
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * ISSUE_PER_SM_CLOCK * clock_info["sm_mhz"] * 1e6 / 1e9
    achieved = warp_instr / (race_ms * 1e-3) / 1e9
    return {"bound": "issue", "kernel": "race (k_race + k_race_token)",
            "achieved": achieved, "peak": peak, "unit": "G warp instructions/s",
            "frac": achieved / peak, "instr_per_entry": RACE_INSTR_PER_ENTRY,
            "entries": entries, "peak_from": f"{sms} SMs x {ISSUE_PER_SM_CLOCK} x sampled SM clock"}


def request_chunks(cu, k):
    """k contiguous, non-empty request ranges [r0, r1) covering the batch,
    about equal in requests (fewer when the batch has fewer requests)."""
    B = len(cu) - 1
    k = max(1, min(int(k), B))
    edges = [round(i * B / k) for i in range(k + 1)]
    return [(edges[i], edges[i + 1]) for i in range(k) if edges[i + 1] > edges[i]]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_oracle_rate_all_cores(batch, seconds: float):
    """The unchanged oracle on every host core: disjoint request sets (every
    t-th request) verified by one thread each (the oracle call releases the
    GIL); returns (positions/s, description, seconds, threads)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cu = batch["cu_num_draft"]
    gam = np.diff(cu)
    B = batch["B"]
    threads = host_cores()
    t0 = time.perf_counter()
    oracle.verify(batch, requests=[0, 1])
    per_req = max((time.perf_counter() - t0) / 2, 1e-4)
    n = int(max(threads, min(B, threads * seconds / per_req)))
    n = min(n, B)
    parts = [list(range(t, n, threads)) for t in range(threads)]
    parts = [p for p in parts if p]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(len(parts)) as ex:
        list(ex.map(lambda reqs: oracle.verify(batch, requests=reqs), parts))
    dt = time.perf_counter() - t0
    pos = int(gam[:n].sum())
    desc = (f"first {n} of {B} requests ({pos} draft positions), {len(parts)} threads "
            f"on disjoint request sets")
    return pos / dt, desc, dt, len(parts)


def cpu_oracle_rate(batch, seconds: float, steps: int = 1):
    """Time the CPU oracle on a bounded sample of requests; returns
    (positions/s, description, seconds used)."""
    import oracle
    cu = batch["cu_num_draft"]
    gam = np.diff(cu)
    B = batch["B"]
    t0 = time.perf_counter()
    oracle.verify(batch, requests=[0, 1])
    per_req = max((time.perf_counter() - t0) / 2, 1e-4)
    n = int(max(1, min(B, seconds / per_req)))
    reqs = list(range(n))
    t0 = time.perf_counter()
    oracle.verify(batch, requests=reqs)
    dt = time.perf_counter() - t0
    pos = int(gam[:n].sum())
    return pos / dt, f"first {n} of {B} requests ({pos} draft positions), one thread", dt


def run_reference(args, rank, world):
    if rank != 0:
        return
    batch = synth.make(args.config)
    import oracle
    cu = batch["cu_num_draft"]
    gam = np.diff(cu)
    budget = 90.0
    t0 = time.perf_counter()
    oracle.verify(batch, requests=[0, 1])
    per_req = max((time.perf_counter() - t0) / 2, 1e-4)
    per_step = max(1, int(budget / max(1, args.steps + args.warmup) / per_req))
    per_step = min(per_step, batch["B"])
    B = batch["B"]

    def step(i):
        lo = (i * per_step) % B
        reqs = [(lo + t) % B for t in range(per_step)]
        oracle.verify(batch, requests=reqs)
        return int(gam[reqs].sum())

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    pos = 0
    for i in range(args.steps):
        pos += step(args.warmup + i)
    dt = time.perf_counter() - t0
    v = pos / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": v,
        "unit": "draft_positions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config}: {WORKLOADS[args.config]}",
                   "sample": f"{per_step} requests per step"},
        "cpu_baseline": {"value": v, "unit": "draft_positions/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} requests per step of {args.config}, one thread"},
        "e2e": {"value": v, "unit": "draft_positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    import speculative_decoding_rejection_02_gb300 as sv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    batch = synth.make(args.config, B=args.B, V=args.V)
    if args.top_p is not None:
        batch["top_p"] = np.full(batch["B"], args.top_p, np.float32)
    if args.top_k is not None:
        batch["top_k"] = np.full(batch["B"], args.top_k, np.int32)
    B, V = batch["B"], batch["V"]
    batch["request_base"] = rank_request_base(rank, B)
    if args.accept == "sampler-match":
        batch["flags"] = sv.FLAG_SAMPLER_MATCH
    if args.early_exit:
        batch["flags"] = int(batch.get("flags", 0)) | sv.FLAG_EARLY_EXIT
    cu = batch["cu_num_draft"]
    N = int(cu[-1])
    R = N + B
    positions = N

    ver = sv.Verifier(max_batch=B, max_rows=R, max_vocab=V, device=local,
                      config_flags=sv.CONFIG_EARLY_RESIDENT if args.resident else 0)
    db = sv.upload(batch, dev, with_p=False)
    stream = torch.cuda.current_stream(dev)
    in_bytes = sum(v for v in synth.batch_bytes(batch).values())
    flush = flush_buffer(batch, dev)

    # Warm-up (also fixes the deterministic outcome used for the byte count).
    for _ in range(max(3, args.warmup)):
        ver.run(db, stream)
    torch.cuda.synchronize(dev)
    assert ver.status() == 0, "device status bits set"
    n_acc = db.num_accepted.cpu().numpy()
    bytes_ = algorithmic_bytes(batch, n_acc)

    # Timed region: K calls, per-call events and per-phase events.
    K = args.steps
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    step_ms, phases = timed_calls(ver, db, stream, dev, K, flush)
    clock_info = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dev)
    ms_per_step = total_ms / K
    value = world * positions / (ms_per_step * 1e-3)
    rows_avg = phases["rows"]

    peak, peak_kind = measured_hbm_peak()
    fr = fractions(bytes_, ms_per_step, rows_avg, peak)
    achieved = fr["rows_gbs"]
    step_gbs = fr["call_gbs"]

    # End to end through the public API with host buffers. draft_probs stays
    # in page-locked host memory, which the library reads in place (only the
    # gathered q(x) and the rows of rejected requests cross the host link);
    # the other inputs are copied to the device every step.
    e2e = None
    if args.e2e_steps > 0:
        host = {}
        for k in ("cu_num_draft", "draft_token_ids", "target_logits",
                  "temperature", "top_k", "top_p"):
            a = batch.get(k)
            if a is None:
                continue
            if k == "target_logits" and batch["logits_dtype"] == "bf16":
                a = np.ascontiguousarray(a).view(np.int16)
            host[k] = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        dst = {"cu_num_draft": db.cu_num_draft, "draft_token_ids": db.draft_token_ids,
               "target_logits": db.target_logits,
               "temperature": db.temperature, "top_k": db.top_k, "top_p": db.top_p}
        hb = sv.DeviceBatch(cu_num_draft=db.cu_num_draft, draft_token_ids=db.draft_token_ids,
                            target_logits=db.target_logits, draft_probs=None,
                            temperature=db.temperature, top_k=db.top_k, top_p=db.top_p,
                            seed=db.seed, request_base=db.request_base, flags=db.flags,
                            out_tokens=db.out_tokens, num_accepted=db.num_accepted,
                            N=db.N, V=db.V)
        q_read = 0
        if batch["draft_probs"] is not None:
            hb.draft_probs = torch.from_numpy(batch["draft_probs"]).pin_memory()
            q_read = bytes_["race_q"] + bytes_["q_gathers"]
        out_tok = torch.empty(R, dtype=torch.int32).pin_memory()
        out_acc = torch.empty(B, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + q_read
        d2h = out_tok.numel() * 4 + out_acc.numel() * 4
        tok_ref = db.out_tokens.cpu().numpy()
        chunks = request_chunks(batch["cu_num_draft"], args.e2e_chunks)
        parts = []
        if len(chunks) > 1:
            # Each request range is its own call (request_base = its first
            # request, so the draws are those of the whole batch); a copy
            # stream moves range c + 1 while range c is verified.
            cu_np = batch["cu_num_draft"]
            h2d = q_read
            for r0, r1 in chunks:
                a, z = int(cu_np[r0]), int(cu_np[r1])
                row0, row1 = a + r0, z + r1
                cu_h = torch.from_numpy((cu_np[r0:r1 + 1] - cu_np[r0]).astype(np.int32))
                cu_h = cu_h.pin_memory()
                cu_d = torch.empty(r1 - r0 + 1, dtype=torch.int32, device=dev)
                sl = {"target_logits": (row0, row1), "draft_token_ids": (a, z)}
                copies = [(cu_d, cu_h)]
                for k, t in host.items():
                    if k == "cu_num_draft":
                        continue
                    i0, i1 = sl.get(k, (r0, r1))
                    copies.append((dst[k][i0:i1], t[i0:i1]))
                h2d += sum(t.numel() * t.element_size() for _, t in copies)
                part = sv.DeviceBatch(
                    cu_num_draft=cu_d, draft_token_ids=db.draft_token_ids[a:z],
                    target_logits=db.target_logits[row0:row1],
                    draft_probs=None if hb.draft_probs is None else hb.draft_probs[a:z],
                    temperature=db.temperature[r0:r1],
                    top_k=None if db.top_k is None else db.top_k[r0:r1],
                    top_p=None if db.top_p is None else db.top_p[r0:r1],
                    seed=db.seed, request_base=db.request_base + r0, flags=db.flags,
                    out_tokens=db.out_tokens[row0:row1], num_accepted=db.num_accepted[r0:r1],
                    N=z - a, V=db.V)
                parts.append((part, copies, torch.cuda.Event(), torch.cuda.Event()))
            cs = torch.cuda.Stream(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        if parts:
            cs.wait_event(e0)
        for _ in range(args.e2e_steps):
            if parts:
                for part, copies, copied, done in parts:
                    with torch.cuda.stream(cs):
                        # the previous step's call on this range has finished with it
                        cs.wait_event(done)
                        for d, t in copies:
                            d.view(t.dtype).reshape(-1).copy_(t.reshape(-1), non_blocking=True)
                        copied.record(cs)
                    stream.wait_event(copied)
                    ver.run(part, stream)
                    done.record(stream)
            else:
                for k, t in host.items():
                    d = dst[k]
                    d.view(t.dtype).reshape(-1).copy_(t.reshape(-1), non_blocking=True)
                ver.run(hb, stream)
            out_tok.copy_(db.out_tokens, non_blocking=True)
            out_acc.copy_(db.num_accepted, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.e2e_steps
        torch.cuda.synchronize(dev)
        assert ver.status() == 0, "device status bits set (end-to-end calls)"
        assert np.array_equal(out_acc.numpy(), n_acc), "end-to-end outcome differs"
        assert np.array_equal(out_tok.numpy(), tok_ref), "end-to-end tokens differ"
        e2e = {"value": world * positions / (e2e_ms * 1e-3), "unit": "draft_positions/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms, "request_ranges": len(chunks),
               "draft_probs": ("page-locked host memory read in place" if q_read
                               else "none (one-hot draft)")}

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, secs = cpu_oracle_rate(batch, args.cpu_seconds)
        cpu = {"value": rate, "unit": "draft_positions/s", "cores": 1, "kind": "oracle",
               "sample": desc, "seconds": round(secs, 2)}
        rate, desc, secs, thr = cpu_oracle_rate_all_cores(batch, args.cpu_seconds)
        cpu_all = {"value": rate, "unit": "draft_positions/s", "cores": thr, "kind": "oracle",
                   "sample": desc, "seconds": round(secs, 2)}

    per_cfg = None
    if (rank == 0 and world == 1 and args.B is None and args.V is None and args.top_p is None
            and args.top_k is None and not args.no_per_config
            and args.config == "c5" and args.accept == "rejection" and not args.early_exit):
        per_cfg = per_config_timings(sv, dev, stream, peak, batch)

    # row pass, accept scan, race, race tokens; with top-k / top-p also the
    # kernel for the rows the row pass leaves unsettled
    filters = batch.get("top_k") is not None or batch.get("top_p") is not None
    launches_per_step = 4 + (1 if filters else 0)
    if args.accept == "sampler-match":
        launches_per_step += 1  # k_match
    if args.early_exit:
        launches_per_step = 4  # queue init, row pass, race, race tokens
        if args.resident and not filters:
            launches_per_step = 1  # the cluster kernel
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value, "unit": "draft_positions/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{args.config}: {WORKLOADS[args.config]}", "B": B, "V": V,
                       "target_rows": R, "draft_positions": positions,
                       "logits_dtype": batch["logits_dtype"], "input_bytes": int(in_bytes),
                       "l2": ("inputs larger than L2" if flush is None
                              else "L2 flushed between timed calls (512 MB write)"),
                       "acceptance": args.accept,
                       "early_exit": bool(args.early_exit),
                       "top_p_all": args.top_p, "top_k_all": args.top_k,
                       "resident_rows": bool(args.early_exit and args.resident),
                       "parallelism": f"replicas x{world}"},
            "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak,
            "hbm_frac_nominal": fr["call_frac_nominal"],
            "algorithmic_bytes_per_step": bytes_,
            "phases_ms": phases,
            "roofline": {"bound": "hbm", "kernel": "target-row pass", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)",
                         "frac_nominal": fr["rows_frac_nominal"],
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "traffic": ncu_traffic(args.config)},
            "race_issue": race_issue(batch, n_acc, phases["race"], args, clock_info, dev),
            "per_config": per_cfg,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "gpu_launches": K * launches_per_step,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    ver.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
