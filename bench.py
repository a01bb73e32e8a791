#!/usr/bin/env python3
"""Throughput of the speculative-sampling verification hot path on GB300.

One step = one pass of the whole hot path over one batch: `spec_sample_draft`
(draw the K draft tokens of every sequence from the adjusted draft rows) and
`spec_verify` (accept tests, residual / bonus draw) -- one kernel launch each.
Metric: vocabulary rows processed per second (rows read from HBM by the two
kernels), with the achieved HBM GB/s of the dominant kernel against the
measured copy bandwidth as the roofline.

Input sets: three device-resident sets of the workload rotate (together larger
than L2).  Step j draws the tokens of set (j+1) % 3 and verifies set j % 3 with
the tokens drawn one step earlier, so no kernel reads rows that the previous
kernel left in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--impl reference]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); timing is max over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verify vocab-rows/s and achieved HBM GB/s (% of GB300 peak) on 1 GPU"
NSETS = 3


def rows_per_step(w):
    """(sample_draft rows, verify rows) read from HBM per step."""
    B, K = w["B"], w["K"]
    return B * K, B * (K + 1 if w["greedy"] else 2 * K + 1)


def esize(w):
    return 2 if w["dtype"] == "bf16" else 4


def workload_desc(name, w):
    cfg = workloads.CONFIGS[name]
    return "%s: %s, Zipf+Gaussian synthetic logits" % (name, cfg.describe()) if cfg.kind == "zipf" \
        else "%s: %s, Gaussian synthetic logits" % (name, cfg.describe())


def kernel_source_sha():
    """SHA-256 over the library's CUDA sources (csrc/, in name order)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "speculative_sampling_verification_spec_gb300", "csrc", "*"))):
        if p.endswith((".cu", ".cuh", ".h")):
            with open(p, "rb") as f:
                h.update(os.path.basename(p).encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload):
    """DRAM bytes (read + write) of one spec_verify call on this workload, as an
    ncu capture recorded them in profiles/traffic.json -- only while the kernel
    sources are the ones that were captured (else None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        if rec.get("source_sha256") == kernel_source_sha() and workload in rec.get("verify_bytes_per_call", {}):
            return float(rec["verify_bytes_per_call"][workload])
    except Exception:
        pass
    return None


def verify_kernel_name(w):
    """The kernels one spec_verify call launches on this workload (rows start on
    16-byte boundaries here): the one-launch streaming kernel for greedy,
    top-k <= 64 and top-p alone, else the segment kernel and the dependent row
    kernel."""
    V = w["V"]
    use_k = 0 < w["top_k"] < V
    if w["greedy"] or (use_k and w["top_k"] <= 64) or (not use_k and w["top_p"] < 1.0):
        return "spec_stream_kernel (one launch per spec_verify call)"
    return "spec_seg_kernel + spec_row_kernel (one spec_verify call)"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


# ---------------------------------------------------------------------------
# oracle on the host cores (cpu_baseline leg and the reference arm)

def oracle_step(w, seqs, threads):
    """Oracle sample_draft + verify over the sequence subset `seqs` on `threads` host
    threads (ctypes releases the GIL).  Returns the vocab rows processed."""
    import oracle
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    parts = np.array_split(np.asarray(seqs), max(1, min(threads, len(seqs))))

    def work(idx):
        if len(idx) == 0:
            return
        sd = oracle.sample_draft(w["draft"][idx], w["u_draft"][idx], **prm)
        oracle.verify(w["target"][idx], w["draft"][idx], sd["tokens"], w["u_verify"][idx], **prm)

    ts = [threading.Thread(target=work, args=(p,)) for p in parts]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    rs, rv = rows_per_step(dict(w, B=len(seqs)))
    return rs + rv


def cpu_baseline(w, threads):
    """Time the oracle as it stands on one full batch of the workload (bounded sample)."""
    import oracle
    oracle.build()
    seqs = np.arange(w["B"])
    t0 = time.perf_counter()
    rows = oracle_step(w, seqs, threads)
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": "one step over all %d sequences of the workload (%d vocab rows), "
                      "%d host threads, %.2f s wall" % (w["B"], rows, threads, dt)}


def run_reference(args, name):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = workloads.make(name)
    threads = os.cpu_count() or 1
    # size each step so the whole run stays within a few minutes
    t0 = time.perf_counter()
    oracle_step(w, np.arange(min(threads, w["B"])), threads)
    t_one = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    nseq = min(w["B"], threads) if t_one <= budget else 1
    seqs = np.arange(nseq)
    for _ in range(args.warmup):
        oracle_step(w, seqs, threads)
    rows = 0
    t0 = time.perf_counter()
    for j in range(args.steps):
        rows += oracle_step(w, (seqs + j * nseq) % w["B"], threads)
    dt = time.perf_counter() - t0
    val = rows / dt
    cfg = dict(workload=workload_desc(name, w), input_dtype=w["dtype"], global_batch=w["B"],
               vocab=w["V"], draft_len=w["K"], parallelism="host threads")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * dt / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": val, "unit": "rows/s", "cores": threads, "kind": "oracle",
                             "sample": "%d sequence(s) of the workload per step" % nseq},
            "e2e": {"value": val, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm

def verify_only(name, steps, dev, sv):
    """Device time of spec_verify alone on another workload: NSETS rotating
    device input sets (drafts drawn once per set), `steps` timed calls after
    three warm-up calls, each bracketed by CUDA events on the launching stream."""
    import torch
    stream = torch.cuda.current_stream(dev)
    base = workloads.CONFIGS[name]
    sets = []
    for s in range(NSETS):
        w = workloads.make(name, seed=base.seed + 17 * s)
        conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if w["dtype"] == "bf16" \
            else torch.from_numpy
        st = dict(tgt=conv(w["target"]).to(dev), drf=conv(w["draft"]).to(dev),
                  ud=torch.from_numpy(w["u_draft"]).to(dev), uv=torch.from_numpy(w["u_verify"]).to(dev))
        prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
        st["tok"] = sv.spec_sample_draft(st["drf"], None if w["greedy"] else st["ud"], **prm)
        sets.append(st)
    B, K, V = w["B"], w["K"], w["V"]
    dt_code = sv.SPEC_BF16 if w["dtype"] == "bf16" else sv.SPEC_F32
    ws = torch.zeros(sv.spec_verify_workspace_size(B, K, V, dt_code, w["greedy"]), dtype=torch.uint8, device=dev)
    out_t = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)

    def verify(s):
        st = sets[s]
        sv.spec_verify(st["tgt"], None if w["greedy"] else st["drf"], st["tok"], None if w["greedy"] else st["uv"],
                       out_tokens=out_t, out_num_accepted=out_n, ws=ws, **prm)

    for j in range(3):
        verify(j % NSETS)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for j in range(steps):
        ev[j][0].record(stream)
        verify(j % NSETS)
        ev[j][1].record(stream)
    torch.cuda.synchronize(dev)
    avg_us = sum(a.elapsed_time(b) for a, b in ev) / steps * 1e3
    rows = rows_per_step(w)[1]
    nbytes = rows * V * esize(w)
    peak, _ = measured_peaks()
    gbs = nbytes / (avg_us / 1e6) / 1e9
    del sets, ws
    torch.cuda.empty_cache()
    return {"workload": workload_desc(name, w), "avg_us": avg_us, "rows": rows, "bytes": nbytes, "gbs": gbs,
            "frac": gbs / peak, "rows_per_s": rows / (avg_us / 1e6), "steps": steps}


def run_gpu(args, name):
    import torch
    import speculative_sampling_verification_spec_gb300 as sv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sv.binding.lib()

    # inputs: NSETS seeded sets per rank (rank offsets the seed: weak scaling)
    base = workloads.CONFIGS[name]
    sets = []
    host_first = None
    for s in range(NSETS):
        w = workloads.make(name, seed=base.seed + 1000 * rank + 17 * s)
        if s == 0:
            host_first = w
        conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if w["dtype"] == "bf16" \
            else torch.from_numpy
        sets.append(dict(tgt=conv(w["target"]).to(dev), drf=conv(w["draft"]).to(dev),
                         ud=torch.from_numpy(w["u_draft"]).to(dev),
                         uv=torch.from_numpy(w["u_verify"]).to(dev),
                         tok=torch.zeros((w["B"], w["K"]), dtype=torch.int32, device=dev)))
    w = host_first
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    B, K, V = w["B"], w["K"], w["V"]
    dt_code = sv.SPEC_BF16 if w["dtype"] == "bf16" else sv.SPEC_F32
    ws_v = torch.zeros(sv.spec_verify_workspace_size(B, K, V, dt_code, w["greedy"]), dtype=torch.uint8, device=dev)
    ws_s = torch.zeros(sv.spec_sample_draft_workspace_size(B, K, V, dt_code, w["greedy"]), dtype=torch.uint8, device=dev)
    out_t = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)

    def sample(s):
        st = sets[s]
        sv.spec_sample_draft(st["drf"], None if w["greedy"] else st["ud"], out_tokens=st["tok"], ws=ws_s, **prm)

    def verify(s):
        st = sets[s]
        sv.spec_verify(st["tgt"], None if w["greedy"] else st["drf"], st["tok"],
                       None if w["greedy"] else st["uv"], out_tokens=out_t, out_num_accepted=out_n,
                       ws=ws_v, **prm)

    for s in range(NSETS):
        sample(s)
    for j in range(args.warmup):
        sample((j + 1) % NSETS)
        verify(j % NSETS)
    torch.cuda.synchronize(dev)

    rs, rv = rows_per_step(w)
    es = esize(w)
    bytes_s, bytes_v = rs * V * es, rv * V * es

    def timed(steps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        n0 = sv.spec_launch_count()
        clk = ClockSampler(local)
        clk.start()
        time.sleep(0.25)  # let the sampler come up before the timed region
        t_host = time.perf_counter()
        for j in range(steps):
            e0, e1, e2 = ev[j]
            e0.record(stream)
            sample((j + 1) % NSETS)
            e1.record(stream)
            verify(j % NSETS)
            e2.record(stream)
        torch.cuda.synchronize(dev)
        t_host = time.perf_counter() - t_host
        clocks = clk.stop()
        launches = sv.spec_launch_count() - n0
        t_s = [ev[j][0].elapsed_time(ev[j][1]) for j in range(steps)]
        t_v = [ev[j][1].elapsed_time(ev[j][2]) for j in range(steps)]
        total_ms = ev[0][0].elapsed_time(ev[-1][2])
        return dict(total_ms=total_ms, t_s=t_s, t_v=t_v, launches=launches, clocks=clocks, t_host=t_host)

    r = timed(args.steps)
    note = None
    if set(r["clocks"]["reasons"]) & BAD_REASONS:
        note = "first measurement saw %s; re-measured once" % sorted(set(r["clocks"]["reasons"]) & BAD_REASONS)
        r = timed(args.steps)
    total_ms = r["total_ms"]
    if dist is not None:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_step = total_ms / args.steps
    rows_step = rs + rv
    value = world * rows_step * args.steps / (total_ms / 1e3)
    avg_v = sum(r["t_v"]) / len(r["t_v"])
    avg_s = sum(r["t_s"]) / len(r["t_s"])
    peak, peak_kind = measured_peaks()
    achieved = bytes_v / (avg_v / 1e3) / 1e9

    # end to end through the public API: host (pinned) inputs -> device -> outputs -> host
    e2e_steps = max(3, min(args.steps, 50))
    conv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)) if w["dtype"] == "bf16" \
        else torch.from_numpy
    h_t = conv(w["target"]).pin_memory()
    h_d = conv(w["draft"]).pin_memory()
    h_ud = torch.from_numpy(w["u_draft"]).pin_memory()
    h_uv = torch.from_numpy(w["u_verify"]).pin_memory()
    h_out_t = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    h_out_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    d_t, d_d = torch.empty_like(h_t, device=dev), torch.empty_like(h_d, device=dev)
    d_ud, d_uv = torch.empty_like(h_ud, device=dev), torch.empty_like(h_uv, device=dev)
    d_tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    h2d = (h_t.numel() * h_t.element_size() + (0 if w["greedy"] else
           h_d.numel() * h_d.element_size() + h_ud.numel() * 8 + h_uv.numel() * 8))
    if w["greedy"]:
        h2d += h_d.numel() * h_d.element_size()  # greedy drafts are still drawn from the draft rows
    d2h = h_out_t.numel() * 4 + h_out_n.numel() * 4

    def e2e_step():
        d_t.copy_(h_t, non_blocking=True)
        d_d.copy_(h_d, non_blocking=True)
        if not w["greedy"]:
            d_ud.copy_(h_ud, non_blocking=True)
            d_uv.copy_(h_uv, non_blocking=True)
        sv.spec_sample_draft(d_d, None if w["greedy"] else d_ud, out_tokens=d_tok, ws=ws_s, **prm)
        sv.spec_verify(d_t, None if w["greedy"] else d_d, d_tok, None if w["greedy"] else d_uv,
                       out_tokens=out_t, out_num_accepted=out_n, ws=ws_v, **prm)
        h_out_t.copy_(out_t, non_blocking=True)
        h_out_n.copy_(out_n, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(2):
        e2e_step()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = time.perf_counter() - t0
    if dist is not None:
        t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_val = world * rows_step * e2e_steps / e2e_s

    # acceptance telemetry on the last verify's counts (outside the timed step):
    # launch latency, as it reads only B int32
    hist = torch.zeros((K + 2,), dtype=torch.int32, device=dev)
    for _ in range(3):
        sv.spec_accept_histogram(out_n, K, hist=hist)
    nh = 200
    h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0.record(stream)
    for _ in range(nh):
        sv.spec_accept_histogram(out_n, K, hist=hist)
    h1.record(stream)
    torch.cuda.synchronize(dev)
    hist_us = h0.elapsed_time(h1) * 1e3 / nh
    hist_ok = int(hist.sum().item()) == B * (nh + 3)

    # spec_verify alone on the other bandwidth-sized workloads (not part of the step)
    others = {}
    if rank == 0 and world == 1 and not args.no_others:
        for o in ("c3", "c4", "c4_bf16", "c5"):
            if o != name:
                others[o] = verify_only(o, 50, dev, sv)

    base_cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base_cpu = cpu_baseline(host_first, os.cpu_count() or 1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(name, w), "input_dtype": w["dtype"],
                       "global_batch": B * world, "vocab": V, "draft_len": K,
                       "rows_per_step": rows_step, "step": "spec_sample_draft + spec_verify",
                       "l2": "%d rotating device input sets (%.0f MB) > L2; step j samples set j+1, verifies set j"
                             % (NSETS, NSETS * (bytes_v) / 1e6),
                       "parallelism": "dp%d (independent batches)" % world},
            "gbs": (bytes_s + bytes_v) * world / (ms_step / 1e3) / 1e9,
            "kernels": {"spec_verify": {"avg_us": avg_v * 1e3, "rows": rv, "bytes": bytes_v,
                                        "gbs": achieved, "rows_per_s": rv / (avg_v / 1e3)},
                        "spec_sample_draft": {"avg_us": avg_s * 1e3, "rows": rs, "bytes": bytes_s,
                                              "gbs": bytes_s / (avg_s / 1e3) / 1e9,
                                              "rows_per_s": rs / (avg_s / 1e3)},
                        "spec_accept_histogram": {"avg_us": hist_us, "sequences": B, "counts_ok": hist_ok,
                                                  "accepted_per_round": float(
                                                      (torch.arange(K + 1, device=dev) * hist[:K + 1]).sum().item()
                                                      / max(1, int(hist[:K + 1].sum().item())))}},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(args.workload),
                         "kernel": verify_kernel_name(w),
                         "peak_kind": peak_kind},
            "e2e": {"value": e2e_val, "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "steps": e2e_steps},
            "gpu_launches": int(r["launches"]),
            "clocks": {k: r["clocks"][k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples")},
        }
        if others:
            line["verify_other_workloads"] = others
        if note:
            line["clocks"]["note"] = note
        if base_cpu is not None:
            line["cpu_baseline"] = base_cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_decode(args):
    """Decode rounds through the driver (spec_sample_draft x K, then spec_verify)
    on a source with acceptance exactly 0.8 at the c5 shape: tokens per round
    against the closed form, and the round rate."""
    import torch
    from speculative_sampling_verification_spec_gb300 import decode
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    alpha, B, K, V, rounds = 0.8, 32, 8, 256000, max(10, args.steps // 50)
    src = workloads.synthetic_source(V=V, S=64, alpha=alpha, seed=12, dtype="bf16")
    conv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    tt, dt = conv(src.target), conv(src.draft)
    first = torch.from_numpy(np.random.default_rng(4).integers(0, V // 2, B)).to(dev)
    state = lambda last, pos: workloads.state_of(last, pos, src.S)
    unis = [workloads.round_uniforms(13, r, B, K) for r in range(rounds + 3)]
    decode.decode_rounds(tt, dt, state, first, K, 3, lambda r: unis[r])
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    got = decode.decode_rounds(tt, dt, state, first, K, rounds, lambda r: unis[r])
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    n1 = torch.cat([n for _, n in got]).double() + 1
    line = {"mode": "decode", "metric": "tokens per round and rounds/s of the decode loop", "B": B, "K": K, "V": V,
            "dtype": "bf16", "alpha": alpha, "rounds": rounds,
            "tokens_per_round": float(n1.mean()), "tokens_per_round_sd": float(n1.std()),
            "closed_form": decode.expected_tokens_per_round(alpha, K),
            "ms_per_round": ms / rounds, "rounds_per_s": rounds / (ms / 1e3),
            "tokens_per_s": float(n1.sum()) / (ms / 1e3),
            "round": "K spec_sample_draft calls (B rows each) + row gathers standing in for the model calls "
                     "+ one spec_verify; uniforms copied from the host each round"}
    print(json.dumps(line), flush=True)
    return 0


def run_sweep_k(args):
    """spec_verify time against K at the c5 shape (B=32, V=256000 bf16, top-k 50),
    and the speed-up the latency model gives with that cost added to the pages'
    round (Chinchilla 70B target 14.1 ms per call, 4B draft 1.8 ms per call)."""
    import torch
    import speculative_sampling_verification_spec_gb300 as sv
    from speculative_sampling_verification_spec_gb300 import decode
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    t_target, t_draft = 14.1, 1.8
    c = t_draft / t_target
    rows = []
    for K in range(1, 9):
        w = workloads.make("c5", K=K)
        prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
        conv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        tgt, drf = conv(w["target"]), conv(w["draft"])
        tok = sv.spec_sample_draft(drf, torch.from_numpy(w["u_draft"]).to(dev), **prm)
        uv = torch.from_numpy(w["u_verify"]).to(dev)
        for _ in range(5):
            sv.spec_verify(tgt, drf, tok, uv, **prm)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = 50
        e0.record()
        for _ in range(n):
            sv.spec_verify(tgt, drf, tok, uv, **prm)
        e1.record()
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / n
        rows.append({"K": K, "verify_us": us, "rows": w["B"] * (2 * K + 1)})
    # K = 1: the fused drafting step + verification against the two separate calls
    w = workloads.make("c5", K=1)
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    conv = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    tgt, drf = conv(w["target"]), conv(w["draft"])
    ud2 = torch.from_numpy(w["u_draft"]).to(dev)
    ud1 = ud2[:, 0].contiguous()
    uv = torch.from_numpy(w["u_verify"]).to(dev)

    def fused():
        sv.spec_sample_verify(tgt, drf, ud1, uv, **prm)

    def separate():
        d = sv.spec_sample_draft(drf, ud2, **prm)
        sv.spec_verify(tgt, drf, d, uv, **prm)

    k1 = {}
    for nm, fn in (("fused_us", fused), ("separate_us", separate)):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(50):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        k1[nm] = e0.elapsed_time(e1) * 1e3 / 50
    k1["bytes_fused"] = w["B"] * 3 * w["V"] * 2
    k1["bytes_separate"] = w["B"] * 4 * w["V"] * 2
    # ragged batch at the c5 shape: draft lengths spread over 1..8, against the padded call
    w = workloads.make("c5")
    prm = dict(temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], greedy=w["greedy"])
    tgt, drf = conv(w["target"]), conv(w["draft"])
    tok = sv.spec_sample_draft(drf, torch.from_numpy(w["u_draft"]).to(dev), **prm)
    uv = torch.from_numpy(w["u_verify"]).to(dev)
    lens = (np.arange(w["B"]) % w["K"] + 1).astype(np.int32)
    rg = {}
    for nm, fn in (("ragged_us", lambda: sv.spec_verify_ragged(tgt, drf, tok, uv, lens, **prm)),
                   ("padded_us", lambda: sv.spec_verify(tgt, drf, tok, uv, **prm))):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(50):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        rg[nm] = e0.elapsed_time(e1) * 1e3 / 50
    rg["rows_ragged"] = int((2 * lens + 1).sum())
    rg["rows_padded"] = w["B"] * (2 * w["K"] + 1)
    vc = {r["K"]: r["verify_us"] / 1e3 / t_target for r in rows}
    model = []
    for alpha in (0.75, 0.8):
        model.append({"alpha": alpha, "c": c,
                      "speedup": {r["K"]: decode.speedup(alpha, r["K"], c, vc[r["K"]]) for r in rows},
                      "speedup_without_verify": {r["K"]: decode.speedup(alpha, r["K"], c) for r in rows},
                      "best_k": decode.best_k(alpha, c, lambda k: vc.get(k, vc[8]), 8),
                      "best_k_without_verify": decode.best_k(alpha, c, lambda k: 0.0, 8)})
    line = {"mode": "sweep_k", "metric": "spec_verify time vs K (c5 shape) and modelled speed-up",
            "workload": "c5 with K = 1..8 (B=32, V=256000 bf16, top_k=50)", "verify": rows,
            "model": model, "t_target_ms": t_target, "t_draft_ms": t_draft,
            "k1_sample_verify": k1, "ragged_c5": rg}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="c5", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the spec_verify-only lines of the other workloads")
    ap.add_argument("--decode", action="store_true", help="decode-loop line instead of the verify line")
    ap.add_argument("--sweep-k", action="store_true", help="verify time vs K and the latency model")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode:
        return run_decode(args)
    if args.sweep_k:
        return run_sweep_k(args)
    if args.impl == "reference":
        return run_reference(args, args.workload)
    return run_gpu(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
