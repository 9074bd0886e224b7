"""Throughput of the DSpark decode-cycle hot path on GB300.

One step = one whole decode cycle of the workload through the library's C ABI:
prefix selection -> Markov-head block draft -> lossless verify -> commit
lengths, on seeded synthetic inputs already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched_sampling]

Prints one JSON line.  For N > 1 it runs under torch.distributed.run, one
rank per GPU; every rank runs its own replica of the workload (requests are
independent, no collective is needed), the time is the max over ranks and
`value` counts the cycles of all ranks.  `--impl reference` times the CPU
oracle (single-threaded C++) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_decoding_dspark_gb300 import inputs  # noqa: E402

METRIC = "draft+verify cycles/s"
UNIT = "cycles/s"
DEFAULT_WORKLOAD = "batched_sampling"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stage", choices=["cycle", "draft", "verify"], default="cycle",
                    help="time the whole cycle (default) or one call of it (profiling)")
    ap.add_argument("--gamma", type=int, default=None, help="override the workload's block size")
    ap.add_argument("--temperature", type=float, default=None, help="override the workload's T")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world, device="cuda"):
    """The largest x over the ranks of the job (its slowest replica's time);
    x itself when the job has one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units per second of the whole job: every rank processed units_per_rank
    in at most ms milliseconds."""
    return world * units_per_rank / (ms / 1000.0)


L2_BYTES = 129 * 2**20  # GB300 L2


def input_bytes(w):
    """Input bytes of one cycle: W2 once per draft position, U, and the presented
    target rows (fp32; verify reads them only up to each first rejection)."""
    R, V, gamma, rank = w["R"], w["V"], w["gamma"], w["rank"]
    return gamma * V * rank * 2 + R * gamma * V * 2 + R * (gamma + 1) * V * 4


def workload_config(w):
    nb = input_bytes(w)
    l2 = (f"inputs larger than L2 (no flush): W2 per draft position, U and the presented target "
          f"logits total ~{nb / 1e9:.2f} GB per step"
          if nb > L2_BYTES else f"inputs ({nb / 1e6:.1f} MB per step) fit in L2: not a bench workload")
    return {"workload": w["name"], "R": w["R"], "V": w["V"], "gamma": w["gamma"],
            "rank": w["rank"], "temperature": float(w["temperature"]), "l2": l2}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w, d, full, n_req, cycle):
    """Time the oracle on n_req requests of the workload (draft all gamma
    positions + verify); returns (seconds per request, sample text)."""
    import oracle
    oracle.build()
    R, gamma = w["R"], w["gamma"]
    T = float(w["temperature"])
    rows = list(np.linspace(0, R - 1, n_req).astype(int))
    l = np.full(len(rows), gamma, np.int32)
    t0 = time.perf_counter()
    o = oracle.markov_draft(d["U"][rows], d["W1"], d["W2"], d["anchor"][rows], d["seeds"][rows],
                            cycle, T, req_ids=rows)
    oracle.verify(inputs.pack_rows(full[rows], l), inputs.cu_from_lengths(l), o["y"], o["q_logits"],
                  d["seeds"][rows], cycle, T, req_ids=rows)
    oracle.commit_lengths(np.zeros(len(rows), np.int32), l, gamma)
    dt = time.perf_counter() - t0
    return dt / len(rows), f"{len(rows)} of {R} requests, whole cycle each (draft {gamma} positions + verify), scaled x{R}"


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = inputs.workload(args.workload)
    d = inputs.draft_inputs(w)
    full = inputs.target_full(w, d["U"])
    per_req = []
    sample = ""
    for step in range(args.warmup + args.steps):
        s, sample = oracle_sample(w, d, full, 1, step)
        if step >= args.warmup:
            per_req.append(s)
    cyc_s = 1.0 / (statistics.mean(per_req) * w["R"])
    line = {"metric": METRIC, "value": cyc_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 / cyc_s, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w), "impl": "reference",
            "cpu_baseline": {"value": cyc_s, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "each step: " + sample.replace("1 of", "1 request of")},
            "e2e": {"value": cyc_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.idx = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        top = max(mx)
        loaded = [s for s in sm if s > 0.5 * top] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": top, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm
def source_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def traffic_from_profile(kernel, digest):
    """dram bytes per launch recorded for this kernel's current source, or None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == kernel and f[1] == digest:
            return float(f[2])
    return None


def run_ours(args):
    import torch
    import torch.distributed as dist
    from speculative_decoding_dspark_gb300 import binding as B

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    over = {}
    if args.gamma is not None:
        over["gamma"] = args.gamma
    if args.temperature is not None:
        over["temperature"] = args.temperature
    w = inputs.workload(args.workload, **over)
    R, V, gamma, rank_r = w["R"], w["V"], w["gamma"], w["rank"]
    T = float(w["temperature"])
    d = inputs.draft_inputs(w)
    full = inputs.target_full(w, d["U"])
    ci = inputs.confidence_inputs(w)
    if w.get("confidence"):
        K_cap, mode = ci["K_cap"], B.DSPARK_SELECT_HISTORY
    else:  # fixed-length workloads: the capacity admits every draft position
        K_cap, mode = R * (gamma + 1), B.DSPARK_SELECT_FIXED
    max_rows = min(K_cap, R * (gamma + 1))

    def dev(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).cuda()
        return torch.from_numpy(x).cuda()

    U, W1, W2 = dev(d["U"]), dev(d["W1"]), dev(d["W2"])
    anchor, seeds = dev(d["anchor"]), dev(d["seeds"])
    c, c_hist = dev(ci["c"]), dev(ci["c_hist"])
    sizes, sps = dev(ci["capture_sizes"]), dev(ci["sps"])
    # target rows in full [R, gamma+1, V]; with every position selected the packed
    # layout equals it, otherwise the first max_rows rows of the buffer are read
    target = dev(full.reshape(R * (gamma + 1), V))
    del full
    i32 = dict(dtype=torch.int32, device="cuda")
    y = torch.empty((R, gamma), **i32)
    q_lse = torch.empty((R, gamma), device="cuda")
    q_tok = torch.empty((R, gamma), device="cuda")
    # the verify recomputes the drafter's rejected rows from its factors, so the
    # draft keeps no logits in memory
    q_logits = None
    a = torch.empty((R, gamma), device="cuda")
    l = torch.empty(R, **i32)
    cu = torch.empty(R + 1, **i32)
    K_used = torch.empty(1, **i32)
    n_acc = torch.empty(R, **i32)
    out = torch.empty((R, gamma + 1), **i32)
    p_tok = torch.empty((R, gamma), device="cuda")
    cl = torch.empty(R, **i32)
    cuc = torch.empty(R + 1, **i32)
    disc = torch.empty(R, **i32)
    tot = torch.empty(1, **i32)
    status = torch.zeros(1, **i32)
    ws_d = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank_r, 0, B.DSPARK_BF16))
    ws_v = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY_MARKOV, R, gamma, V, rank_r, max_rows))
    stream = torch.cuda.current_stream()
    uses_tc = B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, R, V, rank_r)

    run_select = run_commit = args.stage == "cycle"
    run_draft = args.stage in ("cycle", "draft")
    run_verify = args.stage in ("cycle", "verify")
    if args.stage == "verify":  # the verify stage needs lengths and a draft once
        B.dspark_select_prefix(c, c_hist, sizes, sps, K_cap, mode, a, l, cu, K_used, None, status)
        B.dspark_markov_draft(U, W1, W2, anchor, seeds, 0, T, y, q_lse, q_tok, q_logits, ws_d, status)

    def step(cycle, ev=None, inp=None):
        # inp: the per-cycle inputs (U, target, c, c_hist, anchor, seeds); default the resident ones
        U_, tgt_, c_, ch_, anc_, sd_ = inp if inp is not None else (U, target, c, c_hist, anchor, seeds)
        if ev is not None: ev[0].record(stream)
        if run_select:
            B.dspark_select_prefix(c_, ch_, sizes, sps, K_cap, mode, a, l, cu, K_used, None, status)
        if ev is not None: ev[1].record(stream)
        if run_draft:
            B.dspark_markov_draft(U_, W1, W2, anc_, sd_, cycle, T, y, q_lse, q_tok, q_logits, ws_d,
                                  status)
        if ev is not None: ev[2].record(stream)
        if run_verify:
            B.dspark_verify_markov(tgt_, cu, y, U_, W1, W2, anc_, q_lse, q_tok, sd_, cycle, T,
                                   max_rows, n_acc, out, p_tok, ws_v, status)
        if ev is not None: ev[3].record(stream)
        if run_commit:
            B.dspark_commit_lengths(n_acc, l, gamma, cl, cuc, disc, tot, status)
        if ev is not None: ev[4].record(stream)

    # launches of this library per step
    # tensor cores: every position and the finalize in one launch; CUDA cores:
    # counter reset, then bias and sample kernels per position
    draft_launches = 1 if uses_tc else 1 + 2 * gamma
    verify_launches = 4 if T > 0 else 2  # prologue, rounds, (residual draw, finalize)
    launches_per_step = (int(run_select) + draft_launches * int(run_draft) +
                         verify_launches * int(run_verify) + int(run_commit))

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i, evs[i])
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(start.elapsed_time(stop), world)
    per = {k: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
           for j, k in enumerate(["select", "draft", "verify", "commit"])}
    ms_step = ms / args.steps
    value = whole_job_rate(args.steps, world, ms)

    # roofline of the dominant kernel.  Algorithmic bytes of one Markov draft
    # step (one vocabulary pass): W2 once, U_k once, q_logits if written.  The
    # tensor-core kernel runs all gamma steps in one launch, timed as the whole
    # draft call (which adds the workspace reset, so the fraction is a lower
    # bound); the CUDA-core path is timed per step.
    step_bytes = V * rank_r * 2 + R * V * 2 + (R * V * 4 if q_logits is not None else 0)
    steps_per_launch = gamma if uses_tc else 1
    launch_bytes = step_bytes * steps_per_launch
    launch_ms = per["draft"] / gamma * steps_per_launch
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    hbm = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    achieved = launch_bytes / (launch_ms / 1000.0) / 1e9
    kname = "markov_tc_kernel<draft>" if uses_tc else "draft_bias_simt+draft_sample"
    digest = source_digest(["speculative_decoding_dspark_gb300/csrc/draft_tc.cu" if uses_tc else
                            "speculative_decoding_dspark_gb300/csrc/draft_simt.cu",
                            "speculative_decoding_dspark_gb300/csrc/common.cuh"])
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic_from_profile(kname, digest), "kernel": kname,
            "algorithmic_bytes_per_launch": launch_bytes, "steps_per_launch": steps_per_launch,
            "launch_ms": launch_ms,
            "peak_source": peak_src}

    # end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e and args.stage == "cycle":
        hU = U.cpu().pin_memory(); htgt = target.cpu().pin_memory(); hc = c.cpu().pin_memory()
        hch = c_hist.cpu().pin_memory(); ha = anchor.cpu().pin_memory(); hs = seeds.cpu().pin_memory()
        h_out = torch.empty((R, gamma + 1), dtype=torch.int32).pin_memory()
        h_n = torch.empty(R, dtype=torch.int32).pin_memory()
        h_cl = torch.empty(R + 1, dtype=torch.int32).pin_memory()
        bi = sum(t.numel() * t.element_size() for t in (hU, htgt, hc, hch, ha, hs))
        bo = sum(t.numel() * t.element_size() for t in (h_out, h_n, h_cl))

        # Each cycle's inputs go host -> device as chunks spread over four copy
        # streams (several copy engines), into one of two device input sets, so
        # the copies of cycle i + 1 overlap the kernels of cycle i; the kernels
        # of a cycle wait for its own copies, and a set is refilled only after
        # the cycle that read it has finished.
        copy_streams = [torch.cuda.Stream() for _ in range(4)]
        sets = [(U, target, c, c_hist, anchor, seeds),
                tuple(torch.empty_like(t) for t in (U, target, c, c_hist, anchor, seeds))]
        hosts = (hU, htgt, hc, hch, ha, hs)
        freed = [None, None]

        def issue_copies(b, after):
            for cs in copy_streams:
                if after is not None: cs.wait_event(after)
                if freed[b] is not None: cs.wait_event(freed[b])
            k = 0
            for dst, src in zip(sets[b], hosts):
                fd, fs = dst.view(-1), src.view(-1)
                n = fd.numel()
                pieces = max(1, min(16, (n * dst.element_size()) >> 25))  # ~32 MB pieces
                per = (n + pieces - 1) // pieces
                for j in range(pieces):
                    with torch.cuda.stream(copy_streams[k % len(copy_streams)]):
                        fd[j * per:(j + 1) * per].copy_(fs[j * per:(j + 1) * per], non_blocking=True)
                    k += 1
            done = []
            for cs in copy_streams:
                e = torch.cuda.Event()
                e.record(cs)
                done.append(e)
            return done

        def e2e_run(n, first_cycle, start_ev=None):
            pending = issue_copies(0, start_ev)
            for i in range(n):
                b = i & 1
                for e in pending:
                    stream.wait_event(e)
                if i + 1 < n:
                    pending = issue_copies((i + 1) & 1, None)
                step(first_cycle + i, inp=sets[b])
                fe = torch.cuda.Event()
                fe.record(stream)
                freed[b] = fe
                h_out.copy_(out, non_blocking=True); h_n.copy_(n_acc, non_blocking=True)
                h_cl.copy_(cuc, non_blocking=True)

        n_e2e = max(3, min(args.steps, 20))
        e2e_run(2, 0)
        torch.cuda.synchronize()
        freed[0] = freed[1] = None
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        e2e_run(n_e2e, 100, s0)
        s1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(s0.elapsed_time(s1), world)
        e2e = {"value": whole_job_rate(n_e2e, world, e_ms), "unit": UNIT,
               "h2d_gb_s": bi * n_e2e / (e_ms / 1000.0) / 1e9, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "steps": n_e2e}

    # verify reads target rows only up to each request's first rejection: its
    # data-dependent algorithmic bytes (those rows, plus for T > 0 the residual
    # draw's W2 pass and one target row and one U row per request) per verify call
    verify_roof = None
    if run_verify:
        n_h = n_acc.cpu().numpy().astype(np.int64)
        l_h = l.cpu().numpy().astype(np.int64)
        ok = n_h >= 0
        rows_read = int((np.minimum(n_h[ok], l_h[ok]) + 1).sum())
        vbytes = rows_read * V * 4
        if T > 0:
            vbytes += V * rank_r * 2 + int(ok.sum()) * V * (4 + 2)
        v_ms = per["verify"]
        verify_roof = {"bound": "hbm", "achieved": vbytes / (v_ms / 1000.0) / 1e9, "peak": hbm, "unit": "GB/s",
                       "frac": vbytes / (v_ms / 1000.0) / 1e9 / hbm, "algorithmic_bytes_per_call": vbytes,
                       "rows_read": rows_read, "rows_presented": int((l_h + 1).sum()), "call_ms": v_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.stage == "cycle":
        per_req, sample = oracle_sample(w, d, inputs.target_full(w, d["U"]), 4, 0)
        cpu = {"value": 1.0 / (per_req * R), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 GEMM (fp32 accumulate) + fp32 softmax/verify",
                "data": "synthetic (seeded; shapes and laws of the workload)",
                "config": dict(workload_config(w), parallelism=f"replicas x{world}"),
                "roofline": roof, "verify_roofline": verify_roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": launches_per_step * args.steps,
                "stage": args.stage, "stage_ms": per, "logits_gb_s": (R * (gamma + 1) * V * 4 + R * gamma * V * 2) /
                (ms_step / 1000.0) / 1e9, "draft_path": "tcgen05" if uses_tc else "simt"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
