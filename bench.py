"""Throughput of the DSpark decode-cycle hot path on GB300.

One step = one whole decode cycle of the workload through the library's C ABI:
prefix selection -> Markov-head block draft -> lossless verify -> commit
lengths, on seeded synthetic inputs already resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload batched_sampling]

Prints one JSON line.  For N > 1 it runs under torch.distributed.run, one
rank per GPU; every rank runs its own replica of the workload (requests are
independent, no collective is needed), the time is the max over ranks and
`value` counts the cycles of all ranks.

Timing: after W warm-up steps, blocks of exactly K steps are timed with CUDA
events on the launching stream, one block after another until about a second
has passed; `value` comes from the median block.  Each timed block replays one
CUDA graph of its K steps, captured once from the same library calls (stream
launches if the capture fails; `timing.launch` says which); the per-stage times
come from further stream-launched blocks with an event between the calls.  The
line also carries the other workloads of the pages (`workloads`: the tiny
exhaustive cycle in microseconds, the DeepSeek-style R=512, gamma=5, rank-512
confidence-scheduled cycle with its tensor-core fraction, the variable-length
verify timed alone, the greedy Qwen3-8B-shaped cycle, and the fused drafter
logits beside the unfused route).

`--impl reference` times the CPU oracle (single-threaded C++, one request per
task) over a pool of host processes, one per core: each timed step is one
whole cycle of every request of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import platform
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
BLOCK_SECONDS = 1.0  # timed blocks of K steps are repeated until this much time has passed
SIDE_SECONDS = 0.3   # the same for each side workload
STAGE_BLOCKS = 3     # blocks with an event between the calls of each step (per-stage times)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stage", choices=["cycle", "draft", "verify", "fused_draft"], default="cycle",
                    help="time the whole cycle (default) or one call of it (profiling); fused_draft: "
                         "the fused drafter logits on the fused_logits workload alone")
    ap.add_argument("--gamma", type=int, default=None, help="override the workload's block size")
    ap.add_argument("--temperature", type=float, default=None, help="override the workload's T")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="skip the other workloads (profiling runs)")
    ap.add_argument("--blocks", type=int, default=None,
                    help="timed blocks of K steps (default: repeat for about a second)")
    return ap.parse_args(argv)


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


def workload_config(w, world=1):
    """The `config` object; both arms print the same one."""
    nb = input_bytes(w)
    l2 = (f"inputs larger than L2 (no flush): W2 per draft position, U and the presented target "
          f"logits total ~{nb / 1e9:.2f} GB per step"
          if nb > L2_BYTES else f"inputs ({nb / 1e6:.1f} MB per step) fit in L2: not a bench workload")
    return {"workload": w["name"], "R": w["R"], "V": w["V"], "gamma": w["gamma"],
            "rank": w["rank"], "temperature": float(w["temperature"]), "l2": l2,
            "parallelism": f"replicas x{world}"}


def host_cpu():
    """CPU model and the number of cores this process may use."""
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return model, n


# ---------------------------------------------------------------- CPU oracle
# The oracle is single-threaded; the requests of a cycle are independent (their
# draws are addressed by request index), so a pool of worker processes, one per
# host core, each replays whole requests.  The pool is forked before this
# process makes any CUDA call, after the inputs exist, so the workers share the
# input arrays instead of copying them.
_ORC = {}


def _oracle_request(job):
    """Draft all gamma positions and verify one request on the oracle; returns
    its number of accepted drafts."""
    r, cycle = job
    import oracle
    w, d, full = _ORC["w"], _ORC["d"], _ORC["full"]
    gamma, T = w["gamma"], float(w["temperature"])
    rows = [r]
    l = np.full(1, gamma, np.int32)
    o = oracle.markov_draft(d["U"][rows], d["W1"], d["W2"], d["anchor"][rows], d["seeds"][rows],
                            cycle, T, req_ids=rows)
    v = oracle.verify(inputs.pack_rows(full[rows], l), inputs.cu_from_lengths(l), o["y"], o["q_logits"],
                      d["seeds"][rows], cycle, T, req_ids=rows)
    return int(v["n_acc"][0])


class OraclePool:
    """Worker processes for the CPU oracle (fork: create it before any CUDA call)."""

    def __init__(self, w, d, full, n_proc):
        import oracle
        oracle.build()
        _ORC.update(w=w, d=d, full=full)
        self.n = max(1, min(n_proc, w["R"]))
        self.pool = mp.get_context("fork").Pool(self.n)
        self.w = w

    def cycle(self, cycle, requests=None):
        """One cycle of the given requests (default: all), with the whole-batch
        steps (commit lengths) in this process; returns the seconds it took."""
        import oracle
        R, gamma = self.w["R"], self.w["gamma"]
        reqs = list(range(R)) if requests is None else list(requests)
        t0 = time.perf_counter()
        n_acc = self.pool.map(_oracle_request, [(r, cycle) for r in reqs], chunksize=1)
        oracle.commit_lengths(np.asarray(n_acc, np.int32), np.full(len(reqs), gamma, np.int32), gamma)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = inputs.workload(args.workload)
    d = inputs.draft_inputs(w)
    full = inputs.target_full(w, d["U"])
    model, ncpu = host_cpu()
    pool = OraclePool(w, d, full, ncpu)
    R = w["R"]
    try:
        # warm-up steps: one request per worker (untimed); timed steps: whole cycles
        for step in range(args.warmup):
            pool.cycle(step, [(step * pool.n + i) % R for i in range(pool.n)])
        secs = [pool.cycle(args.warmup + step) for step in range(args.steps)]
    finally:
        pool.close()
    ms_step = 1000.0 * statistics.mean(secs)
    cyc_s = 1000.0 / ms_step
    sample = (f"each timed step: one whole cycle of all {R} requests (draft {w['gamma']} positions + "
              f"verify + commit), requests spread over {pool.n} worker processes")
    line = {"metric": METRIC, "value": cyc_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, world), "impl": "reference",
            "cpu_baseline": {"value": cyc_s, "unit": UNIT, "cores": pool.n, "kind": "oracle",
                             "sample": sample, "cpu_model": model, "nproc": ncpu},
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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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


def load_peaks():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(pk)) if os.path.exists(pk) else {}


class Cycle:
    """Device tensors and the launch sequence of one workload's decode cycle."""

    def __init__(self, w, host, stage="cycle"):
        import torch
        from speculative_decoding_dspark_gb300 import binding as B
        self.B, self.torch, self.w, self.stage = B, torch, w, stage
        d, full, ci = host["d"], host["full"], host["ci"]
        R, V, gamma, rank = w["R"], w["V"], w["gamma"], w["rank"]
        self.R, self.V, self.gamma, self.rank = R, V, gamma, rank
        self.T = float(w["temperature"])
        if w.get("confidence"):
            self.K_cap, self.mode = ci["K_cap"], B.DSPARK_SELECT_HISTORY
        else:  # fixed-length workloads: the capacity admits every draft position
            self.K_cap, self.mode = R * (gamma + 1), B.DSPARK_SELECT_FIXED
        self.max_rows = min(self.K_cap, R * (gamma + 1))
        self.varlen = bool(w.get("varlen"))

        def dev(x):
            x = np.ascontiguousarray(x)
            if x.dtype == np.uint16:
                return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
            if x.dtype == np.uint64:
                return torch.from_numpy(x.view(np.int64)).cuda()
            return torch.from_numpy(x).cuda()

        self.U, self.W1, self.W2 = dev(d["U"]), dev(d["W1"]), dev(d["W2"])
        self.anchor, self.seeds = dev(d["anchor"]), dev(d["seeds"])
        self.c, self.c_hist = dev(ci["c"]), dev(ci["c_hist"])
        self.sizes, self.sps = dev(ci["capture_sizes"]), dev(ci["sps"])
        i32 = dict(dtype=torch.int32, device="cuda")
        if self.varlen:
            # variable verify lengths drawn by the workload: packed rows and fixed
            # cu_seqlens (no selection step)
            l = inputs.verify_lengths(w)
            self.target = dev(inputs.pack_rows(full, l))
            self.l = dev(l)
            self.cu = dev(inputs.cu_from_lengths(l))
            self.max_rows = int(self.target.shape[0])
        else:
            # target rows in full [R, gamma+1, V]; with every position selected the
            # packed layout equals it, otherwise the first max_rows rows are read
            self.target = dev(full.reshape(R * (gamma + 1), V))
            self.l = torch.empty(R, **i32)
            self.cu = torch.empty(R + 1, **i32)
        self.y = torch.empty((R, gamma), **i32)
        self.q_lse = torch.empty((R, gamma), device="cuda")
        self.q_tok = torch.empty((R, gamma), device="cuda")
        self.a = torch.empty((R, gamma), device="cuda")
        self.K_used = torch.empty(1, **i32)
        self.n_acc = torch.empty(R, **i32)
        self.out = torch.empty((R, gamma + 1), **i32)
        self.p_tok = torch.empty((R, gamma), device="cuda")
        self.cl = torch.empty(R, **i32)
        self.cuc = torch.empty(R + 1, **i32)
        self.disc = torch.empty(R, **i32)
        self.tot = torch.empty(1, **i32)
        self.status = torch.zeros(1, **i32)
        self.ws_d = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank, 0,
                                                        B.DSPARK_BF16))
        self.ws_v = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY_MARKOV, R, gamma, V, rank,
                                                        self.max_rows))
        self.stream = torch.cuda.current_stream()
        self.uses_tc = B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, R, V, rank)
        self.run_select = stage == "cycle" and not self.varlen
        self.run_commit = stage == "cycle"
        self.run_draft = stage in ("cycle", "draft")
        self.run_verify = stage in ("cycle", "verify")
        if not self.run_draft or not self.run_select:  # lengths and a draft exist once
            if not self.varlen:
                self._select()
            if not self.run_draft:
                self._draft(0, self.U, self.anchor, self.seeds)
        # launches of this library per step: tensor cores, every position and the
        # finalize in one launch; CUDA cores, counter reset then bias and sample
        # kernels per position.  Verify: prologue, rounds (and the residual draw).
        draft_launches = 1 if self.uses_tc else 1 + 2 * gamma
        verify_launches = 3 if self.T > 0 else 2
        self.launches_per_step = (int(self.run_select) + draft_launches * int(self.run_draft) +
                                  verify_launches * int(self.run_verify) + int(self.run_commit))

    def _select(self, c=None, ch=None):
        self.B.dspark_select_prefix(self.c if c is None else c, self.c_hist if ch is None else ch, self.sizes,
                                    self.sps, self.K_cap, self.mode, self.a, self.l, self.cu, self.K_used,
                                    None, self.status)

    def _draft(self, cycle, U, anchor, seeds):
        self.B.dspark_markov_draft(U, self.W1, self.W2, anchor, seeds, cycle, self.T, self.y, self.q_lse,
                                   self.q_tok, None, self.ws_d, self.status)

    def step(self, cycle, ev=None, inp=None, ws_v=None):
        # inp: the per-cycle inputs (U, target, c, c_hist, anchor, seeds); default the resident ones
        U_, tgt_, c_, ch_, anc_, sd_ = inp if inp is not None else (self.U, self.target, self.c, self.c_hist,
                                                                    self.anchor, self.seeds)
        ws_v = self.ws_v if ws_v is None else ws_v
        s = self.stream
        if ev is not None: ev[0].record(s)
        if self.run_select:
            self._select(c_, ch_)
        if ev is not None: ev[1].record(s)
        if self.run_draft:
            self._draft(cycle, U_, anc_, sd_)
        if ev is not None: ev[2].record(s)
        if self.run_verify:
            self.B.dspark_verify_markov(tgt_, self.cu, self.y, U_, self.W1, self.W2, anc_, self.q_lse, self.q_tok,
                                        sd_, cycle, self.T, self.max_rows, self.n_acc, self.out, self.p_tok,
                                        ws_v, self.status)
        if ev is not None: ev[3].record(s)
        if self.run_commit:
            self.B.dspark_commit_lengths(self.n_acc, self.l, self.gamma, self.cl, self.cuc, self.disc, self.tot,
                                         self.status)
        if ev is not None: ev[4].record(s)

    def timed_blocks(self, steps, first_cycle, seconds, n_blocks=None, stage_blocks=STAGE_BLOCKS):
        """Blocks of exactly `steps` steps, each bracketed by CUDA events on the
        launching stream, repeated until `seconds` have passed (or n_blocks); then
        `stage_blocks` more blocks with an event between the calls of every step,
        which give the per-stage times (the timed blocks carry no events inside,
        so the markers do not add to the measured time).  The timed blocks replay
        one CUDA graph of the block's `steps` steps (captured once: every replay
        runs the same cycles' kernels again); if the capture fails they launch on
        the stream and self.launch_mode says why.
        Returns (per-block ms, per-stage mean ms, steps in the timed blocks,
        median ms of the blocks with stage events)."""
        torch = self.torch
        blocks, evs_all, staged, cyc = [], [], [], first_cycle

        def block(evs):
            nonlocal cyc
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(self.stream)
            for i in range(steps):
                self.step(cyc, evs[i] if evs else None)
                cyc += 1
            b1.record(self.stream)
            torch.cuda.synchronize()
            return b0.elapsed_time(b1)

        graph = None
        try:
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                for i in range(steps):
                    self.step(first_cycle + i)
            graph.replay()
            torch.cuda.synchronize()
            self.launch_mode = "cuda_graph"
        except Exception as exc:  # noqa: BLE001 -- any capture failure falls back to the stream
            graph = None
            torch.cuda.synchronize()
            self.launch_mode = "stream (graph capture failed: %s)" % str(exc).splitlines()[0][:160]
            try:  # a call that picks up the failed capture's error state
                self.step(first_cycle)
            except Exception:  # noqa: BLE001
                pass
            torch.cuda.synchronize()

        def graph_block():
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(self.stream)
            graph.replay()
            b1.record(self.stream)
            torch.cuda.synchronize()
            return b0.elapsed_time(b1)

        t_end = time.perf_counter() + seconds
        while (n_blocks is None and (not blocks or time.perf_counter() < t_end)) or \
                (n_blocks is not None and len(blocks) < n_blocks):
            blocks.append(graph_block() if graph is not None else block(None))
        for _ in range(max(1, stage_blocks)):
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
            staged.append(block(evs))
            evs_all.extend(evs)
        per = {k: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs_all)
               for j, k in enumerate(["select", "draft", "verify", "commit"])}
        assert int(self.status.item()) == 0, f"device status {int(self.status.item())} after the timed blocks"
        return blocks, per, len(blocks) * steps, statistics.median(staged)

    def rows_read(self):
        """Target rows the last verify read: up to each request's first rejection."""
        n_h = self.n_acc.cpu().numpy().astype(np.int64)
        l_h = self.l.cpu().numpy().astype(np.int64)
        ok = n_h >= 0
        return int((np.minimum(n_h[ok], l_h[ok]) + 1).sum()), int((l_h + 1).sum()), int(ok.sum())

    def verify_bytes(self):
        """Data-dependent algorithmic bytes of the last verify call: the rows read,
        plus for T > 0 the residual draw's W2 pass and one target row and one U
        row per request."""
        rows, presented, n_ok = self.rows_read()
        b = rows * self.V * 4
        if self.T > 0:
            b += self.V * self.rank * 2 + n_ok * self.V * (4 + 2)
        return b, rows, presented

    def draft_bytes(self):
        """Algorithmic bytes of one draft call: W2 and U_k once per position."""
        return self.gamma * (self.V * self.rank * 2 + self.R * self.V * 2)

    def draft_flops(self):
        return 2.0 * self.R * self.V * self.rank * self.gamma


def host_inputs(w):
    d = inputs.draft_inputs(w)
    return dict(d=d, full=inputs.target_full(w, d["U"]), ci=inputs.confidence_inputs(w))


def side_workload(name, args, peaks):
    """One of the pages' other workloads, measured on its own: cycles/s, the
    draft's HBM and tensor fractions, and the verify call's HBM fraction (for
    the variable-length workload, verify timed alone)."""
    import torch
    w = inputs.workload(name)
    host = host_inputs(w)
    verify_alone = bool(w.get("varlen"))
    cyc = Cycle(w, host, stage="verify" if verify_alone else "cycle")
    del host
    for i in range(args.warmup):
        cyc.step(i)
    torch.cuda.synchronize()
    assert int(cyc.status.item()) == 0, f"{name}: device status {int(cyc.status.item())}"
    blocks, per, n, _ = cyc.timed_blocks(args.steps, args.warmup, SIDE_SECONDS)
    ms_block = statistics.median(blocks)
    hbm = peaks.get("hbm_gbs") or 6800.0
    tens = peaks.get("bf16_tflops_sustained") or 1700.0
    out = {"R": w["R"], "V": w["V"], "gamma": w["gamma"], "rank": w["rank"],
           "temperature": float(w["temperature"]), "blocks": len(blocks), "steps_per_block": args.steps,
           "stage_ms": per}
    vb, rows, presented = cyc.verify_bytes()
    v_ms = per["verify"]
    out["verify"] = {"ms": v_ms, "algorithmic_bytes": vb, "rows_read": rows, "rows_presented": presented,
                     "achieved_gbs": vb / (v_ms / 1e3) / 1e9, "frac_hbm": vb / (v_ms / 1e3) / 1e9 / hbm}
    if verify_alone:
        out["metric"] = "verify calls/s (verify timed alone)"
        out["value"] = 1000.0 * args.steps / ms_block
    else:
        out["metric"] = METRIC
        out["value"] = 1000.0 * args.steps / ms_block
        d_ms = per["draft"]
        fl = cyc.draft_flops()
        out["draft"] = {"ms": d_ms, "algorithmic_bytes": cyc.draft_bytes(),
                        "achieved_gbs": cyc.draft_bytes() / (d_ms / 1e3) / 1e9,
                        "frac_hbm": cyc.draft_bytes() / (d_ms / 1e3) / 1e9 / hbm,
                        "flops": fl, "achieved_tflops": fl / (d_ms / 1e3) / 1e12,
                        "frac_tensor": fl / (d_ms / 1e3) / 1e12 / tens,
                        "tensor_peak_tflops": tens, "tensor_peak": "bf16_tflops_sustained (measured)",
                        "path": "tcgen05" if cyc.uses_tc else "simt"}
        if w.get("confidence"):
            out["K_used"] = int(cyc.K_used.item())
    out["peak_hbm_gbs"] = hbm
    del cyc
    torch.cuda.empty_cache()
    return out


def graph_timed(torch, step, steps, warmup, seconds):
    """Median ms of blocks of `steps` calls of step(cycle), each block one replayed
    CUDA graph captured once (stream launches if the capture fails), after `warmup`
    plain steps.  Returns (median block ms, blocks, launch mode)."""
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    graph, mode = None, "cuda_graph"
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            for i in range(steps):
                step(warmup + i)
        graph.replay()
        torch.cuda.synchronize()
    except Exception as exc:  # noqa: BLE001 -- any capture failure falls back to the stream
        graph, mode = None, "stream (graph capture failed: %s)" % str(exc).splitlines()[0][:160]
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    blocks, t_end = [], time.perf_counter() + seconds
    while not blocks or time.perf_counter() < t_end:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for i in range(steps):
                step(warmup + i)
        e1.record(stream)
        torch.cuda.synchronize()
        blocks.append(e0.elapsed_time(e1))
    return statistics.median(blocks), len(blocks), mode


def tiny_study(args):
    """The tiny exhaustive workload (R = 1, V = 64, gamma = 5, rank 8, fp32 factors and
    base logits): select, the CUDA-core draft keeping its logits, the verify on stored
    logits and commit, at T = 1 and greedy.  Bound by launch latency: microseconds per
    cycle, no roofline fraction."""
    import torch
    from speculative_decoding_dspark_gb300 import binding as B

    def dev(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).cuda()
        return torch.from_numpy(x).cuda()

    out = {}
    for T in (1.0, 0.0):
        w = inputs.workload("tiny_exhaustive", temperature=T)
        d, ci = inputs.draft_inputs(w), inputs.confidence_inputs(w)
        R, V, gamma, rank = w["R"], w["V"], w["gamma"], w["rank"]
        rows = R * (gamma + 1)
        target = dev(inputs.target_full(w, d["U"]).reshape(rows, V))
        U, W1, W2, anc, seeds, c = (dev(d["U"]), dev(d["W1"]), dev(d["W2"]), dev(d["anchor"]), dev(d["seeds"]),
                                    dev(ci["c"]))
        f32 = dict(device="cuda")
        i32 = dict(dtype=torch.int32, device="cuda")
        y, q_lse, q_tok = torch.empty((R, gamma), **i32), torch.empty((R, gamma), **f32), torch.empty((R, gamma), **f32)
        q_logits = torch.empty((R, gamma, V), **f32)
        a, l, cu, K = torch.empty((R, gamma), **f32), torch.empty(R, **i32), torch.empty(R + 1, **i32), torch.empty(1, **i32)
        n_acc, outt, p_tok = torch.empty(R, **i32), torch.empty((R, gamma + 1), **i32), torch.empty((R, gamma), **f32)
        cl, cuc, disc, tot = torch.empty(R, **i32), torch.empty(R + 1, **i32), torch.empty(R, **i32), torch.empty(1, **i32)
        status = torch.zeros(1, **i32)
        ws_d = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank, 0, B.DSPARK_F32))
        ws_v = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY, R, gamma, V, 0, rows))
        samp = T > 0

        def step(cycle):
            B.dspark_select_prefix(c, None, None, None, rows, B.DSPARK_SELECT_FIXED, a, l, cu, K, None, status)
            B.dspark_markov_draft(U, W1, W2, anc, seeds if samp else None, cycle, T, y, q_lse, q_tok, q_logits,
                                  ws_d, status)
            B.dspark_verify(target, cu, y, q_logits if samp else None, q_lse if samp else None,
                            q_tok if samp else None, seeds if samp else None, cycle, T, rows, n_acc, outt, p_tok,
                            ws_v, status)
            B.dspark_commit_lengths(n_acc, l, gamma, cl, cuc, disc, tot, status)

        ms, nb, mode = graph_timed(torch, step, args.steps, args.warmup, SIDE_SECONDS)
        assert int(status.item()) == 0, f"tiny_exhaustive: device status {int(status.item())}"
        out["T%g" % T] = {"us_per_cycle": 1000.0 * ms / args.steps, "cycles_per_s": 1000.0 * args.steps / ms,
                          "blocks": nb, "steps_per_block": args.steps, "launch": mode,
                          "draft_path": "simt (fp32 factors, rank 8)"}
    out.update({"R": 1, "V": 64, "gamma": 5, "rank": 8, "bound": "launch latency"})
    return out


def fused_study(args, peaks, unfused_route=True, **over):
    """The fused drafter logits (dspark_markov_draft_fused, q_logits not kept) on the
    fused_logits workload (or a variant): one draft call per step, timed in blocks
    like the cycle.  Beside it, for context, the route it replaces: the lm_head GEMM
    writing U (torch.matmul, i.e. cuBLAS, bf16 out) followed by dspark_markov_draft."""
    import torch
    from speculative_decoding_dspark_gb300 import binding as B
    w = inputs.workload("fused_logits", **over)
    f = inputs.fused_inputs(w)
    R, V, gamma, rank, d = w["R"], w["V"], w["gamma"], w["rank"], w["d"]
    T = float(w["temperature"])

    def dev(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
        if x.dtype == np.uint64:
            return torch.from_numpy(x.view(np.int64)).cuda()
        return torch.from_numpy(x).cuda()

    t = {k: dev(f[k]) for k in ("h", "W_lm", "W1", "W2", "anchor", "seeds")}
    del f
    stream = torch.cuda.Stream()
    y = torch.empty((R, gamma), dtype=torch.int32, device="cuda")
    q_lse = torch.empty((R, gamma), device="cuda")
    q_tok = torch.empty((R, gamma), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT_FUSED, R, gamma, V, rank, 0, B.DSPARK_BF16, 0))
    ws_u = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank, 0, B.DSPARK_BF16, 0))
    U = torch.empty((R, gamma, V), dtype=torch.bfloat16, device="cuda")

    def fused(c):
        B.dspark_markov_draft_fused(t["h"], t["W_lm"], t["W1"], t["W2"], t["anchor"], t["seeds"], c, T, y,
                                    q_lse, q_tok, None, ws, status, stream=stream)

    def unfused(c):
        torch.matmul(t["h"].view(R * gamma, d), t["W_lm"].t(), out=U.view(R * gamma, V))
        B.dspark_markov_draft(U, t["W1"], t["W2"], t["anchor"], t["seeds"], c, T, y, q_lse, q_tok, None, ws_u,
                              status, stream=stream)

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                fn(i)
            torch.cuda.synchronize()
            blocks, c = [], args.warmup
            t_end = time.perf_counter() + SIDE_SECONDS
            while (args.blocks is None and (not blocks or time.perf_counter() < t_end)) or \
                    (args.blocks is not None and len(blocks) < args.blocks):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.steps):
                    fn(c)
                    c += 1
                e1.record(stream)
                torch.cuda.synchronize()
                blocks.append(e0.elapsed_time(e1) / args.steps)
        return statistics.median(blocks), len(blocks)

    ms, nb = timed(fused)
    assert int(status.item()) == 0, f"fused draft: device status {int(status.item())}"
    ms_u = None
    if unfused_route:
        ms_u, _ = timed(unfused)
        assert int(status.item()) == 0, f"unfused draft: device status {int(status.item())}"
    hbm = peaks.get("hbm_gbs") or 6800.0
    tens = peaks.get("bf16_tflops_sustained") or 1700.0
    # algorithmic bytes: [W_lm | W2] once per position, h once
    byts = gamma * V * (d + rank) * 2 + R * gamma * d * 2
    fl = 2.0 * R * V * (d + rank) * gamma
    del t, U
    torch.cuda.empty_cache()
    return {"R": R, "V": V, "gamma": gamma, "rank": rank, "d": d, "temperature": T, "blocks": nb,
            "steps_per_block": args.steps, "metric": "fused draft calls/s", "value": 1000.0 / ms,
            "draft_ms": ms, "algorithmic_bytes": byts, "achieved_gbs": byts / (ms / 1e3) / 1e9,
            "frac_hbm": byts / (ms / 1e3) / 1e9 / hbm, "flops": fl, "achieved_tflops": fl / (ms / 1e3) / 1e12,
            "frac_tensor": fl / (ms / 1e3) / 1e12 / tens, "tensor_peak": "bf16_tflops_sustained (measured)",
            "unfused_route_ms": ms_u,
            "unfused_route": "cuBLAS lm_head GEMM (torch.matmul, bf16 U written) + dspark_markov_draft"}


PLAN_MODES = [("fixed", 0, 0.0), ("history", 1, 0.0), ("current", 2, 0.0), ("first_stop", 3, 0.0),
              ("conf_cutoff_0.6", 4, 0.6), ("conf_cutoff_0.3", 4, 0.3), ("survival_cutoff_0.3", 5, 0.3)]


def planner_study(n_cycles=1000, repeats=5):
    """The planner on the workload as given (R = 512) and on two variants that
    make the capacity choice matter: 384 request slots (between two capture
    sizes), and the same with a wandering batch-wide confidence shift."""
    return {"R512": planner_run(n_cycles, repeats),
            "R384": planner_run(n_cycles, repeats, R=384),
            "R384_drift": planner_run(n_cycles, repeats, R=384, drift=0.6)}


def planner_run(n_cycles=1000, repeats=5, R=None, drift=0.0):
    """The scheduler over a run of consecutive cycles of the confidence-scheduled
    workload (R = 512, gamma = 5, K_cap = 1024, the synthetic SPS staircase),
    one dspark_plan_cycles launch per policy: the capacity planned on the
    confidences of two cycles back (HISTORY) against the non-causal CURRENT
    mode, the paper's first-stop greedy, the fixed capacity and static
    per-request cutoffs.  The target's verdicts are synthetic (each draft
    survives with its calibrated confidence)."""
    import torch
    from speculative_decoding_dspark_gb300 import binding as B
    w = inputs.workload("confidence_scheduled", **({} if R is None else {"R": R}))
    seq = inputs.confidence_sequence(w, n_cycles, drift=drift)
    R = w["R"]
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    c, nf = dev(seq["c"]), dev(seq["n_full"])
    sizes, sps = dev(seq["capture_sizes"]), dev(seq["sps"])
    l = torch.empty((n_cycles, R), dtype=torch.int32, device="cuda")
    K = torch.empty(n_cycles, dtype=torch.int32, device="cuda")
    st = torch.empty((n_cycles, 4), dtype=torch.float64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = {"cycles": n_cycles, "R": R, "gamma": w["gamma"], "K_cap": seq["K_cap"], "lag": 2, "drift": drift,
           "verdicts": "synthetic: draft k survives with probability c[t, r, k] given the ones before",
           "policies": {}}
    stream = torch.cuda.current_stream()
    for name, mode, conf_min in PLAN_MODES:
        run = lambda: B.dspark_plan_cycles(c, nf, sizes, sps, seq["K_cap"], mode, l, K, st, conf_min=conf_min,
                                           lag=2, dev_status=status)
        run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(repeats):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        s_h = st.cpu().numpy()
        k_h = K.cpu().numpy()
        out["policies"][name] = {
            "mode": mode, "conf_min": conf_min,
            "theta_achieved_mean": float(s_h[:, 1].mean()), "theta_predicted_mean": float(s_h[:, 0].mean()),
            "accepted_per_cycle": float(s_h[:, 2].mean()), "wasted_rows_per_cycle": float(s_h[:, 3].mean()),
            "rows_per_cycle": float(k_h.mean()),
            "launch_ms": e0.elapsed_time(e1) / repeats}
    assert int(status.item()) == 0
    out["unit_theta"] = "tokens/s of the synthetic engine: SPS(B) x (R + accepted drafts)"
    return out


def calibration_study(n_samples=512_000, repeats=5):
    """dspark_fit_temperatures on labels drawn from the workload's per-position
    temperatures: time per fit and the temperatures it recovers."""
    import torch
    from speculative_decoding_dspark_gb300 import binding as B
    w = inputs.workload("confidence_scheduled")
    cs = inputs.calibration_samples(w, n_samples)
    gamma = w["gamma"]
    z = torch.from_numpy(cs["z"]).cuda()
    acc = torch.from_numpy(cs["accepted"]).cuda()
    tau = torch.empty(gamma, device="cuda")
    nll = torch.empty(gamma, dtype=torch.float64, device="cuda")
    cnt = torch.empty(gamma, dtype=torch.int32, device="cuda")
    ws = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_CALIBRATE, 0, gamma, 0))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run = lambda: B.dspark_fit_temperatures(z, acc, tau, nll, cnt, ws, status)
    run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(repeats):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ms = e0.elapsed_time(e1) / repeats
    bytes_read = n_samples * gamma * 5  # z and labels once; the Newton steps re-read them from L2
    return {"samples": n_samples, "gamma": gamma, "ms": ms, "samples_per_s": n_samples / (ms / 1e3),
            "tau_true": [float(x) for x in cs["tau_true"]], "tau_fit": [float(x) for x in tau.cpu()],
            "samples_per_position": [int(x) for x in cnt.cpu()],
            "note": f"latency-bound: {bytes_read / 1e6:.1f} MB of inputs, a few Newton steps each with a "
                    "barrier of the position's CTAs"}


R_SPARE = 512 * 24  # pages for 50 cycles of growth of 512 requests (at most 6 tokens a cycle each)


def kv_study(cycles=50):
    """dspark_kv_reserve + dspark_kv_commit per cycle on a 512-request paged KV
    cache (page size 16): microseconds per cycle (one CTA each: latency-bound)."""
    import torch
    from speculative_decoding_dspark_gb300 import binding as B
    w = inputs.workload("confidence_scheduled")
    kv = inputs.kv_state(w, page_size=16, max_len=4096, spare_pages=R_SPARE, headroom=6 * cycles)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    g = np.random.default_rng(3)
    R, gamma = w["R"], w["gamma"]
    ls = [dev(g.integers(0, gamma + 1, size=R).astype(np.int32)) for _ in range(cycles)]
    nas = [dev((g.random(R) * (ls[i].cpu().numpy() + 1)).astype(np.int32)) for i in range(cycles)]
    d_len, d_bt = dev(kv["kv_len"]), dev(kv["block_table"])
    d_free, d_top = dev(kv["free_pages"]), dev(np.array([kv["free_top"]], np.int32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(cycles):
        B.dspark_kv_reserve(d_len, ls[i], 16, d_bt, d_free, d_top, None, status)
        B.dspark_kv_commit(d_len, ls[i], nas[i], 16, d_bt, d_free, d_top, status)
    e1.record(stream)
    torch.cuda.synchronize()
    # the first cycles may run out of pages as contexts grow: report the status
    return {"R": R, "page_size": 16, "cycles": cycles, "us_per_cycle": 1000.0 * e0.elapsed_time(e1) / cycles,
            "status": int(status.item()), "note": "reserve + commit, one CTA each (latency-bound)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    over = {}
    if args.gamma is not None:
        over["gamma"] = args.gamma
    if args.temperature is not None:
        over["temperature"] = args.temperature
    w = inputs.workload(args.workload, **over)
    host = host_inputs(w)
    R, V, gamma, rank_r = w["R"], w["V"], w["gamma"], w["rank"]
    T = float(w["temperature"])
    # the oracle's worker pool is forked now, before this process touches CUDA
    pool = None
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline and args.stage == "cycle"
    model, ncpu = host_cpu()
    if want_cpu:
        pool = OraclePool(w, host["d"], host["full"], ncpu)

    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    cyc = Cycle(w, host, stage=args.stage)
    stream = cyc.stream

    for i in range(args.warmup):
        cyc.step(i)
    torch.cuda.synchronize()
    assert int(cyc.status.item()) == 0, f"device status {int(cyc.status.item())}"

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    t0 = time.perf_counter()
    blocks, per, n_timed, ms_staged = cyc.timed_blocks(args.steps, args.warmup, BLOCK_SECONDS, args.blocks)
    launch_mode = cyc.launch_mode
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms_block = statistics.median(blocks)
    ms = max_over_ranks(ms_block, world)
    ms_step = ms / args.steps
    value = whole_job_rate(args.steps, world, ms)
    if clk is not None:
        clk["timed_region_s"] = wall
        clk["sm_mhz_x_ms_per_step"] = clk["sm_mhz"] * ms_step

    # roofline of the dominant kernel.  Algorithmic bytes of one Markov draft
    # step (one vocabulary pass): W2 once, U_k once.  The tensor-core kernel
    # runs all gamma steps in one launch, timed as the whole draft call (which
    # adds the workspace reset, so the fraction is a lower bound); the CUDA-core
    # path is timed per step.
    step_bytes = V * rank_r * 2 + R * V * 2
    steps_per_launch = gamma if cyc.uses_tc else 1
    launch_bytes = step_bytes * steps_per_launch
    launch_ms = per["draft"] / gamma * steps_per_launch
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm else "fallback"
    hbm = hbm or 6800.0
    achieved = launch_bytes / (launch_ms / 1000.0) / 1e9
    kname = "markov_tc_kernel<draft>" if cyc.uses_tc else "draft_bias_simt+draft_sample"
    digest = source_digest(["speculative_decoding_dspark_gb300/csrc/draft_tc.cu" if cyc.uses_tc else
                            "speculative_decoding_dspark_gb300/csrc/draft_simt.cu",
                            "speculative_decoding_dspark_gb300/csrc/common.cuh",
                            "speculative_decoding_dspark_gb300/csrc/tc_ptx.cuh"])
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic_from_profile(kname, digest), "kernel": kname,
            "algorithmic_bytes_per_launch": launch_bytes, "steps_per_launch": steps_per_launch,
            "launch_ms": launch_ms, "peak_source": peak_src}
    tens = peaks.get("bf16_tflops_sustained") or 1700.0
    fl = cyc.draft_flops()
    roof["tensor"] = {"achieved_tflops": fl / (launch_ms / 1e3) / 1e12, "peak_tflops": tens,
                      "frac": fl / (launch_ms / 1e3) / 1e12 / tens, "peak": "bf16_tflops_sustained"}

    # end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e and args.stage == "cycle":
        e2e = measure_e2e(cyc, args, world, host_target=True)
        e2e["copy_all"] = measure_e2e(cyc, args, world, host_target=False)

    verify_roof = None
    if cyc.run_verify:
        vbytes, rows_read, rows_presented = cyc.verify_bytes()
        v_ms = per["verify"]
        verify_roof = {"bound": "hbm", "achieved": vbytes / (v_ms / 1000.0) / 1e9, "peak": hbm, "unit": "GB/s",
                       "frac": vbytes / (v_ms / 1000.0) / 1e9 / hbm, "algorithmic_bytes_per_call": vbytes,
                       "rows_read": rows_read, "rows_presented": rows_presented, "call_ms": v_ms}
    else:
        rows_read = rows_presented = 0

    side = None
    if rank == 0 and args.stage == "cycle" and not args.no_side_workloads and args.workload == DEFAULT_WORKLOAD:
        del cyc
        torch.cuda.empty_cache()
        side = {name: side_workload(name, args, peaks)
                for name in ("confidence_scheduled", "varlen_verify", "qwen3_8b_greedy")}
        side["tiny_exhaustive"] = tiny_study(args)
        side["fused_logits"] = fused_study(args, peaks)
        side["fused_logits_R512"] = fused_study(args, peaks, R=512, V=129280, gamma=5, temperature=1.0)
        side["planner"] = planner_study()
        side["calibration"] = calibration_study()
        side["kv_bookkeeping"] = kv_study()

    cpu = None
    if pool is not None:
        secs = pool.cycle(0)
        pool.close()
        cpu = {"value": 1.0 / secs, "unit": UNIT, "cores": pool.n, "kind": "oracle",
               "sample": f"one whole cycle of all {R} requests (draft {gamma} positions + verify + commit), "
                         f"requests spread over {pool.n} worker processes",
               "cpu_model": model, "nproc": ncpu}

    if rank == 0:
        logits_read = rows_read * V * 4 + R * gamma * V * 2
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 GEMM (fp32 accumulate) + fp32 softmax/verify",
                "data": "synthetic (seeded; shapes and laws of the workload)",
                "config": workload_config(w, world),
                "timing": {"blocks": len(blocks), "steps_per_block": args.steps,
                           "block_ms_min_median_max": [min(blocks), ms_block, max(blocks)],
                           "stage_event_block_ms_median": ms_staged,
                           "launch": launch_mode,
                           "stage_ms_from": f"{max(1, STAGE_BLOCKS)} further blocks with an event between the calls",
                           "rule": "median of timed blocks of exactly K steps, repeated for about "
                                   f"{BLOCK_SECONDS:g} s"},
                "roofline": roof, "verify_roofline": verify_roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": cyc_launches(args, w) * n_timed,
                "stage": args.stage, "stage_ms": per,
                "logits_gb_s": logits_read / (ms_step / 1000.0) / 1e9,
                "logits_gb_s_rule": "target rows verify read (up to each first rejection) + U, per cycle",
                "presented_logits_gb_s": (R * (gamma + 1) * V * 4 + R * gamma * V * 2) / (ms_step / 1000.0) / 1e9,
                "draft_path": "tcgen05" if roof["kernel"].startswith("markov_tc") else "simt",
                "workloads": side}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cyc_launches(args, w):
    """Launches of this library per step of the headline workload (recomputed
    after the side workloads freed its tensors)."""
    from speculative_decoding_dspark_gb300 import binding as B
    R, V, gamma, rank = w["R"], w["V"], w["gamma"], w["rank"]
    uses_tc = B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, R, V, rank)
    draft = (1 if uses_tc else 1 + 2 * gamma) * int(args.stage in ("cycle", "draft"))
    verify = (3 if float(w["temperature"]) > 0 else 2) * int(args.stage in ("cycle", "verify"))
    varlen = bool(w.get("varlen"))
    return int(args.stage == "cycle" and not varlen) + draft + verify + int(args.stage == "cycle")


def measure_e2e(cyc, args, world, host_target=True):
    """The cycle end to end: every step takes its inputs from pinned host memory
    and reads its results back, inside the timed region.  U, the confidences,
    anchors and seeds are copied each step.  The target logits are either left in
    pinned host memory, where the verify kernels read only the rows they examine
    across the host link (host_target, the library's host-target mode), or copied
    whole like the rest."""
    import torch
    B = cyc.B
    stream = cyc.stream
    R, gamma = cyc.R, cyc.gamma
    dev_in = (cyc.U, cyc.target, cyc.c, cyc.c_hist, cyc.anchor, cyc.seeds)
    hosts = tuple(t.cpu().pin_memory() for t in dev_in)
    h_out = torch.empty((R, gamma + 1), dtype=torch.int32).pin_memory()
    h_n = torch.empty(R, dtype=torch.int32).pin_memory()
    h_cl = torch.empty(R + 1, dtype=torch.int32).pin_memory()
    copied = [i for i in range(len(dev_in)) if not (host_target and i == 1)]
    bi = sum(hosts[i].numel() * hosts[i].element_size() for i in copied)
    bo = sum(t.numel() * t.element_size() for t in (h_out, h_n, h_cl))
    ws_v = None
    if host_target:
        ws_v = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY_MARKOV, R, gamma, cyc.V, cyc.rank, cyc.max_rows,
                                                   B.DSPARK_BF16, B.DSPARK_VERIFY_HOST_TARGET))

    # Each cycle's inputs go host -> device as chunks spread over four copy
    # streams (several copy engines), into one of two device input sets, so
    # the copies of cycle i + 1 overlap the kernels of cycle i; the kernels
    # of a cycle wait for its own copies, and a set is refilled only after
    # the cycle that read it has finished.
    copy_streams = [torch.cuda.Stream() for _ in range(4)]
    second = list(torch.empty_like(t) for t in dev_in)
    if host_target:
        second[1] = hosts[1]
    first = list(dev_in)
    if host_target:
        first[1] = hosts[1]
    sets = [tuple(first), tuple(second)]
    freed = [None, None]
    n_acc_log = []

    def issue_copies(b, after):
        for cs in copy_streams:
            if after is not None: cs.wait_event(after)
            if freed[b] is not None: cs.wait_event(freed[b])
        k = 0
        for i in copied:
            dst, src = sets[b][i], hosts[i]
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

    def e2e_run(n, first_cycle, start_ev=None, log=None):
        pending = issue_copies(0, start_ev)
        for i in range(n):
            b = i & 1
            for e in pending:
                stream.wait_event(e)
            if i + 1 < n:
                pending = issue_copies((i + 1) & 1, None)
            cyc.step(first_cycle + i, inp=sets[b], ws_v=ws_v)
            fe = torch.cuda.Event()
            fe.record(stream)
            freed[b] = fe
            h_out.copy_(cyc.out, non_blocking=True); h_n.copy_(cyc.n_acc, non_blocking=True)
            h_cl.copy_(cyc.cuc, non_blocking=True)
            if log is not None:
                log.append(cyc.n_acc.clone())

    n_e2e = max(3, min(args.steps, 20))
    e2e_run(2, 0)
    torch.cuda.synchronize()
    freed[0] = freed[1] = None
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    e2e_run(n_e2e, 100000, s0, n_acc_log)
    s1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(s0.elapsed_time(s1), world)
    out = {"value": whole_job_rate(n_e2e, world, e_ms), "unit": UNIT, "steps": n_e2e, "d2h_bytes_per_step": bo}
    if host_target:
        # the target bytes the kernels read across the link: every row up to each
        # first rejection (the residual draw reads the device copy of the last one)
        l_h = cyc.l.cpu().numpy().astype(np.int64)
        rows = [int((np.minimum(n.cpu().numpy().astype(np.int64), l_h) + 1).sum()) for n in n_acc_log]
        zc = statistics.mean(rows) * cyc.V * 4
        out.update({"h2d_bytes_per_step": int(bi + zc), "h2d_copied_bytes_per_step": bi,
                    "h2d_target_rows_read_bytes_per_step": int(zc),
                    "target": "left in pinned host memory; the verify kernels read the rows they examine"})
    else:
        out.update({"h2d_bytes_per_step": bi, "target": "copied whole every step"})
    out["h2d_gb_s"] = out["h2d_bytes_per_step"] * n_e2e / (e_ms / 1000.0) / 1e9
    del sets
    return out


def main():
    args = parse()
    if args.impl == "ours" and args.stage == "fused_draft":
        print(json.dumps({"stage": "fused_draft", **fused_study(args, load_peaks(), unfused_route=False)}), flush=True)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
