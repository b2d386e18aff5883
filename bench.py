#!/usr/bin/env python
"""Draft + verify throughput of the DSpark step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
Markov-head draft loop (one cooperative launch over the gamma positions)
with the verification stream (log-sum-exps of target rows 0..gamma) running
beside it on the same SMs, confidence + STS + survival, prefix scheduler,
accept walk, residual and bonus draws, compaction: 7 kernel launches
(--fuse-target off: the verification stream as its own launch after the
draft, also 7).  Default workload: B=64, V=151936, r=256, gamma=7, d=4096,
bf16 draft-head weights, fp32 base and target logits, full-prefix
verification (scheduler call made in OFF mode, K_b = 7).

Prints one JSON line (rank 0).  `value` = emitted tokens per second over all
ranks with inputs resident in HBM (CUDA-graph replay of the step, CUDA
events on the launching stream, inputs 1.13 GB > L2 so no flush).
`e2e` = the same metric through the public API (HostPipeline) with every
step's activations copied from pinned host memory and its emitted tokens
copied back inside the timed region; the copy of step t+1 overlaps the
compute of step t.  `roofline` = the draft launch (the dominant one: per launch
it streams W2 and one row block of U for each of the gamma positions), with
the target rows its side stream reads when that runs beside it.

With several ranks each owns B requests of a batch of B * ranks (weak
scaling).  With the scheduler off no data crosses ranks; with it on
(--sched spec) the survival lists are all-gathered and every rank runs the
scheduler on the whole list.

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the reference arm of this tier).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workload  # noqa: E402

MIN_TIMED_S = 0.5      # the timed region lasts at least this long (clock samples inside it)
METRIC = "draft+verify tokens/s (B=64, V=151936, γ=7) and % of HBM roofline on 1 GB300"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons while running."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.monotonic())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock and the throttle reasons seen in the samples taken
        between mark("start") and mark("end") (the timed region)."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t_start", None), getattr(self, "t_end", None)
        for t, ln in self.lines:
            if t0 is not None and not (t0 <= t <= t1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0])); mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": "timed region"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        return dist, ws, rank, local
    return None, 1, 0, 0


def _max_over_ranks(dist, x, dev):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _sum_over_ranks(dist, x, dev):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _quick_steps(vm, dev):
    """Extra records beside the headline: the step of the latency case (b1),
    of b256 and of b64 with its scheduler on (the stepped capacity table,
    synchronous mode), each by CUDA-graph replay of device-resident inputs
    for at least 0.3 s."""
    out = {}
    for label, name, sched in (("b1", "b1", False), ("b256", "b256", False), ("b64_scheduled", "b64", True)):
        w = workload.WORKLOADS[name]
        mode = w.mode if sched else 0
        inp = workload.inputs(w, device=dev)
        buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r, device=dev)
        stream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize(dev)

        def one():
            vm.run_step(inp, buf, mode=mode, seed=w.seed, step=0, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                one()
        stream.synchronize()
        st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
        if st != 0:
            raise SystemExit(f"{label}: device status {st} bits {bits}")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one()
        with torch.cuda.stream(stream):
            for _ in range(5):
                g.replay()
        stream.synchronize()
        n, t = 0, 0.0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        while t < 300.0:
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(50):
                    g.replay()
                e1.record(stream)
            stream.synchronize()
            t += e0.elapsed_time(e1)
            n += 50
        emitted = int(buf.out_off[-1].item())
        ms = t / n
        out[label] = {"ms_per_step": ms, "tokens_per_s": emitted / (ms / 1e3), "emitted_tokens_per_step": emitted,
                      "steps": n, "workload": f"B={w.B} V={w.V} r={w.r} gamma={w.gamma}, "
                      + (f"scheduler mode {mode} ({w.sps_fn.__name__} capacity table)" if sched else "scheduler off")}
        del inp, buf, g
        torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import verify_markov_head_gb300 as vm

    dist, world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload.WORKLOADS[args.workload]
    mode = {"off": 0, "spec": w.mode}[args.sched]
    B, gamma, V, r = w.B, w.gamma, w.V, w.r
    req_base = rank * B        # each rank owns its own B requests (weak scaling)
    inp = workload.inputs(w, step=rank, device=dev)
    head = args.head
    # scheduler off: the target stream runs beside the draft where it fits
    # (one chunk of B <= 64 requests), else the separate verify stream
    fuse_target = {"on": True, "off": False, "auto": vm.target_stream_preferred(inp)}[args.fuse_target]
    if head == "rnn":
        inp["rnn"] = vm.rnn_prepare(workload.rnn_head(w, device=dev))
    buf = vm.StepBuffers(B, gamma, V, r, device=dev)
    stream = torch.cuda.Stream(device=dev)
    seed = w.seed
    torch.cuda.synchronize(dev)       # inputs are made on the default stream; the step runs on `stream`

    if world > 1 and mode != 0:
        # the scheduler ranks the whole batch: a capacity table for B * world
        inp["sps"] = workload.custom(w.name, B=B * world).sps_table().to(dev)
        sched = vm.GlobalSchedule(B, gamma, world, device=dev)

        if head != "markov":
            raise SystemExit("the scheduled multi-rank step runs the Markov head only")

        def one_step():
            vm.run_step_dp(inp, buf, sched, mode=mode, seed=seed, step=0, stream=stream)
    else:
        def one_step():
            vm.run_step(inp, buf, mode=mode, seed=seed, step=0, req_base=req_base, stream=stream, head=head,
                        fuse_target=fuse_target)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    stream.synchronize()
    st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            graph.replay()
    stream.synchronize()

    # ---- timed region: graph replays of the whole step, at least K of them
    #      and at least MIN_TIMED_S seconds' worth, so the clock sampler (one
    #      sample every 50 ms) sees the timed region itself
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the same replays for ~1 s first: the sampler starts and the clocks
        # settle under load before the timed region
        t_pre = time.monotonic()
        n_pre = 0
        with torch.cuda.stream(stream):
            while time.monotonic() - t_pre < 1.0:
                for _ in range(20):
                    graph.replay()
                n_pre += 20
                stream.synchronize()
        est_s = (time.monotonic() - t_pre) / max(1, n_pre)
        steps = int(max(args.steps, math.ceil(MIN_TIMED_S / max(est_s, 1e-6))))
        steps = int(_max_over_ranks(dist, steps, dev))
        _barrier(dist)
        torch.cuda.synchronize()
        clk.mark("start")
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                graph.replay()
            e1.record(stream)
        stream.synchronize()
        clk.mark("end")
    torch.cuda.synchronize()
    _barrier(dist)
    ms = e0.elapsed_time(e1) / steps
    ms_max = _max_over_ranks(dist, ms, dev)
    emitted = int(buf.out_off[-1].item())
    emitted_all = _sum_over_ranks(dist, emitted, dev)
    value = emitted_all / (ms_max / 1e3)

    # ---- dominant kernel: the draft call, timed alone on the same stream (with
    #      the scheduler off the step drafts with the target stream: the call
    #      run_step makes)
    fused = fuse_target and head == "markov" and mode == 0 and vm.target_stream_supported(inp)
    # one cooperative launch covers the gamma positions (the RNN head runs its
    # GRU steps inside it)
    draft_launches = 1
    reps = max(5, min(args.steps, 1000))
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        d0.record(stream)
        for _ in range(reps):
            if head == "rnn":
                vm.dspark_draft_rnn(inp["U"], inp["rnn"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                                    buf.z_tok, buf.state, buf.ws, seed=seed, req_base=req_base, stream=stream)
            elif fused:
                vm.dspark_draft_markov_target(inp["U"], inp["W1"], inp["W2"], inp["target"], inp["anchor"],
                                              buf.draft_tok, buf.lse_q, buf.z_tok, buf.ws, seed=seed,
                                              req_base=req_base, logits_out=buf.logits, stream=stream)
            else:
                vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                                       buf.z_tok, buf.ws, seed=seed, req_base=req_base, stream=stream)
        d1.record(stream)
    stream.synchronize()
    draft_launch_ms = d0.elapsed_time(d1) / (reps * draft_launches)
    w2_bytes = r * V * inp["W2"].element_size()
    u_bytes_k = B * V * inp["U"].element_size()
    # per position: W2 once + one row block of U; a launch covers gamma /
    # draft_launches positions.  With the target stream (beside the draft,
    # B <= 64: rows 0..gamma, the bonus row's law included; in the epilogue:
    # rows 0..gamma-1) the launch also reads those target rows.
    t_rows = (gamma + 1 if vm.target_stream_beside(inp) else gamma) if fused else 0
    draft_bytes = (w2_bytes + u_bytes_k) * gamma // draft_launches + \
        B * t_rows * V * inp["target"].element_size() // draft_launches
    peak, peak_kind = _peaks()
    achieved = draft_bytes / (draft_launch_ms / 1e3) / 1e9
    formula_bytes = gamma * w2_bytes + inp["U"].numel() * inp["U"].element_size() + \
        inp["target"].numel() * inp["target"].element_size()
    step_gbs = formula_bytes / (ms_max / 1e3) / 1e9

    # ---- end to end through the public API from pinned host memory
    host = {k: inp[k].cpu().pin_memory() for k in ("U", "target", "h", "anchor")}
    host_out = {"out_tok": torch.empty(B * (gamma + 1), dtype=torch.int32).pin_memory(),
                "out_off": torch.empty(B + 1, dtype=torch.int32).pin_memory(),
                "next_anchor": torch.empty(B, dtype=torch.int32).pin_memory()}
    # the copy of step t+1's inputs overlaps step t's compute (two input slots)
    e2e_steps = max(3, min(args.steps, 20))
    pipe = vm.HostPipeline(inp, buf, stream)
    for _ in range(2):
        pipe.step(host, host_out, mode=mode, seed=seed, head=head, fuse_target=fuse_target)
    torch.cuda.synchronize()
    _barrier(dist)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    pipe.copy_stream.wait_event(f0)
    for _ in range(e2e_steps):
        h2d, d2h = pipe.step(host, host_out, mode=mode, seed=seed, head=head, fuse_target=fuse_target)
    f1.record(stream)
    stream.synchronize()
    e2e_ms = _max_over_ranks(dist, f0.elapsed_time(f1) / e2e_steps, dev)
    e2e_emitted = _sum_over_ranks(dist, int(host_out["out_off"][-1]), dev)

    st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")

    # draft, confidence, schedule, verify stream (bonus rows only when fused), accept walk,
    # residual draw, compaction
    launches_per_step = draft_launches + 6
    cpu = None
    ties = None
    extra = None
    if rank == 0 and world == 1 and w.name == "b64" and head == "markov" and mode == 0 and not args.no_extras:
        extra = _quick_steps(vm, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, mode, budget_s=args.cpu_budget, dev_inp=inp, min_seconds=10.0, head=head)
        if _LAST_SAMPLE and head == "markov" and mode == 0:
            off = buf.out_off.cpu().numpy()
            ties = near_ties(buf.draft_tok.cpu().numpy(), buf.z_tok.cpu().numpy(), buf.accepted.cpu().numpy(),
                             buf.out_tok.cpu().numpy()[off[1:] - 1], _LAST_SAMPLE, device_gumbel_error(vm, dev))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "steps_requested": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 weights, f32 logits, f32 accumulate", "data": "synthetic",
            "config": {"workload": f"{w.name}: B={B} V={V} r={r} gamma={gamma} d={d_of(w)} "
                                   f"verify={'full prefix (scheduler off)' if mode == 0 else 'scheduled'}"
                                   + (", RNN draft head" if head == "rnn" else ""),
                       "global_batch": B * world, "seq_len": gamma, "parallelism": f"dp{world} over requests",
                       "l2": "inputs 1.13 GB per step > 129 MB L2; no flush", "graph": "CUDA graph replay"},
            "emitted_tokens_per_step": emitted_all, "drafted_tokens_per_step": B * gamma * world,
            "step_formula_bytes": formula_bytes, "step_formula_gbs": step_gbs,
            "step_formula_frac": step_gbs / peak,
            "roofline": {"kernel": ("rows_kernel<draft> + verify_stream_side_kernel beside it "
                                    "(dspark_draft_markov_target, %d position(s) per launch)"
                                    % (gamma // draft_launches)) if fused and vm.target_stream_beside(inp) else
                                   ("rows_kernel<draft, target stream> (dspark_draft_markov_target, %d "
                                    "position(s) per launch)" % (gamma // draft_launches)) if fused else
                                   ("rows_kernel<draft> (dspark_draft_markov, %d position(s) per launch)"
                                    % (gamma // draft_launches)) if head == "markov" else
                                   ("rows_kernel<draft, RNN head> (dspark_draft_rnn, %d position(s) per "
                                    "launch, the GRU steps inside)" % (gamma // draft_launches)),
                         "bound": "hbm", "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": achieved / peak,
                         "traffic": _draft_traffic(w.name, fused) if draft_launches == 1 and head == "markov"
                         else None,
                         "algorithmic_bytes_per_launch": draft_bytes, "launch_ms": draft_launch_ms},
            "e2e": {"value": e2e_emitted / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "near_ties": ties,
            "extra_steps": extra,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_chain(args):
    """The workload's chained steps (16 for b512) with its scheduler mode:
    step t+1 starts from step t's next anchors, the asynchronous scheduler
    takes its capacity from the survivals of step t-2, and every step's
    activations are its own (generated up front, resident in HBM).  One CUDA
    graph per step; the chain is replayed and timed as a whole."""
    import verify_markov_head_gb300 as vm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workload.WORKLOADS[args.workload]
    mode = {"off": 0, "spec": w.mode}[args.sched]
    B, gamma, V, r = w.B, w.gamma, w.V, w.r
    n = w.steps
    W = workload.weights(w, device=dev)
    steps = [workload.step_inputs(w, step=t, device=dev) for t in range(n)]
    anchor0 = steps[0]["anchor"].clone()
    anchor = torch.empty_like(anchor0)
    ring = [torch.zeros((B, gamma), dtype=torch.float32, device=dev) for _ in range(3)]
    emitted = torch.zeros((n,), dtype=torch.int32, device=dev)
    buf = vm.StepBuffers(B, gamma, V, r, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)

    def step(t):
        inp = dict(W)
        inp.update(steps[t])
        inp["anchor"] = anchor
        hist = ring[(t - 2) % 3] if t >= 2 else None
        vm.run_step(inp, buf, mode=mode, seed=w.seed, step=t, log_surv_hist=hist, stream=stream)
        anchor.copy_(buf.next_anchor)
        ring[t % 3].copy_(buf.log_surv)
        emitted[t:t + 1].copy_(buf.out_off[-1:])

    with torch.cuda.stream(stream):
        anchor.copy_(anchor0)
        for t in range(n):
            step(t)
    stream.synchronize()
    st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")
    graphs = []
    for t in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(t)
        graphs.append(g)

    def chain():
        anchor.copy_(anchor0)
        for g in graphs:
            g.replay()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            chain()
    stream.synchronize()
    reps = max(1, args.steps // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        t_pre = time.monotonic()
        with torch.cuda.stream(stream):
            while time.monotonic() - t_pre < 1.0:
                chain()
                stream.synchronize()
        clk.mark("start")
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                chain()
            e1.record(stream)
        stream.synchronize()
        clk.mark("end")
    ms_chain = e0.elapsed_time(e1) / reps
    tokens = int(emitted.sum())
    st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")
    line = {"metric": f"chained draft+verify tokens/s (B={B}, V={V}, γ={gamma}, {n}-step chain)",
            "value": tokens / (ms_chain / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": reps * n,
            "warmup": max(3, args.warmup) * n, "ms_per_step": ms_chain / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 weights, f32 logits, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: B={B} V={V} r={r} gamma={gamma} d={w.d}, {n} chained steps, "
                                   f"scheduler {['off', 'sync', 'async'][mode]}",
                       "global_batch": B, "seq_len": gamma, "parallelism": "dp1 over requests",
                       "l2": "every step's inputs resident (3.4 GB per step at b512) > 129 MB L2; no flush",
                       "graph": "one CUDA graph per step"},
            "emitted_tokens_per_chain": tokens, "drafted_tokens_per_step": B * gamma,
            "gpu_launches": 7 * n * reps, "clocks": clk.summary(), "cpu_baseline": None}
    print(json.dumps(line), flush=True)


# Special-function-unit (XU pipe) results per SM per clock on GB300: ncu
# rates the pipe at one warp instruction per clock per SM.
SFU_PER_SM_CLK = 32


def run_sts(args):
    """The STS temperature fit (dspark_sts_fit) on the benchmark's validation
    set: 2^20 blocks, 256 candidate temperatures, 15 bins, gamma = 7.  One
    fit is gamma launches of the evaluation kernel; each fit is timed alone
    with CUDA events, L2 flushed in between (the inputs, 33 MB, fit in L2)."""
    import verify_markov_head_gb300 as vm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = dict(workload.STS_FIT)
    if args.sts_blocks:
        c["N"] = args.sts_blocks
    N, gamma, G, M = c["N"], c["gamma"], c["G"], c["M"]
    score, acc_len = workload.sts_validation(N, gamma=gamma, seed=c["seed"], device=dev)
    grid = workload.sts_grid(G, c["lo"], c["hi"]).to(dev)
    T = torch.empty(gamma, dtype=torch.float32, device=dev)
    idx = torch.empty(gamma, dtype=torch.int32, device=dev)
    ece = torch.empty(gamma, G, dtype=torch.float64, device=dev)
    ws = torch.zeros(vm.dspark_sts_workspace_bytes(gamma, G, M), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)

    def fit():
        vm.dspark_sts_fit(score, acc_len, grid, M=M, T_out=T, idx_out=idx, ece_out=ece, ws=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fit()
    st, bits = vm.dspark_sync_status(ws, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")
    reps = max(3, min(args.steps, 200))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with ClockSampler(0) as clk:
        t_pre = time.monotonic()
        with torch.cuda.stream(stream):
            while time.monotonic() - t_pre < 1.0:
                fit()
                stream.synchronize()
        clk.mark("start")
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush.fill_(1)
                a.record(stream)
                fit()
                b.record(stream)
        stream.synchronize()
        clk.mark("end")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    evals = N * G * gamma
    value = evals / (ms / 1e3)
    clocks = clk.summary()
    mhz = clocks.get("sm_max_mhz") or 2070.0
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = n_sm * SFU_PER_SM_CLK * mhz * 1e6 / 2 / 1e9      # two SFU operations per evaluation

    # end to end: host (pinned) inputs copied in, results read back, per fit
    h_score, h_acc = score.cpu().pin_memory(), acc_len.cpu().pin_memory()
    h_T = torch.empty(gamma, dtype=torch.float32).pin_memory()
    h_idx = torch.empty(gamma, dtype=torch.int32).pin_memory()
    h_ece = torch.empty(gamma, G, dtype=torch.float64).pin_memory()
    d_score, d_acc = torch.empty_like(score), torch.empty_like(acc_len)

    def fit_e2e():
        d_score.copy_(h_score, non_blocking=True)
        d_acc.copy_(h_acc, non_blocking=True)
        vm.dspark_sts_fit(d_score, d_acc, grid, M=M, T_out=T, idx_out=idx, ece_out=ece, ws=ws, stream=stream)
        h_T.copy_(T, non_blocking=True)
        h_idx.copy_(idx, non_blocking=True)
        h_ece.copy_(ece, non_blocking=True)

    with torch.cuda.stream(stream):
        fit_e2e()
    stream.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_reps = max(3, min(args.steps, 20))
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(e2e_reps):
            fit_e2e()
        f1.record(stream)
    stream.synchronize()
    e2e_ms = f0.elapsed_time(f1) / e2e_reps
    if not torch.equal(h_idx, idx.cpu()):
        raise SystemExit("end-to-end fit disagrees with the device-resident fit")
    st, bits = vm.dspark_sync_status(ws, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")

    cpu = None
    if not args.no_cpu_baseline:
        cpu = sts_cpu_baseline(score.cpu(), acc_len.cpu(), grid.cpu(), M, budget_s=args.cpu_budget)
    line = {"metric": f"STS fit candidate evaluations/s (N={N} blocks, G={G}, M={M}, γ={gamma})",
            "value": value, "unit": "evaluations/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32 survivals and bins, int64 fixed-point bin totals", "data": "synthetic",
            "config": {"workload": f"sts_fit: N={N} gamma={gamma} G={G} M={M}, grid [{c['lo']}, {c['hi']}]",
                       "l2": "256 MB buffer written between timed fits", "parallelism": "dp1"},
            "roofline": {"kernel": "sts_eval_kernel<4> (dspark_sts_fit, one launch per position)",
                         "note": "2^x + reciprocal per evaluation on the SFU; the shared-memory bin update shares their issue path",
                         "bound": "alu", "achieved": value / 1e9, "peak": peak,
                         "peak_kind": f"derived: {n_sm} SMs x {SFU_PER_SM_CLK} SFU results/clk x "
                                      f"{mhz:.0f} MHz / 2 per evaluation",
                         "unit": "Geval/s", "frac": value / 1e9 / peak, "traffic": None,
                         "launch_ms": ms / gamma},
            "e2e": {"value": evals / (e2e_ms / 1e3), "unit": "evaluations/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h_score.numel() * 4 + h_acc.numel() * 4,
                    "d2h_bytes_per_step": h_T.numel() * 4 + h_idx.numel() * 4 + h_ece.numel() * 8},
            "gpu_launches": gamma * reps, "clocks": clocks, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)


def sts_cpu_baseline(score, acc_len, grid, M, budget_s=20.0):
    """The oracle's STS fit, as it stands, on the first S blocks of the
    validation set with the whole grid (S sized to a ~budget_s run)."""
    import oracle

    gamma, G = score.shape[1], grid.numel()
    t = time.perf_counter()
    oracle.sts_fit(score[:4096], acc_len[:4096], grid.double(), M=M)
    per_block = (time.perf_counter() - t) / 4096
    S = int(max(4096, min(score.shape[0], budget_s / max(per_block, 1e-9))))
    t = time.perf_counter()
    oracle.sts_fit(score[:S], acc_len[:S], grid.double(), M=M)
    dt = time.perf_counter() - t
    return {"value": S * G * gamma / dt, "unit": "evaluations/s", "cores": 1, "kind": "oracle",
            "sample": f"first {S} of {score.shape[0]} blocks, all {G} temperatures, {dt:.1f} s", "seconds": dt}


def d_of(w):
    return w.d


def run_kernel(args):
    """One ABI call, repeated, on the workload's shapes with only the inputs it
    reads on the device (no embedding table), for profiler captures of a
    single kernel; prints the status and no metric.  draft: dspark_draft_markov;
    verify: one draft, then dspark_verify with every K_b = gamma (verify
    stream, accept walk, residual draw, compaction); fused: the draft with the
    target stream beside it (dspark_draft_markov_target); fused-verify: one
    such draft, then dspark_verify in full-prefix mode (accept walk, residual
    and bonus draws, compaction); confidence: one draft, then
    dspark_confidence_sts (this mode also holds the embedding table)."""
    import verify_markov_head_gb300 as vm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = workload.WORKLOADS[args.workload]
    B, gamma, V, r = w.B, w.gamma, w.V, w.r
    inp = (workload.weights if args.kernel == "confidence" else workload.draft_weights)(w, device=dev)
    st = workload.step_inputs(w, device=dev)
    inp.update(U=st["U"], target=st["target"], anchor=st["anchor"])
    ws = vm.Workspace(B, gamma, V, r, dev)
    i32 = dict(dtype=torch.int32, device=dev)
    tok = torch.empty((B, gamma), **i32)
    lse = torch.empty((B, gamma), device=dev)
    zt = torch.empty((B, gamma), device=dev)
    K = torch.full((B,), gamma, **i32)
    acc, nxt = torch.empty((B,), **i32), torch.empty((B,), **i32)
    out_tok, out_req, out_pos = (torch.empty((B * (gamma + 1),), **i32) for _ in range(3))
    out_off = torch.empty((B + 1,), **i32)

    def draft():
        vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, zt, ws, seed=w.seed)

    def verify(k=K):
        vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, zt, k, acc,
                         out_tok, out_req, out_pos, out_off, nxt, ws, seed=w.seed)

    def fused():
        vm.dspark_draft_markov_target(inp["U"], inp["W1"], inp["W2"], inp["target"], inp["anchor"], tok, lse, zt,
                                      ws, seed=w.seed)

    def confidence():
        vm.dspark_confidence_sts(st["h"], inp["emb"], inp["anchor"], tok, inp["w_c"], inp["b_c"], inp["T"], conf,
                                 surv, ws)

    conf, surv = torch.empty((B, gamma), device=dev), torch.empty((B, gamma), device=dev)
    calls = {"draft": draft, "verify": verify, "fused": fused, "fused-verify": lambda: verify(None),
             "confidence": confidence}
    if args.kernel in ("verify", "confidence"):
        draft()
    if args.kernel == "fused-verify":
        fused()
    for _ in range(args.calls):
        calls[args.kernel]()
    status, bits = vm.dspark_sync_status(ws.buf)
    print(json.dumps({"kernel_run": args.kernel, "workload": w.name, "calls": args.calls, "status": status,
                      "bits": bits}), flush=True)
    if status != 0:
        raise SystemExit(1)


# Sources the draft kernel is compiled from: DRAM traffic taken from an ncu
# capture is reported only while they are unchanged since the capture.
_DRAFT_SOURCES = ("draft_rows.cu", "verify.cu", "common.cuh", "sm100_ptx.cuh", "internal.h", "vstream.cuh",
                  "pdl.cuh", "resid_tail.cuh")


def _normalised_source_hash(texts):
    """SHA-256 (first 16 hex digits) of source texts with comments and blank
    space removed: edits to comments keep the hash, edits to code change it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for text in texts:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def _draft_source_hash():
    """The normalised hash of the draft kernel's sources."""
    texts = []
    for f in _DRAFT_SOURCES:
        with open(os.path.join(ROOT, "verify_markov_head_gb300", "csrc", f)) as fh:
            texts.append(fh.read())
    return _normalised_source_hash(texts)


def _draft_traffic(workload_name, fused=False):
    """dram__bytes_read.sum + dram__bytes_write.sum per draft launch from ncu
    captures recorded in profiles/traffic.json beside the summaries (with the
    target stream beside the draft: the two kernels' captures added), or None
    when one is missing or the kernels' sources changed after it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        total = 0
        for name in (("draft_rows", "target_side") if fused else ("draft_rows",)):
            r = rec[name][workload_name]
            if r.get("source_sha256") != _draft_source_hash():
                return None
            total += int(r["dram_bytes_per_launch"])
        return total
    except (OSError, KeyError, ValueError, TypeError):
        return None


_CPU_INPUTS = {}


def _cpu_inputs(w, dev_inp=None):
    """Host copies of the workload (from the device tensors when given)."""
    if w.name not in _CPU_INPUTS:
        if dev_inp is not None:
            src = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in dev_inp.items()}
        else:
            src = workload.inputs(w)
        src["W1_64"] = src["W1"].double().numpy()
        src["W2_64"] = src["W2"].double().numpy()
        _CPU_INPUTS[w.name] = src
    return _CPU_INPUTS[w.name]


def cpu_baseline(w, mode, budget_s=20.0, dev_inp=None, min_seconds=0.0, head="markov"):
    """The float64 oracle, as it stands, on a bounded sample of the workload:
    the first S requests of the batch through the whole step (draft,
    confidence, schedule, verify, compaction), S sized to a ~budget_s run,
    repeated until min_seconds have passed."""
    import oracle

    inp = _cpu_inputs(w, dev_inp)
    W1, W2 = inp["W1_64"], inp["W2_64"]
    if head == "rnn" and "rnn64" not in inp:
        src = dev_inp["rnn"] if dev_inp is not None and "rnn" in dev_inp else workload.rnn_head(w)
        inp["rnn64"] = {k: v.double().cpu().numpy() for k, v in src.items() if k != "P"}
    threads = oracle.num_threads()
    t = time.perf_counter()
    _ = oracle.draft_markov(inp["U"][:1], W1, W2, inp["anchor"][:1], seed=w.seed)
    per_req = 2.2 * (time.perf_counter() - t)         # draft + the verify's recompute of q
    S = int(max(1, min(w.B, budget_s * threads / max(per_req, 1e-3))))
    if S >= threads:
        S = (S // threads) * threads
    sub = {k: inp[k][:S] for k in ("U", "target", "h", "anchor")}
    _LAST_SAMPLE.clear()
    reps, tokens, dt = 0, 0, 0.0
    while reps == 0 or dt < min_seconds:
        t = time.perf_counter()
        tokens += _oracle_sample_step(w, mode, inp, sub, W1, W2, S, head)
        dt += time.perf_counter() - t
        reps += 1
    return {"value": tokens / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{S} of {w.B} requests of {w.name}, whole step (draft+confidence+schedule+verify+compact"
                      f"{', RNN head' if head == 'rnn' else ''}), {reps} run(s), {dt:.1f} s", "seconds": dt / reps}


def _oracle_sample_step(w, mode, inp, sub, W1, W2, S, head="markov"):
    """One oracle step over the sample; returns the tokens it emits."""
    import numpy as np

    import oracle

    arows = None
    if head == "rnn":
        p = inp["rnn64"]
        d = oracle.draft_rnn(sub["U"], p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"], W2,
                             sub["anchor"], seed=w.seed)
        arows = d["arows"]
    else:
        d = oracle.draft_markov(sub["U"], W1, W2, sub["anchor"], seed=w.seed)
    # the confidence head reads emb rows of the anchors and drafts only
    prev = np.concatenate([sub["anchor"].numpy()[:, None], d["tok"][:, :-1]], axis=1)
    ids, remap = np.unique(prev, return_inverse=True)
    remap = remap.reshape(prev.shape).astype(np.int32)
    emb = inp["emb"][torch.from_numpy(ids)]
    # position k reads the row of x~_{k-1}: anchors, then drafts 1..gamma-1 (the
    # last draft's row is never read, so its slot repeats the anchor's)
    tok_remap = np.concatenate([remap[:, 1:], remap[:, :1]], axis=1)
    c = oracle.confidence_sts(sub["h"], emb, remap[:, 0], tok_remap, inp["w_c"], inp["b_c"], inp["T"])
    if mode == 0:
        K = np.full(S, w.gamma, np.int32)
    else:
        K = oracle.schedule(c["log_surv"], inp["sps"], mode)["K"]
    v = oracle.verify(sub["target"], sub["U"], None if arows is not None else W1, W2, sub["anchor"], d["tok"], K,
                      seed=w.seed, arows=arows)
    o = oracle.compact(d["tok"], v["accepted"], v["final_tok"])
    _LAST_SAMPLE.update(S=S, draft=d, verify=v)
    return int(o["out_off"][-1])


_LAST_SAMPLE = {}       # the oracle's outputs of the last cpu_baseline sample (first S requests)


def near_ties(g_tok, g_ztok, g_acc, g_fin, sample, dg):
    """The device's decisions on the cpu_baseline sample against the oracle's:
    draws compared, mismatches, and near-ties at the published thresholds
    (Gumbel top-2 gap 1e-3, acceptance margin 1e-5) and at eps = max(4 *
    (max |z_tok error| + max |Gumbel error|), 1e-5); a mismatch that is no
    near-tie at 1e-3 / 1e-5 counts as unflagged."""
    import numpy as np
    d, v, S = sample["draft"], sample["verify"], sample["S"]
    tok, gap = d["tok"], d["gap"]
    g_tok = g_tok[:S]
    valid = np.ones(tok.shape, bool)
    for b in range(S):
        bad = np.nonzero(g_tok[b] != tok[b])[0]
        if bad.size:
            valid[b, bad[0]:] = False
    dz = float(np.abs(g_ztok[:S][valid] - d["z_tok"][valid]).max()) if valid.any() else 0.0
    eps = max(4.0 * (dz + dg), 1e-5)
    c = dict(draws=0, mismatches=0, unflagged=0, flagged_1e3=0, flagged_eps=0)
    for b in range(S):
        for k in range(tok.shape[1]):
            c["draws"] += 1
            c["flagged_1e3"] += int(gap[b, k] < 1e-3)
            c["flagged_eps"] += int(gap[b, k] < eps)
            if g_tok[b, k] != tok[b, k]:
                c["mismatches"] += 1
                c["unflagged"] += int(gap[b, k] >= 1e-3)
                break
    for b in np.nonzero(valid.all(axis=1))[0]:
        margin, fgap = v["diag"][b, 0], v["diag"][b, 1]
        c["draws"] += 2                      # the accept walk and the final draw
        c["flagged_1e3"] += int(margin < 1e-5) + int(fgap < 1e-3)
        c["flagged_eps"] += int(margin < 1e-5) + int(fgap < eps)
        if g_acc[b] != v["accepted"][b]:
            c["mismatches"] += 1
            c["unflagged"] += int(margin >= 1e-5)
        elif g_fin[b] != v["final_tok"][b]:
            c["mismatches"] += 1
            c["unflagged"] += int(fgap >= 1e-3)
    c.update(eps=eps, rate_eps=c["flagged_eps"] / max(1, c["draws"]), requests=int(S),
             sample="the cpu_baseline requests, whole step")
    return c


def device_gumbel_error(vm, dev, n=1 << 18):
    """max |G_device - G_exact| over n columns of two random streams (the
    device's uniforms are exact; G_exact = -log(-log u) in binary64)."""
    import numpy as np
    g = torch.empty(n, device=dev)
    u = torch.empty(n, device=dev)
    worst = 0.0
    for seed, dom, row in ((0, 0, 0), (2, 2, 77)):
        vm.dspark_gumbel_stream(seed, 0, dom, row, n, g, u)
        torch.cuda.synchronize(dev)
        gu = u.cpu().double().numpy()
        worst = max(worst, float(np.abs(g.cpu().double().numpy() + np.log(-np.log(gu))).max()))
    return worst


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload.WORKLOADS[args.workload]
    mode = {"off": 0, "spec": w.mode}[args.sched]
    # each step a sample sized so the whole run stays within a few minutes
    # (at least one request: about 0.3 s on 16 cores at the b64 sizes)
    budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, mode, budget_s=budget)
    vals, secs = [], 0.0
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(w, mode, budget_s=budget)
        vals.append(last["value"]); secs += last["seconds"]
    value = statistics.mean(vals)
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(1, args.steps), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: B={w.B} V={w.V} r={w.r} gamma={w.gamma} d={w.d}, bounded sample"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="b64", choices=sorted(workload.WORKLOADS))
    ap.add_argument("--sched", default="off", choices=["off", "spec"],
                    help="off: full-prefix verification; spec: the workload's scheduler mode")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the extra step records (b1, b256, b64 with its scheduler) of the default line")
    ap.add_argument("--chain", action="store_true",
                    help="time the workload's chained steps (b512: 16 steps, async scheduler) instead of one step")
    ap.add_argument("--head", default="markov", choices=["markov", "rnn"],
                    help="draft head: the Markov head (default) or the RNN head")
    ap.add_argument("--fuse-target", default="auto", choices=["auto", "on", "off"],
                    help="scheduler off: draft with the target stream (dspark_draft_markov_target) and verify "
                         "in full-prefix mode; auto takes it where the stream beside the draft pays (B <= 256)")
    ap.add_argument("--sts", action="store_true",
                    help="time the STS temperature fit (2^20 validation blocks, 256 temperatures)")
    ap.add_argument("--kernel", default=None, choices=["draft", "verify", "fused", "fused-verify", "confidence"],
                    help="run one ABI call --calls times on the workload's shapes (for profiler captures); "
                         "prints no metric")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--sts-blocks", type=int, default=None,
                    help="validation blocks of the STS fit (default 2^20; smaller for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.kernel:
        run_kernel(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.chain:
        run_chain(args)
    elif args.sts:
        run_sts(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
