#!/usr/bin/env python
"""Draft + verify throughput of the DSpark step on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
Markov-head draft loop (gamma launches), confidence + STS + survival,
prefix scheduler, verification stream + accept walk + residual draw +
compaction.  Default workload: B=64, V=151936, r=256, gamma=7, d=4096,
bf16 draft-head weights, fp32 base and target logits, full-prefix
verification (scheduler call made in OFF mode, K_b = 7).

Prints one JSON line (rank 0).  `value` = emitted tokens per second over all
ranks with inputs resident in HBM (CUDA-graph replay of the step, CUDA
events on the launching stream, inputs 1.13 GB > L2 so no flush).
`e2e` = the same metric through the public API with the step's activations
copied from pinned host memory and the emitted tokens copied back inside the
timed region.  `roofline` = the draft kernel (the dominant one: gamma
launches per step, each streaming W2 and one row block of U).

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the reference arm of this tier).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workload  # noqa: E402

METRIC = "draft+verify tokens/s (B=64, V=151936, γ=7) and % of HBM roofline on 1 GB300"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

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
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
                "samples": len(sm)}


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
    buf = vm.StepBuffers(B, gamma, V, r, device=dev)
    stream = torch.cuda.Stream(device=dev)
    seed = w.seed

    def one_step():
        vm.run_step(inp, buf, mode=mode, seed=seed, step=0, req_base=req_base, stream=stream)

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

    # ---- timed region: K graph replays of the whole step
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        stream.synchronize()
        if args.steps * 0.2 < 1.0:     # keep sampling long enough for a few clock readings
            time.sleep(0.5)
    torch.cuda.synchronize()
    _barrier(dist)
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = _max_over_ranks(dist, ms, dev)
    emitted = int(buf.out_off[-1].item())
    emitted_all = _sum_over_ranks(dist, emitted, dev)
    value = emitted_all / (ms_max / 1e3)

    # ---- dominant kernel: the draft launches, timed alone on the same stream
    reps = max(5, args.steps)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        d0.record(stream)
        for _ in range(reps):
            vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                                   buf.z_tok, buf.ws, seed=seed, req_base=req_base, stream=stream)
        d1.record(stream)
    stream.synchronize()
    draft_launch_ms = d0.elapsed_time(d1) / (reps * gamma)
    w2_bytes = r * V * inp["W2"].element_size()
    u_bytes_k = B * V * inp["U"].element_size()
    draft_bytes = w2_bytes + u_bytes_k                   # per launch: W2 once + one position of U
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
    e2e_steps = max(3, min(args.steps, 10))
    with torch.cuda.stream(stream):
        vm.run_step_host(host, inp, buf, host_out, mode=mode, seed=seed, stream=stream)
    stream.synchronize()
    _barrier(dist)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(e2e_steps):
            h2d, d2h = vm.run_step_host(host, inp, buf, host_out, mode=mode, seed=seed, stream=stream)
        f1.record(stream)
    stream.synchronize()
    e2e_ms = _max_over_ranks(dist, f0.elapsed_time(f1) / e2e_steps, dev)
    e2e_emitted = _sum_over_ranks(dist, int(host_out["out_off"][-1]), dev)

    st, bits = vm.dspark_sync_status(buf.ws.buf, stream)
    if st != 0:
        raise SystemExit(f"device status {st} bits {bits}")

    launches_per_step = gamma + 1 + 1 + 4
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, mode, budget_s=args.cpu_budget, dev_inp=inp)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 weights, f32 logits, f32 accumulate", "data": "synthetic",
            "config": {"workload": f"{w.name}: B={B} V={V} r={r} gamma={gamma} d={d_of(w)} "
                                   f"verify={'full prefix (scheduler off)' if mode == 0 else 'scheduled'}",
                       "global_batch": B * world, "seq_len": gamma, "parallelism": f"dp{world} over requests",
                       "l2": "inputs 1.13 GB per step > 129 MB L2; no flush", "graph": "CUDA graph replay"},
            "emitted_tokens_per_step": emitted_all, "drafted_tokens_per_step": B * gamma * world,
            "step_formula_bytes": formula_bytes, "step_formula_gbs": step_gbs,
            "step_formula_frac": step_gbs / peak,
            "roofline": {"kernel": "draft_markov (per position launch)", "bound": "hbm", "achieved": achieved,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "algorithmic_bytes_per_launch": draft_bytes,
                         "launch_ms": draft_launch_ms},
            "e2e": {"value": e2e_emitted / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def d_of(w):
    return w.d


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


def cpu_baseline(w, mode, budget_s=20.0, dev_inp=None):
    """The float64 oracle, as it stands, on a bounded sample of the workload:
    the first S requests of the batch through the whole step (draft,
    confidence, schedule, verify, compaction), S sized to a ~budget_s run."""
    import numpy as np

    import oracle

    inp = _cpu_inputs(w, dev_inp)
    W1, W2 = inp["W1_64"], inp["W2_64"]
    threads = oracle.num_threads()
    t = time.perf_counter()
    _ = oracle.draft_markov(inp["U"][:1], W1, W2, inp["anchor"][:1], seed=w.seed)
    per_req = 2.2 * (time.perf_counter() - t)         # draft + the verify's recompute of q
    S = int(max(1, min(w.B, budget_s * threads / max(per_req, 1e-3))))
    if S >= threads:
        S = (S // threads) * threads
    sub = {k: inp[k][:S] for k in ("U", "target", "h", "anchor")}
    t = time.perf_counter()
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
    v = oracle.verify(sub["target"], sub["U"], W1, W2, sub["anchor"], d["tok"], K, seed=w.seed)
    o = oracle.compact(d["tok"], v["accepted"], v["final_tok"])
    dt = time.perf_counter() - t
    return {"value": int(o["out_off"][-1]) / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{S} of {w.B} requests of {w.name}, whole step (draft+confidence+schedule+verify+compact), "
                      f"{dt:.1f} s", "seconds": dt}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload.WORKLOADS[args.workload]
    mode = {"off": 0, "spec": w.mode}[args.sched]
    budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="b64", choices=sorted(workload.WORKLOADS))
    ap.add_argument("--sched", default="off", choices=["off", "spec"],
                    help="off: full-prefix verification; spec: the workload's scheduler mode")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
