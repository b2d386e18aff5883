"""One rank of the request-sharded step on the CPU (gloo), with the oracle
standing in for the device kernels.  Run as a process with RANK, WORLD_SIZE,
MASTER_ADDR and MASTER_PORT set; argv: workload name, B, scheduler mode,
output file (written by rank 0)."""
import importlib.util
import os
import sys

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workload  # noqa: E402


def _shard_module():
    spec = importlib.util.spec_from_file_location(
        "dspark_shard", os.path.join(ROOT, "verify_markov_head_gb300", "shard.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def history(B, gamma, seed):
    """A survival list two steps old: non-increasing, <= 0, seeded."""
    rng = np.random.default_rng(seed)
    return -np.cumsum(rng.exponential(0.3, size=(B, gamma)), axis=1)


def main():
    name, B, mode, out = sys.argv[1], int(sys.argv[2]), int(sys.argv[3]), sys.argv[4]
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    shard = _shard_module()
    w = workload.custom(name, B=B)
    inp = workload.inputs(w)                      # the whole batch, identical on every rank
    start, n = shard.shard_of(rank, world, w.B)
    sl = slice(start, start + n)
    req = np.arange(start, start + n, dtype=np.int32)
    d = oracle.draft_markov(inp["U"][sl], inp["W1"], inp["W2"], inp["anchor"][sl], seed=w.seed, req=req)
    c = oracle.confidence_sts(inp["h"][sl], inp["emb"], inp["anchor"][sl], d["tok"], inp["w_c"], inp["b_c"],
                              inp["T"])
    hist = torch.from_numpy(history(w.B, w.gamma, 7)[sl].copy()) if mode == 2 else None
    sps = inp["sps"].double().numpy()

    def schedule(all_surv, all_hist):
        s = oracle.schedule(all_surv.numpy(), sps, mode, None if all_hist is None else all_hist.numpy())
        return torch.from_numpy(s["K"]), s["n_total"], s["theta"]

    K, n_total, theta, _ = shard.global_schedule(torch.from_numpy(c["log_surv"]), hist, schedule)
    v = oracle.verify(inp["target"][sl], inp["U"][sl], inp["W1"], inp["W2"], inp["anchor"][sl], d["tok"],
                      K.numpy(), seed=w.seed, req=req)
    g = {k: shard.gather_rows(torch.from_numpy(np.ascontiguousarray(x)))
         for k, x in (("tok", d["tok"]), ("lse_q", d["lse_q"]), ("log_surv", c["log_surv"]), ("K", K.numpy()),
                      ("accepted", v["accepted"]), ("final_tok", v["final_tok"]))}
    if rank == 0:
        np.savez(out, n_total=n_total, theta=theta, **{k: t.numpy() for k, t in g.items()})
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
