"""One rank of the vocabulary-split draft and verification on the CPU
(gloo), with the oracle's slice functions standing in for the device
kernels.  Run with RANK, WORLD_SIZE, MASTER_ADDR and MASTER_PORT set; argv:
B, V, output file (written by rank 0)."""
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


def main():
    B, V, out = int(sys.argv[1]), int(sys.argv[2]), sys.argv[3]
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    shard = _shard_module()
    w = workload.custom("b1", B=B, V=V, r=32, d=16, seed=9)
    inp = workload.inputs(w)
    U = inp["U"].double().numpy(); T = inp["target"].double().numpy()
    W1 = inp["W1"].double().numpy(); W2 = inp["W2"].double().numpy()
    anchor = inp["anchor"].numpy()
    g1 = w.gamma + 1
    bounds = np.linspace(0, V, world + 1).astype(int)     # uneven slices are fine
    v0, v1 = int(bounds[rank]), int(bounds[rank + 1])
    seed, step = 41, 3

    def slice_draft(k, prev):
        rows = []
        for b in range(B):
            d = oracle.slice_draft(U[b, k - 1, v0:v1], W1[int(prev[b])], W2[:, v0:v1], v0, seed=seed, step=step,
                                   row=b * g1 + (k - 1))
            rows.append([d["best"], d["idx"], d["zb"], d["lse"]])
        return np.array(rows)

    tok, lse_q, z_tok = shard.split_v_draft(slice_draft, anchor, w.gamma)
    tk = tok.numpy()
    K = np.full(B, w.gamma, np.int32)

    def row_lse():
        return np.array([[oracle.slice_lse(T[b, k, v0:v1]) for k in range(w.gamma)] for b in range(B)])

    def token_logit():
        x = np.full((B, w.gamma), -np.inf)
        for b in range(B):
            for k in range(w.gamma):
                if v0 <= tk[b, k] < v1:
                    x[b, k] = T[b, k, tk[b, k]]
        return x

    def uniform(b, k):
        return oracle.uniform(seed, step, 1, b * g1 + (k - 1), 0)

    def residual(b, j, lp, lq):
        prev = anchor[b] if j == 0 else tk[b, j - 1]
        z = U[b, j, v0:v1] + W1[prev] @ W2[:, v0:v1]
        d = oracle.slice_residual(T[b, j, v0:v1], z, lp, lq, v0, seed=seed, step=step, row=b * g1 + j)
        return [d["best_r"], d["idx_r"], d["best_p"], d["idx_p"]]

    def bonus(b, k):
        d = oracle.slice_bonus(T[b, k, v0:v1], v0, seed=seed, step=step, row=b * g1 + k)
        return [d["best"], d["idx"]]

    acc, fin = shard.split_v_verify(row_lse, token_logit, uniform, residual, bonus, tok, lse_q, z_tok, K)
    if rank == 0:
        np.savez(out, tok=tk, lse_q=lse_q.numpy(), z_tok=z_tok.numpy(), accepted=acc.numpy(), final=fin.numpy())
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
