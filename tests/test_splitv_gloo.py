"""The vocabulary split of the latency case on two and three CPU ranks
(gloo): every rank holds a slice of V (slices of unequal size), the draft
gathers one (draw, log-sum-exp) state per request and position, verification
gathers the rows' log-sum-exps and the residual or bonus draw's winners.
Splitting must not change a result: the gathered drafts, log-normalisers,
accepted counts and final tokens equal the oracle's on the whole vocabulary.
Host logic only; not measured on GPUs."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,B,V", [(2, 1, 1000), (3, 3, 1026)])
def test_vocabulary_split_matches_the_whole_vocabulary(tmp_path, world, B, V):
    out = str(tmp_path / "splitv.npz")
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "tests", "_splitv_worker.py"), str(B),
                                       str(V), out], env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                      text=True))
    logs = []
    for p in procs:
        try:
            logs.append(p.communicate(timeout=240)[0])
        except subprocess.TimeoutExpired:
            p.kill()
            logs.append(p.communicate()[0])
    for p, log in zip(procs, logs):
        assert p.returncode == 0, log[-3000:]
    got = np.load(out)
    w = workload.custom("b1", B=B, V=V, r=32, d=16, seed=9)
    inp = workload.inputs(w)
    d = oracle.draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], seed=41, step=3)
    np.testing.assert_array_equal(got["tok"], d["tok"])
    np.testing.assert_allclose(got["lse_q"], d["lse_q"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["z_tok"], d["z_tok"], rtol=0, atol=1e-12)
    K = np.full(B, w.gamma, np.int32)
    v = oracle.verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], d["tok"], K, seed=41, step=3)
    np.testing.assert_array_equal(got["accepted"], v["accepted"])
    np.testing.assert_array_equal(got["final"], v["final_tok"])


def test_slice_functions_on_the_whole_row_equal_the_oracle():
    """One slice covering the whole vocabulary reproduces the oracle's draw,
    log-normaliser and drawn logit (a pin of the slice functions)."""
    w = workload.custom("tiny", B=2, V=512, r=16, seed=4)
    inp = workload.inputs(w)
    U = inp["U"].double().numpy(); W1 = inp["W1"].double().numpy(); W2 = inp["W2"].double().numpy()
    d = oracle.draft_markov(U, W1, W2, inp["anchor"].numpy(), seed=2, step=0)
    for b in range(w.B):
        prev = int(inp["anchor"][b])
        for k in range(w.gamma):
            s = oracle.slice_draft(U[b, k], W1[prev], W2, 0, seed=2, step=0, row=b * (w.gamma + 1) + k)
            assert s["idx"] == d["tok"][b, k]
            assert abs(s["lse"] - d["lse_q"][b, k]) < 1e-12 and abs(s["zb"] - d["z_tok"][b, k]) < 1e-12
            prev = int(d["tok"][b, k])
    np.testing.assert_allclose(oracle.gumbel_span(3, 1, 2, 9, 100, 8),
                               [oracle.gumbel(3, 1, 2, 9, 100 + i) for i in range(8)], rtol=0, atol=0)
