"""The request-sharded step on two CPU ranks (gloo): drafting, confidence
and verification per rank with global request indices, the scheduler on the
all-gathered survival lists.  Sharding must not change a single result: the
gathered outputs equal the whole batch run in one process."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workload
from tests._dp_worker import history

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(name, B, mode, out, world=2):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "tests", "_dp_worker.py"), name,
                                       str(B), str(mode), out], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    logs = []
    for p in procs:
        try:
            logs.append(p.communicate(timeout=240)[0])
        except subprocess.TimeoutExpired:
            p.kill()
            logs.append(p.communicate()[0])
    for p, log in zip(procs, logs):
        assert p.returncode == 0, log[-3000:]


@pytest.mark.parametrize("B,mode", [(4, 1), (8, 1), (8, 2), (8, 0)])
def test_two_ranks_match_one_process(tmp_path, B, mode):
    out = str(tmp_path / "ranks.npz")
    _run_ranks("tiny", B, mode, out)
    got = np.load(out)
    w = workload.custom("tiny", B=B)
    inp = workload.inputs(w)
    hist = history(w.B, w.gamma, 7) if mode == 2 else None
    ref = oracle.step(inp, mode=mode, seed=w.seed, log_surv_hist=hist)
    np.testing.assert_array_equal(got["tok"], ref["draft"]["tok"])
    np.testing.assert_allclose(got["lse_q"], ref["draft"]["lse_q"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["log_surv"], ref["conf"]["log_surv"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(got["K"], ref["sched"]["K"])
    assert int(got["n_total"]) == ref["sched"]["n_total"]
    np.testing.assert_array_equal(got["accepted"], ref["verify"]["accepted"])
    np.testing.assert_array_equal(got["final_tok"], ref["verify"]["final_tok"])


def test_uneven_split_is_refused():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "dspark_shard", os.path.join(ROOT, "verify_markov_head_gb300", "shard.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    assert m.shard_of(1, 2, 8) == (4, 4)
    with pytest.raises(ValueError):
        m.shard_of(0, 3, 8)
    with pytest.raises(ValueError):
        m.shard_of(2, 2, 8)
