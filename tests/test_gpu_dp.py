"""The request-sharded step on the device (run_step_dp) in a one-rank NCCL
group equals the single-process step: the gather, the scheduler on the
gathered list and the verify lengths it hands back are plumbing only."""
import pytest
import torch

import workload

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None


@pytest.fixture(scope="module")
def group():
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1)
    yield None
    dist.destroy_process_group()


@pytest.mark.parametrize("base,kw,mode", [("tiny", dict(B=8), 1), ("tiny", dict(B=8), 2),
                                          ("b64", dict(V=16384), 1), ("b64", dict(V=16384), 0)])
def test_dp_step_one_rank_equals_step(group, base, kw, mode):
    w = workload.custom(base, **kw)
    inp = workload.inputs(w, device="cuda")
    hist = None
    if mode == 2:
        g = torch.Generator(device="cuda").manual_seed(5)
        hist = -torch.cumsum(torch.rand((w.B, w.gamma), generator=g, device="cuda"), dim=1)
    a = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    b = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    sched = vm.GlobalSchedule(w.B, w.gamma, 1)
    vm.run_step(inp, a, mode=mode, seed=w.seed, log_surv_hist=hist)
    vm.run_step_dp(inp, b, sched, mode=mode, seed=w.seed, log_surv_hist=hist)
    for buf in (a, b):
        st, bits = vm.dspark_sync_status(buf.ws.buf)
        assert st == 0, bits
    assert torch.equal(a.K, b.K)
    assert torch.equal(a.n_total, b.n_total)
    assert torch.equal(a.accepted, b.accepted)
    n = int(a.out_off[-1])
    assert torch.equal(a.out_off, b.out_off) and torch.equal(a.out_tok[:n], b.out_tok[:n])
