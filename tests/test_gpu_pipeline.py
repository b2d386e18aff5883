"""Steps from host memory through HostPipeline (the copy of step t+1
overlapping step t) give the same results as steps run one at a time on
device inputs, with several steps in flight before anything is read."""
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

PER_STEP = ("U", "target", "h", "anchor")


@pytest.mark.parametrize("base,kw", [("tiny", dict(B=8)), ("b64", dict(V=16384))])
def test_pipeline_equals_sequential_steps(base, kw):
    w = workload.custom(base, **kw)
    W = workload.weights(w, device="cuda")
    steps = [workload.step_inputs(w, step=t, device="cpu") for t in range(4)]
    # sequential reference on device inputs
    ref = []
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    for t, si in enumerate(steps):
        inp = dict(W)
        inp.update({k: v.to("cuda") for k, v in si.items()})
        vm.run_step(inp, buf, mode=0, seed=w.seed, step=t)
        n = int(buf.out_off[-1])
        ref.append((buf.out_off.cpu().clone(), buf.out_tok[:n].cpu().clone(), buf.next_anchor.cpu().clone()))
    # pipelined: every step enqueued before any result is read
    dev_inp = dict(W)
    dev_inp.update({k: v.to("cuda") for k, v in steps[0].items()})
    pbuf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    stream = torch.cuda.Stream()
    pipe = vm.HostPipeline(dev_inp, pbuf, stream)
    hosts = [{k: si[k].pin_memory() for k in PER_STEP} for si in steps]
    outs = [{"out_tok": torch.empty(w.B * (w.gamma + 1), dtype=torch.int32).pin_memory(),
             "out_off": torch.empty(w.B + 1, dtype=torch.int32).pin_memory(),
             "next_anchor": torch.empty(w.B, dtype=torch.int32).pin_memory()} for _ in steps]
    for t in range(len(steps)):
        pipe.step(hosts[t], outs[t], mode=0, seed=w.seed, step=t)
    torch.cuda.synchronize()
    st, bits = vm.dspark_sync_status(pbuf.ws.buf)
    assert st == 0, bits
    for t, (off, tok, nxt) in enumerate(ref):
        assert torch.equal(outs[t]["out_off"], off), t
        assert torch.equal(outs[t]["out_tok"][: int(off[-1])], tok), t
        assert torch.equal(outs[t]["next_anchor"], nxt), t
