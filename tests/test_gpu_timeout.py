"""The timeout path of the device waits, made to run on purpose.

dspark_workspace_set_wait_limit bounds every wait of a kernel on another role
or on other CTAs (copy rings, accumulator hand-offs, grid barriers, the verify
stream's ring).  With a bound of a few hundred cycles those waits give up
before the copies they wait for can land: each kernel must then raise the
timeout bit, drain the copies it issued (their own fixed bounds), free its
tensor memory and return, so that dspark_sync_status reports
DSPARK_ERR_TIMEOUT, the context stays usable, and after dspark_workspace_init
the same calls again match the oracle.  No fault, trap or unbounded wait is
involved: every wait on the path is bounded."""
import numpy as np
import pytest
import torch

import oracle
import workload
from tests._parity import LOGIT_ATOL, U_EPS, assert_close_where, compare_draft

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None

DEV = "cuda"
TIMEOUT = -3
TIMEOUT_BIT = 1 << 2
SHORT = 300          # SM cycles: far below one copy's latency


def _cpu(inp):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _draft(inp, buf, seed):
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                           buf.ws, seed=seed)


def _verify(inp, buf, seed, K):
    vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                     buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off, buf.next_anchor,
                     buf.ws, seed=seed)


def test_expired_waits_report_a_timeout_and_the_workspace_recovers():
    # the tensor-core draft (one cooperative launch, grid barriers) and the
    # verify stream plus the tensor-core residual draw
    w = workload.custom("tiny", B=24, V=8200, r=128, w_dtype=torch.bfloat16, w_std=0.1, seed=13)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    seed = 5

    vm.dspark_workspace_set_wait_limit(buf.ws.buf, SHORT)
    _draft(inp, buf, seed)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == TIMEOUT and bits & TIMEOUT_BIT, (st, hex(bits))

    vm.dspark_workspace_init(buf.ws.buf)
    _draft(inp, buf, seed)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, (st, hex(bits))
    ci = _cpu(inp)
    ref = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=seed)
    _, _, valid = compare_draft(buf.draft_tok.cpu().numpy(), ref["tok"], ref["gap"])
    assert_close_where(buf.lse_q.cpu().numpy(), ref["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")

    K = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    vm.dspark_workspace_set_wait_limit(buf.ws.buf, SHORT)
    _verify(inp, buf, seed, K)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == TIMEOUT and bits & TIMEOUT_BIT, (st, hex(bits))

    vm.dspark_workspace_init(buf.ws.buf)
    _verify(inp, buf, seed, K)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, (st, hex(bits))
    tok = buf.draft_tok.cpu().numpy()
    v = oracle.verify(ci["target"], ci["U"], ci["W1"], ci["W2"], ci["anchor"], tok, np.full(w.B, w.gamma, np.int32),
                      seed=seed)
    acc = buf.accepted.cpu().numpy()
    for b in np.nonzero(acc != v["accepted"])[0]:
        assert v["diag"][b, 0] < U_EPS, f"accept mismatch at request {b} after recovery"


def test_expired_waits_with_the_target_stream_beside_the_draft():
    # the draft and the lean target stream on the same SMs, then the
    # full-prefix verify (residual and bonus draws in one kernel)
    w = workload.custom("tiny", B=24, V=8200, r=128, w_dtype=torch.bfloat16, w_std=0.1, seed=14)
    inp = workload.inputs(w, device=DEV)
    assert vm.target_stream_beside(inp)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    seed = 6

    def fused():
        vm.dspark_draft_markov_target(inp["U"], inp["W1"], inp["W2"], inp["target"], inp["anchor"], buf.draft_tok,
                                      buf.lse_q, buf.z_tok, buf.ws, seed=seed)
        _verify(inp, buf, seed, None)

    vm.dspark_workspace_set_wait_limit(buf.ws.buf, SHORT)
    fused()
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == TIMEOUT and bits & TIMEOUT_BIT, (st, hex(bits))

    vm.dspark_workspace_init(buf.ws.buf)
    fused()
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, (st, hex(bits))
    ci = _cpu(inp)
    tok = buf.draft_tok.cpu().numpy()
    ref = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=seed)
    compare_draft(tok, ref["tok"], ref["gap"])
    v = oracle.verify(ci["target"], ci["U"], ci["W1"], ci["W2"], ci["anchor"], tok, np.full(w.B, w.gamma, np.int32),
                      seed=seed)
    acc = buf.accepted.cpu().numpy()
    for b in np.nonzero(acc != v["accepted"])[0]:
        assert v["diag"][b, 0] < U_EPS, f"accept mismatch at request {b} after recovery"


def test_default_bound_is_restored_by_zero():
    w = workload.custom("tiny", B=4, V=1024, r=64, w_dtype=torch.bfloat16, seed=2)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_workspace_set_wait_limit(buf.ws.buf, SHORT)
    vm.dspark_workspace_set_wait_limit(buf.ws.buf, 0)
    _draft(inp, buf, seed=1)
    assert vm.dspark_sync_status(buf.ws.buf) == (0, 0)
