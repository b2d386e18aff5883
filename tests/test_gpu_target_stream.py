"""GPU parity of the draft with the target stream (dspark_draft_markov_target)
and of the full-prefix verify that uses it (K = None), against the float64
oracle ("DSpark：半自回归生成与置信度调度的投机解码", section 形式化定义: each
draft position is verified against the target's distribution at that
position, the bonus token drawn from the row after the last one).

The fused draft runs the same race and log-sum-exp as dspark_draft_markov, so
its drafts must equal that call's bit for bit.  The full-prefix verify takes
rows 0..gamma-1's log-sum-exps from the draft's partials; its decisions are
compared with the oracle's verify at K_b = gamma for every request, with the
same near-tie flags as the other verify tests.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
from tests._parity import GAP_EPS, PROB_RTOL, U_EPS, assert_close_where, compare_draft

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None
DEV = "cuda"
KERNEL_BADINPUT = 1 << 3


def _cpu(inp):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _fused_draft(inp, w, buf, seed, step=0, req_base=0, tau=1.0, logits=None):
    vm.dspark_draft_markov_target(inp["U"], inp["W1"], inp["W2"], inp["target"], inp["anchor"], buf.draft_tok,
                                  buf.lse_q, buf.z_tok, buf.ws, seed=seed, step=step, req_base=req_base, tau=tau,
                                  logits_out=logits)


def _plain_draft(inp, w, seed, step=0, req_base=0, tau=1.0):
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                           buf.ws, seed=seed, step=step, req_base=req_base, tau=tau)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    return buf


def _full_verify(inp, buf, seed, step=0, req_base=0, tau=1.0, logits=None):
    args = (buf.draft_tok, buf.lse_q, buf.z_tok, None, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos,
            buf.out_off, buf.next_anchor, buf.ws)
    kw = dict(seed=seed, step=step, req_base=req_base, tau=tau, p_tok=buf.p_tok, near_ties=buf.near_ties)
    if logits is None:
        vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], *args, **kw)
    else:
        vm.dspark_verify_logits(inp["target"], inp["U"], inp["W1"], inp["W2"], logits, inp["anchor"], *args, **kw)


def _check_against_oracle(inp, w, buf, seed, step=0, req_base=0, tau=1.0):
    ci = _cpu(inp)
    tok = buf.draft_tok.cpu().numpy()
    K = np.full(w.B, w.gamma, np.int32)
    req = np.arange(req_base, req_base + w.B)
    ref = oracle.verify(ci["target"], ci["U"], ci["W1"], ci["W2"], ci["anchor"], tok, K, seed=seed, step=step,
                        req=req, tau=tau)
    acc = buf.accepted.cpu().numpy()
    bad = acc != ref["accepted"]
    for b in np.nonzero(bad)[0]:
        assert ref["diag"][b, 0] < U_EPS, f"unflagged accept mismatch at request {b}"
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[1:] - 1]
    for b in range(w.B):
        if not bad[b] and fin[b] != ref["final_tok"][b]:
            assert ref["diag"][b, 1] < GAP_EPS, f"unflagged final-token mismatch at request {b}"
    walked = ~np.isnan(ref["p_tok"])          # positions up to the first rejection
    assert walked[:, 0].all()
    assert_close_where(buf.p_tok.cpu().numpy(), ref["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")
    assert off[0] == 0 and (np.diff(off) == acc + 1).all()
    np.testing.assert_array_equal(buf.next_anchor.cpu().numpy(), fin)
    return ref


@pytest.mark.parametrize("B,V,r,tdt", [(4, 1024, 64, torch.float32), (7, 4104, 64, torch.float32),
                                       (64, 2048, 256, torch.float32), (33, 8200, 128, torch.float32),
                                       (130, 2056, 64, torch.float32), (1, 4104, 128, torch.float32),
                                       (40, 4104, 128, torch.bfloat16), (200, 2056, 64, torch.bfloat16)])
def test_fused_draft_equals_plain_draft_and_verifies_like_the_oracle(B, V, r, tdt):
    # V = 4104, 8200, 2056: the last tile's column blocks straddle the end of the
    # vocabulary (masked tail); B = 130, 200: two request chunks (RF = 1); B = 1:
    # the one-request epilogue; bf16 targets: the stream beside the draft reads
    # half the bytes per entry
    w = workload.custom("tiny", B=B, V=V, r=r, w_dtype=torch.bfloat16, w_std=0.1, seed=5 * B + r,
                        target_dtype=tdt)
    inp = workload.inputs(w, device=DEV)
    seed = B + 11
    plain = _plain_draft(inp, w, seed)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    _fused_draft(inp, w, buf, seed)
    np.testing.assert_array_equal(buf.draft_tok.cpu().numpy(), plain.draft_tok.cpu().numpy())
    np.testing.assert_array_equal(buf.lse_q.cpu().numpy(), plain.lse_q.cpu().numpy())
    np.testing.assert_array_equal(buf.z_tok.cpu().numpy(), plain.z_tok.cpu().numpy())
    _full_verify(inp, buf, seed)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    _check_against_oracle(inp, w, buf, seed)


def test_full_prefix_verify_equals_the_streamed_verify():
    """The same drafts verified twice: K = gamma through the verify stream, and
    K = None from the draft's partials.  Decisions agree; p(x~) to rounding."""
    w = workload.custom("tiny", B=48, V=8192, r=128, w_dtype=torch.bfloat16, w_std=0.1, seed=3)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    _fused_draft(inp, w, buf, seed=9, step=2)
    _full_verify(inp, buf, seed=9, step=2)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    acc_f, p_f = buf.accepted.cpu().numpy(), buf.p_tok.cpu().numpy()
    fin_f = buf.next_anchor.cpu().numpy()
    K = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                     buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                     buf.next_anchor, buf.ws, seed=9, step=2, p_tok=buf.p_tok, near_ties=buf.near_ties)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    np.testing.assert_allclose(p_f, buf.p_tok.cpu().numpy(), rtol=1e-5, atol=0)
    np.testing.assert_array_equal(acc_f, buf.accepted.cpu().numpy())
    np.testing.assert_array_equal(fin_f, buf.next_anchor.cpu().numpy())


def test_temperature_request_base_and_stored_logits():
    w = workload.custom("tiny", B=3, V=4104, r=64, w_dtype=torch.bfloat16, w_std=0.1, seed=12)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    logits = torch.empty((w.B, w.gamma, w.V), device=DEV)
    _fused_draft(inp, w, buf, seed=4, step=3, req_base=500, tau=0.7, logits=logits)
    _full_verify(inp, buf, seed=4, step=3, req_base=500, tau=0.7, logits=logits)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    ci = _cpu(inp)
    d = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=4, step=3, tau=0.7,
                            req=np.arange(500, 503))
    compare_draft(buf.draft_tok.cpu().numpy(), d["tok"], d["gap"])
    _check_against_oracle(inp, w, buf, seed=4, step=3, req_base=500, tau=0.7)


@pytest.mark.parametrize("tdt", [torch.float32, torch.bfloat16])
def test_stream_beside_the_draft_short_chain_temperature_request_base(tdt):
    """gamma = 2 (the shortest chain the stream beside the draft takes), a
    temperature, a request base and a vocabulary whose last segment is short;
    the residual launch also draws the bonus tokens (full-prefix dspark_verify)."""
    w = workload.custom("tiny", B=24, V=33800, r=128, gamma=2, w_dtype=torch.bfloat16, w_std=0.1, seed=31,
                        target_dtype=tdt)
    inp = workload.inputs(w, device=DEV)
    assert vm.target_stream_beside(inp)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    _fused_draft(inp, w, buf, seed=7, step=5, req_base=100, tau=0.8)
    _full_verify(inp, buf, seed=7, step=5, req_base=100, tau=0.8)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    ci = _cpu(inp)
    d = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=7, step=5, tau=0.8,
                            req=np.arange(100, 100 + w.B))
    compare_draft(buf.draft_tok.cpu().numpy(), d["tok"], d["gap"])
    _check_against_oracle(inp, w, buf, seed=7, step=5, req_base=100, tau=0.8)


def test_single_position_target_stream():
    """gamma = 1 runs the target-stream draft as one single-position launch
    (the epilogue form, the launch every position uses where cooperative
    launch is unavailable), then the full-prefix verify."""
    w = workload.custom("tiny", B=20, V=4104, r=128, gamma=1, w_dtype=torch.bfloat16, w_std=0.1, seed=8)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    _fused_draft(inp, w, buf, seed=6)
    _full_verify(inp, buf, seed=6)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    _check_against_oracle(inp, w, buf, seed=6)


def test_full_size_b64_step_sampled_requests():
    """The b64 workload (B=64, V=151936, r=256) through run_step with the
    scheduler off and the fused path; sampled requests recomputed by the
    oracle along the device's drafts."""
    w = workload.WORKLOADS["b64"]
    inp = workload.inputs(w, device=DEV)
    assert vm.target_stream_supported(inp)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=0, seed=w.seed, p_tok=True, fuse_target=True)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    S = np.array([0, 17, 40, 63])
    Sd = torch.from_numpy(S).to(DEV).long()
    ci = {k: inp[k][Sd].cpu() for k in ("U", "target", "anchor")}
    W1 = inp["W1"].cpu()
    W2 = inp["W2"].cpu()
    tok = buf.draft_tok.cpu().numpy()[S]
    K = np.full(len(S), w.gamma, np.int32)
    ref = oracle.verify(ci["target"], ci["U"], W1, W2, ci["anchor"], tok, K, seed=w.seed, req=S)
    acc = buf.accepted.cpu().numpy()[S]
    for i in np.nonzero(acc != ref["accepted"])[0]:
        assert ref["diag"][i, 0] < U_EPS
    assert_close_where(buf.p_tok.cpu().numpy()[S], ref["p_tok"], ~np.isnan(ref["p_tok"]), rtol=PROB_RTOL,
                       what="p_tok")


def test_mismatched_inputs_raise_the_status_bit():
    """A full-prefix verify whose inputs differ from the last target-stream
    draft on the workspace (here: the seed) is flagged, not silently wrong."""
    w = workload.custom("tiny", B=4, V=1024, r=64, w_dtype=torch.bfloat16, w_std=0.1, seed=2)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    _fused_draft(inp, w, buf, seed=1)
    _full_verify(inp, buf, seed=2)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st != 0 and bits & KERNEL_BADINPUT
    # a fresh workspace (no target-stream draft at all) is flagged too
    buf2 = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf2.draft_tok, buf2.lse_q, buf2.z_tok,
                           buf2.ws, seed=1)
    _full_verify(inp, buf2, seed=1)
    st, bits = vm.dspark_sync_status(buf2.ws.buf)
    assert st != 0 and bits & KERNEL_BADINPUT


def test_unsupported_inputs_are_refused():
    w = workload.custom("tiny", B=4, V=1024, r=32, w_dtype=torch.float32, seed=2)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    with pytest.raises(vm.DsparkError):          # fp32 weights: no tensor-core draft
        _fused_draft(inp, w, buf, seed=1)
    w = workload.custom("tiny", B=4, V=1024, r=64, gamma=1, w_dtype=torch.bfloat16, target_dtype=torch.bfloat16,
                        seed=2)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    with pytest.raises(vm.DsparkError):          # bf16 target with the epilogue form (gamma = 1)
        _fused_draft(inp, w, buf, seed=1)
