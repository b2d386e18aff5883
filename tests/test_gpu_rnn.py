"""GPU parity of the RNN draft head (dspark_draft_rnn, dspark_verify_rnn)
against the float64 oracle ("DSpark：半自回归生成与置信度调度的投机解码",
section RNN Head：长程依赖).

Tokens must match except flagged near-ties (Gumbel top-2 gap below 1e-3),
after which a request's later positions are not compared: their states
condition on another token.  Log-normalisers and drawn logits agree to 1e-3.
The states agree to STATE_ATOL: the device runs the GRU in binary32 (sums of
2r products, accurate expf/tanhf), the oracle in binary64.  The bias is formed
from the state rounded to bfloat16 on both sides; near a rounding midpoint the
two roundings may differ by one bfloat16 step, which moves a bias entry by at
most |W2| * 2^-8 |s| and stays inside the 1e-3 logit tolerance.
"""
import numpy as np
import pytest
import torch

import oracle
import workload
from tests._parity import GAP_EPS, LOGIT_ATOL, PROB_RTOL, U_EPS, assert_close_where, compare_draft

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None
DEV = "cuda"
STATE_ATOL = 2e-5


def _case(B, V, r, seed):
    w = workload.custom("b64", B=B, V=V, r=r, seed=seed)
    W = workload.weights(w, device=DEV)
    inp = dict(W)
    inp.update(workload.step_inputs(w, device=DEV))
    inp["rnn"] = vm.rnn_prepare(workload.rnn_head(w, device=DEV))
    return w, inp


def _rnn64(inp):
    return {k: v.double().cpu().numpy() for k, v in inp["rnn"].items() if k != "P"}


def _draft(w, inp, seed, req_base=0):
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_draft_rnn(inp["U"], inp["rnn"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                        buf.state, buf.ws, seed=seed, req_base=req_base)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    return buf


@pytest.mark.parametrize("B,V,r", [(16, 8192, 64), (5, 4104, 128), (64, 16384, 256), (130, 2048, 64)])
def test_rnn_draft_parity(B, V, r):
    w, inp = _case(B, V, r, seed=B + r)
    buf = _draft(w, inp, seed=w.seed)
    p = _rnn64(inp)
    ref = oracle.draft_rnn(inp["U"].cpu(), p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"],
                           inp["W2"].double().cpu().numpy(), inp["anchor"].cpu(), seed=w.seed)
    compared, flagged, valid = compare_draft(buf.draft_tok.cpu().numpy(), ref["tok"], ref["gap"])
    assert flagged <= max(1, compared // 1000)
    assert_close_where(buf.lse_q.cpu().numpy(), ref["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")
    assert_close_where(buf.z_tok.cpu().numpy(), ref["z_tok"], valid, atol=LOGIT_ATOL, what="z_tok")
    states = buf.state.cpu().numpy().transpose(1, 0, 2)      # [B, gamma, r]
    assert_close_where(states, ref["states"], np.broadcast_to(valid[..., None], states.shape), atol=STATE_ATOL,
                       what="states")


def test_rnn_draft_request_base_and_steps():
    w, inp = _case(24, 4096, 64, seed=9)
    buf = _draft(w, inp, seed=5, req_base=1000)
    p = _rnn64(inp)
    ref = oracle.draft_rnn(inp["U"].cpu(), p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"],
                           inp["W2"].double().cpu().numpy(), inp["anchor"].cpu(), seed=5,
                           req=np.arange(1000, 1024))
    compare_draft(buf.draft_tok.cpu().numpy(), ref["tok"], ref["gap"])


@pytest.mark.parametrize("B,V,r,tdt", [(16, 8192, 64, torch.float32), (33, 2056, 128, torch.bfloat16),
                                       (64, 4096, 256, torch.float32)])
def test_rnn_verify_parity(B, V, r, tdt):
    """Verification of the device's RNN drafts: the oracle rebuilds q along the
    same tokens from its own float64 states."""
    w, inp = _case(B, V, r, seed=3 * B + r)
    if tdt == torch.bfloat16:
        inp["target"] = inp["target"].to(torch.bfloat16).contiguous()
    seed = B + 7
    buf = _draft(w, inp, seed=seed)
    K = np.random.default_rng(seed).integers(0, w.gamma + 1, w.B).astype(np.int32)
    Kd = torch.tensor(K, device=DEV)
    vm.dspark_verify_rnn(inp["target"], inp["U"], buf.state, inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                         buf.z_tok, Kd, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                         buf.next_anchor, buf.ws, seed=seed, p_tok=buf.p_tok, near_ties=buf.near_ties)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    p = _rnn64(inp)
    tok = buf.draft_tok.cpu().numpy()
    _, arows = oracle.rnn_states(p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"],
                                 inp["anchor"].cpu(), tok)
    ref = oracle.verify(inp["target"].cpu(), inp["U"].cpu(), None, inp["W2"].double().cpu().numpy(),
                        inp["anchor"].cpu(), tok, K, seed=seed, arows=arows)
    acc = buf.accepted.cpu().numpy()
    diag = ref["diag"]
    bad = acc != ref["accepted"]
    for b in np.nonzero(bad)[0]:
        assert diag[b, 0] < U_EPS, f"unflagged accept mismatch at request {b}"
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[1:] - 1]
    for b in range(w.B):
        if not bad[b] and fin[b] != ref["final_tok"][b]:
            assert diag[b, 1] < GAP_EPS, f"unflagged final-token mismatch at request {b}"
    walked = ~np.isnan(ref["p_tok"])
    assert_close_where(buf.p_tok.cpu().numpy(), ref["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")
    assert off[0] == 0 and (np.diff(off) == acc + 1).all()


def test_rnn_whole_step_matches_oracle_chain():
    w, inp = _case(12, 4096, 64, seed=21)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=0, seed=w.seed, head="rnn", p_tok=True)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    p = _rnn64(inp)
    W2 = inp["W2"].double().cpu().numpy()
    d = oracle.draft_rnn(inp["U"].cpu(), p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"], W2,
                         inp["anchor"].cpu(), seed=w.seed)
    compared, flagged, valid = compare_draft(buf.draft_tok.cpu().numpy(), d["tok"], d["gap"])
    full = valid.all(axis=1)
    K = np.full(w.B, w.gamma, np.int32)
    v = oracle.verify(inp["target"].cpu(), inp["U"].cpu(), None, W2, inp["anchor"].cpu(), d["tok"], K,
                      seed=w.seed, arows=d["arows"])
    acc = buf.accepted.cpu().numpy()
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[1:] - 1]
    for b in np.nonzero(full)[0]:
        if acc[b] != v["accepted"][b]:
            assert v["diag"][b, 0] < U_EPS
        elif fin[b] != v["final_tok"][b]:
            assert v["diag"][b, 1] < GAP_EPS
    assert full.sum() >= w.B - 1


def test_rnn_full_size_b64_sampled_requests():
    """The b64 workload (B=64, V=151936, r=256) drafted with the RNN head and
    verified over the full prefix, in the launch configuration run_step uses;
    sampled requests recomputed by the oracle."""
    w = workload.WORKLOADS["b64"]
    inp = workload.inputs(w, device=DEV)
    inp["rnn"] = vm.rnn_prepare(workload.rnn_head(w, device=DEV))
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=0, seed=w.seed, head="rnn", p_tok=True)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    S = np.array([0, 21, 42, 63], dtype=np.int32)
    Sd = torch.from_numpy(S).to(DEV).long()
    p = _rnn64(inp)
    W2 = inp["W2"].double().cpu().numpy()
    U = inp["U"][Sd].cpu()
    T = inp["target"][Sd].cpu()
    anchor = inp["anchor"].cpu().numpy()[S]
    d = oracle.draft_rnn(U, p["E"], p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], p["s0"], W2, anchor,
                         seed=w.seed, req=S)
    compared, flagged, valid = compare_draft(buf.draft_tok.cpu().numpy()[S], d["tok"], d["gap"])
    assert_close_where(buf.lse_q.cpu().numpy()[S], d["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")
    states = buf.state.cpu().numpy().transpose(1, 0, 2)[S]
    assert_close_where(states, d["states"], np.broadcast_to(valid[..., None], states.shape), atol=STATE_ATOL,
                       what="states")
    K = np.full(len(S), w.gamma, np.int32)
    v = oracle.verify(T, U, None, W2, anchor, d["tok"], K, seed=w.seed, req=S, arows=d["arows"])
    acc = buf.accepted.cpu().numpy()[S]
    for i in np.nonzero(valid.all(axis=1))[0]:
        if acc[i] != v["accepted"][i]:
            assert v["diag"][i, 0] < U_EPS
    allacc = buf.accepted.cpu().numpy()
    off = buf.out_off.cpu().numpy()
    assert (np.diff(off) == allacc + 1).all() and ((allacc >= 0) & (allacc <= w.gamma)).all()


def test_rnn_input_table():
    """P = E W_ih^T + b_ih for every token, against float64 numpy on the same
    bf16 values (fp32 accumulation over r products)."""
    for V, r in ((1000, 64), (4099, 256), (77, 128)):
        w = workload.custom("b64", B=4, V=V - V % 8 if V % 8 else V, r=r, seed=V)
        rnn = workload.rnn_head(w, device=DEV)
        P = vm.dspark_rnn_input_table(rnn["E"], rnn["W_ih"], rnn["b_ih"])
        torch.cuda.synchronize()
        ref = rnn["E"].double().cpu().numpy() @ rnn["W_ih"].double().cpu().numpy().T + rnn["b_ih"].double().cpu().numpy()
        np.testing.assert_allclose(P.cpu().numpy(), ref, rtol=0, atol=2e-5)


def test_rnn_rejects_unsupported_shapes():
    w, inp = _case(4, 1024, 64, seed=1)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    with pytest.raises(vm.DsparkError):
        vm.dspark_draft_rnn(inp["U"].to(torch.bfloat16).contiguous(), inp["rnn"], inp["W2"], inp["anchor"],
                            buf.draft_tok, buf.lse_q, buf.z_tok, buf.state, buf.ws)
