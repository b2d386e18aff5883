"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (the whole step through run_step), on sampled requests the
oracle recomputes one by one, plus properties that hold at any size."""
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


def _sample(B):
    s = sorted({0, B // 3, B // 2, B - 1})
    return np.array(s, dtype=np.int32)


def _emb_rows(emb, anchor, tok):
    """The embedding rows position k reads (x~_{k-1}), remapped to a small table."""
    prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
    ids, inv = np.unique(prev, return_inverse=True)
    inv = inv.reshape(prev.shape).astype(np.int32)
    table = emb[torch.from_numpy(ids).to(emb.device)].cpu()
    return table, inv[:, 0].copy(), np.concatenate([inv[:, 1:], inv[:, :1]], axis=1)


@pytest.mark.parametrize("name", ["b1", "b64", "b256", "b512"])
def test_full_size_step_on_sampled_requests(name):
    w = workload.WORKLOADS[name]
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=0, seed=w.seed, p_tok=True)          # full-prefix verification
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    S = _sample(w.B)
    W1 = inp["W1"].double().cpu().numpy()
    W2 = inp["W2"].double().cpu().numpy()
    U = inp["U"][torch.from_numpy(S).to(DEV).long()].cpu()
    T = inp["target"][torch.from_numpy(S).to(DEV).long()].cpu()
    anchor = inp["anchor"].cpu().numpy()[S]
    d = oracle.draft_markov(U, W1, W2, anchor, seed=w.seed, req=S)
    gtok = buf.draft_tok.cpu().numpy()[S]
    compared, flagged, valid = compare_draft(gtok, d["tok"], d["gap"])
    assert_close_where(buf.lse_q.cpu().numpy()[S], d["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")
    assert_close_where(buf.z_tok.cpu().numpy()[S], d["z_tok"], valid, atol=LOGIT_ATOL, what="z_tok")

    # confidence on the oracle's own drafts; compared where the drafts agree
    table, a_idx, t_idx = _emb_rows(inp["emb"], anchor, d["tok"])
    c = oracle.confidence_sts(inp["h"][torch.from_numpy(S).to(DEV).long()].cpu(), table, a_idx, t_idx,
                              inp["w_c"].cpu(), inp["b_c"], inp["T"].cpu())
    assert_close_where(buf.conf_cal.cpu().numpy()[S], c["conf_cal"], valid, rtol=PROB_RTOL, what="conf_cal")
    assert_close_where(np.exp(buf.log_surv.cpu().numpy()[S]), np.exp(c["log_surv"]), valid, rtol=PROB_RTOL,
                       what="survival")

    # verification of the requests whose whole draft matched
    K = np.full(len(S), w.gamma, np.int32)
    v = oracle.verify(T, U, W1, W2, anchor, d["tok"], K, seed=w.seed, req=S)
    full = valid.all(axis=1)
    acc = buf.accepted.cpu().numpy()[S]
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[S + 1] - 1]
    for i in np.nonzero(full)[0]:
        if acc[i] != v["accepted"][i]:
            assert v["diag"][i, 0] < U_EPS, f"{name}: unflagged accept mismatch at request {S[i]}"
            continue
        if fin[i] != v["final_tok"][i]:
            assert v["diag"][i, 1] < GAP_EPS, f"{name}: unflagged final-token mismatch at request {S[i]}"
    walked = ~np.isnan(v["p_tok"]) & valid
    assert_close_where(buf.p_tok.cpu().numpy()[S], v["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")

    # properties over the whole batch
    allacc = buf.accepted.cpu().numpy()
    assert off[0] == 0 and (np.diff(off) == allacc + 1).all() and ((allacc >= 0) & (allacc <= w.gamma)).all()
    toks = buf.out_tok.cpu().numpy()[:off[-1]]
    assert ((toks >= 0) & (toks < w.V)).all()
    ls = buf.log_surv.cpu().numpy()
    assert (np.diff(ls, axis=1) <= 0).all() and (ls <= 0).all()


def _theta_curve(log_surv, sps, B):
    a = np.exp(log_surv.astype(np.float64)).ravel()
    order = np.lexsort((np.arange(a.size), -log_surv.astype(np.float64).ravel()))
    cum = np.concatenate([[0.0], np.cumsum(a[order])])
    return (B + cum) * sps[B - 1 + np.arange(a.size + 1)], order


def test_b512_async_chain_of_sixteen_steps():
    """Sixteen chained steps: anchors follow next_anchor, the capacity comes
    from survivals two steps old and the ranking from the current ones."""
    w = workload.WORKLOADS["b512"]
    W = workload.weights(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    sps = W["sps"].double().cpu().numpy()
    hist = []
    anchor = None
    emitted = 0
    for t in range(w.steps):
        inp = dict(W)
        inp.update(workload.step_inputs(w, step=t, device=DEV, anchor=anchor))
        old = hist[-2] if len(hist) >= 2 else None
        vm.run_step(inp, buf, mode=2, seed=w.seed, step=t, log_surv_hist=old)
        st, bits = vm.dspark_sync_status(buf.ws.buf)
        assert st == 0, bits
        ls = buf.log_surv.clone()
        K = buf.K.cpu().numpy()
        n = int(buf.n_total.item())
        assert K.sum() == n and ((K >= 0) & (K <= w.gamma)).all()
        # capacity: first argmax of Theta over the list two steps old (current list at t < 2)
        ref_ls = (old if old is not None else ls).cpu().numpy()
        curve, _ = _theta_curve(ref_ls, sps, w.B)
        best = int(np.argmax(curve))
        if best != n:
            assert abs(curve[best] - curve[n]) <= 1e-6 * abs(curve[best])
        # admitted set = the n best current candidates (ties by request, position)
        cur = ls.cpu().numpy()
        _, order = _theta_curve(cur, sps, w.B)
        expect = np.bincount(order[:n] // w.gamma, minlength=w.B)
        if not np.array_equal(expect, K):
            srt = np.sort(cur.ravel())[::-1]
            assert abs(srt[n - 1] - srt[n]) < 1e-5           # a near-tie at the cut
        off = buf.out_off.cpu().numpy()
        acc = buf.accepted.cpu().numpy()
        assert (np.diff(off) == acc + 1).all() and (acc <= K).all()
        emitted += int(off[-1])
        anchor = buf.next_anchor.clone()
        hist.append(ls)
    assert emitted >= w.B * w.steps
