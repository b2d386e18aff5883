"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (the whole step through run_step), against the oracle on
the same requests: every request at b1 and b64 (b64 over four seeds), 32
requests spread over every request chunk at b256 and b512; plus a large
sample that bounds the near-tie rate, and properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import workload
from tests._parity import (GAP_EPS, LOGIT_ATOL, PROB_RTOL, RATE_CAP, NearTieLedger, assert_close_where,
                           compare_draft, max_abs_where, score_eps)

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise
    vm = None

DEV = "cuda"


def _sample(B):
    """Every request up to 64; otherwise 32 spread evenly (every request chunk)."""
    if B <= 64:
        return np.arange(B, dtype=np.int32)
    return np.unique(np.linspace(0, B - 1, 32).round().astype(np.int32))


def _emb_rows(emb, anchor, tok):
    """The embedding rows position k reads (x~_{k-1}), remapped to a small table."""
    prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
    ids, inv = np.unique(prev, return_inverse=True)
    inv = inv.reshape(prev.shape).astype(np.int32)
    table = emb[torch.from_numpy(ids).to(emb.device)].cpu()
    return table, inv[:, 0].copy(), np.concatenate([inv[:, 1:], inv[:, :1]], axis=1)


def _step_against_oracle(inp, w, S, seeds, dg, check_conf=True):
    """run_step (full-prefix verification, the benchmark's call) for each seed,
    the sampled requests S against the oracle: draft tokens, lse_q, z_tok,
    confidences and survivals, p(x~), accepted counts, final tokens and the
    emitted segments.  Returns the near-tie ledger over all seeds."""
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    Sd = torch.from_numpy(S).to(DEV).long()
    W1 = inp["W1"].double().cpu().numpy()
    W2 = inp["W2"].double().cpu().numpy()
    U = inp["U"][Sd].double().cpu().numpy()
    T = inp["target"][Sd].double().cpu().numpy()
    anchor = inp["anchor"].cpu().numpy()[S]
    runs = []
    for seed in seeds:
        vm.run_step(inp, buf, mode=0, seed=seed, p_tok=True)
        st, bits = vm.dspark_sync_status(buf.ws.buf)
        assert st == 0, bits
        g = {k: getattr(buf, k).cpu().numpy() for k in ("draft_tok", "lse_q", "z_tok", "conf_cal", "log_surv",
                                                       "p_tok", "accepted", "out_off", "out_tok")}
        d = oracle.draft_markov(U, W1, W2, anchor, seed=seed, req=S)
        runs.append((seed, g, d))
    # the device's own error bound: drawn logits over positions whose prefix matched
    dz = 0.0
    for seed, g, d in runs:
        _, _, valid = compare_draft(g["draft_tok"][S], d["tok"], d["gap"])
        dz = max(dz, max_abs_where(g["z_tok"][S], d["z_tok"], valid))
    ledger = NearTieLedger(score_eps(dz, dg))
    for seed, g, d in runs:
        gtok = g["draft_tok"][S]
        valid = ledger.draft(gtok, d["tok"], d["gap"])
        assert_close_where(g["lse_q"][S], d["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")
        assert_close_where(g["z_tok"][S], d["z_tok"], valid, atol=LOGIT_ATOL, what="z_tok")
        if check_conf:
            # the confidence head on the oracle's own drafts, compared where the drafts agree
            table, a_idx, t_idx = _emb_rows(inp["emb"], anchor, d["tok"])
            c = oracle.confidence_sts(inp["h"][Sd].cpu(), table, a_idx, t_idx, inp["w_c"].cpu(), inp["b_c"],
                                      inp["T"].cpu())
            assert_close_where(g["conf_cal"][S], c["conf_cal"], valid, rtol=PROB_RTOL, what="conf_cal")
            assert_close_where(np.exp(g["log_surv"][S]), np.exp(c["log_surv"]), valid, rtol=PROB_RTOL,
                               what="survival")
        K = np.full(len(S), w.gamma, np.int32)
        v = oracle.verify(T, U, W1, W2, anchor, d["tok"], K, seed=seed, req=S)
        full = np.nonzero(valid.all(axis=1))[0]
        off = g["out_off"]
        acc = g["accepted"][S]
        fin = g["out_tok"][off[S + 1] - 1]
        ledger.verify(acc, fin, v, full)
        walked = ~np.isnan(v["p_tok"]) & valid
        assert_close_where(g["p_tok"][S], v["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")
        # emitted segments of the requests whose walk and final token matched
        o = oracle.compact(d["tok"], v["accepted"], v["final_tok"])
        for i in full:
            if acc[i] == v["accepted"][i] and fin[i] == v["final_tok"][i]:
                seg = g["out_tok"][off[S[i]]:off[S[i] + 1]]
                np.testing.assert_array_equal(seg, o["out_tok"][o["out_off"][i]:o["out_off"][i + 1]])
        # properties over the whole batch
        allacc = g["accepted"]
        assert off[0] == 0 and (np.diff(off) == allacc + 1).all() and ((allacc >= 0) & (allacc <= w.gamma)).all()
        toks = g["out_tok"][:off[-1]]
        assert ((toks >= 0) & (toks < w.V)).all()
        ls = g["log_surv"]
        assert (np.diff(ls, axis=1) <= 0).all() and (ls <= 0).all()
    return ledger


@pytest.mark.parametrize("name", ["b1", "b64", "b256", "b512"])
def test_full_size_step_against_the_oracle(name, device_gumbel_error):
    w = workload.WORKLOADS[name]
    inp = workload.inputs(w, device=DEV)
    seeds = [w.seed + 1000 * i for i in range(4 if name == "b64" else 1)]
    ledger = _step_against_oracle(inp, w, _sample(w.B), seeds, device_gumbel_error)
    print(name, "near-ties", ledger.summary())


def test_near_tie_rate_on_a_large_sample(device_gumbel_error):
    """The near-tie budget: draws flagged at the device's error bound eps stay
    under 0.01% of all draws, on 512 requests x 12 seeds of the b64 logit
    distribution (N(0, 2^2) plus the decaying mode boost) at V = 4096, so
    that the oracle covers ~55k decisions (draft draws, accept walks, final
    draws) in seconds."""
    w = workload.custom("b64", B=512, V=4096, r=64, d=64, seed=77)
    inp = workload.inputs(w, device=DEV)
    ledger = _step_against_oracle(inp, w, np.arange(w.B, dtype=np.int32), list(range(5, 17)),
                                  device_gumbel_error, check_conf=False)
    summ = ledger.summary()
    print("large-sample near-ties", summ)
    assert ledger.draws() > 50000
    assert ledger.rate_eps() < RATE_CAP, summ


def _sched_matches(K, ref, ls, what):
    """K from the device against oracle.schedule's K on the same lists: equal,
    or a near-tie at the cut (adjacent sorted log-survivals within 1e-5, or a
    Theta step within 1e-6 relative: the two sides rank or compare in
    different precisions).  Returns whether K is equal."""
    if np.array_equal(K, ref["K"]):
        return True
    n = ref["n_total"]
    srt = np.sort(np.asarray(ls, np.float64).ravel())[::-1]
    curve = ref["curve"]
    near_rank = any(abs(srt[m] - srt[m + 1]) < 1e-5 for m in range(max(0, n - 2), min(srt.size - 1, n + 1)))
    near_theta = any(abs(curve[m + 1] - curve[m]) <= 1e-6 * abs(curve[m])
                     for m in range(max(0, n - 1), min(curve.size - 1, n + 1)))
    assert near_rank or near_theta, f"{what}: scheduler differs from the oracle without a near-tie"
    return False


def test_b512_async_chain_of_sixteen_steps():
    """Sixteen chained steps at full size: anchors follow next_anchor, the
    capacity comes from survivals two steps old and the ranking from the
    current ones; every step's verify lengths equal oracle.schedule on the
    device's own survival lists."""
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
        ref = oracle.schedule(ls.cpu().numpy(), sps, 2, log_surv_hist=None if old is None else old.cpu().numpy())
        if _sched_matches(K, ref, ls.cpu().numpy(), f"step {t}"):
            assert int(buf.n_total.item()) == ref["n_total"]
        off = buf.out_off.cpu().numpy()
        acc = buf.accepted.cpu().numpy()
        assert (np.diff(off) == acc + 1).all() and (acc <= K).all()
        emitted += int(off[-1])
        anchor = buf.next_anchor.clone()
        hist.append(ls)
    assert emitted >= w.B * w.steps


def test_async_chain_against_the_oracle(device_gumbel_error):
    """The sixteen-step asynchronous chain of the b512 workload (B = 512,
    gamma = 7, its stepped capacity table, seed-chained anchors) at V = 8192
    so that the oracle runs every step whole: each step's drafts, verify
    lengths, accepted counts, emitted tokens and next anchors against
    oracle.step on the same inputs, the same anchors (the device's
    next_anchor of the step before) and the same survival lists two steps
    old."""
    w = workload.custom("b512", V=8192, d=256)
    W = workload.weights(w, device=DEV)
    Wc = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in W.items()}
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    hist = []
    anchor = None
    ledger = NearTieLedger(score_eps(0.0, device_gumbel_error))
    dz = 0.0
    sched_equal = 0
    for t in range(w.steps):
        inp = dict(W)
        inp.update(workload.step_inputs(w, step=t, device=DEV, anchor=anchor))
        old = hist[-2] if len(hist) >= 2 else None
        vm.run_step(inp, buf, mode=2, seed=w.seed, step=t, log_surv_hist=old)
        st, bits = vm.dspark_sync_status(buf.ws.buf)
        assert st == 0, bits
        ci = dict(Wc)
        ci.update({k: inp[k].cpu() for k in ("U", "target", "h", "anchor")})
        ref = oracle.step(ci, mode=2, seed=w.seed, step=t, log_surv_hist=None if old is None else old.cpu().numpy())
        tok = buf.draft_tok.cpu().numpy()
        # the device's error bound so far: drawn logits where the prefix matched
        _, _, pre = compare_draft(tok, ref["draft"]["tok"], ref["draft"]["gap"])
        dz = max(dz, max_abs_where(buf.z_tok.cpu().numpy(), ref["draft"]["z_tok"], pre))
        ledger.eps = score_eps(dz, device_gumbel_error)
        valid = ledger.draft(tok, ref["draft"]["tok"], ref["draft"]["gap"])
        ls = buf.log_surv.cpu().numpy()
        K = buf.K.cpu().numpy()
        same_K = _sched_matches(K, ref["sched"], ls, f"step {t}")
        sched_equal += int(same_K)
        if same_K:
            acc = buf.accepted.cpu().numpy()
            off = buf.out_off.cpu().numpy()
            fin = buf.out_tok.cpu().numpy()[off[1:] - 1]
            rows = np.nonzero(valid.all(axis=1))[0]
            ledger.verify(acc, fin, ref["verify"], rows)
            o = ref["out"]
            nxt = buf.next_anchor.cpu().numpy()
            for i in rows:
                if acc[i] == ref["verify"]["accepted"][i] and fin[i] == ref["verify"]["final_tok"][i]:
                    np.testing.assert_array_equal(buf.out_tok.cpu().numpy()[off[i]:off[i + 1]],
                                                  o["out_tok"][o["out_off"][i]:o["out_off"][i + 1]])
                    assert nxt[i] == o["next_anchor"][i]
        anchor = buf.next_anchor.clone()
        hist.append(buf.log_surv.clone())
    print("async chain: steps with the oracle's verify lengths", sched_equal, "of", w.steps,
          "near-ties", ledger.summary())
    assert sched_equal >= w.steps - 2
