"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs (tiny and ragged shapes the oracle finishes in
seconds), plus the lossless chi-square on the GPU itself."""
import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
import workload
from tests._parity import (GAP_EPS, LOGIT_ATOL, PROB_RTOL, U_EPS, NearTieLedger, assert_close_where,
                           compare_draft, max_abs_where, score_eps)

pytestmark = pytest.mark.gpu

try:
    import verify_markov_head_gb300 as vm
except ImportError:
    if torch.cuda.is_available():
        raise                      # on a GPU the library must load: no silent skip
    vm = None
DEV = "cuda"


def _cpu(inp):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _draft_gpu(inp, B, gamma, V, r, seed, step=0, logits=False, req_base=0, tau=1.0):
    ws = vm.Workspace(B, gamma, V, r)
    tok = torch.empty((B, gamma), dtype=torch.int32, device=DEV)
    lse = torch.empty((B, gamma), device=DEV)
    zt = torch.empty((B, gamma), device=DEV)
    lo = torch.empty((B, gamma, V), device=DEV) if logits else None
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, zt, ws,
                           seed=seed, step=step, logits_out=lo, req_base=req_base, tau=tau)
    st, bits = vm.dspark_sync_status(ws.buf)
    assert st == 0, bits
    return tok.cpu().numpy(), lse.cpu().numpy(), zt.cpu().numpy(), (lo.cpu().numpy() if logits else None)


def _check_draft(inp, w, seed, step=0, tau=1.0, dg=3e-6):
    """The draft against the oracle: tokens bit-exact except near-ties, the
    log-normalisers, drawn logits and the whole logits dump within 1e-3.
    Every token mismatch must be a near-tie at the device's own error bound
    eps (from the measured logit error and the device Gumbel error dg).
    Returns the ledger."""
    tok, lse, zt, lo = _draft_gpu(inp, w.B, w.gamma, w.V, w.r, seed, step, logits=True, tau=tau)
    ci = _cpu(inp)
    ref = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=seed, step=step,
                              want_logits=True, tau=tau)
    compared, flagged, valid = compare_draft(tok, ref["tok"], ref["gap"])
    vmask = np.broadcast_to(valid[..., None], lo.shape)
    assert_close_where(lse, ref["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")
    assert_close_where(zt, ref["z_tok"], valid, atol=LOGIT_ATOL, what="z_tok")
    assert_close_where(lo, ref["logits"], vmask, atol=LOGIT_ATOL, what="draft logits")
    ledger = NearTieLedger(score_eps(max_abs_where(lo, ref["logits"], vmask), dg))
    ledger.draft(tok, ref["tok"], ref["gap"])
    return ledger


# ----------------------------------------------------------------- whole step

def test_tiny_workload_end_to_end():
    w = workload.WORKLOADS["tiny"]
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=w.mode, seed=w.seed, p_tok=True)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    ref = oracle.step(_cpu(inp), mode=w.mode, seed=w.seed)
    np.testing.assert_array_equal(buf.draft_tok.cpu().numpy(), ref["draft"]["tok"])
    np.testing.assert_allclose(buf.lse_q.cpu().numpy(), ref["draft"]["lse_q"], atol=LOGIT_ATOL, rtol=0)
    np.testing.assert_allclose(buf.z_tok.cpu().numpy(), ref["draft"]["z_tok"], atol=LOGIT_ATOL, rtol=0)
    np.testing.assert_allclose(buf.conf_cal.cpu().numpy(), ref["conf"]["conf_cal"], rtol=PROB_RTOL)
    np.testing.assert_allclose(np.exp(buf.log_surv.cpu().numpy()), np.exp(ref["conf"]["log_surv"]),
                               rtol=PROB_RTOL)
    np.testing.assert_array_equal(buf.K.cpu().numpy(), ref["sched"]["K"])
    assert int(buf.n_total.item()) == ref["sched"]["n_total"]
    np.testing.assert_allclose(buf.theta.item(), ref["sched"]["theta"], rtol=1e-6)
    np.testing.assert_array_equal(buf.accepted.cpu().numpy(), ref["verify"]["accepted"])
    n = int(buf.out_off[-1].item())
    np.testing.assert_array_equal(buf.out_off.cpu().numpy(), ref["out"]["out_off"])
    np.testing.assert_array_equal(buf.out_tok[:n].cpu().numpy(), ref["out"]["out_tok"])
    np.testing.assert_array_equal(buf.out_req[:n].cpu().numpy(), ref["out"]["out_req"])
    np.testing.assert_array_equal(buf.out_pos[:n].cpu().numpy(), ref["out"]["out_pos"])
    np.testing.assert_array_equal(buf.next_anchor.cpu().numpy(), ref["out"]["next_anchor"])
    walked = ~np.isnan(ref["verify"]["p_tok"])
    assert_close_where(buf.p_tok.cpu().numpy(), ref["verify"]["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_tiny_workload_all_scheduler_modes(mode):
    w = workload.custom("tiny", B=6, seed=21)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.run_step(inp, buf, mode=mode, seed=5, step=3)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    ref = oracle.step(_cpu(inp), mode=mode, seed=5, step=3)
    np.testing.assert_array_equal(buf.draft_tok.cpu().numpy(), ref["draft"]["tok"])
    np.testing.assert_array_equal(buf.K.cpu().numpy(), ref["sched"]["K"])
    n = int(buf.out_off[-1].item())
    np.testing.assert_array_equal(buf.out_tok[:n].cpu().numpy(), ref["out"]["out_tok"])


# ----------------------------------------------------------------- draft

@pytest.mark.parametrize("B,V,r,wdt", [
    (1, 1024, 32, torch.float32),
    (5, 4104, 64, torch.float32),        # ragged last tile (4104 = 32*128 + 8)
    (1, 2048, 256, torch.bfloat16),
    (1, 4104, 64, torch.bfloat16),       # one request, ragged vocabulary tail
    (3, 4104, 256, torch.bfloat16),
    (17, 1032, 128, torch.bfloat16),     # ragged request chunk
    (64, 4096, 256, torch.bfloat16),
    (130, 1024, 64, torch.bfloat16),
    (32, 2056, 128, torch.bfloat16),     # 4 vocabulary tiles per accumulator, ragged tail
    (40, 1032, 256, torch.bfloat16),     # 2 tiles per accumulator, partly filled rows
])
def test_draft_parity(B, V, r, wdt, device_gumbel_error):
    w = workload.custom("tiny", B=B, V=V, r=r, w_dtype=wdt, w_std=0.1, seed=B + V + r)
    inp = workload.inputs(w, device=DEV)
    ledger = _check_draft(inp, w, seed=11, step=2, dg=device_gumbel_error)
    print("near-ties", ledger.summary())


def test_draft_temperature_and_request_base():
    w = workload.custom("tiny", B=3, V=1024, r=64, w_dtype=torch.bfloat16, seed=4)
    inp = workload.inputs(w, device=DEV)
    _check_draft(inp, w, seed=9, tau=0.8)
    tok, *_ = _draft_gpu(inp, w.B, w.gamma, w.V, w.r, seed=9, req_base=7)
    ci = _cpu(inp)
    ref = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=9, req=[7, 8, 9])
    compare_draft(tok, ref["tok"], ref["gap"])


def test_draft_one_request_temperature_and_request_base():
    """B = 1 takes the one-request epilogue (every lane races one column)."""
    w = workload.custom("tiny", B=1, V=2056, r=128, w_dtype=torch.bfloat16, seed=12)
    inp = workload.inputs(w, device=DEV)
    _check_draft(inp, w, seed=21, tau=0.7)
    tok, lse, zt, _ = _draft_gpu(inp, w.B, w.gamma, w.V, w.r, seed=21, req_base=40)
    ci = _cpu(inp)
    ref = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=21, req=[40])
    compared, flagged, valid = compare_draft(tok, ref["tok"], ref["gap"])
    assert_close_where(lse, ref["lse_q"], valid, atol=LOGIT_ATOL, what="lse_q")


def test_draft_gamma_one_and_sixteen():
    for g in (1, 16):
        w = workload.custom("tiny", B=2, V=1024, r=32, gamma=g, seed=g)
        inp = workload.inputs(w, device=DEV)
        _check_draft(inp, w, seed=3)


# ----------------------------------------------------------------- confidence

@pytest.mark.parametrize("jumps", [(16,), (8, 24)])
def test_draft_reference_moves_after_a_winner(jumps, device_gumbel_error):
    """Logits that rise by 60 nats (87 in base 2) at the given columns of every
    32-column block, so that the race's log-sum-exp reference (the first quad's
    maximum) moves up after the thread has a winner: the winner key and the
    screen threshold must grow with it, and the draw then comes from the high
    columns, as the oracle's does."""
    w = workload.custom("tiny", B=8, V=4096, r=64, w_dtype=torch.bfloat16, seed=21)
    inp = workload.inputs(w, device=DEV)
    v = torch.arange(w.V, device=DEV)
    bump = torch.zeros(w.V, device=DEV)
    for j in jumps:
        bump += 60.0 * ((v % 32) >= j).float()
    inp["U"] = inp["U"] + bump
    for seed in (3, 4):
        ledger = _check_draft(inp, w, seed=seed, dg=device_gumbel_error)
        assert ledger.c["draft_draws"] >= w.B


def test_confidence_parity_fp32_and_bf16_embeddings():
    for edt, d in ((torch.float32, 64), (torch.float32, 4096), (torch.bfloat16, 256), (torch.float32, 30)):
        w = workload.custom("tiny", B=9, d=d, seed=d)
        inp = workload.inputs(w, device=DEV)
        emb = inp["emb"].to(edt)
        tok = torch.randint(0, w.V, (w.B, w.gamma), device=DEV, dtype=torch.int32)
        cal = torch.empty((w.B, w.gamma), device=DEV)
        ls = torch.empty((w.B, w.gamma), device=DEV)
        ws = vm.Workspace(w.B, w.gamma, w.V, w.r)
        vm.dspark_confidence_sts(inp["h"], emb, inp["anchor"], tok, inp["w_c"], inp["b_c"], inp["T"], cal, ls, ws)
        assert vm.dspark_sync_status(ws.buf)[0] == 0
        ref = oracle.confidence_sts(inp["h"].cpu(), emb.float().cpu(), inp["anchor"].cpu(), tok.cpu(),
                                    inp["w_c"].cpu(), inp["b_c"], inp["T"].cpu())
        np.testing.assert_allclose(cal.cpu().numpy(), ref["conf_cal"], rtol=PROB_RTOL)
        np.testing.assert_allclose(np.exp(ls.cpu().numpy()), np.exp(ref["log_surv"]), rtol=PROB_RTOL)
        assert (np.diff(ls.cpu().numpy(), axis=1) <= 0).all()


# ----------------------------------------------------------------- scheduler

def _synthetic_survival(B, gamma, seed, mean=1.0, std=2.0):
    g = np.random.default_rng(seed)
    c = 1 / (1 + np.exp(-g.normal(mean, std, (B, gamma))))
    return np.cumsum(np.log(c), axis=1).astype(np.float32)


def _sched_gpu(ls, sps, mode, hist=None):
    B, gamma = ls.shape
    ws = vm.Workspace(B, gamma, 8, 1)
    K = torch.empty(B, dtype=torch.int32, device=DEV)
    nt = torch.empty(1, dtype=torch.int32, device=DEV)
    th = torch.empty(1, device=DEV)
    h = None if hist is None else torch.tensor(hist, device=DEV)
    vm.dspark_schedule(torch.tensor(ls, device=DEV), torch.as_tensor(sps, device=DEV).float(), mode, K, nt, th,
                       ws, log_surv_hist=h)
    torch.cuda.synchronize()
    return K.cpu().numpy(), int(nt.item()), float(th.item())


@pytest.mark.parametrize("name", ["tiny", "b64", "b256", "b512"])
@pytest.mark.parametrize("mode", [1, 2])
def test_schedule_parity(name, mode):
    w = workload.WORKLOADS[name]
    sps = w.sps_table()
    for trial in range(4):
        # survivals both as the workloads produce them and raised so admissions happen
        ls = _synthetic_survival(w.B, w.gamma, seed=trial, mean=1.0 + 3 * (trial % 2))
        hist = _synthetic_survival(w.B, w.gamma, seed=100 + trial) if mode == 2 and trial >= 2 else None
        K, nt, th = _sched_gpu(ls, sps.numpy(), mode, hist)
        ref = oracle.schedule(ls, sps.numpy(), mode, log_surv_hist=hist)
        curve = ref["curve"]
        if not np.array_equal(K, ref["K"]):
            # only a Theta near-tie at the cut may differ
            n = ref["n_total"]
            near = [abs(curve[m + 1] - curve[m]) <= 1e-6 * abs(curve[m]) for m in range(max(0, n - 1), min(len(curve) - 1, n + 1))]
            assert any(near), (name, mode, trial)
        else:
            assert nt == ref["n_total"]
            assert th == pytest.approx(ref["theta"], rel=1e-6)


def test_schedule_ties_and_flat_survival():
    ls = np.zeros((5, 3), np.float32)
    sps = np.ones(5 + 15, np.float32)
    K, nt, _ = _sched_gpu(ls, sps, 1)
    assert K.tolist() == [3] * 5 and nt == 15
    ls = np.full((4, 7), -0.0, np.float32)
    sps = np.array([1000 / (10 + 0.5 * n) for n in range(1, 33)], np.float32)
    K, nt, _ = _sched_gpu(ls, sps, 1)
    ref = oracle.schedule(ls, sps, 1)
    np.testing.assert_array_equal(K, ref["K"])


def test_schedule_off_and_limits():
    ls = _synthetic_survival(512, 8, seed=1)
    sps = np.ones(512 + 4096, np.float32)
    K, nt, _ = _sched_gpu(ls, sps, 0)
    assert (K == 8).all() and nt == 4096
    K, nt, _ = _sched_gpu(ls, sps, 1)
    ref = oracle.schedule(ls, sps, 1)
    np.testing.assert_array_equal(K, ref["K"])


# ----------------------------------------------------------------- verify

def _verify_case(w, seed, K=None, req_base=0):
    inp = workload.inputs(w, device=DEV)
    ci = _cpu(inp)
    d = oracle.draft_markov(ci["U"], ci["W1"], ci["W2"], ci["anchor"], seed=seed)
    tok = torch.tensor(d["tok"], device=DEV)
    lse = torch.tensor(d["lse_q"], dtype=torch.float32, device=DEV)
    zt = torch.tensor(d["z_tok"], dtype=torch.float32, device=DEV)
    if K is None:
        K = np.random.default_rng(seed).integers(0, w.gamma + 1, w.B).astype(np.int32)
    Kd = torch.tensor(K, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], tok, lse, zt, Kd,
                     buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off, buf.next_anchor, buf.ws,
                     seed=seed, p_tok=buf.p_tok, near_ties=buf.near_ties, req_base=req_base)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    req = np.arange(req_base, req_base + w.B)
    ref = oracle.verify(ci["target"], ci["U"], ci["W1"], ci["W2"], ci["anchor"], d["tok"], K, seed=seed, req=req)
    return buf, ref, d, K


@pytest.mark.parametrize("B,V,r,wdt,tdt", [
    (4, 1024, 32, torch.float32, torch.float32),
    (7, 4104, 64, torch.bfloat16, torch.float32),
    (33, 2056, 128, torch.bfloat16, torch.bfloat16),
    (64, 1024, 256, torch.bfloat16, torch.float32),
    (32, 1032, 128, torch.bfloat16, torch.bfloat16),
    (130, 2048, 64, torch.bfloat16, torch.float32),
])
def test_verify_parity(B, V, r, wdt, tdt):
    w = workload.custom("tiny", B=B, V=V, r=r, w_dtype=wdt, target_dtype=tdt, w_std=0.1, seed=B * 3 + r)
    buf, ref, d, K = _verify_case(w, seed=B + 1)
    acc = buf.accepted.cpu().numpy()
    diag = ref["diag"]
    bad = acc != ref["accepted"]
    for b in np.nonzero(bad)[0]:
        assert diag[b, 0] < U_EPS, f"unflagged accept mismatch at request {b}"
    off = buf.out_off.cpu().numpy()
    tok = buf.out_tok.cpu().numpy()
    fin = tok[off[1:] - 1]
    for b in range(w.B):
        if bad[b]:
            continue
        if fin[b] != ref["final_tok"][b]:
            assert diag[b, 1] < GAP_EPS, f"unflagged final-token mismatch at request {b}"
    walked = ~np.isnan(ref["p_tok"])
    assert_close_where(buf.p_tok.cpu().numpy(), ref["p_tok"], walked, rtol=PROB_RTOL, what="p_tok")
    # layout invariants
    assert off[0] == 0 and (np.diff(off) == acc + 1).all()
    np.testing.assert_array_equal(buf.next_anchor.cpu().numpy(), fin)


def test_verify_zero_and_full_lengths():
    w = workload.custom("tiny", B=8, seed=77)
    for K in (np.zeros(8, np.int32), np.full(8, 7, np.int32)):
        buf, ref, d, _ = _verify_case(w, seed=4, K=K, req_base=3)
        np.testing.assert_array_equal(buf.accepted.cpu().numpy(), ref["accepted"])
        off = buf.out_off.cpu().numpy()
        np.testing.assert_array_equal(buf.out_tok.cpu().numpy()[off[1:] - 1], ref["final_tok"])


def test_lossless_chi_square_on_gpu():
    """Emitted tokens follow the target law (V=16, 2^16 independent requests)."""
    n, gamma, V, r = 65536, 3, 16, 8
    g = np.random.default_rng(0)
    urows = g.normal(0, 1.5, (gamma, V)).astype(np.float32)
    trows = (np.concatenate([urows, g.normal(0, 1.5, (1, V))]) + g.normal(0, 0.8, (gamma + 1, V))).astype(np.float32)
    U = torch.tensor(urows, device=DEV).expand(n, gamma, V).contiguous()
    T = torch.tensor(trows, device=DEV).expand(n, gamma + 1, V).contiguous()
    W1 = torch.randn((V, r), device=DEV)
    W2 = torch.zeros((r, V), device=DEV)
    anchor = torch.zeros(n, dtype=torch.int32, device=DEV)
    inp = dict(U=U, target=T, W1=W1, W2=W2, anchor=anchor)
    buf = vm.StepBuffers(n, gamma, V, r)
    vm.dspark_draft_markov(U, W1, W2, anchor, buf.draft_tok, buf.lse_q, buf.z_tok, buf.ws, seed=31)
    K = torch.full((n,), gamma, dtype=torch.int32, device=DEV)
    vm.dspark_verify(T, U, W1, W2, anchor, buf.draft_tok, buf.lse_q, buf.z_tok, K, buf.accepted, buf.out_tok,
                     buf.out_req, buf.out_pos, buf.out_off, buf.next_anchor, buf.ws, seed=31)
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0
    off = buf.out_off.cpu().numpy()
    tok = buf.out_tok.cpu().numpy()
    p = special.softmax(trows.astype(np.float64), axis=-1)
    length = np.diff(off)
    for pos in range(gamma + 1):
        has = length > pos
        y = tok[off[:-1][has] + pos]
        if y.size < 2000:
            continue
        counts = np.bincount(y, minlength=V)
        assert stats.chisquare(counts, p[pos] * y.size).pvalue > 1e-4, pos


def test_cuda_graph_replay_matches_eager():
    w = workload.custom("tiny", B=8, V=2048, r=64, w_dtype=torch.bfloat16, seed=12)
    inp = workload.inputs(w, device=DEV)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        vm.run_step(inp, buf, mode=1, seed=2, stream=s)
    s.synchronize()
    eager = buf.out_tok.clone(), buf.out_off.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        vm.run_step(inp, buf, mode=1, seed=2, stream=s)
    for _ in range(3):
        buf.out_tok.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager[1], buf.out_off)
    n = int(eager[1][-1])
    assert torch.equal(eager[0][:n], buf.out_tok[:n])


def test_device_range_checks_raise_status_not_faults():
    w = workload.custom("tiny", B=2, seed=1)
    inp = workload.inputs(w, device=DEV)
    inp["anchor"] = torch.tensor([5, w.V + 10], dtype=torch.int32, device=DEV)   # out of range
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                           buf.ws, seed=0)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == -5 and bits & 1
    assert vm.dspark_sync_status(buf.ws.buf)[0] == 0          # reading clears it
    K = torch.tensor([3, 99], dtype=torch.int32, device=DEV)    # verify length beyond gamma
    vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                     buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                     buf.next_anchor, buf.ws, seed=0)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == -5 and bits & 2
    torch.cuda.synchronize()


def test_host_pointers_are_rejected():
    w = workload.custom("tiny", B=2, seed=1)
    inp = workload.inputs(w, device="cpu")
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    with pytest.raises(vm.DsparkError):
        vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                               buf.z_tok, buf.ws, seed=0)


def test_draft_single_position_launch_tensor_cores():
    """gamma = 1 takes the single-position launch of the tensor-core draft (the
    launch every position uses where cooperative launch is unavailable): the
    last CTA of each request chunk merges the partial states."""
    for B in (1, 70):
        w = workload.custom("tiny", B=B, V=2056, r=256, gamma=1, w_dtype=torch.bfloat16, w_std=0.1, seed=5 + B)
        inp = workload.inputs(w, device=DEV)
        ledger = _check_draft(inp, w, seed=7, step=1)
        assert ledger.c["draft_draws"] == B


def test_device_random_stream_matches_definition():
    """Uniforms bit-exact, Gumbel variates within 3e-6 of the binary64 value,
    over 2^20 columns of several streams."""
    import oracle as ora
    n = 1 << 20
    g = torch.empty(n, device=DEV)
    u = torch.empty(n, device=DEV)
    for seed, step, dom, row in ((0, 0, 0, 0), (2**40 + 7, 3, 2, 1234), (99, 2**33 + 5, 3, 77)):
        vm.dspark_gumbel_stream(seed, step, dom, row, n, g, u)
        torch.cuda.synchronize()
        gu = u.cpu().double().numpy()
        gg = g.cpu().double().numpy()
        idx = np.random.default_rng(seed % 1000).choice(n, 4000, replace=False)
        ref_u = np.array([ora.uniform(seed, step, dom, row, int(c)) for c in idx])
        np.testing.assert_array_equal(gu[idx], ref_u)
        # exact Gumbel of the exact uniforms, everywhere
        exact = -np.log(-np.log(gu))
        err = np.abs(gg - exact)
        assert err.max() < 3e-6, err.max()
        # the extreme tail (1 - u < 2^-10), where the winners come from
        tail = gu > 1 - 2.0 ** -10
        assert tail.sum() > 100 and err[tail].max() < 3e-6


@pytest.mark.parametrize("B,V,r,wdt", [(1, 151936, 256, torch.bfloat16), (3, 4104, 64, torch.bfloat16),
                                       (5, 2048, 32, torch.float32)])
def test_verify_from_stored_draft_logits(B, V, r, wdt):
    """dspark_verify_logits: the residual draw reads the rejected row from the
    draft's own stored logits; checked against the oracle on the device's drafts."""
    w = workload.custom("tiny", B=B, V=V, r=r, w_dtype=wdt, w_std=0.1, seed=B * 7 + r)
    inp = workload.inputs(w, device=DEV)
    seed = B + 3
    ws = vm.Workspace(w.B, w.gamma, w.V, w.r)
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    logits = torch.empty((w.B, w.gamma, w.V), device=DEV)
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok, ws,
                           seed=seed, logits_out=logits)
    K = np.random.default_rng(seed).integers(0, w.gamma + 1, w.B).astype(np.int32)
    K[0] = w.gamma
    vm.dspark_verify_logits(inp["target"], inp["U"], inp["W1"], inp["W2"], logits, inp["anchor"], buf.draft_tok,
                            buf.lse_q, buf.z_tok, torch.tensor(K, device=DEV), buf.accepted, buf.out_tok,
                            buf.out_req, buf.out_pos, buf.out_off, buf.next_anchor, ws, seed=seed, p_tok=buf.p_tok,
                            near_ties=buf.near_ties)
    st, bits = vm.dspark_sync_status(ws.buf)
    assert st == 0, bits
    ci = _cpu(inp)
    tok = buf.draft_tok.cpu().numpy()
    ref = oracle.verify(ci["target"], ci["U"], ci["W1"], ci["W2"], ci["anchor"], tok, K, seed=seed)
    acc = buf.accepted.cpu().numpy()
    bad = acc != ref["accepted"]
    for b in np.nonzero(bad)[0]:
        assert ref["diag"][b, 0] < U_EPS, f"unflagged accept mismatch at request {b}"
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[1:] - 1]
    for b in range(w.B):
        if not bad[b] and fin[b] != ref["final_tok"][b]:
            assert ref["diag"][b, 1] < GAP_EPS, f"unflagged final-token mismatch at request {b}"
    assert (np.diff(off) == acc + 1).all()


@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float32])
def test_residual_without_mass_draws_from_p(wdt):
    """The fallback of the residual draw ("DSpark：半自回归生成与置信度调度的投机解码",
    section 形式化定义: at the first rejection the token comes from
    max(0, p - q), and from p when that has no mass).  lse_q is passed 20
    nats too low, so q = e^20 q_true: the first draft is rejected and
    p - q < 0 at every entry.  The emitted token must be the draw from p on
    the rejected row with the residual's noise, argmax_v t_v / tau + G(domain
    2, row (b)(gamma+1) + 0, v), computed here with the oracle's Gumbel
    stream; every request is counted as a fallback draw."""
    w = workload.custom("tiny", B=5, V=4104, r=64, w_dtype=wdt, w_std=0.1, seed=61)
    inp = workload.inputs(w, device=DEV)
    seed, tau = 7, 1.0
    buf = vm.StepBuffers(w.B, w.gamma, w.V, w.r)
    vm.dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok, buf.ws,
                           seed=seed)
    lse_fake = (buf.lse_q - 20.0).contiguous()
    K = torch.full((w.B,), w.gamma, dtype=torch.int32, device=DEV)
    buf.near_ties.zero_()
    vm.dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, lse_fake,
                     buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off, buf.next_anchor,
                     buf.ws, seed=seed, tau=tau, near_ties=buf.near_ties)
    st, bits = vm.dspark_sync_status(buf.ws.buf)
    assert st == 0, bits
    acc = buf.accepted.cpu().numpy()
    assert (acc == 0).all()
    assert int(buf.near_ties[1]) == w.B
    off = buf.out_off.cpu().numpy()
    fin = buf.out_tok.cpu().numpy()[off[:-1]]
    t = inp["target"].double().cpu().numpy()
    for b in range(w.B):
        row = b * (w.gamma + 1) + 0
        g = np.array([oracle.gumbel(seed, 0, 2, row, v) for v in range(w.V)])
        score = t[b, 0] / tau + g
        order = np.argsort(-score, kind="stable")
        if fin[b] != order[0]:
            assert score[order[0]] - score[order[1]] < GAP_EPS, f"request {b}: {fin[b]} != {order[0]}"
