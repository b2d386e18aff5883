"""Pins of the oracle's confidence head + STS + survival (a4) and of the
hardware-aware prefix scheduler (a5): invariants the pages state, closed-form
special cases, exhaustive search on tiny instances, hand arithmetic."""
import itertools
import math

import numpy as np
import pytest
from scipy import stats

import oracle
import workload


def _conf_inputs(seed=0, nb=6, gamma=7, d=16, V=30):
    rng = np.random.default_rng(seed)
    h = rng.normal(0, 1, (nb, gamma, d))
    emb = rng.normal(0, 1, (V, d))
    w_c = rng.normal(0, 0.4, 2 * d)
    anchor = rng.integers(0, V, nb).astype(np.int32)
    tok = rng.integers(0, V, (nb, gamma)).astype(np.int32)
    T = np.array([1 + 0.1 * k for k in range(1, gamma + 1)])
    return h, emb, w_c, anchor, tok, T


def test_survival_is_monotone_and_a_product():
    h, emb, w_c, anchor, tok, T = _conf_inputs()
    out = oracle.confidence_sts(h, emb, anchor, tok, w_c, 0.5, T)
    ls = out["log_surv"]
    assert (np.diff(ls, axis=1) <= 0).all() and (ls <= 0).all()
    np.testing.assert_allclose(np.exp(ls), np.cumprod(out["conf_cal"], axis=1), rtol=1e-12)


def test_unit_temperature_is_identity():
    h, emb, w_c, anchor, tok, T = _conf_inputs(seed=1)
    out = oracle.confidence_sts(h, emb, anchor, tok, w_c, -0.3, np.ones_like(T))
    np.testing.assert_allclose(out["conf_cal"], out["conf_raw"], rtol=1e-13)


def test_closed_form_special_cases():
    h, emb, w_c, anchor, tok, T = _conf_inputs(seed=2)
    d = h.shape[2]
    # w = 0: c = sigmoid(b) everywhere, c~_k = sigmoid(b / T_k)
    out = oracle.confidence_sts(h, emb, anchor, tok, np.zeros_like(w_c), math.log(4.0), T)
    np.testing.assert_allclose(out["conf_raw"], 0.8, rtol=1e-14)
    np.testing.assert_allclose(out["conf_cal"][0], 1 / (1 + 4.0 ** (-1 / T)), rtol=1e-13)
    # w selects h_k[3]: c = sigmoid(h_k[3])
    w = np.zeros_like(w_c); w[3] = 1.0
    out = oracle.confidence_sts(h, emb, anchor, tok, w, 0.0, T)
    np.testing.assert_allclose(out["conf_raw"], 1 / (1 + np.exp(-h[:, :, 3])), rtol=1e-13)
    # w selects emb(x~_{k-1})[5]: position 1 reads the anchor, position k the draft k-1
    w = np.zeros_like(w_c); w[d + 5] = 1.0
    out = oracle.confidence_sts(h, emb, anchor, tok, w, 0.0, T)
    prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
    np.testing.assert_allclose(out["conf_raw"], 1 / (1 + np.exp(-emb[prev, 5])), rtol=1e-13)


def test_sts_preserves_per_position_ranking():
    h, emb, w_c, anchor, tok, T = _conf_inputs(seed=3, nb=40)
    out = oracle.confidence_sts(h, emb, anchor, tok, w_c, 0.5, T)
    for k in range(T.size):
        tau, _ = stats.kendalltau(out["conf_raw"][:, k], out["conf_cal"][:, k])
        assert tau == pytest.approx(1.0)


# ---------------------------------------------------------------- scheduler


def _theta(la, K, sps):
    B = la.shape[0]
    tau = B + sum(np.exp(la[b, :K[b]]).sum() for b in range(B))
    return tau * sps[B + int(np.sum(K)) - 1]


def _unimodal(curve):
    i = int(np.argmax(curve))
    return (np.diff(curve[: i + 1]) > 0).all() and (np.diff(curve[i:]) < 0).all()


def test_sync_greedy_equals_exhaustive_search_when_unimodal():
    rng = np.random.default_rng(7)
    checked = 0
    for trial in range(400):
        B, gamma = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        c = 1 / (1 + np.exp(-rng.normal(1.0, 1.5, (B, gamma))))
        la = np.cumsum(np.log(c), axis=1)
        a, b = rng.uniform(5, 15), rng.uniform(0.2, 1.5)
        sps = np.array([1000 / (a + b * n) for n in range(1, B + B * gamma + 1)])
        out = oracle.schedule(la, sps, oracle.MODE_SYNC)
        if not _unimodal(out["curve"]):
            continue
        best = max(_theta(la, K, sps) for K in itertools.product(range(gamma + 1), repeat=B))
        got = _theta(la, out["K"], sps)
        assert got == pytest.approx(best, rel=1e-12)
        assert out["theta"] == pytest.approx(best, rel=1e-12)
        checked += 1
    assert checked > 100


def test_sync_stops_at_first_non_rise():
    # a capacity curve with a dip: greedy stops before it even though a
    # later n would be better (the sawtooth trap)
    la = np.log(np.array([[0.9, 0.85, 0.8, 0.75]]))
    la = np.cumsum(la, axis=1)
    sps = np.array([100, 100, 10, 200, 200], dtype=float)   # SPS(1..5)
    out = oracle.schedule(la, sps, oracle.MODE_SYNC)
    # Theta(0)=100, Theta(1)=(1+.9)*100=190, Theta(2)=(1.9+.765)*10 <190 -> stop at 1
    assert out["K"].tolist() == [1] and out["n_total"] == 1
    assert out["theta"] == pytest.approx(190.0)
    curve = out["curve"]
    assert curve[4] > curve[1]                     # a later n was better


def test_async_is_global_argmax_without_break():
    la = np.cumsum(np.log(np.array([[0.9, 0.85, 0.8, 0.75]])), axis=1)
    sps = np.array([100, 100, 10, 200, 200], dtype=float)
    out = oracle.schedule(la, sps, oracle.MODE_ASYNC)
    # Theta = 100, 190, 26.65, 655.4, 747.1: the maximum is past the dip
    np.testing.assert_allclose(out["curve"], [100, 190, 26.65, 655.4, 747.135], rtol=1e-4)
    assert out["n_total"] == 4 and out["K"].tolist() == [4]


def test_async_capacity_from_history_ranking_from_current():
    rng = np.random.default_rng(11)
    for _ in range(50):
        B, gamma = 5, 4
        cur = np.cumsum(np.log(1 / (1 + np.exp(-rng.normal(1, 2, (B, gamma))))), axis=1)
        old = np.cumsum(np.log(1 / (1 + np.exp(-rng.normal(1, 2, (B, gamma))))), axis=1)
        sps = np.array([1000 / (5 + 0.7 * n) for n in range(1, B + B * gamma + 1)])
        out = oracle.schedule(cur, sps, oracle.MODE_ASYNC, log_surv_hist=old)
        hist_curve = oracle.schedule(old, sps, oracle.MODE_ASYNC)["curve"]
        n_star = int(np.argmax(hist_curve))            # first maximum
        assert out["n_total"] == n_star
        # the admitted set is the n* largest current survivals, ties by (b, j)
        items = sorted(((-cur[b, j], b, j) for b in range(B) for j in range(gamma)))[:n_star]
        K = np.zeros(B, int)
        for _, b, _j in items:
            K[b] += 1
        np.testing.assert_array_equal(out["K"], K)


def test_ties_break_by_request_then_position():
    la = np.zeros((3, 2))                     # every survival equals 1
    sps = np.array([1.0] * 3 + [1.0] * 6)     # flat: Theta rises with every admission
    out = oracle.schedule(la, sps, oracle.MODE_SYNC)
    assert out["order"].tolist() == [0, 1, 2, 3, 4, 5]
    assert out["K"].tolist() == [2, 2, 2]


def test_mode_off_verifies_whole_block():
    la = np.cumsum(np.full((4, 7), -1.0), axis=1)
    out = oracle.schedule(la, np.ones(40), oracle.MODE_OFF)
    assert out["K"].tolist() == [7] * 4 and out["n_total"] == 28


def test_stepped_table_admits_nothing(golden_dir):
    vals = {}
    for line in open(f"{golden_dir}/sched_b64_zero_admission.txt"):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    w = workload.WORKLOADS["b64"]
    sps = w.sps_table().double().numpy()
    # survivals as high as they can be: every confidence equal to 1
    la = np.zeros((w.B, w.gamma))
    out = oracle.schedule(la, sps, oracle.MODE_SYNC)
    assert out["curve"][0] == pytest.approx(vals["theta0"], rel=1e-6)
    assert out["curve"][1] == pytest.approx(vals["theta1_upper"], rel=1e-6)
    assert out["n_total"] == int(vals["admitted"]) and out["K"].sum() == 0


def test_sawtooth_table_matches_its_recipe():
    w = workload.WORKLOADS["b256"]
    s = w.sps_table().double().numpy()
    base = lambda n: 1000 / (6 + 0.004 * n)
    assert s[0] == pytest.approx(base(1), rel=1e-6)            # n = 1: no drop
    assert s[128] == pytest.approx(base(129) * 0.85, rel=1e-6)  # n = 129: full 15 % drop
    assert s[128 + 16] == pytest.approx(base(145) * (1 - 0.15 * 0.5), rel=1e-6)
    assert s[128 + 32] == pytest.approx(base(161), rel=1e-6)   # recovered after 32
    assert s[256] == pytest.approx(base(257) * 0.85, rel=1e-6)
