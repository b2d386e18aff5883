"""Pins of the oracle's STS fit ("DSpark：半自回归生成与置信度调度的投机解码",
section 校准问题：原始置信度不可靠; "DeepSeek-AI与北京大学联手破局", section 四).

Each case fixes something other than the oracle's own code: closed-form
survivals built from sigmoid(log 3) = 3/4, the half-open bin rule, the ratio
form of the expected calibration error, recovery of known temperatures from
data drawn from a calibrated model, and invariances.
"""
import math

import numpy as np
import pytest

import oracle
import workload

LN3 = math.log(3.0)


def test_single_sample_closed_form():
    # score 2 ln 3: T = 2 gives 3/4, T = 1 gives 9/10, T = 1/2 gives 81/82.
    grid = [2.0, 1.0, 0.5]
    acc = oracle.sts_fit([[2 * LN3]], [1], grid, M=15)
    np.testing.assert_allclose(acc["ece"][0], [1 / 4, 1 / 10, 1 / 82], rtol=0, atol=1e-14)
    assert acc["idx"][0] == 2 and acc["T"][0] == 0.5
    rej = oracle.sts_fit([[2 * LN3]], [0], grid, M=15)
    np.testing.assert_allclose(rej["ece"][0], [3 / 4, 9 / 10, 81 / 82], rtol=0, atol=1e-14)
    assert rej["idx"][0] == 0 and rej["T"][0] == 2.0


def test_sequential_product_keeps_earlier_temperature():
    # One block, first draft accepted, second rejected (acc_len 1).
    # Position 1 (label 1): T = 2 gives 3/4, T = 3 gives 1/(1 + 3^(-2/3)); 2 wins.
    # Position 2 (label 0) with T_1 = 2 kept: T = 3 gives (3/4)(3/4) = 9/16,
    # T = 2 gives (3/4) * 3^1.5 / (3^1.5 + 1); 3 wins.
    score = [[2 * LN3, 3 * LN3]]
    r = oracle.sts_fit(score, [1], [2.0, 3.0], M=10)
    s15 = 3 ** 1.5
    np.testing.assert_allclose(r["ece"][0], [1 / 4, 1 - 1 / (1 + 3 ** (-2 / 3))], atol=1e-14)
    np.testing.assert_allclose(r["ece"][1], [0.75 * s15 / (s15 + 1), 9 / 16], atol=1e-14)
    assert list(r["idx"]) == [0, 1]
    # Forcing T_1 = 3 changes only position 2: its factor 1 becomes 1/(1 + 3^(-2/3)).
    f = oracle.sts_fit(score, [1], [2.0, 3.0], M=10, T_fixed=[3.0, 3.0])
    np.testing.assert_allclose(f["ece"][0], r["ece"][0], atol=0)
    c1 = 1 / (1 + 3 ** (-2 / 3))
    np.testing.assert_allclose(f["ece"][1], [c1 * s15 / (s15 + 1), c1 * 0.75], atol=1e-14)


def test_half_open_bins():
    # M = 2.  A: score 0 (a = 1/2 for every T), label 0.  B: score ln 9 (a = 9/10), label 1.
    # With bins [0, 1/2) and [1/2, 1], A shares B's bin: ECE = |(0 - 1/2) + (1 - 9/10)| / 2 = 0.2.
    r = oracle.sts_fit([[0.0], [math.log(9.0)]], [0, 1], [1.0], M=2)
    assert r["ece"][0, 0] == pytest.approx(0.2, abs=1e-14)
    # M = 3 puts them apart (1/2 in [1/3, 2/3), 9/10 in [2/3, 1]): (1/2 + 1/10) / 2 = 0.3.
    r3 = oracle.sts_fit([[0.0], [math.log(9.0)]], [0, 1], [1.0], M=3)
    assert r3["ece"][0, 0] == pytest.approx(0.3, abs=1e-14)


def test_one_bin_is_calibration_in_the_large():
    rng = np.random.default_rng(5)
    score = rng.normal(0.5, 2.0, size=(300, 3))
    acc_len = rng.integers(0, 4, size=300)
    grid = np.array([0.5, 1.0, 1.7])
    r = oracle.sts_fit(score, acc_len, grid, M=1)
    prev = []
    for k in range(1, 4):
        a = oracle.sts_survival(score, prev, k, grid)
        y = (acc_len >= k).astype(float)
        np.testing.assert_allclose(r["ece"][k - 1], np.abs(y.mean() - a.mean(axis=0)), atol=1e-13)
        prev.append(r["T"][k - 1])


def test_ratio_form_by_brute_force():
    # ECE = sum_m (|B_m| / N) * |acc(B_m) - conf(B_m)|, bins gathered one sample at a time.
    rng = np.random.default_rng(11)
    N, gamma, M = 257, 3, 7
    score = rng.normal(1.0, 2.5, size=(N, gamma))
    acc_len = rng.integers(0, gamma + 1, size=N)
    grid = np.array([0.4, 0.9, 1.3, 2.2, 3.1])
    r = oracle.sts_fit(score, acc_len, grid, M=M)
    prev = []
    for k in range(1, gamma + 1):
        a = oracle.sts_survival(score, prev, k, grid)
        for g in range(grid.size):
            bins = [[] for _ in range(M)]
            for n in range(N):
                m = M - 1
                for j in range(M):
                    if a[n, g] < (j + 1) / M:
                        m = j
                        break
                bins[m].append((1.0 if acc_len[n] >= k else 0.0, a[n, g]))
            e = 0.0
            for b in bins:
                if b:
                    acc = sum(y for y, _ in b) / len(b)
                    conf = sum(p for _, p in b) / len(b)
                    e += len(b) / N * abs(acc - conf)
            assert r["ece"][k - 1, g] == pytest.approx(e, abs=1e-12)
        prev.append(r["T"][k - 1])


def test_recovers_known_temperatures():
    T_true = [0.5, 2.0, 1.0, 3.0]
    score, acc_len = workload.sts_validation(100_000, gamma=4, seed=3, T_true=T_true)
    grid = np.round(np.arange(0.25, 4.01, 0.25), 2)
    r = oracle.sts_fit(score, acc_len, grid, M=15)
    np.testing.assert_allclose(r["T"], T_true, atol=0.25)
    assert (r["ece"].min(axis=1) < 0.01).all()
    # The raw confidences (T = 1) are clearly miscalibrated wherever T* != 1.
    # (Reading the page's formula with T_k on every factor instead would need
    # one temperature to fit 0.5 and 2.0 at once at position 2, and misses T*.)
    one = np.where(grid == 1.0)[0][0]
    assert (r["ece"][[0, 1, 3], one] > 3 * r["ece"].min(axis=1)[[0, 1, 3]]).all()


def test_sample_order_and_ties():
    rng = np.random.default_rng(2)
    score = rng.normal(0.0, 3.0, size=(500, 4))
    acc_len = rng.integers(0, 5, size=500)
    grid = np.array([0.7, 1.0, 1.6, 2.5])
    r = oracle.sts_fit(score, acc_len, grid)
    perm = rng.permutation(500)
    q = oracle.sts_fit(score[perm], acc_len[perm], grid)
    np.testing.assert_allclose(q["ece"], r["ece"], atol=1e-13)
    assert list(q["idx"]) == list(r["idx"])
    # Equal grid values tie: the lower index is chosen.
    d = oracle.sts_fit(score, acc_len, np.array([1.6, 1.6, 0.7]))
    assert (d["ece"][:, 0] == d["ece"][:, 1]).all() and (d["idx"] != 1).all()
    # Score 0 makes every temperature equal: index 0 everywhere.
    z = oracle.sts_fit(np.zeros((50, 3)), acc_len[:50], np.array([3.0, 1.0, 2.0]))
    assert (z["idx"] == 0).all()
