"""Pins of the oracle's Markov-head draft loop (steps a1-a3).

Each check compares the oracle with something other than itself: numpy's
matmul and scipy's logsumexp on the same values, the softmax law of a
Gumbel-max draw (chi-square), and closed-form special cases."""
import numpy as np
import pytest
from scipy import special, stats

import oracle
import workload


def _tiny(seed=5, nb=3, gamma=4, V=40, r=8, wstd=0.5):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2.0, (nb, gamma, V))
    W1 = rng.normal(0, wstd, (V, r))
    W2 = rng.normal(0, wstd, (r, V))
    anchor = rng.integers(0, V, nb).astype(np.int32)
    return U, W1, W2, anchor


@pytest.mark.parametrize("tau", [1.0, 0.7])
def test_logits_equal_numpy_matmul(tau):
    U, W1, W2, anchor = _tiny()
    out = oracle.draft_markov(U, W1, W2, anchor, seed=1, tau=tau, want_logits=True)
    tok, z = out["tok"], out["logits"]
    for b in range(U.shape[0]):
        prev = anchor[b]
        for k in range(U.shape[1]):
            expect = (U[b, k] + W1[prev] @ W2) / tau        # B_k = W1[x_{k-1}] W2, added to U_k
            np.testing.assert_allclose(z[b, k], expect, rtol=0, atol=1e-12)
            prev = tok[b, k]                                 # the next position conditions on this draw


def test_lse_and_drawn_logit():
    U, W1, W2, anchor = _tiny(seed=9)
    out = oracle.draft_markov(U, W1, W2, anchor, seed=2, want_logits=True)
    z = out["logits"]
    np.testing.assert_allclose(out["lse_q"], special.logsumexp(z, axis=-1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.exp(z - out["lse_q"][..., None]).sum(-1), 1.0, atol=1e-12)
    got = np.take_along_axis(z, out["tok"][..., None].astype(np.int64), -1)[..., 0]
    np.testing.assert_array_equal(out["z_tok"], got)
    assert (out["gap"] >= 0).all()


def test_gumbel_argmax_is_the_max_of_perturbed_scores():
    # brute force on a tiny row: the drawn token maximises z_v + G_v with
    # G_v taken from the stream at (row k-1, col v), lowest index on ties
    U, W1, W2, anchor = _tiny(seed=4, nb=2, gamma=2, V=12)
    out = oracle.draft_markov(U, W1, W2, anchor, seed=77, step=3, want_logits=True, req=[5, 9])
    gamma = U.shape[1]
    for b, rq in enumerate([5, 9]):
        for k in range(gamma):
            s = [out["logits"][b, k, v] + oracle.gumbel(77, 3, 0, rq * (gamma + 1) + k, v) for v in range(12)]
            assert out["tok"][b, k] == int(np.argmax(s))
            top2 = np.sort(s)[-2:]
            assert out["gap"][b, k] == pytest.approx(top2[1] - top2[0], abs=1e-12)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_sampling_law_chi_square(tau):
    # W2 = 0 removes the bias, so x~_1 ~ softmax(U_1 / tau); 10^5 independent
    # requests (distinct Philox rows) give 10^5 draws.
    V, n = 16, 100000
    rng = np.random.default_rng(0)
    u1 = rng.normal(0, 1.5, V)
    U = np.broadcast_to(u1, (n, 1, V)).copy()
    W1 = rng.normal(0, 1, (V, 4)); W2 = np.zeros((4, V))
    anchor = np.zeros(n, np.int32)
    out = oracle.draft_markov(U, W1, W2, anchor, seed=123, tau=tau)
    counts = np.bincount(out["tok"][:, 0], minlength=V)
    p = special.softmax(u1 / tau)
    assert stats.chisquare(counts, p * n).pvalue > 1e-4


def test_markov_bias_changes_the_law_with_the_previous_token():
    # a bias that forces "token (prev+1) mod V": with a one-hot W1 and a
    # shifted identity W2 scaled by 60, every draw follows its predecessor
    V = 10
    W1 = np.eye(V)
    W2 = 60.0 * np.roll(np.eye(V), 1, axis=1)
    U = np.zeros((2, 5, V))
    anchor = np.array([3, 8], np.int32)
    out = oracle.draft_markov(U, W1, W2, anchor, seed=0)
    np.testing.assert_array_equal(out["tok"], [[4, 5, 6, 7, 8], [9, 0, 1, 2, 3]])


def test_request_ids_select_independent_streams():
    U, W1, W2, anchor = _tiny(seed=1, nb=2)
    a = oracle.draft_markov(U, W1, W2, anchor, seed=3, req=[0, 1])
    b = oracle.draft_markov(U[::-1].copy(), W1, W2, anchor[::-1].copy(), seed=3, req=[1, 0])
    np.testing.assert_array_equal(a["tok"], b["tok"][::-1])


def test_tiny_workload_runs():
    w = workload.WORKLOADS["tiny"]
    inp = workload.inputs(w)
    out = oracle.draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], seed=w.seed)
    assert out["tok"].shape == (w.B, w.gamma)
    assert ((out["tok"] >= 0) & (out["tok"] < w.V)).all()
