"""Pins of the oracle's lossless verification (a6-a7) and ragged compaction
(a8): the emitted tokens follow the target law (chi-square on V=16), a
hand-worked three-token example, closed-form special cases and the layout
invariants of the flattened output."""
import numpy as np
import pytest
from scipy import special, stats

import oracle


def _golden(golden_dir):
    vals = {}
    for line in open(f"{golden_dir}/spec_sampling_v3.txt"):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            vals[k] = np.array([float(t) for t in v])
    return vals


def _replicated_case(n, gamma, V, seed, *, target_rows=None, u_rows=None, r=4):
    """n requests that share the same logits rows but draw from distinct
    Philox rows: n independent trials of one draft + verify step.  The Markov
    bias is switched off (W2 = 0) so the target's conditionals (which ignore
    the history) are a valid autoregressive target."""
    rng = np.random.default_rng(seed)
    if u_rows is None:
        u_rows = rng.normal(0, 1.5, (gamma, V))
    if target_rows is None:
        target_rows = np.concatenate([u_rows, rng.normal(0, 1.5, (1, V))]) + rng.normal(0, 0.8, (gamma + 1, V))
    U = np.broadcast_to(u_rows, (n, gamma, V)).copy()
    T = np.broadcast_to(target_rows, (n, gamma + 1, V)).copy()
    W1 = rng.normal(0, 1, (V, r)); W2 = np.zeros((r, V))
    anchor = np.zeros(n, np.int32)
    return U, T, W1, W2, anchor, u_rows, target_rows


def _run(U, T, W1, W2, anchor, K, seed):
    d = oracle.draft_markov(U, W1, W2, anchor, seed=seed)
    v = oracle.verify(T, U, W1, W2, anchor, d["tok"], K, seed=seed)
    o = oracle.compact(d["tok"], v["accepted"], v["final_tok"])
    return d, v, o


def _emitted(o, n, pos):
    """token emitted at 0-based position pos for each request (-1 if none)."""
    out = np.full(n, -1)
    length = np.diff(o["out_off"])
    has = length > pos
    out[has] = o["out_tok"][o["out_off"][:-1][has] + pos]
    return out


@pytest.mark.parametrize("Kfull", [True, False])
def test_lossless_chi_square(Kfull):
    n, gamma, V = 200000, 3, 16
    U, T, W1, W2, anchor, _, trows = _replicated_case(n, gamma, V, seed=1)
    rng = np.random.default_rng(2)
    K = np.full(n, gamma, np.int32) if Kfull else rng.integers(0, gamma + 1, n).astype(np.int32)
    d, v, o = _run(U, T, W1, W2, anchor, K, seed=99)
    p = special.softmax(trows, axis=-1)
    for pos in range(gamma + 1):
        y = _emitted(o, n, pos)
        y = y[y >= 0]
        if y.size < 2000:
            continue
        counts = np.bincount(y, minlength=V)
        assert stats.chisquare(counts, p[pos] * y.size).pvalue > 1e-4, pos
    # given the first token and that the step goes on, the second token is
    # still p_2: whether the step continues depends on y_1, never on y_2
    y1, y2 = _emitted(o, n, 0), _emitted(o, n, 1)
    m = y2 >= 0
    joint = np.bincount(y1[m] * V + y2[m], minlength=V * V)
    first = np.bincount(y1[m], minlength=V)
    expect = np.outer(first, p[1]).ravel()
    keep = expect > 5
    assert stats.chisquare(joint[keep], expect[keep] * joint[keep].sum() / expect[keep].sum()).pvalue > 1e-4


def test_zero_verify_length_emits_one_token_from_p1():
    n, gamma, V = 100000, 2, 16
    U, T, W1, W2, anchor, _, trows = _replicated_case(n, gamma, V, seed=3)
    d, v, o = _run(U, T, W1, W2, anchor, np.zeros(n, np.int32), seed=5)
    assert (v["accepted"] == 0).all() and (np.diff(o["out_off"]) == 1).all()
    counts = np.bincount(o["out_tok"], minlength=V)
    assert stats.chisquare(counts, special.softmax(trows[0]) * n).pvalue > 1e-4


def test_hand_worked_three_token_example(golden_dir):
    g = _golden(golden_dir)
    n = 100000
    U, T, W1, W2, anchor, _, _ = _replicated_case(
        n, 1, 3, seed=0, u_rows=np.log(g["q"])[None], target_rows=np.log(np.stack([g["p"], g["p"]])))
    d, v, o = _run(U, T, W1, W2, anchor, np.ones(n, np.int32), seed=17)
    x = d["tok"][:, 0]
    acc = v["accepted"] == 1
    # acceptance rate sum_v min(p, q)
    assert stats.binomtest(int(acc.sum()), n, g["accept_rate"][0]).pvalue > 1e-4
    # acceptance probability given the draft
    for tok in range(3):
        sel = x == tok
        assert stats.binomtest(int(acc[sel].sum()), int(sel.sum()), g["accept_given_draft"][tok]).pvalue > 1e-4
    # every rejection is corrected to token 0: the residual is one-hot
    assert (v["final_tok"][~acc] == 0).all()
    assert (v["diag"][~acc, 4] == 0).all()               # residual kind
    np.testing.assert_allclose(v["diag"][~acc, 2], 0.3, rtol=1e-12)   # residual mass
    counts = np.bincount(o["out_tok"][o["out_off"][:-1]], minlength=3)
    assert stats.chisquare(counts, g["emit"] * n).pvalue > 1e-4


def test_equal_distributions_accept_everything():
    n, gamma, V = 2000, 4, 16
    U, T, W1, W2, anchor, urows, _ = _replicated_case(n, gamma, V, seed=8)
    T = np.concatenate([U, np.broadcast_to(np.zeros(V), (n, 1, V))], axis=1)   # p_k = q_k
    d, v, o = _run(U, T, W1, W2, anchor, np.full(n, gamma, np.int32), seed=1)
    assert (v["accepted"] == gamma).all() and (v["diag"][:, 4] == 1).all()
    np.testing.assert_allclose(v["p_tok"], v["q_tok"], rtol=1e-12)


def test_one_hot_target_always_emits_its_mode():
    n, gamma, V = 3000, 3, 16
    rng = np.random.default_rng(4)
    urows = rng.normal(0, 1, (gamma, V))
    modes = np.array([3, 7, 11, 2])
    trows = np.full((gamma + 1, V), -1e4); trows[np.arange(gamma + 1), modes] = 0.0
    U, T, W1, W2, anchor, _, _ = _replicated_case(n, gamma, V, seed=4, u_rows=urows, target_rows=trows)
    d, v, o = _run(U, T, W1, W2, anchor, np.full(n, gamma, np.int32), seed=6)
    for pos in range(gamma + 1):
        y = _emitted(o, n, pos)
        assert (y[y >= 0] == modes[pos]).all()


def test_first_position_acceptance_rate_is_one_minus_tv():
    n, gamma, V = 100000, 1, 16
    U, T, W1, W2, anchor, urows, trows = _replicated_case(n, gamma, V, seed=12)
    d, v, o = _run(U, T, W1, W2, anchor, np.ones(n, np.int32), seed=21)
    rate = np.minimum(special.softmax(urows[0]), special.softmax(trows[0])).sum()
    assert stats.binomtest(int((v["accepted"] == 1).sum()), n, rate).pvalue > 1e-4


def test_compaction_layout_invariants():
    n, gamma, V = 500, 5, 16
    U, T, W1, W2, anchor, _, _ = _replicated_case(n, gamma, V, seed=13)
    K = np.random.default_rng(0).integers(0, gamma + 1, n).astype(np.int32)
    d, v, o = _run(U, T, W1, W2, anchor, K, seed=2)
    A, off = v["accepted"], o["out_off"]
    assert off[0] == 0 and off[-1] == (A + 1).sum() == o["out_tok"].size
    assert (np.diff(off) >= 1).all() and (A <= K).all() and (A >= 0).all()
    for b in range(n):
        seg = o["out_tok"][off[b]:off[b + 1]]
        np.testing.assert_array_equal(seg[:-1], d["tok"][b, :A[b]])
        assert seg[-1] == v["final_tok"][b] == o["next_anchor"][b]
        assert (o["out_req"][off[b]:off[b + 1]] == b).all()
        np.testing.assert_array_equal(o["out_pos"][off[b]:off[b + 1]], np.arange(A[b] + 1))
