"""Pins of the oracle's RNN draft head ("DSpark：半自回归生成与置信度调度的投机解码",
section RNN Head：长程依赖; "DeepSeek-AI与北京大学联手破局", section 三).

The GRU cell is checked against PyTorch's GRUCell (float64), the bfloat16
rounding against hand-worked ties and PyTorch's conversion, and the whole
RNN draft against the already pinned Markov draft in the two limits where the
GRU collapses to a lookup table: the update gate shut (the state is the
candidate n computed from the token alone) and the update gate open (the
state stays s0 for ever).
"""
import math

import numpy as np
import torch

import oracle
import workload


def _params(r, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    a = scale / math.sqrt(r)
    return dict(W_ih=rng.uniform(-a, a, (3 * r, r)), W_hh=rng.uniform(-a, a, (3 * r, r)),
                b_ih=rng.uniform(-a, a, 3 * r), b_hh=rng.uniform(-a, a, 3 * r))


def test_gru_cell_matches_torch_grucell():
    r = 24
    p = _params(r, 1, scale=3.0)
    cell = torch.nn.GRUCell(r, r).double()
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(p["W_ih"]))
        cell.weight_hh.copy_(torch.from_numpy(p["W_hh"]))
        cell.bias_ih.copy_(torch.from_numpy(p["b_ih"]))
        cell.bias_hh.copy_(torch.from_numpy(p["b_hh"]))
    rng = np.random.default_rng(2)
    for _ in range(5):
        x = rng.normal(0, 1.5, r)
        h = np.tanh(rng.normal(0, 1, r))
        ref = cell(torch.from_numpy(x)[None], torch.from_numpy(h)[None])[0].detach().numpy()
        got = oracle.gru_cell(x, h, p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"])
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_bf16_rounding():
    e = 2.0 ** -8
    assert oracle.bf16_round(1.0) == 1.0
    assert oracle.bf16_round(1 + e) == 1.0                      # tie, even mantissa below
    assert oracle.bf16_round(1 + 3 * e) == 1 + 4 * e            # tie, even mantissa above
    assert oracle.bf16_round(1 + e + 2.0 ** -30) == 1 + 2 * e   # just above the tie
    assert oracle.bf16_round(-(1 + 3 * e)) == -(1 + 4 * e)
    assert oracle.bf16_round(0.75) == 0.75
    assert math.copysign(1.0, oracle.bf16_round(-0.0)) == -1.0
    # binary32 inputs round once either way: torch's float32 -> bfloat16 conversion agrees
    x = torch.randn(2000, generator=torch.Generator().manual_seed(3)) * 0.7
    ref = x.to(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_round(float(v)) for v in x.double().numpy()])
    np.testing.assert_array_equal(got, ref)


def _draft_inputs(B=3, gamma=5, V=64, r=16, seed=4):
    rng = np.random.default_rng(seed)
    U = rng.normal(0, 2.0, (B, gamma, V))
    W2 = rng.normal(0, 0.5, (r, V))
    E = rng.normal(0, 1.0, (V, r))
    anchor = rng.integers(0, V, B).astype(np.int32)
    s0 = rng.normal(0, 0.5, r)
    return U, W2, E, anchor, s0


def _bf16(a):
    return np.vectorize(oracle.bf16_round)(a)


def test_shut_update_gate_reduces_to_a_markov_table():
    # z = 0 and W_hh = 0: s_k = tanh(W_in E[x~_{k-1}] + b_in), a function of the
    # previous token alone, i.e. the Markov head with W1 = bf16(tanh(E W_in^T + b_in)).
    U, W2, E, anchor, s0 = _draft_inputs()
    r = W2.shape[0]
    p = _params(r, 5, scale=2.0)
    p["W_hh"][:] = 0.0
    p["b_hh"][:] = 0.0
    p["b_ih"][r:2 * r] = -1e4                      # sigma(-1e4) = 0 exactly in binary64
    W1 = _bf16(np.tanh(E @ p["W_ih"][2 * r:].T + p["b_ih"][2 * r:]))
    got = oracle.draft_rnn(U, E, p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], s0, W2, anchor, seed=11)
    ref = oracle.draft_markov(U, W1, W2, anchor, seed=11)
    np.testing.assert_array_equal(got["tok"], ref["tok"])
    np.testing.assert_allclose(got["lse_q"], ref["lse_q"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["z_tok"], ref["z_tok"], rtol=0, atol=1e-12)
    prev = np.concatenate([anchor[:, None], got["tok"][:, :-1]], axis=1)
    np.testing.assert_allclose(got["arows"], W1[prev], rtol=0, atol=1e-12)


def test_open_update_gate_keeps_the_initial_state():
    # z = 1: s_k = s_{k-1} = s0 at every position, whatever the tokens.
    U, W2, E, anchor, s0 = _draft_inputs(seed=6)
    r = W2.shape[0]
    p = _params(r, 7)
    p["b_ih"][r:2 * r] = 1e4
    W1 = np.tile(_bf16(s0), (E.shape[0], 1))
    got = oracle.draft_rnn(U, E, p["W_ih"], p["W_hh"], p["b_ih"], p["b_hh"], s0, W2, anchor, seed=12)
    ref = oracle.draft_markov(U, W1, W2, anchor, seed=12)
    np.testing.assert_array_equal(got["tok"], ref["tok"])
    np.testing.assert_allclose(got["lse_q"], ref["lse_q"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["states"], np.broadcast_to(s0, got["states"].shape), rtol=0, atol=0)


def test_state_carries_the_block_history():
    # Same token at position 1, different anchors: the states at position 2
    # differ (the Markov head's rows would be equal).
    w = workload.custom("tiny", B=2, r=32)
    rnn = {k: v.double().numpy() for k, v in workload.rnn_head(w).items()}
    x1 = 7
    h_a = oracle.gru_cell(rnn["E"][3], rnn["s0"], rnn["W_ih"], rnn["W_hh"], rnn["b_ih"], rnn["b_hh"])
    h_b = oracle.gru_cell(rnn["E"][900], rnn["s0"], rnn["W_ih"], rnn["W_hh"], rnn["b_ih"], rnn["b_hh"])
    s2_a = oracle.gru_cell(rnn["E"][x1], h_a, rnn["W_ih"], rnn["W_hh"], rnn["b_ih"], rnn["b_hh"])
    s2_b = oracle.gru_cell(rnn["E"][x1], h_b, rnn["W_ih"], rnn["W_hh"], rnn["b_ih"], rnn["b_hh"])
    assert np.abs(s2_a - s2_b).max() > 1e-2


def test_verify_with_explicit_rows_equals_the_markov_verify():
    w = workload.WORKLOADS["tiny"]
    inp = workload.inputs(w)
    W1 = inp["W1"].double().numpy()
    d = oracle.draft_markov(inp["U"], W1, inp["W2"], inp["anchor"], seed=3)
    prev = np.concatenate([inp["anchor"].numpy()[:, None], d["tok"][:, :-1]], axis=1)
    K = np.full(w.B, w.gamma, np.int32)
    ref = oracle.verify(inp["target"], inp["U"], W1, inp["W2"], inp["anchor"], d["tok"], K, seed=3)
    got = oracle.verify(inp["target"], inp["U"], None, inp["W2"], inp["anchor"], d["tok"], K, seed=3,
                        arows=W1[prev])
    for key in ("accepted", "final_tok"):
        np.testing.assert_array_equal(got[key], ref[key])
    np.testing.assert_array_equal(got["diag"], ref["diag"])
