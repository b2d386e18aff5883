"""Comparison helpers shared by the GPU parity tests.

Sampling decisions (draft tokens, accept/reject, final tokens) must match the
oracle bit for bit, except draws the oracle flags as near-ties: a Gumbel
top-2 gap below GAP_EPS, or an acceptance uniform within U_EPS of its
threshold.  Both sides then take the decision in different precisions
(binary32 on the device, binary64 in the oracle), so either answer is a
correct draw; the test checks the flag, counts it, and stops comparing that
request's later positions (they condition on a different token)."""
import numpy as np

GAP_EPS = 1e-3     # Gumbel top-2 gap that excuses a token mismatch
U_EPS = 1e-5       # |u - min(1, p/q)| that excuses an accept/reject mismatch
LOGIT_ATOL = 1e-3  # draft logits, biases, log-normalisers
PROB_RTOL = 1e-4   # probabilities, confidences, survivals


def compare_draft(gpu_tok, ora_tok, ora_gap, eps=GAP_EPS):
    """Per request, compare tokens up to the first mismatch; every mismatch
    must be flagged.  Returns (positions compared, flagged mismatches)."""
    gpu_tok = np.asarray(gpu_tok); ora_tok = np.asarray(ora_tok)
    compared, flagged = 0, 0
    valid = np.ones(gpu_tok.shape, bool)
    for b in range(gpu_tok.shape[0]):
        for k in range(gpu_tok.shape[1]):
            compared += 1
            if gpu_tok[b, k] != ora_tok[b, k]:
                assert ora_gap[b, k] < eps, (
                    f"unflagged draft mismatch at b={b} k={k}: gpu {gpu_tok[b, k]} oracle {ora_tok[b, k]} "
                    f"gap {ora_gap[b, k]}")
                flagged += 1
                valid[b, k:] = False
                break
    return compared, flagged, valid


def assert_close_where(a, b, mask, atol=0.0, rtol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)[mask]
    b = np.asarray(b, dtype=np.float64)[mask]
    if a.size == 0:
        return
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    bad = err > lim
    assert not bad.any(), f"{what}: {bad.sum()} of {a.size} outside tolerance, worst {err.max():.3g}"
