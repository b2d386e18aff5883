"""Comparison helpers shared by the GPU parity tests.

Sampling decisions (draft tokens, accept/reject, final tokens) must match the
oracle bit for bit, except draws the oracle flags as near-ties.  Both sides
take such a decision in different precisions (binary32 on the device,
binary64 in the oracle), so either answer is a correct draw.

Two flag thresholds are used ("DSpark：半自回归生成与置信度调度的投机解码", section
形式化定义: the emitted tokens follow the target law exactly; the tolerance
is the build's own):
  - GAP_EPS = 1e-3 on the Gumbel top-2 gap and U_EPS = 1e-5 on the
    acceptance margin |u - min(1, p/q)|, the published bar: every mismatch
    must be flagged at these;
  - eps = max(4 * (measured max |z_gpu - z_oracle| + measured max |G_gpu -
    G_exact|), 1e-5), the device's own error bound: a mismatch needs the two
    scores within twice the score error, so every draft mismatch must also
    lie below eps, and draws flagged at eps must stay under 0.01% of all
    draws (checked on a large sample).
After a draft mismatch the request's later positions condition on a
different token and are not compared."""
import numpy as np

GAP_EPS = 1e-3     # Gumbel top-2 gap that excuses a token mismatch
U_EPS = 1e-5       # |u - min(1, p/q)| that excuses an accept/reject mismatch
LOGIT_ATOL = 1e-3  # draft logits, biases, log-normalisers
PROB_RTOL = 1e-4   # probabilities, confidences, survivals
EPS_FLOOR = 1e-5   # lower bound of the device-error near-tie threshold
RATE_CAP = 1e-4    # draws flagged at eps: at most 0.01 %


def score_eps(dz, dg):
    """The near-tie threshold from the measured logit and Gumbel errors."""
    return max(4.0 * (float(dz) + float(dg)), EPS_FLOOR)


class NearTieLedger:
    """Counts of compared decisions and of near-ties at 1e-3 / 1e-5 and at eps."""

    def __init__(self, eps):
        self.eps = float(eps)
        self.c = dict(draft_draws=0, draft_gap_1e3=0, draft_gap_eps=0, draft_mismatch=0,
                      accept_walks=0, accept_near_1e5=0, accept_mismatch=0,
                      final_draws=0, final_gap_1e3=0, final_gap_eps=0, final_mismatch=0)

    def draft(self, gpu_tok, ora_tok, ora_gap):
        """Per request, compare tokens up to the first mismatch; every mismatch
        must be a near-tie at eps (and so at GAP_EPS).  Returns the mask of
        positions whose prefix matched."""
        gpu_tok = np.asarray(gpu_tok); ora_tok = np.asarray(ora_tok); ora_gap = np.asarray(ora_gap)
        valid = np.ones(gpu_tok.shape, bool)
        for b in range(gpu_tok.shape[0]):
            for k in range(gpu_tok.shape[1]):
                g = ora_gap[b, k]
                self.c["draft_draws"] += 1
                self.c["draft_gap_1e3"] += int(g < GAP_EPS)
                self.c["draft_gap_eps"] += int(g < self.eps)
                if gpu_tok[b, k] != ora_tok[b, k]:
                    assert g < self.eps, (
                        f"draft mismatch at b={b} k={k} is no near-tie: gpu {gpu_tok[b, k]} oracle "
                        f"{ora_tok[b, k]} gap {g:.3g} (eps {self.eps:.3g})")
                    self.c["draft_mismatch"] += 1
                    valid[b, k:] = False
                    break
        return valid

    def verify(self, gpu_acc, gpu_fin, ora, rows):
        """Accept counts and final tokens of the requests `rows` (whose whole
        draft matched) against the oracle's verify output `ora`."""
        diag = ora["diag"]
        for i in rows:
            margin, fgap = diag[i, 0], diag[i, 1]
            self.c["accept_walks"] += 1
            self.c["accept_near_1e5"] += int(margin < U_EPS)
            if gpu_acc[i] != ora["accepted"][i]:
                assert margin < U_EPS, f"accept mismatch at request {i} is no near-tie (margin {margin:.3g})"
                self.c["accept_mismatch"] += 1
                continue
            self.c["final_draws"] += 1
            self.c["final_gap_1e3"] += int(fgap < GAP_EPS)
            self.c["final_gap_eps"] += int(fgap < self.eps)
            if gpu_fin[i] != ora["final_tok"][i]:
                assert fgap < GAP_EPS, f"final-token mismatch at request {i} is no near-tie (gap {fgap:.3g})"
                self.c["final_mismatch"] += 1

    def draws(self):
        return self.c["draft_draws"] + self.c["accept_walks"] + self.c["final_draws"]

    def flagged_eps(self):
        return self.c["draft_gap_eps"] + self.c["accept_near_1e5"] + self.c["final_gap_eps"]

    def rate_eps(self):
        return self.flagged_eps() / max(1, self.draws())

    def summary(self):
        return dict(self.c, eps=self.eps, draws=self.draws(), flagged_eps=self.flagged_eps(),
                    rate_eps=self.rate_eps())


def compare_draft(gpu_tok, ora_tok, ora_gap, eps=GAP_EPS):
    """Per request, compare tokens up to the first mismatch; every mismatch
    must be flagged.  Returns (positions compared, flagged mismatches, mask)."""
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


def max_abs_where(a, b, mask):
    a = np.asarray(a, dtype=np.float64)[mask]
    b = np.asarray(b, dtype=np.float64)[mask]
    return float(np.abs(a - b).max()) if a.size else 0.0
