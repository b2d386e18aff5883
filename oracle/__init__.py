"""Float64 CPU oracle of the DSpark draft + verify step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links or
calls it, and it shares no code with the CUDA sources.

The arithmetic lives in ``dspark_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  Each wrapper names the passage its C function follows:

  [P2] "DSpark：半自回归生成与置信度调度的投机解码" (pinghaoyang.com.cn)
  [P3] "拒绝盲猜与算力空转：深度拆解 DeepSeek 开源投机采样方案 DeepSpec & DSpark"
  [P4] "DeepSeek-AI与北京大学联手破局：AI聊天机器人"慢速打字"的终极解决方案"

Parity pins (see tests/test_oracle_*.py): Philox known-answer vectors, the
bias equal to a numpy matmul, log-sum-exp normalisation, Gumbel-max
chi-square, survival monotonicity, STS identity and rank preservation,
scheduler equal to exhaustive search, lossless chi-square of the whole
draft + verify chain; the STS fit against closed-form survivals, the
half-open bin rule, the ratio form of the calibration error by brute force
and recovery of known temperatures from calibrated synthetic data.  Acceptance length on the synthetic workloads has no
published value: parity unpinned there (reported only).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile dspark_oracle.c into oracle/_build/liboracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
            u32p = np.ctypeslib.ndpointer(np.uint32, flags="C_CONTIGUOUS")
            opt_f64 = C.c_void_p
            lib.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_random_word.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32]
            lib.oracle_random_word.restype = C.c_uint32
            lib.oracle_uniform.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32]
            lib.oracle_uniform.restype = C.c_double
            lib.oracle_gumbel.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32]
            lib.oracle_gumbel.restype = C.c_double
            lib.oracle_gumbel_span.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_int,
                                               f64p]
            lib.oracle_gumbel_span.restype = None
            lib.oracle_draft_markov.argtypes = [
                f64p, f64p, f64p, i32p, i32p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_double,
                C.c_uint64, C.c_uint64, i32p, f64p, f64p, f64p, opt_f64]
            lib.oracle_draft_markov.restype = C.c_int
            lib.oracle_confidence_sts.argtypes = [
                f64p, C.c_int, f64p, C.c_int, i32p, i32p, f64p, C.c_double, f64p,
                C.c_int, C.c_int, f64p, f64p, f64p]
            lib.oracle_confidence_sts.restype = None
            lib.oracle_schedule.argtypes = [
                f64p, opt_f64, f64p, C.c_int, C.c_int, C.c_int, C.c_int,
                i32p, i32p, f64p, i32p, f64p]
            lib.oracle_schedule.restype = C.c_int
            lib.oracle_gru_cell.argtypes = [f64p, f64p, f64p, f64p, f64p, f64p, C.c_int, C.c_int, f64p]
            lib.oracle_gru_cell.restype = None
            lib.oracle_bf16_round.argtypes = [C.c_double]
            lib.oracle_bf16_round.restype = C.c_double
            lib.oracle_rnn_states.argtypes = [f64p, f64p, f64p, f64p, f64p, f64p, i32p, i32p, C.c_int, C.c_int,
                                              C.c_int, C.c_int, f64p, f64p]
            lib.oracle_rnn_states.restype = C.c_int
            lib.oracle_draft_rnn.argtypes = [
                f64p, f64p, f64p, f64p, f64p, f64p, f64p, f64p, i32p, i32p, C.c_int, C.c_int, C.c_int,
                C.c_int, C.c_double, C.c_uint64, C.c_uint64, i32p, f64p, f64p, f64p, f64p, f64p]
            lib.oracle_draft_rnn.restype = C.c_int
            lib.oracle_verify.argtypes = [
                f64p, f64p, opt_f64, f64p, opt_f64, i32p, i32p, i32p, i32p, C.c_int, C.c_int, C.c_int, C.c_int,
                C.c_double, C.c_uint64, C.c_uint64, i32p, i32p, f64p, f64p, f64p]
            lib.oracle_verify.restype = C.c_int
            lib.oracle_compact.argtypes = [i32p, i32p, i32p, C.c_int, C.c_int, i32p, i32p, i32p, i32p, i32p]
            lib.oracle_compact.restype = None
            lib.oracle_sts_survival.argtypes = [f64p, C.c_int, C.c_int, f64p, C.c_int, f64p, C.c_int, f64p]
            lib.oracle_sts_survival.restype = None
            lib.oracle_sts_fit.argtypes = [f64p, i32p, C.c_int, C.c_int, f64p, C.c_int, C.c_int, opt_f64,
                                           f64p, i32p, f64p]
            lib.oracle_sts_fit.restype = C.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = C.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):          # a torch tensor: upcast exactly, then hand over
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# --------------------------------------------------------------------------- #
# Counter-based generator: Philox4x32-10 (Salmon et al., SC'11) and the        #
# stream layout described in dspark_oracle.c.                                 #
# --------------------------------------------------------------------------- #
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(c, k, out)
    return out


def random_word(seed, step, domain, row, col) -> int:
    return int(_load().oracle_random_word(seed, step, domain, row, col))


def uniform(seed, step, domain, row, col) -> float:
    return float(_load().oracle_uniform(seed, step, domain, row, col))


def gumbel(seed, step, domain, row, col) -> float:
    return float(_load().oracle_gumbel(seed, step, domain, row, col))


def gumbel_span(seed, step, domain, row, col0, n) -> np.ndarray:
    """G for columns col0 .. col0+n-1 of one stream."""
    out = np.zeros(n)
    _load().oracle_gumbel_span(seed, step, domain, row, col0, n, out)
    return out


# --------------------------------------------------------------------------- #
# vocabulary slices: the per-slice states a split of V over ranks exchanges   #
# [P2 §Markov Head：一阶转移偏置] (the bias spans the whole vocabulary, so a    #
# split of V shares one draw and one log-sum-exp per position)               #
# --------------------------------------------------------------------------- #
def _lse(x) -> float:
    x = np.asarray(x, np.float64)
    m = x.max() if x.size else -np.inf
    if m == -np.inf:
        return -np.inf
    return float(m + np.log(np.exp(x - m).sum()))


def _argmax_first(score) -> int:
    """Lowest index among the maxima (the draw's tie rule)."""
    return int(np.argmax(score))


def slice_draft(U_row, h, W2_slice, col0, *, seed, step, row, tau=1.0):
    """Position draw on columns col0 .. col0+n-1 of one request's row:
    z = (U + h . W2) / tau over the slice, best = max z + G (domain 0, global
    column index), its index and z, and lse = log sum exp z of the slice."""
    z = (_f64(U_row) + _f64(h) @ _f64(W2_slice)) / tau
    g = gumbel_span(seed, step, 0, row, col0, z.size)
    s = z + g
    i = _argmax_first(s)
    return dict(best=float(s[i]), idx=col0 + i, zb=float(z[i]), lse=_lse(z))


def slice_lse(x_slice, tau=1.0) -> float:
    """log sum exp(x / tau) over a slice of a target row."""
    return _lse(_f64(x_slice) / tau)


def slice_residual(t_slice, z_slice, lse_p, lse_q, col0, *, seed, step, row, tau=1.0):
    """The residual draw on a slice: p = exp(t / tau - lse_p), q = exp(z -
    lse_q), argmax log(max(0, p - q)) + G (domain 2) where p > q (best_r =
    -inf if none), and the fallback draw from p, argmax t / tau + G."""
    t = _f64(t_slice) / tau
    r = np.exp(t - lse_p) - np.exp(_f64(z_slice) - lse_q)
    g = gumbel_span(seed, step, 2, row, col0, t.size)
    with np.errstate(divide="ignore"):
        sr = np.where(r > 0, np.log(np.where(r > 0, r, 1.0)) + g, -np.inf)
    ir = _argmax_first(sr)
    sp = t + g
    ip = _argmax_first(sp)
    return dict(best_r=float(sr[ir]), idx_r=col0 + ir, best_p=float(sp[ip]), idx_p=col0 + ip)


def slice_bonus(t_slice, col0, *, seed, step, row, tau=1.0):
    """The bonus draw on a slice: argmax t / tau + G (domain 3)."""
    s = _f64(t_slice) / tau + gumbel_span(seed, step, 3, row, col0, np.asarray(t_slice).size)
    i = _argmax_first(s)
    return dict(best=float(s[i]), idx=col0 + i)


# --------------------------------------------------------------------------- #
# a1-a3 draft loop [P2 §整体架构, §Markov Head：一阶转移偏置], [P3 §低秩马尔可夫头] #
# --------------------------------------------------------------------------- #
def draft_markov(U, W1, W2, anchor, *, seed, step=0, tau=1.0, req=None, want_logits=False):
    """U [nb,gamma,V], W1 [V,r], W2 [r,V], anchor [nb]; req = global request ids.

    Returns tok [nb,gamma] (int32), lse_q, z_tok, gap (float64 [nb,gamma]) and,
    if asked, the draft logits z [nb,gamma,V]."""
    U = _f64(U); W1 = _f64(W1); W2 = _f64(W2); anchor = _i32(anchor)
    nb, gamma, V = U.shape
    r = W1.shape[1]
    assert W1.shape == (V, r) and W2.shape == (r, V) and anchor.shape == (nb,)
    req = np.arange(nb, dtype=np.int32) if req is None else _i32(req)
    tok = np.zeros((nb, gamma), np.int32)
    lse = np.zeros((nb, gamma)); ztok = np.zeros((nb, gamma)); gap = np.zeros((nb, gamma))
    logits = np.zeros((nb, gamma, V)) if want_logits else None
    rc = _load().oracle_draft_markov(
        U, W1, W2, anchor, req, nb, gamma, V, r, float(tau), int(seed), int(step),
        tok, lse, ztok, gap, logits.ctypes.data if want_logits else None)
    if rc != 0:
        raise ValueError("oracle_draft_markov: invalid arguments")
    out = dict(tok=tok, lse_q=lse, z_tok=ztok, gap=gap)
    if want_logits:
        out["logits"] = logits
    return out


def gru_cell(x, h, W_ih, W_hh, b_ih, b_hh):
    """One GRU step h' = GRU(h, x) (oracle_gru_cell; [P2 §RNN Head：长程依赖])."""
    x = _f64(x); h = _f64(h); W_ih = _f64(W_ih); W_hh = _f64(W_hh); b_ih = _f64(b_ih); b_hh = _f64(b_hh)
    r, r_in = h.size, x.size
    assert W_ih.shape == (3 * r, r_in) and W_hh.shape == (3 * r, r) and b_ih.size == b_hh.size == 3 * r
    out = np.zeros(r)
    _load().oracle_gru_cell(x, h, W_ih, W_hh, b_ih, b_hh, r_in, r, out)
    return out


def bf16_round(x) -> float:
    return float(_load().oracle_bf16_round(float(x)))


def rnn_states(E, W_ih, W_hh, b_ih, b_hh, s0, anchor, tok):
    """The RNN head's states along the tokens tok [nb,gamma] (oracle_rnn_states):
    returns (states, arows), both [nb,gamma,r], arows rounded to bfloat16."""
    E = _f64(E); W_ih = _f64(W_ih); W_hh = _f64(W_hh); b_ih = _f64(b_ih); b_hh = _f64(b_hh); s0 = _f64(s0)
    anchor = _i32(anchor); tok = _i32(tok)
    nb, gamma = tok.shape
    V, r = E.shape
    states = np.zeros((nb, gamma, r)); arows = np.zeros((nb, gamma, r))
    if _load().oracle_rnn_states(E, W_ih, W_hh, b_ih, b_hh, s0, anchor, tok, nb, gamma, V, r, states, arows):
        raise ValueError("oracle_rnn_states: token out of range")
    return states, arows


def draft_rnn(U, E, W_ih, W_hh, b_ih, b_hh, s0, W2, anchor, *, seed, step=0, tau=1.0, req=None):
    """The draft loop with the RNN head (oracle_draft_rnn; [P2 §RNN Head：长程依赖], [P4 §三]).

    U [nb,gamma,V], E [V,r], W_ih/W_hh [3r,r], b_ih/b_hh [3r], s0 [r], W2 [r,V].
    Returns tok, lse_q, z_tok, gap, states [nb,gamma,r] (s_k) and arows
    [nb,gamma,r] (s_k rounded to bfloat16: the rows the biases are formed from)."""
    U = _f64(U); E = _f64(E); W_ih = _f64(W_ih); W_hh = _f64(W_hh); b_ih = _f64(b_ih)
    b_hh = _f64(b_hh); s0 = _f64(s0); W2 = _f64(W2); anchor = _i32(anchor)
    nb, gamma, V = U.shape
    r = s0.size
    assert E.shape == (V, r) and W2.shape == (r, V) and W_ih.shape == (3 * r, r) and W_hh.shape == (3 * r, r)
    req = np.arange(nb, dtype=np.int32) if req is None else _i32(req)
    tok = np.zeros((nb, gamma), np.int32)
    lse = np.zeros((nb, gamma)); ztok = np.zeros((nb, gamma)); gap = np.zeros((nb, gamma))
    states = np.zeros((nb, gamma, r)); arows = np.zeros((nb, gamma, r))
    rc = _load().oracle_draft_rnn(U, E, W_ih, W_hh, b_ih, b_hh, s0, W2, anchor, req, nb, gamma, V, r,
                                  float(tau), int(seed), int(step), tok, lse, ztok, gap, states, arows)
    if rc != 0:
        raise ValueError("oracle_draft_rnn: invalid arguments")
    return dict(tok=tok, lse_q=lse, z_tok=ztok, gap=gap, states=states, arows=arows)


# --------------------------------------------------------------------------- #
# a4 confidence + STS + survival [P2 §置信度头, §校准问题], [P4 §四]            #
# --------------------------------------------------------------------------- #
def confidence_sts(h, emb, anchor, draft_tok, w_c, b_c, T):
    """h [nb,gamma,d], emb [V,e], w_c [d+e], T [gamma] -> conf_raw, conf_cal, log_surv."""
    h = _f64(h); emb = _f64(emb); w_c = _f64(w_c); T = _f64(T)
    anchor = _i32(anchor); draft_tok = _i32(draft_tok)
    nb, gamma, d = h.shape
    e = emb.shape[1]
    assert w_c.shape == (d + e,) and T.shape == (gamma,) and draft_tok.shape == (nb, gamma)
    raw = np.zeros((nb, gamma)); cal = np.zeros((nb, gamma)); ls = np.zeros((nb, gamma))
    _load().oracle_confidence_sts(h, d, emb, e, anchor, draft_tok, w_c, float(b_c), T,
                                  nb, gamma, raw, cal, ls)
    return dict(conf_raw=raw, conf_cal=cal, log_surv=ls)


def sts_survival(score, T_prev, k, grid):
    """Survival of prefix k under each grid temperature, the earlier positions
    at T_prev[:k-1]: [N, G] (oracle_sts_survival; [P2 §校准问题], [P4 §四])."""
    score = _f64(score); grid = _f64(grid)
    N, gamma = score.shape
    T_prev = _f64(np.asarray(T_prev, dtype=np.float64).reshape(-1)[:max(k - 1, 0)])
    T_pad = np.ones(gamma); T_pad[:T_prev.size] = T_prev
    out = np.zeros((N, grid.size))
    _load().oracle_sts_survival(score, N, gamma, np.ascontiguousarray(T_pad), int(k), grid, grid.size, out)
    return out


def sts_fit(score, acc_len, grid, M=15, T_fixed=None):
    """Left-to-right STS fit (oracle_sts_fit; [P2 §校准问题], [P4 §四]).

    score [N, gamma] = logit of the raw confidences, acc_len [N] accepted
    drafts, grid [G] candidate temperatures, M equal-width ECE bins.  With
    T_fixed [gamma] the earlier positions use those temperatures instead of
    the chosen ones.  Returns dict(ece [gamma, G], idx [gamma], T [gamma])."""
    score = _f64(score); acc_len = _i32(acc_len); grid = _f64(grid)
    N, gamma = score.shape
    assert acc_len.shape == (N,) and grid.ndim == 1
    ece = np.zeros((gamma, grid.size)); idx = np.zeros(gamma, np.int32); T = np.zeros(gamma)
    fixed = None if T_fixed is None else _f64(T_fixed)
    rc = _load().oracle_sts_fit(score, acc_len, N, gamma, grid, grid.size, int(M),
                                None if fixed is None else fixed.ctypes.data, ece, idx, T)
    if rc != 0:
        raise ValueError("oracle_sts_fit: bad sizes")
    return dict(ece=ece, idx=idx, T=T)


# --------------------------------------------------------------------------- #
# a5 hardware-aware prefix scheduler [P2 §硬件感知前缀调度器], [P4 §四, §五]     #
# --------------------------------------------------------------------------- #
MODE_OFF, MODE_SYNC, MODE_ASYNC = 0, 1, 2


def schedule(log_surv, sps, mode, log_surv_hist=None):
    """log_surv [B,gamma]; sps[m-1] = SPS(m).  Returns K [B], n_total, theta,
    order (sorted candidate ids b*gamma + j-1) and the Theta curve [B*gamma+1]."""
    ls = _f64(log_surv); sps = _f64(sps)
    B, gamma = ls.shape
    hist = None if log_surv_hist is None else _f64(log_surv_hist)
    K = np.zeros(B, np.int32); nt = np.zeros(1, np.int32); th = np.zeros(1)
    order = np.zeros(B * gamma, np.int32); curve = np.zeros(B * gamma + 1)
    rc = _load().oracle_schedule(ls, None if hist is None else hist.ctypes.data, sps, sps.size,
                                 B, gamma, int(mode), K, nt, th, order, curve)
    if rc != 0:
        raise ValueError("oracle_schedule: invalid arguments")
    return dict(K=K, n_total=int(nt[0]), theta=float(th[0]), order=order, curve=curve)


# --------------------------------------------------------------------------- #
# a6-a8 verification and compaction [P2 §形式化定义], [P4 §四, §五]               #
# --------------------------------------------------------------------------- #
def verify(target, U, W1, W2, anchor, draft_tok, K, *, seed, step=0, tau=1.0, req=None, arows=None):
    """target [nb,gamma+1,V], U [nb,gamma,V]; returns accepted, final_tok,
    p_tok, q_tok and diag [nb,6] (see dspark_oracle.c).  With arows
    [nb,gamma,r] (the RNN head's bias rows) W1 may be None."""
    target = _f64(target); U = _f64(U); W2 = _f64(W2)
    W1 = None if W1 is None else _f64(W1)
    arows = None if arows is None else _f64(arows)
    anchor = _i32(anchor); draft_tok = _i32(draft_tok); K = _i32(K)
    nb, gamma, V = U.shape
    r = W2.shape[0]
    assert (W1 is None or W1.shape == (V, r)) and (arows is None or arows.shape == (nb, gamma, r))
    assert target.shape == (nb, gamma + 1, V) and K.shape == (nb,)
    req = np.arange(nb, dtype=np.int32) if req is None else _i32(req)
    acc = np.zeros(nb, np.int32); fin = np.zeros(nb, np.int32)
    pt = np.full((nb, gamma), np.nan); qt = np.full((nb, gamma), np.nan)
    diag = np.zeros((nb, 6))
    rc = _load().oracle_verify(target, U, None if W1 is None else W1.ctypes.data, W2,
                               None if arows is None else arows.ctypes.data, anchor, draft_tok, K, req, nb, gamma, V, r,
                               float(tau), int(seed), int(step), acc, fin, pt, qt, diag)
    if rc != 0:
        raise ValueError("oracle_verify: invalid arguments")
    return dict(accepted=acc, final_tok=fin, p_tok=pt, q_tok=qt, diag=diag)


def compact(draft_tok, accepted, final_tok):
    draft_tok = _i32(draft_tok); accepted = _i32(accepted); final_tok = _i32(final_tok)
    nb, gamma = draft_tok.shape
    n = int(accepted.sum()) + nb
    tok = np.zeros(n, np.int32); req = np.zeros(n, np.int32); pos = np.zeros(n, np.int32)
    off = np.zeros(nb + 1, np.int32); nxt = np.zeros(nb, np.int32)
    _load().oracle_compact(draft_tok, accepted, final_tok, nb, gamma, tok, req, pos, off, nxt)
    return dict(out_tok=tok, out_req=req, out_pos=pos, out_off=off, next_anchor=nxt)


def step(inp, *, mode, seed, step=0, tau=1.0, log_surv_hist=None):
    """One whole step a1-a8 on a dict of inputs (as produced by the workload
    generator): draft, confidence, schedule, verify, compaction."""
    d = draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], seed=seed, step=step, tau=tau)
    c = confidence_sts(inp["h"], inp["emb"], inp["anchor"], d["tok"], inp["w_c"], inp["b_c"], inp["T"])
    s = schedule(c["log_surv"], inp["sps"], mode, log_surv_hist)
    v = verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], d["tok"], s["K"],
               seed=seed, step=step, tau=tau)
    o = compact(d["tok"], v["accepted"], v["final_tok"])
    return dict(draft=d, conf=c, sched=s, verify=v, out=o)
