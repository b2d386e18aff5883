"""Python binding of libdspark (the C ABI in include/dspark.h).

Argument marshalling only: every function below checks tensor shapes, passes
``data_ptr()`` values and sizes to the C function of the same name, and
raises ``DsparkError`` on a non-OK status.  All arithmetic runs in the CUDA
kernels of the library.  PyTorch provides device memory and streams.

The library must be built first (``python verify_markov_head_gb300/build.py``
or ``__graft_entry__.build()``); importing this package without it raises
ImportError: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import torch


__all__ = [
    "DsparkError", "lib_path", "dspark_version", "dspark_status_string", "dspark_workspace_bytes",
    "dspark_workspace_init", "dspark_workspace_set_wait_limit", "dspark_sync_status", "dspark_draft_markov", "dspark_confidence_sts",
    "dspark_schedule", "dspark_verify", "dspark_draft_markov_target", "target_stream_supported", "dspark_draft_rnn", "dspark_verify_rnn", "dspark_verify_logits", "dspark_rnn_input_table", "rnn_prepare", "dspark_sts_workspace_bytes", "dspark_sts_fit", "dspark_gumbel_stream", "dspark_draft_markov_noalloc", "dspark_noalloc_sync_status", "Workspace", "StepBuffers", "run_step", "run_step_host", "run_step_dp", "GlobalSchedule", "HostPipeline",
    "SCHED_OFF", "SCHED_SYNC", "SCHED_ASYNC",
]

SCHED_OFF, SCHED_SYNC, SCHED_ASYNC = 0, 1, 2
STORE_LOGITS_BYTES = 64 << 20   # StepBuffers keeps the draft logits up to this size
_F32, _BF16 = 0, 1

lib_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libdspark.so")
if not os.path.exists(lib_path):
    raise ImportError(f"libdspark.so is not built ({lib_path}); run verify_markov_head_gb300/build.py")
_lib = C.CDLL(lib_path)

_vp, _i, _f, _u64, _sz = C.c_void_p, C.c_int, C.c_float, C.c_uint64, C.c_size_t
_lib.dspark_version.restype = _i
_lib.dspark_status_string.argtypes = [_i]
_lib.dspark_status_string.restype = C.c_char_p
_lib.dspark_workspace_bytes.argtypes = [_i, _i, _i, _i]
_lib.dspark_workspace_bytes.restype = _sz
_lib.dspark_workspace_init.argtypes = [_vp, _sz, _vp]
_lib.dspark_workspace_init.restype = _i
_lib.dspark_workspace_set_wait_limit.argtypes = [_vp, _sz, _u64, _vp]
_lib.dspark_workspace_set_wait_limit.restype = _i
_lib.dspark_sync_status.argtypes = [_vp, _vp, C.POINTER(C.c_uint32)]
_lib.dspark_sync_status.restype = _i
_lib.dspark_draft_markov.argtypes = [_vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _f, _u64, _u64,
                                     _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_draft_markov.restype = _i
_lib.dspark_draft_markov_target.argtypes = [_vp, _i, _vp, _vp, _i, _vp, _i, _vp, _i, _i, _i, _i, _i, _f, _u64,
                                            _u64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_draft_markov_target.restype = _i
_lib.dspark_confidence_sts.argtypes = [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _f, _vp, _i, _i, _i,
                                       _vp, _vp, _vp, _sz, _vp]
_lib.dspark_confidence_sts.restype = _i
_lib.dspark_schedule.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_schedule.restype = _i
_lib.dspark_verify.argtypes = [_vp, _i, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp,
                               _i, _i, _i, _i, _i, _f, _u64, _u64,
                               _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_verify.restype = _i
_lib.dspark_draft_markov_noalloc.argtypes = [_vp, _i, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _f, _u64, _u64,
                                             _vp, _vp, _vp, _vp, _vp]
_lib.dspark_draft_markov_noalloc.restype = _i
_lib.dspark_noalloc_sync_status.argtypes = [_vp, C.POINTER(C.c_uint32)]
_lib.dspark_noalloc_sync_status.restype = _i
_lib.dspark_draft_rnn.argtypes = [_vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _f,
                                  _u64, _u64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_rnn_input_table.argtypes = [_vp, _vp, _vp, _i, _i, _vp, _vp]
_lib.dspark_rnn_input_table.restype = _i
_lib.dspark_draft_rnn.restype = _i
_lib.dspark_verify_logits.argtypes = [_vp, _i, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _i, _i, _i, _i, _i, _f, _u64, _u64,
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_verify_logits.restype = _i
_lib.dspark_verify_rnn.argtypes = [_vp, _i, _vp, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp,
                                   _i, _i, _i, _i, _i, _f, _u64, _u64,
                                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_verify_rnn.restype = _i
_lib.dspark_sts_workspace_bytes.argtypes = [_i, _i, _i]
_lib.dspark_sts_workspace_bytes.restype = _sz
_lib.dspark_sts_fit.argtypes = [_vp, _vp, _i, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.dspark_sts_fit.restype = _i
_lib.dspark_gumbel_stream.argtypes = [_u64, _u64, C.c_uint32, C.c_uint32, _i, _vp, _vp, _vp]
_lib.dspark_gumbel_stream.restype = _i


class DsparkError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {dspark_status_string(status)} ({status})")


def _check(fn, st):
    if st != 0:
        raise DsparkError(fn, st)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _F32
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def dspark_version() -> int:
    return int(_lib.dspark_version())


def dspark_status_string(status: int) -> str:
    return _lib.dspark_status_string(int(status)).decode()


def dspark_workspace_bytes(B, gamma, V, r) -> int:
    return int(_lib.dspark_workspace_bytes(B, gamma, V, r))


def dspark_workspace_init(ws: torch.Tensor, stream=None):
    _check("dspark_workspace_init", _lib.dspark_workspace_init(_p(ws), ws.numel(), _stream(stream)))


def dspark_workspace_set_wait_limit(ws: torch.Tensor, cycles: int, stream=None):
    """Bound the device waits of calls on this workspace (0: the default)."""
    _check("dspark_workspace_set_wait_limit",
           _lib.dspark_workspace_set_wait_limit(_p(ws), ws.numel(), int(cycles), _stream(stream)))


def dspark_sync_status(ws: torch.Tensor, stream=None):
    """Synchronise the stream; return (status, bits) of the workspace status word."""
    bits = C.c_uint32(0)
    st = _lib.dspark_sync_status(_p(ws), _stream(stream), C.byref(bits))
    return int(st), int(bits.value)


class Workspace:
    """Device scratch for a step of (B, gamma, V, r), cleared once."""

    def __init__(self, B, gamma, V, r, device="cuda", stream=None):
        n = dspark_workspace_bytes(B, gamma, V, r)
        if n == 0:
            raise ValueError("sizes out of range")
        self.tensor = torch.empty(n + 256, dtype=torch.uint8, device=device)
        off = (-self.tensor.data_ptr()) % 256
        self.buf = self.tensor[off:off + n]
        dspark_workspace_init(self.buf, stream)
        # cleared before any stream uses it (side streams do not wait for the
        # stream the clear was issued on)
        torch.cuda.synchronize(self.buf.device)

    def ptr(self):
        return self.buf.data_ptr()

    def nbytes(self):
        return self.buf.numel()


def dspark_draft_markov(U, W1, W2, anchor, draft_tok, lse_q, z_tok, ws: Workspace, *,
                        tau=1.0, seed=0, step=0, req_base=0, logits_out=None, stream=None):
    B, gamma, V = U.shape
    r = W1.shape[1]
    if W1.shape != (V, r) or W2.shape != (r, V) or W1.dtype != W2.dtype:
        raise ValueError("W1 [V,r] and W2 [r,V] must share a dtype")
    for t, shp in ((anchor, (B,)), (draft_tok, (B, gamma)), (lse_q, (B, gamma)), (z_tok, (B, gamma))):
        if tuple(t.shape) != shp:
            raise ValueError(f"shape {tuple(t.shape)} != {shp}")
    _check("dspark_draft_markov", _lib.dspark_draft_markov(
        _p(U), _dt(U), _p(W1), _p(W2), _dt(W1), _p(anchor), B, gamma, V, r, req_base, float(tau),
        int(seed), int(step), _p(draft_tok), _p(lse_q), _p(z_tok), _p(logits_out),
        ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_draft_markov_target(U, W1, W2, target, anchor, draft_tok, lse_q, z_tok, ws: Workspace, *,
                               tau=1.0, seed=0, step=0, req_base=0, logits_out=None, stream=None):
    """dspark_draft_markov that also reduces the target rows of a full-prefix
    verify (dspark_verify / dspark_verify_logits with K=None, same workspace,
    target, seed, step, req_base and tau): rows 0..gamma with a stream kernel
    beside the draft (gamma > 1), else rows 0..gamma-1 in its epilogue."""
    B, gamma, V = U.shape
    r = W1.shape[1]
    if W1.shape != (V, r) or W2.shape != (r, V) or W1.dtype != W2.dtype:
        raise ValueError("W1 [V,r] and W2 [r,V] must share a dtype")
    if tuple(target.shape) != (B, gamma + 1, V):
        raise ValueError("target must be [B, gamma+1, V]")
    for t, shp in ((anchor, (B,)), (draft_tok, (B, gamma)), (lse_q, (B, gamma)), (z_tok, (B, gamma))):
        if tuple(t.shape) != shp:
            raise ValueError(f"shape {tuple(t.shape)} != {shp}")
    _check("dspark_draft_markov_target", _lib.dspark_draft_markov_target(
        _p(U), _dt(U), _p(W1), _p(W2), _dt(W1), _p(target), _dt(target), _p(anchor), B, gamma, V, r, req_base,
        float(tau), int(seed), int(step), _p(draft_tok), _p(lse_q), _p(z_tok), _p(logits_out),
        ws.ptr(), ws.nbytes(), _stream(stream)))


def _target_draft_base(inp: dict) -> bool:
    r = inp["W1"].shape[1]
    return (inp["W1"].dtype == torch.bfloat16 and inp["U"].dtype == torch.float32 and r % 64 == 0
            and r <= 256 and inp["target"].dtype in (torch.float32, torch.bfloat16))


def target_stream_beside(inp: dict) -> bool:
    """Whether dspark_draft_markov_target runs the target stream beside the
    draft on the same SMs (gamma > 1; fp32 or bf16 target): the step's
    fastest form with the scheduler off."""
    return _target_draft_base(inp) and inp["U"].shape[1] > 1


def target_stream_preferred(inp: dict) -> bool:
    """Whether the step with the scheduler off should draft with the target
    stream beside the draft rather than stream the target after it.  Measured
    on one GB300 (graph replay, same outputs): b64 327 -> 301 us, b256 660 ->
    627 us, b512 1319 -> 1325 us (its draft already moves 2 TB/s of U); again
    on the current kernels b256 651 -> 631 us and b512 1316 -> 1331 us, so up
    to 256 requests."""
    return target_stream_beside(inp) and inp["U"].shape[0] <= 256


def target_stream_supported(inp: dict) -> bool:
    """Whether dspark_draft_markov_target takes these inputs: bf16 weights
    with r % 64 == 0 and r <= 256, fp32 U, and a target that is fp32 (or
    bf16 where the stream runs beside the draft)."""
    return _target_draft_base(inp) and (inp["target"].dtype == torch.float32 or target_stream_beside(inp))


def dspark_confidence_sts(h, emb, anchor, draft_tok, w_c, b_c, T, conf_cal, log_surv, ws: Workspace,
                          *, stream=None):
    B, gamma, d = h.shape
    V, e = emb.shape
    if w_c.numel() != d + e or T.numel() != gamma:
        raise ValueError("w_c must hold d+e weights and T gamma temperatures")
    _check("dspark_confidence_sts", _lib.dspark_confidence_sts(
        _p(h), d, _p(emb), _dt(emb), e, _p(anchor), _p(draft_tok), _p(w_c), float(b_c), _p(T),
        B, gamma, V, _p(conf_cal), _p(log_surv), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_sts_workspace_bytes(gamma, G, M) -> int:
    return int(_lib.dspark_sts_workspace_bytes(gamma, G, M))


def dspark_sts_fit(score, acc_len, grid, *, M=15, T_out=None, idx_out=None, ece_out=None, ws=None,
                   stream=None):
    """Left-to-right STS temperature fit on the device: score [N, gamma] fp32,
    acc_len [N] int32, grid [G] fp32.  Returns (T [gamma] fp32, idx [gamma]
    int32, ece [gamma, G] fp64); outputs and the workspace (a uint8 tensor)
    are allocated on score's device when not given."""
    N, gamma = score.shape
    G = grid.numel()
    if score.dtype != torch.float32 or grid.dtype != torch.float32 or acc_len.dtype != torch.int32:
        raise TypeError("score and grid must be float32, acc_len int32")
    if acc_len.numel() != N:
        raise ValueError("acc_len must hold one length per block")
    dev = score.device
    nbytes = dspark_sts_workspace_bytes(gamma, G, M)
    if nbytes == 0:
        raise ValueError("gamma, grid size or bin count out of range")
    T_out = torch.empty(gamma, dtype=torch.float32, device=dev) if T_out is None else T_out
    idx_out = torch.empty(gamma, dtype=torch.int32, device=dev) if idx_out is None else idx_out
    ece_out = torch.empty(gamma, G, dtype=torch.float64, device=dev) if ece_out is None else ece_out
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev) if ws is None else ws
    if T_out.numel() != gamma or idx_out.numel() != gamma or ece_out.numel() != gamma * G:
        raise ValueError("output buffers have the wrong size")
    _check("dspark_sts_fit", _lib.dspark_sts_fit(
        _p(score), _p(acc_len), N, gamma, _p(grid), G, int(M), _p(T_out), _p(idx_out), _p(ece_out),
        _p(ws), ws.numel(), _stream(stream)))
    return T_out, idx_out, ece_out


def dspark_schedule(log_surv, sps, mode, K, n_total, theta, ws: Workspace, *, log_surv_hist=None,
                    stream=None):
    B, gamma = log_surv.shape
    _check("dspark_schedule", _lib.dspark_schedule(
        _p(log_surv), _p(log_surv_hist), _p(sps), sps.numel(), B, gamma, int(mode), _p(K), _p(n_total),
        _p(theta), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_verify(target, U, W1, W2, anchor, draft_tok, lse_q, z_tok, K, accepted, out_tok, out_req,
                  out_pos, out_off, next_anchor, ws: Workspace, *, tau=1.0, seed=0, step=0, req_base=0,
                  p_tok=None, near_ties=None, stream=None):
    B, gamma, V = U.shape
    r = W1.shape[1]
    if tuple(target.shape) != (B, gamma + 1, V):
        raise ValueError("target must be [B, gamma+1, V]")
    if out_tok.numel() < B * (gamma + 1) or out_off.numel() != B + 1:
        raise ValueError("output buffers too small")
    _check("dspark_verify", _lib.dspark_verify(
        _p(target), _dt(target), _p(U), _dt(U), _p(W1), _p(W2), _dt(W1), _p(anchor), _p(draft_tok),
        _p(lse_q), _p(z_tok), _p(K), B, gamma, V, r, req_base, float(tau), int(seed), int(step),
        _p(accepted), _p(out_tok), _p(out_req), _p(out_pos), _p(out_off), _p(next_anchor),
        _p(p_tok), _p(near_ties), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_rnn_input_table(E, W_ih, b_ih, P=None, *, stream=None):
    """The RNN head's per-token input projections P = E W_ih^T + b_ih
    ([V, 3r] fp32), computed on the device once per set of weights."""
    V, r = E.shape
    if tuple(W_ih.shape) != (3 * r, r) or b_ih.numel() != 3 * r:
        raise ValueError("W_ih [3r, r] and b_ih [3r] expected")
    if E.dtype != torch.bfloat16 or W_ih.dtype != torch.bfloat16 or b_ih.dtype != torch.float32:
        raise TypeError("E and W_ih must be bfloat16, b_ih float32")
    P = torch.empty((V, 3 * r), dtype=torch.float32, device=E.device) if P is None else P
    _check("dspark_rnn_input_table", _lib.dspark_rnn_input_table(_p(E), _p(W_ih), _p(b_ih), V, r, _p(P),
                                                                 _stream(stream)))
    return P


def rnn_prepare(rnn: dict, *, stream=None) -> dict:
    """The RNN head's parameters with the input table P added (from E, W_ih
    and b_ih); returns the same dict."""
    if "P" not in rnn:
        rnn["P"] = dspark_rnn_input_table(rnn["E"], rnn["W_ih"], rnn["b_ih"], stream=stream)
    return rnn


def dspark_draft_rnn(U, rnn, W2, anchor, draft_tok, lse_q, z_tok, state, ws: Workspace, *,
                     tau=1.0, seed=0, step=0, req_base=0, stream=None):
    """The draft loop with the RNN head.  rnn = dict(P [V,3r] fp32 (see
    rnn_prepare), W_hh [3r,r] bf16, b_hh [3r], s0 [r] fp32); state
    [gamma,B,r] fp32 receives the states s_1..s_gamma."""
    B, gamma, V = U.shape
    r = W2.shape[0]
    if "P" not in rnn:
        raise ValueError("the RNN head needs its input table: call rnn_prepare first")
    P, W_hh = rnn["P"], rnn["W_hh"]
    if tuple(P.shape) != (V, 3 * r) or P.dtype != torch.float32 or tuple(W_hh.shape) != (3 * r, r):
        raise ValueError("P [V,3r] float32 and W_hh [3r,r] expected")
    if not (W_hh.dtype == W2.dtype == torch.bfloat16):
        raise TypeError("W_hh and W2 must be bfloat16")
    if rnn["b_hh"].numel() != 3 * r or rnn["s0"].numel() != r:
        raise ValueError("b_hh [3r] and s0 [r] expected")
    if tuple(state.shape) != (gamma, B, r) or state.dtype != torch.float32:
        raise ValueError("state must be float32 [gamma, B, r]")
    _check("dspark_draft_rnn", _lib.dspark_draft_rnn(
        _p(U), _dt(U), _p(P), _p(W_hh), _p(rnn["b_hh"]), _p(rnn["s0"]), _p(W2), _dt(W2), _p(anchor),
        B, gamma, V, r, req_base, float(tau), int(seed), int(step), _p(draft_tok), _p(lse_q), _p(z_tok),
        _p(state), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_verify_logits(target, U, W1, W2, draft_logits, anchor, draft_tok, lse_q, z_tok, K, accepted, out_tok,
                         out_req, out_pos, out_off, next_anchor, ws: Workspace, *, tau=1.0, seed=0, step=0,
                         req_base=0, p_tok=None, near_ties=None, stream=None):
    """dspark_verify reading rejected rows from the draft's stored logits
    draft_logits [B, gamma, V] (the draft's logits_out)."""
    B, gamma, V = U.shape
    r = W1.shape[1]
    if tuple(target.shape) != (B, gamma + 1, V) or tuple(draft_logits.shape) != (B, gamma, V):
        raise ValueError("target must be [B, gamma+1, V] and draft_logits [B, gamma, V]")
    if out_tok.numel() < B * (gamma + 1) or out_off.numel() != B + 1:
        raise ValueError("output buffers too small")
    _check("dspark_verify_logits", _lib.dspark_verify_logits(
        _p(target), _dt(target), _p(U), _dt(U), _p(W1), _p(W2), _dt(W1), _p(draft_logits), _p(anchor),
        _p(draft_tok), _p(lse_q), _p(z_tok), _p(K), B, gamma, V, r, req_base, float(tau), int(seed), int(step),
        _p(accepted), _p(out_tok), _p(out_req), _p(out_pos), _p(out_off), _p(next_anchor),
        _p(p_tok), _p(near_ties), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_verify_rnn(target, U, state, W2, anchor, draft_tok, lse_q, z_tok, K, accepted, out_tok, out_req,
                      out_pos, out_off, next_anchor, ws: Workspace, *, tau=1.0, seed=0, step=0, req_base=0,
                      p_tok=None, near_ties=None, stream=None):
    B, gamma, V = U.shape
    r = W2.shape[0]
    if tuple(target.shape) != (B, gamma + 1, V) or tuple(state.shape) != (gamma, B, r):
        raise ValueError("target must be [B, gamma+1, V] and state [gamma, B, r]")
    if out_tok.numel() < B * (gamma + 1) or out_off.numel() != B + 1:
        raise ValueError("output buffers too small")
    _check("dspark_verify_rnn", _lib.dspark_verify_rnn(
        _p(target), _dt(target), _p(U), _dt(U), _p(state), _p(W2), _dt(W2), _p(anchor), _p(draft_tok),
        _p(lse_q), _p(z_tok), _p(K), B, gamma, V, r, req_base, float(tau), int(seed), int(step),
        _p(accepted), _p(out_tok), _p(out_req), _p(out_pos), _p(out_off), _p(next_anchor),
        _p(p_tok), _p(near_ties), ws.ptr(), ws.nbytes(), _stream(stream)))


def dspark_draft_markov_noalloc(U, W1, W2, anchor, draft_tok, lse_q, z_tok, *, tau=1.0, seed=0, step=0,
                                req_base=0, logits_out=None, stream=None):
    """dspark_draft_markov without a workspace, for callers that cannot
    allocate device memory: the library keeps the scratch in a fixed array."""
    B, gamma, V = U.shape
    r = W1.shape[1]
    if W1.shape != (V, r) or W2.shape != (r, V) or W1.dtype != W2.dtype:
        raise ValueError("W1 [V,r] and W2 [r,V] must share a dtype")
    _check("dspark_draft_markov_noalloc", _lib.dspark_draft_markov_noalloc(
        _p(U), _dt(U), _p(W1), _p(W2), _dt(W1), _p(anchor), B, gamma, V, r, req_base, float(tau),
        int(seed), int(step), _p(draft_tok), _p(lse_q), _p(z_tok), _p(logits_out), _stream(stream)))


def dspark_noalloc_sync_status(stream=None):
    """Synchronise the stream; return (status, bits) of the fixed array's
    status word (the scratch of dspark_draft_markov_noalloc)."""
    bits = C.c_uint32(0)
    st = _lib.dspark_noalloc_sync_status(_stream(stream), C.byref(bits))
    return int(st), int(bits.value)


def dspark_gumbel_stream(seed, step, domain, row, n, gumbel_out=None, uniform_out=None, stream=None):
    _check("dspark_gumbel_stream", _lib.dspark_gumbel_stream(
        int(seed), int(step), int(domain), int(row), int(n), _p(gumbel_out), _p(uniform_out), _stream(stream)))


class StepBuffers:
    """Device outputs of one step for B requests of block length gamma."""

    def __init__(self, B, gamma, V, r, device="cuda"):
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.B, self.gamma = B, gamma
        self.draft_tok = torch.empty((B, gamma), **i32)
        self.lse_q = torch.empty((B, gamma), **f32)
        self.z_tok = torch.empty((B, gamma), **f32)
        self.conf_cal = torch.empty((B, gamma), **f32)
        self.log_surv = torch.empty((B, gamma), **f32)
        self.K = torch.empty((B,), **i32)
        self.n_total = torch.empty((1,), **i32)
        self.theta = torch.empty((1,), **f32)
        self.accepted = torch.empty((B,), **i32)
        self.out_tok = torch.empty((B * (gamma + 1),), **i32)
        self.out_req = torch.empty((B * (gamma + 1),), **i32)
        self.out_pos = torch.empty((B * (gamma + 1),), **i32)
        self.out_off = torch.empty((B + 1,), **i32)
        self.next_anchor = torch.empty((B,), **i32)
        self.p_tok = torch.empty((B, gamma), **f32)
        self.near_ties = torch.zeros((4,), dtype=torch.int32, device=device)
        self.state = torch.empty((gamma, B, r), **f32)    # RNN head states s_1..s_gamma
        # the draft's logits, kept when small enough: the residual draw then
        # reads the rejected row instead of rebuilding it (the latency path)
        self.logits = (torch.empty((B, gamma, V), **f32) if B * gamma * V * 4 <= STORE_LOGITS_BYTES else None)
        self.ws = Workspace(B, gamma, V, r, device)
        # scheduler off: the verify lengths are gamma for every request, and
        # the confidence head and the scheduler run beside the verify on a
        # side stream (nothing the verify reads depends on them)
        self.K_full = torch.full((B,), gamma, **i32)
        self.verify_items = B * (gamma + 1) * -(-V // 32768)     # verify-stream work items (32768-entry segments)
        self.sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.side = torch.cuda.Stream(device=device)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()


def run_step(inp: dict, buf: StepBuffers, *, mode, seed, step=0, tau=1.0, req_base=0, log_surv_hist=None,
         stream=None, p_tok=False, head="markov", fuse_target=None):
    """One whole draft + verify step (a1-a8) on device-resident inputs: the
    four ABI calls in order, all on `stream`.  head="rnn" drafts with the RNN
    head (parameters in inp["rnn"]) and verifies against its states.  With
    the scheduler off (every K_b = gamma) and fuse_target, the Markov draft
    also reduces the target rows it drafts against
    (dspark_draft_markov_target) and the verify runs in full-prefix mode.
    fuse_target=None takes that path where the stream runs beside the draft
    and pays (target_stream_preferred), else the separate verify stream."""
    if fuse_target is None:
        fuse_target = target_stream_preferred(inp)
    fused = fuse_target and head == "markov" and int(mode) == 0 and target_stream_supported(inp)
    if head == "rnn":
        dspark_draft_rnn(inp["U"], inp["rnn"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                         buf.state, buf.ws, tau=tau, seed=seed, step=step, req_base=req_base, stream=stream)
    elif fused:
        dspark_draft_markov_target(inp["U"], inp["W1"], inp["W2"], inp["target"], inp["anchor"], buf.draft_tok,
                                   buf.lse_q, buf.z_tok, buf.ws, tau=tau, seed=seed, step=step, req_base=req_base,
                                   logits_out=buf.logits, stream=stream)
    elif head == "markov":
        dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                            buf.ws, tau=tau, seed=seed, step=step, req_base=req_base, logits_out=buf.logits,
                            stream=stream)
    else:
        raise ValueError(f"unknown head {head!r}")
    main = stream if stream is not None else torch.cuda.current_stream()
    # confidence and scheduler off the verify's critical path: with the
    # scheduler off nothing the verify reads depends on them, and a verify
    # stream too small to fill the GPU leaves SMs for them to run beside it
    # (a full one holds every SM's registers, and they would only run later;
    # in full-prefix mode no stream runs in the verify at all)
    side = int(mode) == 0 and (fused or buf.verify_items < 2 * buf.sms)
    if side:
        buf.fork.record(main)
        buf.side.wait_event(buf.fork)
    conf_stream = buf.side if side else stream
    dspark_confidence_sts(inp["h"], inp["emb"], inp["anchor"], buf.draft_tok, inp["w_c"], inp["b_c"], inp["T"],
                          buf.conf_cal, buf.log_surv, buf.ws, stream=conf_stream)
    dspark_schedule(buf.log_surv, inp["sps"], mode, buf.K, buf.n_total, buf.theta, buf.ws,
                    log_surv_hist=log_surv_hist, stream=conf_stream)
    if side:
        buf.join.record(buf.side)
    # full-prefix mode: rows 0..gamma-1 already reduced by the draft (K = None);
    # scheduler off: K_b = gamma from the constant buffer
    K = None if fused else (buf.K_full if side else buf.K)
    if head == "rnn":
        dspark_verify_rnn(inp["target"], inp["U"], buf.state, inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                          buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                          buf.next_anchor, buf.ws, tau=tau, seed=seed, step=step, req_base=req_base,
                          p_tok=buf.p_tok if p_tok else None, near_ties=buf.near_ties, stream=stream)
    elif buf.logits is not None:
        dspark_verify_logits(inp["target"], inp["U"], inp["W1"], inp["W2"], buf.logits, inp["anchor"],
                             buf.draft_tok, buf.lse_q, buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req,
                             buf.out_pos, buf.out_off, buf.next_anchor, buf.ws, tau=tau, seed=seed, step=step,
                             req_base=req_base, p_tok=buf.p_tok if p_tok else None, near_ties=buf.near_ties,
                             stream=stream)
    else:
        dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                      buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                      buf.next_anchor, buf.ws, tau=tau, seed=seed, step=step, req_base=req_base,
                      p_tok=buf.p_tok if p_tok else None, near_ties=buf.near_ties, stream=stream)
    if side:
        main.wait_event(buf.join)      # the step ends when both streams have


class GlobalSchedule:
    """Device buffers of the scheduler over the survival lists of `world`
    ranks of B requests each (see run_step_dp)."""

    def __init__(self, B, gamma, world, device="cuda"):
        Bg = B * world
        f32 = dict(dtype=torch.float32, device=device)
        self.log_surv = torch.empty((Bg, gamma), **f32)
        self.hist = torch.empty((Bg, gamma), **f32)
        self.K = torch.empty((Bg,), dtype=torch.int32, device=device)
        self.n_total = torch.empty((1,), dtype=torch.int32, device=device)
        self.theta = torch.empty((1,), **f32)
        # the scheduler's scratch depends on the list length only: the
        # smallest vocabulary and rank the workspace sizing accepts
        self.ws = Workspace(Bg, gamma, 8, 1, device)


def run_step_dp(inp: dict, buf: StepBuffers, sched: GlobalSchedule, *, mode, seed, step=0, tau=1.0,
                log_surv_hist=None, group=None, stream=None, p_tok=False):
    """One step on this rank's block of a batch sharded over the ranks of
    `group`: rank r owns global requests [r*B, (r+1)*B) and draws their
    random streams.  With the scheduler on, the survival lists (and the
    history, in async mode) are all-gathered and every rank runs the device
    scheduler on the whole list, then verifies its own block with its share
    of the verify lengths; inp["sps"] must cover the global batch.  With the
    scheduler off no data crosses ranks."""
    import torch.distributed as dist

    from . import shard

    rank = dist.get_rank(group)
    B = buf.B
    req_base = rank * B
    dspark_draft_markov(inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q, buf.z_tok,
                        buf.ws, tau=tau, seed=seed, step=step, req_base=req_base, stream=stream)
    dspark_confidence_sts(inp["h"], inp["emb"], inp["anchor"], buf.draft_tok, inp["w_c"], inp["b_c"], inp["T"],
                          buf.conf_cal, buf.log_surv, buf.ws, stream=stream)
    if int(mode) == 0:
        dspark_schedule(buf.log_surv, inp["sps"], 0, buf.K, buf.n_total, buf.theta, buf.ws, stream=stream)
        K = buf.K
    else:
        def device_schedule(all_surv, all_hist):
            dspark_schedule(all_surv, inp["sps"], mode, sched.K, sched.n_total, sched.theta, sched.ws,
                            log_surv_hist=all_hist, stream=stream)
            return sched.K, sched.n_total, sched.theta

        # the gather and the copies are ordered on the step's stream
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream()):
            K, _, _, _ = shard.global_schedule(buf.log_surv, log_surv_hist, device_schedule, group,
                                               surv_out=sched.log_surv, hist_out=sched.hist)
            buf.K.copy_(K)
            buf.n_total.copy_(sched.n_total)
            buf.theta.copy_(sched.theta)
    dspark_verify(inp["target"], inp["U"], inp["W1"], inp["W2"], inp["anchor"], buf.draft_tok, buf.lse_q,
                  buf.z_tok, K, buf.accepted, buf.out_tok, buf.out_req, buf.out_pos, buf.out_off,
                  buf.next_anchor, buf.ws, tau=tau, seed=seed, step=step, req_base=req_base,
                  p_tok=buf.p_tok if p_tok else None, near_ties=buf.near_ties, stream=stream)
    return K


_PER_STEP = ("U", "target", "h", "anchor")


def run_step_host(host_inp: dict, dev_inp: dict, buf: StepBuffers, host_out: dict, *, mode, seed, step=0,
              tau=1.0, stream=None):
    """End-to-end step from host memory: copies the step's activations
    (U, target logits, hidden states, anchors) from pinned host tensors into
    the device inputs, runs the step, and copies the emitted tokens, offsets
    and next anchors back.  Returns (h2d_bytes, d2h_bytes)."""
    h2d = 0
    for k in _PER_STEP:
        dev_inp[k].copy_(host_inp[k], non_blocking=True)
        h2d += host_inp[k].numel() * host_inp[k].element_size()
    run_step(dev_inp, buf, mode=mode, seed=seed, step=step, tau=tau, stream=stream)
    d2h = 0
    for name in ("out_tok", "out_off", "next_anchor"):
        src = getattr(buf, name)
        host_out[name].copy_(src, non_blocking=True)
        d2h += src.numel() * src.element_size()
    return h2d, d2h


class HostPipeline:
    """Steps from pinned host memory with the copy of the next step's inputs
    overlapping the current step's compute.

    Two device copies of the per-step inputs (U, target logits, hidden
    states, anchors) alternate: step t computes from slot t % 2 on the
    compute stream while the copy stream fills slot (t + 1) % 2, which the
    step before last has finished reading.  Each step's emitted tokens,
    offsets and next anchors are copied back to the pinned `host_out`
    tensors on the compute stream.  The weights and every other device input
    are shared by both slots."""

    def __init__(self, dev_inp: dict, buf: StepBuffers, compute_stream, copy_stream=None):
        dev = dev_inp["U"].device
        second = dict(dev_inp)
        for k in _PER_STEP:
            second[k] = torch.empty_like(dev_inp[k])
        self.slots = [dev_inp, second]
        self.buf = buf
        self.compute_stream = compute_stream
        self.copy_stream = copy_stream if copy_stream is not None else torch.cuda.Stream(device=dev)
        self.copied = [torch.cuda.Event(), torch.cuda.Event()]
        self.consumed = [torch.cuda.Event(), torch.cuda.Event()]
        self.used = [False, False]
        self.next = 0
        # the weights, buffers and second slot were made on the current stream
        cur = torch.cuda.current_stream(dev)
        self.compute_stream.wait_stream(cur)
        self.copy_stream.wait_stream(cur)

    def step(self, host_inp: dict, host_out: dict, *, mode, seed, step=0, tau=1.0, head="markov",
             fuse_target=None):
        """Enqueue one step; returns (h2d_bytes, d2h_bytes)."""
        i = self.next
        slot = self.slots[i]
        if self.used[i]:
            self.copy_stream.wait_event(self.consumed[i])     # the step that last read slot i is done
        h2d = 0
        with torch.cuda.stream(self.copy_stream):
            for k in _PER_STEP:
                slot[k].copy_(host_inp[k], non_blocking=True)
                h2d += host_inp[k].numel() * host_inp[k].element_size()
        self.copied[i].record(self.copy_stream)
        self.compute_stream.wait_event(self.copied[i])
        d2h = 0
        with torch.cuda.stream(self.compute_stream):
            run_step(slot, self.buf, mode=mode, seed=seed, step=step, tau=tau, stream=self.compute_stream,
                     head=head, fuse_target=fuse_target)
            for name in ("out_tok", "out_off", "next_anchor"):
                src = getattr(self.buf, name)
                host_out[name].copy_(src, non_blocking=True)
                d2h += src.numel() * src.element_size()
        self.consumed[i].record(self.compute_stream)
        self.used[i] = True
        self.next = i ^ 1
        return h2d, d2h
