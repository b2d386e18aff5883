// api.cu -- the C ABI declared in include/dspark.h: host-side argument
// checks, workspace layout and the launch sequence of each call.
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {

// One NVTX range per ABI call (named after the call), for timeline tools; a
// push and a pop of a few nanoseconds when no tool is attached.
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
};

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(int B, int gamma, int V) {
    WsLayout L;
    L.nseg = (V + kVerifySeg - 1) / kVerifySeg;
    const int ntiles = (V + kPartTile - 1) / kPartTile;
    L.parts = ntiles < kMaxParts ? ntiles : kMaxParts;
    const WsDraftPrefix P = ws_draft_prefix(B, gamma, L.parts);
    L.status = P.status; L.tickets = P.tickets; L.gbar = P.gbar; L.win = P.win; L.vq = P.vq;
    L.draft_part = P.draft_part;
    size_t o = P.end;
    L.verify_part = o; o = align256(o + sizeof(LseDraw) * (size_t)B * (gamma + 1) * L.nseg * kVerifySub);
    L.tgt_part = o;    o = align256(o + sizeof(LseDraw) * (size_t)B * gamma * kTgtSlots);
    L.tgt_token = o;   o = align256(o + sizeof(unsigned long long));
    L.rej = o;         o = align256(o + sizeof(int32_t) * (size_t)B);
    L.acc = o;         o = align256(o + sizeof(int32_t) * (size_t)B);
    L.fin = o;         o = align256(o + sizeof(int32_t) * (size_t)B);
    L.lse_rej = o;     o = align256(o + sizeof(float2) * (size_t)B);
    L.resid_part = o;  o = align256(o + sizeof(Draw2) * (size_t)B * L.parts);
    L.conf = o;        o = align256(o + sizeof(uint32_t) * (size_t)B + sizeof(float) * (size_t)B * gamma);
    L.rnn_gh = o;      o = align256(o + sizeof(float) * (size_t)B * 3 * kMaxRnnRank);
    L.bonus_tickets = o; o = align256(o + sizeof(uint32_t) * (size_t)B);
    L.row_lse = o;     o = align256(o + sizeof(float) * (size_t)B * (gamma + 1));
    L.row_tickets = o; o = align256(o + sizeof(uint32_t) * (size_t)B * (gamma + 1));
    L.rtok = o;        o = align256(o + sizeof(int32_t) * (size_t)B);
    L.total = o;
    return L;
}

WsPtrs ws_ptrs(void* ws, int B, int gamma, int V) {
    const WsLayout L = ws_layout(B, gamma, V);
    char* base = static_cast<char*>(ws);
    WsPtrs P;
    P.status = reinterpret_cast<uint32_t*>(base + L.status);
    P.wait_limit = reinterpret_cast<unsigned long long*>(base + L.status + 8);
    P.tickets_draft = reinterpret_cast<uint32_t*>(base + L.tickets);
    P.tickets_resid = P.tickets_draft + ((size_t)B + kChunk - 1) / kChunk;
    P.gbar = reinterpret_cast<uint32_t*>(base + L.gbar);
    P.win = reinterpret_cast<unsigned long long*>(base + L.win);
    P.vq = reinterpret_cast<uint32_t*>(base + L.vq);
    P.draft_part = reinterpret_cast<DrawLse*>(base + L.draft_part);
    P.verify_part = reinterpret_cast<LseDraw*>(base + L.verify_part);
    P.tgt_part = reinterpret_cast<LseDraw*>(base + L.tgt_part);
    P.tgt_token = reinterpret_cast<unsigned long long*>(base + L.tgt_token);
    P.rej = reinterpret_cast<int32_t*>(base + L.rej);
    P.acc = reinterpret_cast<int32_t*>(base + L.acc);
    P.fin = reinterpret_cast<int32_t*>(base + L.fin);
    P.lse_rej = reinterpret_cast<float2*>(base + L.lse_rej);
    P.resid_part = reinterpret_cast<Draw2*>(base + L.resid_part);
    P.conf_tickets = reinterpret_cast<uint32_t*>(base + L.conf);
    P.conf_score = reinterpret_cast<float*>(base + L.conf + sizeof(uint32_t) * (size_t)B);
    P.rnn_gh = reinterpret_cast<float*>(base + L.rnn_gh);
    P.bonus_tickets = reinterpret_cast<uint32_t*>(base + L.bonus_tickets);
    P.row_lse = reinterpret_cast<float*>(base + L.row_lse);
    P.row_tickets = reinterpret_cast<uint32_t*>(base + L.row_tickets);
    P.rtok = reinterpret_cast<int32_t*>(base + L.rtok);
    P.nseg = L.nseg;
    P.parts = L.parts;
    return P;
}

// A pointer the device can dereference: device memory or managed memory.
bool is_device_ptr(const void* p) {
    if (!p) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) { cudaGetLastError(); return false; }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dspark_status launch_status(cudaError_t e) {
    if (e == cudaSuccess) return DSPARK_OK;
    fprintf(stderr, "dspark: launch failed: %s\n", cudaGetErrorString(e));
    return DSPARK_ERR_CUDA;
}

bool sizes_ok(int B, int gamma, int V, int r) {
    if (B < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 8 || (V % 8) != 0 || r < 1 || r > 1024)
        return false;
    if ((double)B * (gamma + 1) >= 4294967295.0) return false;
    if (B > 1000000) return false;
    return true;
}

// Identifies the inputs of a target-stream draft: the verify call in
// full-prefix mode recomputes it and checks the one the draft left in the
// workspace.  Odd, so a cleared workspace never matches.
static unsigned long long tgt_token_of(const void* target, uint64_t seed, uint64_t step, int req_base, int B,
                                       int gamma, int V, float tau) {
    uint32_t tau_bits;
    memcpy(&tau_bits, &tau, sizeof(tau_bits));
    const uint64_t words[] = {(uint64_t)reinterpret_cast<uintptr_t>(target), seed, step, (uint64_t)(uint32_t)req_base,
                              ((uint64_t)(uint32_t)B << 32) | (uint32_t)gamma, ((uint64_t)(uint32_t)V << 32) | tau_bits};
    uint64_t h = 0x6a09e667f3bcc909ull;
    for (uint64_t w : words) {
        h ^= w + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
        h = (h ^ (h >> 30)) * 0xbf58476d1ce4e5b9ull;
        h = (h ^ (h >> 27)) * 0x94d049bb133111ebull;
        h ^= h >> 31;
    }
    return h | 1ull;
}

dspark_status read_status_word(void* word, cudaStream_t s, uint32_t* bits) {
    uint32_t host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        fprintf(stderr, "dspark: %s\n", cudaGetErrorString(e));
        return DSPARK_ERR_CUDA;
    }
    if (host) {
        e = cudaMemsetAsync(word, 0, sizeof(uint32_t), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (bits) *bits = host;
    if (host & kTimeout) return DSPARK_ERR_TIMEOUT;
    if (host) return DSPARK_ERR_DEVICE;
    return DSPARK_OK;
}

__global__ void set_u64_kernel(unsigned long long* dst, unsigned long long v) { *dst = v; }

}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_version(void) { return 100; }

const char* dspark_status_string(dspark_status s) {
    switch (s) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_INVALID: return "invalid argument";
        case DSPARK_ERR_CUDA: return "CUDA error";
        case DSPARK_ERR_TIMEOUT: return "device wait timed out";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported configuration";
        case DSPARK_ERR_DEVICE: return "device-side range check fired";
    }
    return "unknown status";
}

size_t dspark_workspace_bytes(int B, int gamma, int V, int r) {
    if (!sizes_ok(B, gamma, V, r)) return 0;
    return ws_layout(B, gamma, V).total;
}

dspark_status dspark_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!is_device_ptr(ws) || ws_bytes < 256) return DSPARK_ERR_INVALID;
    return launch_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t cycles, void* stream) {
    if (!is_device_ptr(ws) || ws_bytes < 256) return DSPARK_ERR_INVALID;
    unsigned long long* dst = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + 8);
    set_u64_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(dst, (unsigned long long)cycles);
    return launch_status(cudaGetLastError());
}

dspark_status dspark_sync_status(void* ws, void* stream, uint32_t* bits) {
    if (!is_device_ptr(ws)) return DSPARK_ERR_INVALID;
    return read_status_word(ws, static_cast<cudaStream_t>(stream), bits);
}

dspark_status dspark_draft_markov(const void* U, dspark_dtype U_t, const void* W1, const void* W2,
                                  dspark_dtype W_t, const int32_t* anchor, int B, int gamma, int V,
                                  int r, int req_base, float tau, uint64_t seed, uint64_t step,
                                  int32_t* draft_tok, float* lse_q, float* z_tok, float* logits_out,
                                  void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (!sizes_ok(B, gamma, V, r) || !(tau > 0.f) || req_base < 0) return DSPARK_ERR_INVALID;
    if ((U_t != DSPARK_F32 && U_t != DSPARK_BF16) || (W_t != DSPARK_F32 && W_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    if (!is_device_ptr(U) || !is_device_ptr(W1) || !is_device_ptr(W2) || !is_device_ptr(anchor) ||
        !is_device_ptr(draft_tok) || !is_device_ptr(lse_q) || !is_device_ptr(z_tok) || !is_device_ptr(ws))
        return DSPARK_ERR_INVALID;
    if (logits_out && (!is_device_ptr(logits_out) || !aligned(logits_out, 16))) return DSPARK_ERR_INVALID;
    if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(ws, 256)) return DSPARK_ERR_INVALID;
    if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;

    DraftParams p;
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = W1; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau;
    p.seed = seed; p.step = step;
    p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.logits_out = logits_out;
    p.ws = ws_ptrs(ws, B, gamma, V);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return launch_status(launch_draft(p, s));
}

dspark_status dspark_draft_markov_target(const void* U, dspark_dtype U_t, const void* W1, const void* W2,
                                         dspark_dtype W_t, const void* target, dspark_dtype target_t,
                                         const int32_t* anchor, int B, int gamma, int V, int r, int req_base,
                                         float tau, uint64_t seed, uint64_t step, int32_t* draft_tok, float* lse_q,
                                         float* z_tok, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (!sizes_ok(B, gamma, V, r) || !(tau > 0.f) || req_base < 0) return DSPARK_ERR_INVALID;
    if ((U_t != DSPARK_F32 && U_t != DSPARK_BF16) || (W_t != DSPARK_F32 && W_t != DSPARK_BF16) ||
        (target_t != DSPARK_F32 && target_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    if (!is_device_ptr(U) || !is_device_ptr(W1) || !is_device_ptr(W2) || !is_device_ptr(target) ||
        !is_device_ptr(anchor) || !is_device_ptr(draft_tok) || !is_device_ptr(lse_q) || !is_device_ptr(z_tok) ||
        !is_device_ptr(ws))
        return DSPARK_ERR_INVALID;
    if (logits_out && (!is_device_ptr(logits_out) || !aligned(logits_out, 16))) return DSPARK_ERR_INVALID;
    if (!aligned(U, 16) || !aligned(W1, 16) || !aligned(W2, 16) || !aligned(target, 16) || !aligned(ws, 256))
        return DSPARK_ERR_INVALID;
    if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;

    DraftParams p;
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = W1; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau;
    p.seed = seed; p.step = step;
    p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.logits_out = logits_out;
    p.ws = ws_ptrs(ws, B, gamma, V);
    p.target = static_cast<const float*>(target);
    p.target_bf16 = (target_t == DSPARK_BF16);
    p.tgt_token = tgt_token_of(target, seed, step, req_base, B, gamma, V, tau);
    if (!draft_target_vs(p) && (p.target_bf16 || !draft_target_supported(p))) return DSPARK_ERR_UNSUPPORTED;
    return launch_status(launch_draft_target(p, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_confidence_sts(const float* h, int d, const void* emb, dspark_dtype emb_t, int e,
                                    const int32_t* anchor, const int32_t* draft_tok, const float* w_c,
                                    float b_c, const float* T, int B, int gamma, int V, float* conf_cal,
                                    float* log_surv, void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (B < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || d < 1 || e < 1 || V < 1) return DSPARK_ERR_INVALID;
    if (emb_t != DSPARK_F32 && emb_t != DSPARK_BF16) return DSPARK_ERR_UNSUPPORTED;
    if (!is_device_ptr(h) || !is_device_ptr(emb) || !is_device_ptr(anchor) || !is_device_ptr(draft_tok) ||
        !is_device_ptr(w_c) || !is_device_ptr(T) || !is_device_ptr(conf_cal) || !is_device_ptr(log_surv) ||
        !is_device_ptr(ws))
        return DSPARK_ERR_INVALID;
    if (!aligned(h, 16) || !aligned(emb, 16) || !aligned(w_c, 16) || !aligned(ws, 256)) return DSPARK_ERR_INVALID;
    if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_INVALID;
    ConfParams p;
    p.h = h; p.d = d; p.emb = emb; p.emb_bf16 = (emb_t == DSPARK_BF16); p.e = e;
    p.anchor = anchor; p.draft_tok = draft_tok; p.w_c = w_c; p.b_c = b_c; p.T = T;
    p.B = B; p.gamma = gamma; p.V = V; p.conf_cal = conf_cal; p.log_surv = log_surv;
    const WsPtrs w = ws_ptrs(ws, B, gamma, V);
    p.status = w.status;
    p.tickets = w.conf_tickets;
    p.score = w.conf_score;
    return launch_status(launch_confidence(p, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_schedule(const float* log_surv, const float* log_surv_hist, const float* sps,
                              int sps_len, int B, int gamma, dspark_sched_mode mode, int32_t* K,
                              int32_t* n_total, float* theta, void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    (void)ws; (void)ws_bytes;
    if (B < 1 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || B * gamma > DSPARK_MAX_SCHED_ITEMS)
        return DSPARK_ERR_INVALID;
    if (mode != DSPARK_SCHED_OFF && mode != DSPARK_SCHED_SYNC && mode != DSPARK_SCHED_ASYNC)
        return DSPARK_ERR_INVALID;
    if (sps_len < B + B * gamma) return DSPARK_ERR_INVALID;
    if (!is_device_ptr(log_surv) || !is_device_ptr(sps) || !is_device_ptr(K) || !is_device_ptr(n_total) ||
        !is_device_ptr(theta))
        return DSPARK_ERR_INVALID;
    if (log_surv_hist && !is_device_ptr(log_surv_hist)) return DSPARK_ERR_INVALID;
    SchedParams p;
    p.log_surv = log_surv; p.log_surv_hist = log_surv_hist; p.sps = sps; p.sps_len = sps_len;
    p.B = B; p.gamma = gamma; p.mode = (int)mode; p.K = K; p.n_total = n_total; p.theta = theta;
    return launch_status(launch_schedule(p, static_cast<cudaStream_t>(stream)));
}

static dspark_status verify_impl(const void* target, dspark_dtype target_t, const void* U, dspark_dtype U_t,
                                 const void* W1, const float* state, const float* zlog, const void* W2,
                                 dspark_dtype W_t,
                                 const int32_t* anchor, const int32_t* draft_tok, const float* lse_q,
                                 const float* z_tok, const int32_t* K, int B, int gamma, int V, int r,
                                 int req_base, float tau, uint64_t seed, uint64_t step, int32_t* accepted,
                                 int32_t* out_tok, int32_t* out_req, int32_t* out_pos, int32_t* out_off,
                                 int32_t* next_anchor, float* p_tok, uint32_t* near_ties, void* ws,
                                 size_t ws_bytes, void* stream) {
    if (!sizes_ok(B, gamma, V, r) || !(tau > 0.f) || req_base < 0) return DSPARK_ERR_INVALID;
    if ((target_t != DSPARK_F32 && target_t != DSPARK_BF16) || (U_t != DSPARK_F32 && U_t != DSPARK_BF16) ||
        (W_t != DSPARK_F32 && W_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    const void* rows = state ? static_cast<const void*>(state) : W1;
    const void* need[] = {target, U, rows, W2, anchor, draft_tok, lse_q, z_tok, accepted,
                          out_tok, out_req, out_pos, out_off, next_anchor, ws};
    for (const void* q : need)
        if (!is_device_ptr(q)) return DSPARK_ERR_INVALID;
    if (K && !is_device_ptr(K)) return DSPARK_ERR_INVALID;
    if ((p_tok && !is_device_ptr(p_tok)) || (near_ties && !is_device_ptr(near_ties))) return DSPARK_ERR_INVALID;
    if (!aligned(target, 16) || !aligned(U, 16) || !aligned(rows, 16) || !aligned(W2, 16) || !aligned(ws, 256))
        return DSPARK_ERR_INVALID;
    if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;
    VerifyParams p;
    p.target = target; p.target_bf16 = (target_t == DSPARK_BF16);
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = W1; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor; p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.K = K;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau; p.seed = seed; p.step = step;
    p.accepted = accepted; p.out_tok = out_tok; p.out_req = out_req; p.out_pos = out_pos;
    p.out_off = out_off; p.next_anchor = next_anchor; p.p_tok = p_tok; p.near_ties = near_ties;
    p.ws = ws_ptrs(ws, B, gamma, V);
    p.state = state;
    p.zlog = zlog;
    if (!K) {
        // full prefix after dspark_draft_markov_target on these inputs (the
        // accept kernel checks the token it left): either the stream ran
        // beside its draft (rows 0..gamma), or its epilogue reduced rows
        // 0..gamma-1 (fp32 target)
        if (state) return DSPARK_ERR_UNSUPPORTED;
        DraftParams d = draft_view(p);
        d.target = static_cast<const float*>(target);
        if (draft_target_vs(d)) {
            p.vs_full = 1;
        } else {
            if (target_t != DSPARK_F32) return DSPARK_ERR_UNSUPPORTED;
            p.tgt_slots = draft_rows_grid_x(B, V, p.ws.parts);
            if (p.tgt_slots > kTgtSlots) return DSPARK_ERR_UNSUPPORTED;
        }
        p.tgt_token = tgt_token_of(target, seed, step, req_base, B, gamma, V, tau);
    }
    if (zlog && (!is_device_ptr(zlog) || !aligned(zlog, 16))) return DSPARK_ERR_INVALID;
    if (state && !zlog && !resid_rows_supported(p)) return DSPARK_ERR_UNSUPPORTED;
    return launch_status(launch_verify(p, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_verify(const void* target, dspark_dtype target_t, const void* U, dspark_dtype U_t,
                            const void* W1, const void* W2, dspark_dtype W_t, const int32_t* anchor,
                            const int32_t* draft_tok, const float* lse_q, const float* z_tok,
                            const int32_t* K, int B, int gamma, int V, int r, int req_base, float tau,
                            uint64_t seed, uint64_t step, int32_t* accepted, int32_t* out_tok,
                            int32_t* out_req, int32_t* out_pos, int32_t* out_off, int32_t* next_anchor,
                            float* p_tok, uint32_t* near_ties, void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    return verify_impl(target, target_t, U, U_t, W1, nullptr, nullptr, W2, W_t, anchor, draft_tok, lse_q, z_tok, K, B,
                       gamma, V, r, req_base, tau, seed, step, accepted, out_tok, out_req, out_pos, out_off,
                       next_anchor, p_tok, near_ties, ws, ws_bytes, stream);
}

dspark_status dspark_verify_logits(const void* target, dspark_dtype target_t, const void* U, dspark_dtype U_t,
                                   const void* W1, const void* W2, dspark_dtype W_t, const float* draft_logits,
                                   const int32_t* anchor, const int32_t* draft_tok, const float* lse_q,
                                   const float* z_tok, const int32_t* K, int B, int gamma, int V, int r,
                                   int req_base, float tau, uint64_t seed, uint64_t step, int32_t* accepted,
                                   int32_t* out_tok, int32_t* out_req, int32_t* out_pos, int32_t* out_off,
                                   int32_t* next_anchor, float* p_tok, uint32_t* near_ties, void* ws,
                                   size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (!draft_logits) return DSPARK_ERR_INVALID;
    return verify_impl(target, target_t, U, U_t, W1, nullptr, draft_logits, W2, W_t, anchor, draft_tok, lse_q,
                       z_tok, K, B, gamma, V, r, req_base, tau, seed, step, accepted, out_tok, out_req, out_pos,
                       out_off, next_anchor, p_tok, near_ties, ws, ws_bytes, stream);
}

dspark_status dspark_verify_rnn(const void* target, dspark_dtype target_t, const void* U, dspark_dtype U_t,
                                const float* state, const void* W2, dspark_dtype W_t, const int32_t* anchor,
                                const int32_t* draft_tok, const float* lse_q, const float* z_tok,
                                const int32_t* K, int B, int gamma, int V, int r, int req_base, float tau,
                                uint64_t seed, uint64_t step, int32_t* accepted, int32_t* out_tok,
                                int32_t* out_req, int32_t* out_pos, int32_t* out_off, int32_t* next_anchor,
                                float* p_tok, uint32_t* near_ties, void* ws, size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (!state) return DSPARK_ERR_INVALID;
    return verify_impl(target, target_t, U, U_t, nullptr, state, nullptr, W2, W_t, anchor, draft_tok, lse_q, z_tok, K, B,
                       gamma, V, r, req_base, tau, seed, step, accepted, out_tok, out_req, out_pos, out_off,
                       next_anchor, p_tok, near_ties, ws, ws_bytes, stream);
}

dspark_status dspark_rnn_input_table(const void* E, const void* W_ih, const float* b_ih, int V, int r, float* P,
                                     void* stream) {
    const dspark::CallRange range_(__func__);
    if (V < 1 || r < 1 || r > 1024 || (r % 8) != 0) return DSPARK_ERR_INVALID;
    if (!is_device_ptr(E) || !is_device_ptr(W_ih) || !is_device_ptr(b_ih) || !is_device_ptr(P))
        return DSPARK_ERR_INVALID;
    return launch_status(launch_rnn_input_table(static_cast<const uint16_t*>(E), static_cast<const uint16_t*>(W_ih),
                                                b_ih, V, r, P, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_draft_rnn(const void* U, dspark_dtype U_t, const float* P, const void* W_hh, const float* b_hh,
                               const float* s0, const void* W2, dspark_dtype W_t, const int32_t* anchor, int B,
                               int gamma, int V, int r, int req_base, float tau, uint64_t seed, uint64_t step,
                               int32_t* draft_tok, float* lse_q, float* z_tok, float* state, void* ws,
                               size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (!sizes_ok(B, gamma, V, r) || !(tau > 0.f) || req_base < 0) return DSPARK_ERR_INVALID;
    if ((U_t != DSPARK_F32 && U_t != DSPARK_BF16) || (W_t != DSPARK_F32 && W_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    const void* need[] = {U, P, W_hh, b_hh, s0, W2, anchor, draft_tok, lse_q, z_tok, state, ws};
    for (const void* q : need)
        if (!is_device_ptr(q)) return DSPARK_ERR_INVALID;
    if (!aligned(U, 16) || !aligned(P, 16) || !aligned(W_hh, 16) || !aligned(W2, 16) || !aligned(state, 16) ||
        !aligned(ws, 256))
        return DSPARK_ERR_INVALID;
    if (ws_bytes < ws_layout(B, gamma, V).total) return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;
    DraftParams p;
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = nullptr; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau;
    p.seed = seed; p.step = step;
    p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.logits_out = nullptr;
    p.ws = ws_ptrs(ws, B, gamma, V);
    p.state = state;
    // bf16 weights, fp32 U, r % 64 == 0, r <= 256 (= kMaxRnnRank, the size of the gh scratch rows)
    if (!draft_rows_supported(p) || r > kMaxRnnRank) return DSPARK_ERR_UNSUPPORTED;
    GruParams g;
    g.P = P;
    g.W_hh = static_cast<const uint16_t*>(W_hh);
    g.b_hh = b_hh; g.s0 = s0;
    g.anchor = anchor; g.draft_tok = draft_tok; g.state = state;
    g.gh = p.ws.rnn_gh;
    g.B = B; g.gamma = gamma; g.V = V; g.r = r;
    g.status = p.ws.status;
    return launch_status(launch_draft_rnn(p, g, static_cast<cudaStream_t>(stream)));
}

dspark_status dspark_gumbel_stream(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, int n,
                                   float* gumbel_out, float* uniform_out, void* stream) {
    if (n < 0 || domain > 3 || (!gumbel_out && !uniform_out)) return DSPARK_ERR_INVALID;
    if ((gumbel_out && !is_device_ptr(gumbel_out)) || (uniform_out && !is_device_ptr(uniform_out)))
        return DSPARK_ERR_INVALID;
    if (n == 0) return DSPARK_OK;
    return launch_status(launch_gumbel_stream(seed, step, domain, row, n, gumbel_out, uniform_out,
                                              static_cast<cudaStream_t>(stream)));
}

static size_t sts_tickets_off() { return 256; }
static size_t sts_acc_off(int gamma) { return align256(sts_tickets_off() + sizeof(uint32_t) * (size_t)gamma); }
static size_t sts_ws_total(int gamma, int G, int M) {
    return align256(sts_acc_off(gamma) + sizeof(long long) * (size_t)gamma * M * G);
}

size_t dspark_sts_workspace_bytes(int gamma, int G, int M) {
    if (gamma < 1 || gamma > DSPARK_MAX_GAMMA || G < 1 || G > DSPARK_MAX_STS_GRID || M < 1 || M > DSPARK_MAX_STS_BINS)
        return 0;
    return sts_ws_total(gamma, G, M);
}

dspark_status dspark_sts_fit(const float* score, const int32_t* acc_len, int N, int gamma, const float* grid,
                             int G, int M, float* T_out, int32_t* idx_out, double* ece_out, void* ws,
                             size_t ws_bytes, void* stream) {
    const dspark::CallRange range_(__func__);
    if (N < 1 || dspark_sts_workspace_bytes(gamma, G, M) == 0) return DSPARK_ERR_INVALID;
    if (!is_device_ptr(score) || !is_device_ptr(acc_len) || !is_device_ptr(grid) || !is_device_ptr(T_out) ||
        !is_device_ptr(idx_out) || !is_device_ptr(ece_out) || !is_device_ptr(ws))
        return DSPARK_ERR_INVALID;
    if (!aligned(score, 4) || !aligned(acc_len, 4) || !aligned(grid, 4) || !aligned(T_out, 4) ||
        !aligned(idx_out, 4) || !aligned(ece_out, 8) || !aligned(ws, 256))
        return DSPARK_ERR_INVALID;
    const size_t total = sts_ws_total(gamma, G, M);
    if (ws_bytes < total) return DSPARK_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, total, s);
    if (e != cudaSuccess) return launch_status(e);
    char* base = static_cast<char*>(ws);
    StsFitParams p;
    p.score = score; p.acc_len = acc_len; p.N = N; p.gamma = gamma;
    p.grid = grid; p.G = G; p.M = M;
    p.T_out = T_out; p.idx_out = idx_out; p.ece_out = ece_out;
    p.status = reinterpret_cast<uint32_t*>(base);
    p.tickets = reinterpret_cast<uint32_t*>(base + sts_tickets_off());
    p.acc = reinterpret_cast<long long*>(base + sts_acc_off(gamma));
    return launch_status(launch_sts_fit(p, s));
}

}  // extern "C"
