// internal.h -- parameter blocks, workspace layout and launcher declarations
// shared between the ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dspark.h"

namespace dspark {

struct DrawLse;
struct LseDraw;
struct Draw2;

constexpr int kMaxParts = 1024;        // cap on partial states per request per launch
constexpr int kPartTile = 128;         // vocabulary entries per tile of the partial-producing kernels
constexpr int kVerifySeg = 32768;      // vocabulary entries per verify-stream work item
constexpr int kVerifySub = 8;          // partial states per work item (one per consumer warp)
constexpr int kChunk = 16;             // requests per chunk of the partial-producing kernels
constexpr int kGridBarrierSlots = DSPARK_MAX_GAMMA;   // one grid-barrier counter per draft position
constexpr int kGbarGru = kGridBarrierSlots;           // then one per position for the RNN head's GRU step
constexpr int kGbarExit = 2 * kGridBarrierSlots;      // then the exit counter
constexpr int kWinStride = 16;          // winner keys 128 bytes apart: one cache line each
constexpr int kTgtSlots = 256;          // partial states per (request, target row) of the draft's target
                                        // stream (>= the draft's CTAs along V)

constexpr size_t ws_align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kDrawLseBytes = 16;   // sizeof(DrawLse) (checked in common.cuh)

// The workspace regions the draft kernels touch, in layout order: status
// word, arrival tickets, grid-barrier counters, winner keys, verify-stream
// counters, then the draft's two buffers of partial states.  `end` is the
// first byte past them.  ws_layout places the other regions after these.
struct WsDraftPrefix {
    size_t status, tickets, gbar, win, vq, draft_part, end;
};
constexpr WsDraftPrefix ws_draft_prefix(int B, int gamma, int parts) {
    WsDraftPrefix P{};
    const size_t nchunks = ((size_t)B + kChunk - 1) / kChunk;
    size_t o = 0;
    P.status = o;     o = ws_align256(o + 16);
    P.tickets = o;    o = ws_align256(o + sizeof(uint32_t) * 2 * nchunks);
    P.gbar = o;       o = ws_align256(o + sizeof(uint32_t) * (kGbarExit + 1));
    P.win = o;        o = ws_align256(o + sizeof(unsigned long long) * kWinStride * (size_t)gamma * B);
    P.vq = o;         o = ws_align256(o + sizeof(uint32_t) * 2);
    P.draft_part = o; o = ws_align256(o + kDrawLseBytes * 2 * (size_t)B * parts);
    P.end = o;
    return P;
}

// Byte offsets of the workspace regions (all 256-byte aligned).
struct WsLayout {
    size_t status, tickets, gbar, win, vq, draft_part, verify_part, tgt_part, tgt_token, rej, acc, fin, lse_rej,
        resid_part, conf, rnn_gh, bonus_tickets, row_lse, row_tickets, rtok, total;
    int nseg;    // verify-stream segments per row
    int parts;   // partial-state slots per request (>= CTAs along V of any launch)
};
WsLayout ws_layout(int B, int gamma, int V);

struct WsPtrs {
    uint32_t* status;
    unsigned long long* wait_limit;   // bound on device waits in SM cycles (0: the default, about 2 s)
    uint32_t* tickets_draft;   // [ceil(B/kChunk)] arrival counters, zero between launches
    uint32_t* tickets_resid;   // [ceil(B/kChunk)]
    uint32_t* gbar;            // [kGbarExit + 1] grid-barrier counters, then the exit counter
    uint32_t* vq;              // [2] verify-stream work counter and exit counter, zero between launches
    unsigned long long* win;   // [gamma][B][kWinStride] winner keys of the persistent draft (first of
                               // each line used), zero between launches
    DrawLse* draft_part;       // [2][B][parts] (two buffers alternate between positions)
    LseDraw* verify_part;      // [B][gamma+1][nseg * kVerifySub] verify-stream partials
    LseDraw* tgt_part;         // [B][gamma][kTgtSlots] target-row partials of the draft's target stream
    unsigned long long* tgt_token;   // [1] identifies the call that wrote tgt_part
    int32_t* rej;        // [B] 0-based rejected row, -1 if every walked draft was accepted
    int32_t* acc;        // [B] accepted count
    int32_t* fin;        // [B] final token
    float2* lse_rej;     // [B] (lse_p, lse_q) of the rejected row
    Draw2* resid_part;   // [B][parts]
    uint32_t* conf_tickets;  // [B] confidence-head arrival counters, zero between launches
    float* conf_score;       // [B][gamma]
    float* rnn_gh;           // [B][3 kMaxRnnRank] RNN head scratch
    uint32_t* bonus_tickets; // [B] bonus-draw arrival counters, zero between launches
    // the stream beside the draft: each row's log-sum-exp, merged by the warp
    // that writes the row's last partial (arrival counters zero between launches)
    float* row_lse;          // [B][gamma+1]
    uint32_t* row_tickets;   // [B][gamma+1]
    // [B] the token before the rejected draft (the anchor when the first is
    // rejected; -1 when none is): its W1 row is the residual draw's A row
    int32_t* rtok;
    int nseg;
    int parts;
};
WsPtrs ws_ptrs(void* ws, int B, int gamma, int V);

// Host-side argument checks shared by the ABI entry points (api.cu).
bool is_device_ptr(const void* p);              // device or managed memory
bool sizes_ok(int B, int gamma, int V, int r);  // the limits of dspark_draft_markov
dspark_status launch_status(cudaError_t e);     // DSPARK_OK, or DSPARK_ERR_CUDA with a message
// Synchronise s, read the 32-bit status word at `word` (device memory), clear
// it if set; the status dspark_sync_status returns.
dspark_status read_status_word(void* word, cudaStream_t s, uint32_t* bits);

struct DraftParams {
    const void* U; int U_bf16;
    const void* W1; const void* W2; int W_bf16;
    const int32_t* anchor;
    int B, gamma, V, r, req_base;
    float inv_tau;
    uint64_t seed, step;
    int32_t* draft_tok; float* lse_q; float* z_tok; float* logits_out;
    WsPtrs ws;
    // RNN head: the bias of position k is formed from state[k-1][b] ([gamma][B][r]
    // fp32, rounded to bf16 when staged) instead of W1[x~_{k-1}]
    const float* state = nullptr;
    // target stream (full-prefix verification): position k also reduces target
    // row k-1 ([B][gamma+1][V] fp32) to log-sum-exp partials in ws.tgt_part
    const float* target = nullptr;
    int target_bf16 = 0;                // the target beside the draft may be bf16
    unsigned long long tgt_token = 0;
    // residual draw (full prefix beside the draft): the requests without a
    // rejection draw their bonus token from row gamma's law p in the same launch
    int resid_bonus = 0;
};

// One GRU step of the RNN head for every request: state[k-1] = GRU(state[k-2]
// (s0 for k = 1), E[x~_{k-1}]).
struct GruParams {
    const float* P;                          // [V][3r] input projections E W_ih^T + b_ih, gate blocks (r, z, n)
    const uint16_t* W_hh;                    // [3r][r] bf16, gate rows (r, z, n)
    const float* b_hh;                       // [3r]
    const float* s0;                         // [r] learned initial state
    const int32_t* anchor; const int32_t* draft_tok;
    float* state;                            // [gamma][B][r]
    float* gh;                               // [B][3r] scratch: W_hh h + b_hh of the coming step
    int B, gamma, V, r;
    uint32_t* status;
};
constexpr int kMaxRnnRank = 256;             // the draft rows kernel's limit on r

struct ConfParams {
    const float* h; int d;
    const void* emb; int emb_bf16; int e;
    const int32_t* anchor; const int32_t* draft_tok;
    const float* w_c; float b_c; const float* T;
    int B, gamma, V;
    float* conf_cal; float* log_surv;
    uint32_t* status;
    uint32_t* tickets;   // [B] arrival counters, zero between launches
    float* score;        // [B][gamma] s_k before calibration
};

struct SchedParams {
    const float* log_surv; const float* log_surv_hist;
    const float* sps; int sps_len;
    int B, gamma, mode;
    int32_t* K; int32_t* n_total; float* theta;
};

struct VerifyParams {
    const void* target; int target_bf16;
    const void* U; int U_bf16;
    const void* W1; const void* W2; int W_bf16;
    const int32_t* anchor; const int32_t* draft_tok;
    const float* lse_q; const float* z_tok; const int32_t* K;
    int B, gamma, V, r, req_base;
    float inv_tau;
    uint64_t seed, step;
    int32_t* accepted; int32_t* out_tok; int32_t* out_req; int32_t* out_pos;
    int32_t* out_off; int32_t* next_anchor;
    float* p_tok; uint32_t* near_ties;
    WsPtrs ws;
    const float* state = nullptr;   // RNN head bias rows (see DraftParams)
    const float* zlog = nullptr;    // the draft's stored logits [B][gamma][V] (z / tau), or null
    // full-prefix mode (K == null, every K_b = gamma): rows 0..gamma-1 take
    // their log-sum-exp from the draft's target stream (tgt_slots partials a
    // row in ws.tgt_part, written by the call whose token is tgt_token); the
    // verify stream covers only the bonus rows
    int tgt_slots = 0;
    unsigned long long tgt_token = 0;
    // full-prefix mode after a draft whose verify stream ran beside it: the
    // walked rows' partials and the bonus tokens are already in the workspace
    int vs_full = 0;
    // the tensor-core residual launch left its draws as winner keys: the
    // compaction decodes them (set by the verify launcher)
    int resid_keys = 0;
};

struct StsFitParams {
    const float* score; const int32_t* acc_len; int N, gamma;
    const float* grid; int G, M;
    float* T_out; int32_t* idx_out; double* ece_out;
    long long* acc;      // [gamma][M][G] fixed-point bin totals, zero before the fit
    uint32_t* tickets;   // [gamma] arrival tickets, zero before the fit
    uint32_t* status;
};

int num_sms();

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_draft_simt(const DraftParams& p, int k, cudaStream_t s);
cudaError_t launch_draft(const DraftParams& p, cudaStream_t s);   // all gamma positions
bool draft_rows_supported(const DraftParams& p);
cudaError_t launch_draft_rows(const DraftParams& p, int k_first, int k_last, cudaStream_t s);
int draft_rows_grid_x(int B, int V, int parts);   // CTAs along V of a draft rows launch
bool draft_target_supported(const DraftParams& p);
bool draft_target_vs(const DraftParams& p);       // the target-stream draft runs the verify stream beside it
cudaError_t launch_draft_target(const DraftParams& p, cudaStream_t s);   // the draft with the target stream
bool cooperative_supported();
void* tma_encoder();   // cuTensorMapEncodeTiled from the driver, or NULL
bool resid_rows_supported(const VerifyParams& v);
cudaError_t launch_resid_rows(const VerifyParams& v, cudaStream_t s);
// The walked target rows' log-sum-exps and the bonus draws by a lean stream
// kernel that runs on the SMs beside the draft launched just before it (one
// instance per SM).
cudaError_t launch_target_stream_side(const VerifyParams& v, cudaStream_t s);

// Whether the stream beside the draft also merges each row's partials into
// ws.row_lse (one chunk of requests), which the accept walk then reads.
__host__ __device__ inline bool vs_row_merge(const VerifyParams& v) { return v.vs_full && v.B <= 64; }

// The draft-side view of a verify call (same U, W1, W2, tokens and workspace).
inline DraftParams draft_view(const VerifyParams& v) {
    DraftParams p;
    p.U = v.U; p.U_bf16 = v.U_bf16; p.W1 = v.W1; p.W2 = v.W2; p.W_bf16 = v.W_bf16;
    p.anchor = v.anchor; p.B = v.B; p.gamma = v.gamma; p.V = v.V; p.r = v.r; p.req_base = v.req_base;
    p.inv_tau = v.inv_tau; p.seed = v.seed; p.step = v.step;
    p.draft_tok = const_cast<int32_t*>(v.draft_tok); p.lse_q = nullptr; p.z_tok = nullptr; p.logits_out = nullptr;
    p.ws = v.ws;
    p.state = v.state;
    p.resid_bonus = v.vs_full;
    return p;
}
cudaError_t launch_gumbel_stream(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, int n, float* g,
                                 float* u, cudaStream_t s);
cudaError_t launch_confidence(const ConfParams& p, cudaStream_t s);
cudaError_t launch_schedule(const SchedParams& p, cudaStream_t s);
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s);
cudaError_t launch_sts_fit(const StsFitParams& p, cudaStream_t s);
cudaError_t launch_gru(const GruParams& g, int k, cudaStream_t s);
cudaError_t launch_rnn_input_table(const uint16_t* E, const uint16_t* W_ih, const float* b_ih, int V, int r,
                                   float* P, cudaStream_t s);
cudaError_t launch_draft_rnn(const DraftParams& p, const GruParams& g, cudaStream_t s);
cudaError_t launch_draft_rows_rnn(const DraftParams& p, const GruParams& g, int k_first, int k_last,
                                  cudaStream_t s);

}  // namespace dspark
