/*
 * dspark.h -- C ABI of the DSpark draft + verify step on one GB300 (sm_103a).
 *
 * Sources cited below (page title, then section):
 *   [P2] "DSpark：半自回归生成与置信度调度的投机解码" (pinghaoyang.com.cn/aigc/posts/dspark/)
 *   [P3] "拒绝盲猜与算力空转：深度拆解 DeepSeek 开源投机采样方案 DeepSpec & DSpark"
 *        (val213.github.io/2026/06/28/DSpark&DSpec/)
 *   [P4] "DeepSeek-AI与北京大学联手破局：AI聊天机器人"慢速打字"的终极解决方案"
 *        (techwalker.com/2026/0716/3193540.shtml)
 *
 * Conventions for every call:
 *   - Tensor pointers are CUDA device pointers owned by the caller, row-major and
 *     contiguous, with the shapes given in brackets.  Nothing here allocates
 *     device memory; calls that need scratch take a workspace (ws, ws_bytes)
 *     sized by dspark_workspace_bytes() and cleared once by
 *     dspark_workspace_init().  A workspace must not be shared by calls that
 *     may run concurrently.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return after enqueueing work.  Host-side argument
 *     errors return DSPARK_ERR_INVALID / DSPARK_ERR_UNSUPPORTED before any
 *     work is enqueued; a launch failure returns DSPARK_ERR_CUDA.
 *   - Device-side checks (token ids out of range, verify lengths out of
 *     [0, gamma]) never trap: the offending element is skipped, a bit is set
 *     in the workspace status word, and dspark_sync_status() reports it.
 *   - Results depend only on the inputs, seed, step and request ids: the
 *     random numbers are Philox4x32-10 (Salmon et al., SC'11) with
 *       key = (seed mod 2^32, seed div 2^32),
 *       counter = (col div 4, req*(gamma+1) + row, step mod 2^32,
 *                  domain + 4*(step div 2^32)), word = col mod 4,
 *     u = (2*(x div 2^9) + 1) * 2^-24, Gumbel G = -log(-log u).
 *     Domains: 0 draft, 1 acceptance uniform, 2 residual, 3 bonus.
 *     req = req_base + b.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID = -1,      /* bad argument (null pointer, size, alignment) */
    DSPARK_ERR_CUDA = -2,         /* a CUDA runtime call or launch failed */
    DSPARK_ERR_TIMEOUT = -3,      /* a bounded device wait expired */
    DSPARK_ERR_UNSUPPORTED = -4,  /* valid but not implemented (dtype / shape combination) */
    DSPARK_ERR_DEVICE = -5        /* a device-side range check fired (see dspark_sync_status) */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum {
    DSPARK_SCHED_OFF = 0,    /* every request verifies its whole block: K_b = gamma */
    DSPARK_SCHED_SYNC = 1,   /* greedy admission with early stop [P4 §四] */
    DSPARK_SCHED_ASYNC = 2   /* capacity from survivals two steps old, no early stop [P4 §五] */
} dspark_sched_mode;

/* Limits of the library. */
#define DSPARK_MAX_GAMMA 16
#define DSPARK_MAX_SCHED_ITEMS 4096   /* B * gamma for dspark_schedule */
#define DSPARK_MAX_STS_GRID 65536     /* candidate temperatures for dspark_sts_fit */
#define DSPARK_MAX_STS_BINS 64        /* calibration-error bins for dspark_sts_fit */

/* Library version (major*10000 + minor*100 + patch). */
int dspark_version(void);

/* Human-readable name of a status code (static storage). */
const char* dspark_status_string(dspark_status s);

/* Workspace bytes for a step of B requests, block length gamma, vocabulary V,
 * Markov rank r.  Returns 0 if the sizes are out of range. */
size_t dspark_workspace_bytes(int B, int gamma, int V, int r);

/* Zero a workspace (its status word and the arrival counters the kernels
 * use).  Call once after allocating it; the kernels leave it reusable. */
dspark_status dspark_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Bound the device waits of the calls that use this workspace: a wait on
 * another role of a kernel or on other CTAs (copy rings, accumulator
 * hand-offs, grid barriers, the verify stream's ring) gives up after about
 * `cycles` SM clock cycles, raises the timeout bit (dspark_sync_status then
 * returns DSPARK_ERR_TIMEOUT) and the kernel drains the copies it issued,
 * frees its tensor memory and returns.  0 restores the default, about 2 s
 * at 2 GHz; dspark_workspace_init also restores it.  A small bound exists
 * to exercise that path in tests: with it, results are unspecified, and the
 * workspace needs dspark_workspace_init before its next use.  The value
 * lives in bytes 8-15 of the workspace.  No counterpart on the pages. */
dspark_status dspark_workspace_set_wait_limit(void* ws, size_t ws_bytes, uint64_t cycles, void* stream);

/* Synchronise `stream`, then read and clear the workspace status word.
 * Returns DSPARK_OK, DSPARK_ERR_DEVICE (range check fired), DSPARK_ERR_TIMEOUT,
 * or DSPARK_ERR_CUDA (the stream reported an error).  If bits is non-NULL the
 * raw status bits are stored there: bit 0 a token out of [0, V), bit 1 a
 * block length out of [0, gamma], bit 2 a bounded wait expired, bit 3 a
 * non-finite score or a temperature that is not positive and finite
 * (dspark_sts_fit), and with bit 2 the bits 8-23 name the wait that gave up
 * (for diagnosis only). */
dspark_status dspark_sync_status(void* ws, void* stream, uint32_t* bits);

/*
 * Steps a1-a3: the Markov-head draft loop [P2 §整体架构, §Markov Head：一阶转移偏置],
 * [P3 §DSpark 的解法：半自回归架构与低秩马尔可夫头].  For k = 1..gamma, request b:
 *     h      = W1[x~_{k-1}]                      (x~_0 = anchor[b])
 *     z_k    = (U[b,k-1,:] + h . W2) / tau        (draft logits over V)
 *     lse_q  = log sum_v exp(z_k[v])
 *     x~_k   = argmax_v z_k[v] + G(domain 0, row k-1, col v)   (lowest v on ties)
 * Inputs : U [B,gamma,V] (U_t), W1 [V,r], W2 [r,V] (W_t), anchor [B] in [0,V).
 *          bf16 weights run the W2 contraction on the tensor cores (fp32
 *          accumulation); fp32 weights run it on CUDA cores.
 * Outputs: draft_tok [B,gamma] int32, lse_q [B,gamma], z_tok [B,gamma] = z_k[x~_k].
 *          logits_out, if non-NULL, receives z [B,gamma,V] fp32 (parity checks;
 *          pass NULL on the hot path).
 * Limits : 1 <= gamma <= DSPARK_MAX_GAMMA, V % 8 == 0, 1 <= r <= 1024,
 *          B*(gamma+1) + req_base < 2^32, tau > 0.
 */
dspark_status dspark_draft_markov(
    const void* U, dspark_dtype U_t,
    const void* W1, const void* W2, dspark_dtype W_t,
    const int32_t* anchor,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* draft_tok, float* lse_q, float* z_tok, float* logits_out,
    void* ws, size_t ws_bytes, void* stream);

/*
 * The draft of dspark_draft_markov with the first pass of a full-prefix
 * verification [P2 §形式化定义] (every draft position is checked against the
 * target's distribution at that position) done at the same time: target rows
 * are reduced to partial log-sum-exps of target/tau, kept in ws.  With gamma > 1
 * and cooperative launch, a stream kernel runs beside the draft on the same
 * SMs and reduces rows 0..gamma (the bonus row too); otherwise (fp32 target
 * only) the draft's epilogue reduces rows 0..gamma-1 as position k streams
 * U[b,k-1,:].  A following dspark_verify or dspark_verify_logits with K = NULL
 * uses them instead of reading those rows again.
 * Inputs : those of dspark_draft_markov, plus target [B,gamma+1,V] (target_t:
 *          fp32, or bf16 where the stream runs beside the draft).
 * Outputs: those of dspark_draft_markov (identical values); ws holds the
 *          target partials and a token naming (target, seed, step, req_base,
 *          B, gamma, V, tau).  Leave the target unchanged until the verify call.
 * Limits : those of dspark_draft_markov's tensor-core path (bf16 weights, fp32
 *          U, r % 64 == 0, r <= 256); otherwise, or for a bf16 target without
 *          the stream beside the draft, DSPARK_ERR_UNSUPPORTED.
 */
dspark_status dspark_draft_markov_target(
    const void* U, dspark_dtype U_t,
    const void* W1, const void* W2, dspark_dtype W_t,
    const void* target, dspark_dtype target_t,
    const int32_t* anchor,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* draft_tok, float* lse_q, float* z_tok, float* logits_out,
    void* ws, size_t ws_bytes, void* stream);

/*
 * Step a4: confidence head, sequential temperature scaling and prefix survival
 * [P2 §置信度头：预测自己的命运, §校准问题：原始置信度不可靠], [P4 §四].
 *     s_k        = w_c . [h[b,k-1,:] ; emb[x~_{k-1},:]] + b_c
 *     conf_cal   = sigmoid(s_k / T[k-1])            (= sigmoid(logit(c_k)/T_k))
 *     log_surv   = sum_{i<=k} log conf_cal_i         (log of the survival a_{b,k})
 * Inputs : h [B,gamma,d] fp32, emb [V,e] (emb_t), anchor [B], draft_tok [B,gamma],
 *          w_c [d+e] fp32, T [gamma] fp32 (> 0).  e = d follows the workload
 *          definition (an embedding table); passing W1 with e = r follows
 *          [P2], which reuses the Markov head's W1 rows.
 * Outputs: conf_cal [B,gamma], log_surv [B,gamma] (non-increasing in k).
 * ws     : a workspace of at least dspark_workspace_bytes(B, gamma, V, r) bytes
 *          (any r), 256-byte aligned, cleared once: the call keeps per-request
 *          arrival counters and the raw scores there.
 */
dspark_status dspark_confidence_sts(
    const float* h, int d,
    const void* emb, dspark_dtype emb_t, int e,
    const int32_t* anchor, const int32_t* draft_tok,
    const float* w_c, float b_c, const float* T,
    int B, int gamma, int V,
    float* conf_cal, float* log_surv,
    void* ws, size_t ws_bytes, void* stream);

/*
 * Step a5: hardware-aware greedy prefix scheduler [P2 §硬件感知前缀调度器],
 * [P4 §四, §五].  Candidates (b, j) sorted by survival descending (ties: b,
 * then j); R = B;  Theta(n) = (R + sum of the first n survivals) * sps[R+n-1].
 *   SYNC : admit in order while Theta strictly rises; stop at the first non-rise.
 *   ASYNC: n* = first argmax_n Theta_hist(n) over the list of log_surv_hist
 *          (survivals two steps old; NULL = use log_surv), then admit the n*
 *          best current candidates.
 *   OFF  : K_b = gamma.
 * Inputs : log_surv [B,gamma] fp32 (non-increasing in j), log_surv_hist or
 *          NULL, sps [sps_len] fp32 with sps_len >= B + B*gamma.
 * Outputs: K [B] verify lengths, n_total [1] admitted drafts, theta [1] =
 *          Theta at the admitted count (fp32).
 * Limits : B*gamma <= DSPARK_MAX_SCHED_ITEMS.
 */
dspark_status dspark_schedule(
    const float* log_surv, const float* log_surv_hist,
    const float* sps, int sps_len, int B, int gamma, dspark_sched_mode mode,
    int32_t* K, int32_t* n_total, float* theta,
    void* ws, size_t ws_bytes, void* stream);

/*
 * Steps a6-a8: lossless verification and ragged compaction
 * [P2 §形式化定义], [P4 §四, §五].  For request b, with p_i = softmax(target[b,i,:]/tau):
 *   walk k = 1..K_b: accept x~_k iff u(domain 1, row k-1) < min(1, p_k(x~_k)/q_k(x~_k)),
 *     q_k(x~_k) = exp(z_tok - lse_q);
 *   first rejection j: emit argmax_v log(max(0, p_j - q_j)[v]) + G(domain 2, row j-1, v)
 *     (q_j recomputed over V from U, W1, W2; if p_j <= q_j everywhere, from p_j);
 *   all K_b accepted: emit the bonus argmax_v target[b,K_b,v]/tau + G(domain 3, row K_b, v).
 * Output layout: out_off = exclusive scan of (A_b + 1) over b ([B+1]);
 *   out_tok/out_req/out_pos [B*(gamma+1)] hold the accepted drafts then the
 *   final token of each request at out_off[b]..out_off[b+1]-1; next_anchor [B]
 *   is the last emitted token; accepted [B] = A_b.
 * Inputs : target [B,gamma+1,V] (target_t), U, W1, W2 as for the draft, anchor,
 *          draft_tok, lse_q, z_tok from dspark_draft_markov, K [B] in [0,gamma].
 * K NULL : full prefix (every K_b = gamma) after dspark_draft_markov_target on
 *          the same workspace, target, seed, step, req_base and tau: the
 *          log-sum-exps of the walked rows come from that call.  After the
 *          stream beside the draft the bonus draws run with the residual
 *          draws (dspark_verify) or in a pass after the accept walk
 *          (dspark_verify_logits); after the epilogue form the bonus rows are
 *          streamed here.  A workspace whose last target-stream draft had
 *          other inputs sets status bit 3 (results unspecified).  Not for
 *          dspark_verify_rnn (DSPARK_ERR_UNSUPPORTED).
 * Optional: p_tok [B,gamma] receives p_k(x~_k) for walked rows (others untouched);
 *          near_ties [4] (zeroed by the caller) counts: [0] acceptance
 *          uniforms within 1e-5 of their threshold, [1] residual draws that
 *          fell back to p, [2] final draws, [3] reserved.
 */
dspark_status dspark_verify(
    const void* target, dspark_dtype target_t,
    const void* U, dspark_dtype U_t,
    const void* W1, const void* W2, dspark_dtype W_t,
    const int32_t* anchor, const int32_t* draft_tok,
    const float* lse_q, const float* z_tok, const int32_t* K,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* accepted, int32_t* out_tok, int32_t* out_req, int32_t* out_pos,
    int32_t* out_off, int32_t* next_anchor,
    float* p_tok, uint32_t* near_ties,
    void* ws, size_t ws_bytes, void* stream);

/*
 * dspark_verify with the draft's own logits: draft_logits [B,gamma,V] fp32 is
 * the z / tau that dspark_draft_markov wrote to its logits_out for these
 * drafts.  The residual draw of a rejected position reads its row there
 * instead of rebuilding it from W1, W2 and U, which saves a pass over W2 when
 * B * gamma * V is small enough to store (the latency path).  Otherwise
 * identical to dspark_verify (same outputs, same random streams).
 */
dspark_status dspark_verify_logits(
    const void* target, dspark_dtype target_t,
    const void* U, dspark_dtype U_t,
    const void* W1, const void* W2, dspark_dtype W_t,
    const float* draft_logits,
    const int32_t* anchor, const int32_t* draft_tok,
    const float* lse_q, const float* z_tok, const int32_t* K,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* accepted, int32_t* out_tok, int32_t* out_req, int32_t* out_pos,
    int32_t* out_off, int32_t* next_anchor,
    float* p_tok, uint32_t* near_ties,
    void* ws, size_t ws_bytes, void* stream);

/*
 * The draft loop with the RNN head [P2 §RNN Head：长程依赖], [P4 §三] in place
 * of the Markov head.  A GRU state carries every token of the block so far:
 *     s_k = GRU(s_{k-1}, E[x~_{k-1}])   (s_0 learned, x~_0 = anchor[b])
 *     z_k = (U[b,k-1,:] + bf16(s_k) . W2) / tau,  x~_k drawn as in
 *     dspark_draft_markov (same random stream, same outputs).
 * The GRU cell is the standard one (the pages print no formula), gate rows
 * stacked (r, z, n):
 *     r = sigma(W_ir x + b_ir + W_hr h + b_hr), z = sigma(W_iz x + b_iz + W_hz h + b_hz),
 *     n = tanh(W_in x + b_in + r * (W_hn h + b_hn)), h' = (1 - z) n + z h.
 * The input side enters through its per-token table P = E W_ih^T + b_ih
 * (dspark_rnn_input_table, computed once per set of weights).
 * Inputs : U [B,gamma,V] fp32, P [V,3r] fp32 (gate blocks r, z, n), W_hh
 *          [3r,r] bf16, b_hh [3r] and s0 [r] fp32, W2 [r,V] bf16 (W_t must
 *          be DSPARK_BF16), anchor [B].
 * Outputs: draft_tok, lse_q, z_tok as dspark_draft_markov; state
 *          [gamma,B,r] fp32 receives s_1..s_gamma (dspark_verify_rnn reads it).
 * ws     : as dspark_draft_markov (the GRU's scratch lives there too).
 * Limits : those of dspark_draft_markov, plus r % 64 == 0, r <= 256, fp32 U
 *          (else DSPARK_ERR_UNSUPPORTED).  One cooperative launch (2*gamma
 *          launches where cooperative launch is unavailable).
 */
dspark_status dspark_draft_rnn(
    const void* U, dspark_dtype U_t,
    const float* P, const void* W_hh, const float* b_hh, const float* s0,
    const void* W2, dspark_dtype W_t,
    const int32_t* anchor,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* draft_tok, float* lse_q, float* z_tok, float* state,
    void* ws, size_t ws_bytes, void* stream);

/*
 * The RNN head's input projections for every token: P[v][j] = sum_i E[v][i]
 * W_ih[j][i] + b_ih[j], j < 3r, fp32 accumulation.  E [V,r] and W_ih [3r,r]
 * bf16, b_ih [3r] fp32, P [V,3r] fp32 (caller-owned).  r % 8 == 0.
 */
dspark_status dspark_rnn_input_table(const void* E, const void* W_ih, const float* b_ih, int V, int r, float* P,
                                     void* stream);

/*
 * dspark_verify for drafts of the RNN head: identical, except that the
 * draft distribution of a rejected position k is rebuilt from
 * bf16(state[k-1]) . W2 (state as written by dspark_draft_rnn) instead of
 * W1[x~_{k-1}] . W2.  Same limits as dspark_draft_rnn.
 */
dspark_status dspark_verify_rnn(
    const void* target, dspark_dtype target_t,
    const void* U, dspark_dtype U_t,
    const float* state, const void* W2, dspark_dtype W_t,
    const int32_t* anchor, const int32_t* draft_tok,
    const float* lse_q, const float* z_tok, const int32_t* K,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* accepted, int32_t* out_tok, int32_t* out_req, int32_t* out_pos,
    int32_t* out_off, int32_t* next_anchor,
    float* p_tok, uint32_t* near_ties,
    void* ws, size_t ws_bytes, void* stream);

/*
 * The draft loop of dspark_draft_markov for callers that cannot allocate
 * device memory -- for example code inside a framework that owns all device
 * allocations, or a latency-critical loop that must not enter an allocator
 * (cudaMalloc may take locks and synchronise the device).  Arguments and
 * results are those of dspark_draft_markov without the workspace: the
 * kernels' scratch (status word, arrival and barrier counters, winner keys,
 * partial states) lives in a fixed array inside the library, 8.5 MiB + 1 KiB
 * per GPU, held until the process exits.  No counterpart on the pages: it is
 * a deployment option.
 *   - Limit: B <= 256 (any V, any gamma <= DSPARK_MAX_GAMMA).  Larger batches
 *     return DSPARK_ERR_UNSUPPORTED with a message on stderr.
 *   - Argument checks and error codes are those of dspark_draft_markov (host
 *     pointers: DSPARK_ERR_INVALID).
 *   - The first call on a device looks up the array's device address with
 *     that device current and keeps it for the life of the process; make
 *     that first call before any stream capture.  A cudaDeviceReset after it
 *     is not supported (the kept address would be stale).
 *   - Every call on a device shares the one array and clears its counters
 *     first: calls that may overlap on the GPU (different streams, or
 *     concurrent host threads) race and must be serialised by the caller.
 *   - Device-side range checks set bits in the array's status word; read and
 *     clear it with dspark_noalloc_sync_status.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 */
dspark_status dspark_draft_markov_noalloc(
    const void* U, dspark_dtype U_t,
    const void* W1, const void* W2, dspark_dtype W_t,
    const int32_t* anchor,
    int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step,
    int32_t* draft_tok, float* lse_q, float* z_tok, float* logits_out,
    void* stream);

/*
 * dspark_sync_status for the fixed array of dspark_draft_markov_noalloc on
 * the current device: synchronise `stream`, read and clear the array's status
 * word, same return values and bits.  Allocates nothing.
 */
dspark_status dspark_noalloc_sync_status(void* stream, uint32_t* bits);

/*
 * Sequential temperature scaling fit [P2 §校准问题：原始置信度不可靠], [P4 §四].
 * Off the decode path: it chooses the temperatures T that
 * dspark_confidence_sts applies, from a validation set of N drafted blocks.
 *   score   [N,gamma] fp32: logit(c_k), the confidence head's pre-sigmoid
 *           score of each draft position (finite).
 *   acc_len [N] int32: drafts of the block the target accepted (0..gamma);
 *           prefix k counts as accepted when acc_len >= k.
 *   grid    [G] fp32: candidate temperatures (positive, finite).
 * Left to right, for k = 1..gamma, with T_1..T_{k-1} already chosen:
 *   a_n(T)   = prod_{i<k} sigmoid(score[n,i] / T_i) * sigmoid(score[n,k] / T)
 *   ECE_k(T) = (1/N) sum_m | sum_{n: bin(a_n) = m} ([acc_len_n >= k] - a_n) |,
 *              bin(a) = min(floor(a*M), M-1)  (M equal-width bins of [0, 1])
 *   T_k      = grid[idx_k], idx_k the lowest index minimising ECE_k.
 * Outputs: T_out [gamma] fp32, idx_out [gamma] int32, ece_out [gamma,G] fp64.
 * Precision: survivals and bins in binary32 (a sample within about
 *   M*k*6e-7 of a bin edge in units of 1/M may land in the neighbouring
 *   bin), bin totals in 2^-24 fixed point, so equal candidates tie exactly.
 * ws     : dspark_sts_workspace_bytes(gamma, G, M) bytes, 256-byte aligned;
 *          the call clears it (no init needed) and keeps its status word at
 *          offset 0 (read it with dspark_sync_status: bit 3 reports a bad
 *          score or temperature; the results are then unspecified).
 * Limits : 1 <= gamma <= DSPARK_MAX_GAMMA, 1 <= G <= DSPARK_MAX_STS_GRID,
 *          1 <= M <= DSPARK_MAX_STS_BINS, N >= 1.  gamma launches on stream.
 */
size_t dspark_sts_workspace_bytes(int gamma, int G, int M);
dspark_status dspark_sts_fit(const float* score, const int32_t* acc_len, int N, int gamma,
                             const float* grid, int G, int M,
                             float* T_out, int32_t* idx_out, double* ece_out,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Diagnostics: the random stream as the kernels draw it.  For columns
 * v = 0..n-1 of stream (seed, step, domain, row) writes the uniform
 * u = (2*(x div 2^9) + 1) * 2^-24 and the Gumbel variate G = -log(-log u) the
 * kernels use (either output may be NULL, not both).  G is formed in binary32
 * with the hardware log2 and, for 1 - u < 1/8, a series for -log(1 - w);
 * it stays within ~2e-6 of the exact value.  No counterpart on the pages: it
 * exists so tests can check the device generator against the definition.
 */
dspark_status dspark_gumbel_stream(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, int n,
                                   float* gumbel_out, float* uniform_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DSPARK_H */
