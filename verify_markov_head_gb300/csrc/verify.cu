// verify.cu -- lossless verification and ragged compaction
// ("DSpark：半自回归生成与置信度调度的投机解码" section 形式化定义;
//  "DeepSeek-AI与北京大学联手破局" sections 四 and 五).
//
// Four or five launches, all stream-ordered and free of waits:
//   verify_stream   rows i = 0..K_b-1 of the target logits in 32768-entry
//                   segments: online log-sum-exp of t/tau, bulk copies into
//                   shared memory (evict-first).  With an fp32 target it also
//                   draws the bonus token of every request on row K_b
//                   (Gumbel-max, domain 3), hidden under the streaming.
//                   Full-prefix mode skips it (the draft reduced the rows).
//   verify_accept   one warp per request: merges the partials into lse_p per
//                   row, walks k = 1..K_b with the acceptance uniforms
//                   (domain 1), records the first rejection.
//   verify_residual rejected requests only: recomputes the draft logits of
//                   the rejected row (bias h . W2 plus U), forms
//                   max(0, p - q) and draws from it by Gumbel-max (domain 2),
//                   with the draw from p kept as the fallback.
//   verify_stream   (bf16 target, full-prefix mode, stored logits) the bonus
//                   draw of the requests that accepted all K_b drafts only:
//                   the draw needs a random number per entry, and with
//                   nothing to hide it, drawing it only where it is emitted
//                   saves most of that work.
//   verify_compact  one CTA: exclusive scan of A_b + 1, scatter of the
//                   accepted drafts and the final token of every request.
// The last warp to finish a request's bonus segments merges them into its
// token.
#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"
#include "vstream.cuh"
#include "pdl.cuh"
#include "resid_tail.cuh"

namespace dspark {
namespace {

template <typename T>
__device__ __forceinline__ float load_scalar(const T* p, size_t i) { return to_f32(p[i]); }

// The standalone verify stream: one instance per CTA, two CTAs per SM.
template <typename TT, int kMode>
__global__ void __launch_bounds__(kStreamThreads, 2)
verify_stream_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    grid_dependency_wait();
    vstream_run<TT, kMode>(p, smem_raw + (base - raw), base, (int)threadIdx.x, 1, blockIdx.x == 0, gridDim.x);
}

// The lean instance that runs beside the draft: 4 consumer warps (2 for one
// chunk of several requests, 1 < B <= 64, whose stream is short: at half the
// rate it disturbs the draft less) and a 2-stage ring (about 65 KB of shared memory,
// at most 160 threads of at most 72 registers), which fits next to one draft
// CTA on an SM.  It reduces rows
// 0..gamma of every request (vs_full): the walked rows and the bonus row,
// whose draw then runs in the residual kernel (a random number per entry
// beside the draft would compete with the draft's own).  It needs nothing
// the draft writes, so it starts without waiting on it; it waits at its end,
// so that the launches behind it see the draft's outputs too.
constexpr int kSideStages = 2;

template <typename TT, int kCons>
__global__ void __maxnreg__(72) verify_stream_side_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    // the launch behind this one (the accept walk) is scheduled now and
    // waits for this grid, so its launch latency hides under the draft
    if (threadIdx.x == 0) grid_launch_dependents();
    vstream_run<TT, kStreamLse, kCons, kSideStages, kSidePiece>(p, smem_raw + (base - raw), base, (int)threadIdx.x, 1,
                                                    blockIdx.x == 0, gridDim.x);
    if (threadIdx.x == 0 && blockIdx.x == 0) *p.ws.tgt_token = p.tgt_token;
    grid_dependency_wait();
}

constexpr int kAcceptStaged = 2048;   // partials staged in shared memory (32 KB)

// One warp per request: lse_p of the walked rows 0..K_b-1 from the partials,
// then the accept test of every walked position at once (lane k-1 tests draft
// k), the first rejection found by a ballot.  The partials of a row are the
// verify stream's segment partials, or in full-prefix mode (K null) the
// draft's target-stream partials.
template <typename TT>
__global__ void __launch_bounds__(32)
verify_accept_kernel(const VerifyParams p) {
    // the residual launch behind this one starts its set-up (TMEM, barriers,
    // the W2 prefetch) during the walk; it waits for the walk before reading
    if (threadIdx.x == 0) grid_launch_dependents();
    grid_dependency_wait();
    const int b = blockIdx.x, lane = threadIdx.x;
    const int gamma = p.gamma, V = p.V, nseg = p.ws.nseg;
    const bool full = p.tgt_slots > 0;              // the walked rows' partials are the draft's own
    int Kb = p.K ? p.K[b] : gamma;
    Kb = Kb < 0 ? 0 : (Kb > gamma ? gamma : Kb);
    // full-prefix mode needs the target-stream results of this very call's inputs
    if (!p.K && b == 0 && lane == 0 && *p.ws.tgt_token != p.tgt_token) raise_status(p.ws.status, kBadInput);
    const TT* target = static_cast<const TT*>(p.target);
    const uint32_t row0 = (uint32_t)(p.req_base + b) * (uint32_t)(gamma + 1);
    // per-lane draft data for position k = lane + 1 (issued before the merges)
    int x = 0, x_raw = -1;
    float t = 0.f, lq = 0.f, u = 1.f;
    const bool walk = lane < Kb;
    // the token before draft k+1, whose W1 row the residual draw gathers if
    // draft k+1 is rejected: lane k holds draft k, lane 31 the anchor
    if (lane == 31 && Kb > 0) x_raw = p.anchor[b];
    if (walk) {
        const size_t o = (size_t)b * gamma + lane;
        x = x_raw = p.draft_tok[o];
        if (x < 0 || x >= V) { raise_status(p.ws.status, kBadToken); x = 0; }
        t = load_scalar(target, ((size_t)b * (gamma + 1) + lane) * V + x) * p.inv_tau;
        lq = p.z_tok[o] - p.lse_q[o];
        u = uniform_of(Stream(p.seed, p.step, 1u, row0 + (uint32_t)lane).word(0));
    }
    // every row the residual may gather, on its way to L2 during the walk
    // (the stored-logits residual and the RNN head read no W1 row)
    if (!p.zlog && !p.state && (lane == 31 || lane + 1 < Kb) && x_raw >= 0 && x_raw < V) {
        const size_t rb = (size_t)p.r * (p.W_bf16 ? 2 : 4);
        ptx::prefetch_l2(static_cast<const char*>(p.W1) + (size_t)x_raw * rb, (uint32_t)rb);
    }
    float lse_mine = 0.f;        // lse_p of row `lane` (walked rows 0..K_b-1)
    const int nsub = nseg * kVerifySub;            // verify-stream partials per row
    const LseDraw* parts = p.ws.verify_part + (size_t)b * (gamma + 1) * nsub;
    const int ns = full ? p.tgt_slots : nsub;      // partials per walked row
    const LseDraw* rows = full ? p.ws.tgt_part + (size_t)b * gamma * kTgtSlots : parts;
    const size_t rstride = full ? (size_t)kTgtSlots : (size_t)nsub;
    // full prefix beside the draft: row K_b too (the bonus draw's law)
    const int nrows = Kb + (p.vs_full ? 1 : 0);
    const int nparts = nrows * ns;                 // rows 0..nrows-1, staged row after row
    if (vs_row_merge(p)) {
        // the stream beside the draft merged every row already
        if (lane < nrows) lse_mine = __ldcg(&p.ws.row_lse[(size_t)b * (gamma + 1) + lane]);
    } else if (nrows > 0 && nparts <= kAcceptStaged) {
        // the partials of the walked rows, every load in flight, through shared
        // memory (row i from index i * ns); then lanes fold their row
        __shared__ float4 s_part[kAcceptStaged];
        for (int i0 = lane; i0 < nparts; i0 += 12 * 32) {
            float4 c[12];
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                const int i = i0 + 32 * u;
                if (i < nparts) {
                    const int row = i / ns;
                    c[u] = __ldcg(reinterpret_cast<const float4*>(rows + row * rstride) + (i - row * ns));
                }
            }
#pragma unroll
            for (int u = 0; u < 12; ++u) {
                const int i = i0 + 32 * u;
                if (i < nparts) s_part[i] = c[u];
            }
        }
        __syncwarp();
        // LPR lanes per row (a power of two with K_b * LPR <= 32) fold every
        // LPR-th partial of their row, then a shuffle tree joins them
        int LPR = 32;
        while (LPR > 1 && nrows * LPR > 32) LPR >>= 1;
        const int row = lane / LPR, sub = lane - row * LPR;
        LseDraw a = lsedraw_empty();
        if (row < nrows)
            for (int sg = sub; sg < ns; sg += LPR) {
                const float4 c = s_part[row * ns + sg];
                a = lsedraw_merge(a, LseDraw{c.x, c.y, c.z, __float_as_int(c.w)});
            }
        for (int m = 1; m < LPR; m <<= 1) a = lsedraw_merge(a, shfl_xor(a, m));
        const float lse_row = a.m + logf(a.s);         // on lanes row * LPR
        lse_mine = __shfl_sync(0xffffffffu, lse_row, (lane * LPR) & 31);
    } else {
        for (int i = 0; i < nrows; ++i) {
            const LseDraw* part = rows + i * rstride;
            LseDraw a = lsedraw_empty();
            for (int sg = lane; sg < ns; sg += 32) a = lsedraw_merge(a, part[sg]);
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) a = lsedraw_merge(a, shfl_xor(a, m));
            if (lane == i) lse_mine = a.m + logf(a.s);
        }
    }
    bool reject = false, near = false;
    if (walk) {
        const float lp = t - lse_mine;
        if (p.p_tok) p.p_tok[(size_t)b * gamma + lane] = expf(lp);
        const float thr = fminf(1.f, expf(lp - lq));
        reject = !(u < thr);
        near = fabsf(u - thr) < 1e-5f;
    }
    const unsigned rej_mask = __ballot_sync(0xffffffffu, reject);
    const int rej = rej_mask ? __ffs(rej_mask) - 1 : -1;     // 0-based row of the first rejection
    if (p.near_ties && near && (rej < 0 || lane <= rej)) atomicAdd(&p.near_ties[0], 1u);   // decisions taken
    const float lse_rej = __shfl_sync(0xffffffffu, lse_mine, rej < 0 ? 0 : rej);
    const float lse_bonus = __shfl_sync(0xffffffffu, lse_mine, Kb & 31);   // row K_b (full prefix beside the draft)
    const int x_prev = __shfl_sync(0xffffffffu, x_raw, rej <= 0 ? 31 : rej - 1);
    if (lane == 0) {
        const int A = rej < 0 ? Kb : rej;
        p.ws.acc[b] = A;
        p.ws.rej[b] = rej;      // the final token: the residual draw (rej >= 0) or the bonus pass
        p.ws.rtok[b] = rej < 0 ? -1 : x_prev;
        if (rej >= 0) p.ws.lse_rej[b] = make_float2(lse_rej, p.lse_q[(size_t)b * gamma + rej]);
        // the bonus draw in the residual kernel: the law p of row K_b (q taken as 0)
        else if (p.vs_full) p.ws.lse_rej[b] = make_float2(lse_bonus, INFINITY);
        p.accepted[b] = A;
    }
}

// ----------------------------------------------------------------- residual
constexpr int kTV = 128;
constexpr int kBC = dspark::kChunk;   // requests per residual chunk
constexpr int kResThreads = 256;

// kStored: the draft logits z [B][gamma][V] (already divided by tau) were
// stored by the draft (p.zlog): the rejected row is read from there instead
// of being rebuilt from W1, W2 and U.
template <typename WT, typename UT, typename TT, bool kStored = false>
__global__ void __launch_bounds__(kResThreads)
verify_residual_simt_kernel(const VerifyParams p) {
    extern __shared__ __align__(16) float smem[];
    const int r = p.r, V = p.V, gamma = p.gamma;
    float* sh = smem;                                   // [kBC][r] (not in the stored mode)
    float* tile = smem + (kStored ? 0 : kBC * r);       // [kBC][kTV + 4] draft logits z
    constexpr int kLd = kTV + 4;
    __shared__ int s_row[kBC];
    __shared__ int s_any;

    const int tid = threadIdx.x, chunk = blockIdx.y, b0 = chunk * kBC;
    const int nb = min(kBC, p.B - b0);
    if (tid == 0) s_any = 0;
    __syncthreads();
    // the stored-logits draw after the stream beside the draft (vs_full) also
    // takes the bonus token of every request that rejected nothing: row gamma
    // of the target, q taken as 0 (its log-normaliser is +inf), the bonus
    // noise (domain 3); such a request is marked with row gamma here
    const bool bonus_here = kStored && p.vs_full;
    if (tid < kBC) {
        int row = (tid < nb) ? __ldcg(&p.ws.rej[b0 + tid]) : -1;
        if (bonus_here && tid < nb && row < 0) row = gamma;
        s_row[tid] = row;
        if (row >= 0) atomicOr(&s_any, 1);
    }
    __syncthreads();
    const WT* W1 = static_cast<const WT*>(p.W1);
    const WT* W2 = static_cast<const WT*>(p.W2);
    const UT* U = static_cast<const UT*>(p.U);
    const TT* target = static_cast<const TT*>(p.target);

    const int warp = tid / 32, lane = tid % 32;
    const int bl_e = tid / 16, seg = tid % 16;
    Draw2 st = draw2_empty();
    if (s_any) {
        for (int i = tid; i < (kStored ? 0 : kBC * r); i += kResThreads) {
            const int bl = i / r, rho = i - bl * r;
            float v = 0.f;
            const int row = s_row[bl];
            if (row >= 0) {
                const int b = b0 + bl;
                int x = (row == 0) ? p.anchor[b] : p.draft_tok[(size_t)b * gamma + row - 1];
                if (x >= 0 && x < V) v = to_f32(W1[(size_t)x * r + rho]);
            }
            sh[i] = v;
        }
        __syncthreads();
        const int v_local = tid % kTV, bh = tid / kTV;
        const int ntiles = (V + kTV - 1) / kTV;
        const int my_row = (bl_e < nb) ? s_row[bl_e] : -1;
        const float2 lse = (my_row >= 0) ? p.ws.lse_rej[b0 + bl_e] : make_float2(0.f, 0.f);
        const Stream rng(p.seed, p.step, (kStored && my_row == gamma) ? 3u : 2u,
                         (uint32_t)(p.req_base + b0 + bl_e) * (uint32_t)(gamma + 1) + (uint32_t)(my_row < 0 ? 0 : my_row));
        const TT* trow = target + ((size_t)(b0 + bl_e) * (gamma + 1) + (my_row < 0 ? 0 : my_row)) * V;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int v0 = t * kTV;
            const int v = v0 + v_local;
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
            if (!kStored && v < V) {
                const float* hb = sh + (bh * 8) * r;
                for (int rho = 0; rho < r; ++rho) {
                    const float w = to_f32(W2[(size_t)rho * V + v]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = fmaf(hb[j * r + rho], w, acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int bl = bh * 8 + j;
                const int row = s_row[bl];
                float z = 0.f;
                if (row >= 0 && v < V) {
                    if constexpr (kStored)
                        z = row < gamma ? p.zlog[((size_t)(b0 + bl) * gamma + row) * V + v] : 0.f;
                    else
                        z = (to_f32(U[((size_t)(b0 + bl) * gamma + row) * V + v]) + acc[j]) * p.inv_tau;
                }
                tile[bl * kLd + v_local] = z;
            }
            __syncthreads();
            if (my_row >= 0) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int vl = seg * 8 + q * 4;
                    const int vq = v0 + vl;
                    if (vq < V) {
                        const uint4 w = rng.quad((uint32_t)vq >> 2);
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                        const float4 t4 = Vec4<TT>::load(trow + vq);
                        const float ts[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float z = tile[bl_e * kLd + vl + e];
                            const float tv = ts[e] * p.inv_tau;
                            const float g = gumbel_of(ws[e]);
                            const float pr = expf(tv - lse.x) - expf(z - lse.y);
                            const int idx = vq + e;
                            if (pr > 0.f) {
                                const float sc = logf(pr) + g;
                                if (wins(sc, idx, st.best_r, st.idx_r)) { st.best_r = sc; st.idx_r = idx; }
                            }
                            const float sp = tv + g;
                            if (wins(sp, idx, st.best_p, st.idx_p)) { st.best_p = sp; st.idx_p = idx; }
                        }
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int m = 1; m < 16; m <<= 1) st = draw2_merge(st, shfl_xor(st, m));
        if (seg == 0 && my_row >= 0) p.ws.resid_part[(size_t)(b0 + bl_e) * p.ws.parts + blockIdx.x] = st;
    }

    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&p.ws.tickets_resid[chunk], 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int bl = warp; bl < nb; bl += kResThreads / 32) {
        if (s_row[bl] < 0) continue;
        const int b = b0 + bl;
        const Draw2* part = p.ws.resid_part + (size_t)b * p.ws.parts;
        Draw2 a = draw2_empty();
        for (int i = lane; i < (int)gridDim.x; i += 32) {
            Draw2 c;
            c.best_r = __ldcg(&part[i].best_r); c.idx_r = __ldcg(&part[i].idx_r);
            c.best_p = __ldcg(&part[i].best_p); c.idx_p = __ldcg(&part[i].idx_p);
            a = draw2_merge(a, c);
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) a = draw2_merge(a, shfl_xor(a, m));
        if (lane == 0) {
            if (a.best_r > -INFINITY) {
                p.ws.fin[b] = a.idx_r;
            } else {
                p.ws.fin[b] = a.idx_p;
                if (p.near_ties) atomicAdd(&p.near_ties[1], 1u);
            }
        }
    }
    if (tid == 0) p.ws.tickets_resid[chunk] = 0u;
}

// ----------------------------------------------------------------- compaction
constexpr int kCompactThreads = 1024;

// After the tensor-core residual launch (p.resid_keys) the final tokens of
// the requests it drew (every rejected one, and with the stream beside the
// draft the bonus draws too) are still winner keys: they are decoded here
// first, the keys cleared for the next draft, and a request whose residual
// had no mass at all draws from p itself (the fallback law).
template <typename TT>
__global__ void __launch_bounds__(kCompactThreads)
verify_compact_kernel(const VerifyParams p) {
    __shared__ int s_warp[kCompactThreads / 32];
    __shared__ int s_carry;
    __shared__ int s_nfb;
    __shared__ int s_fb[kCompactThreads];
    grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int gamma = p.gamma;
    if (tid == 0) s_carry = 0;
    for (int base = 0; base < p.B; base += kCompactThreads) {
        const int b = base + tid;
        const bool in = b < p.B;
        if (tid == 0) s_nfb = 0;
        // every load of request b at once: its accepted count, its final token
        // or winner key, and its drafts
        int A = 0, rej = -1, fin = 0;
        unsigned long long key = 0ull;
        int tk[DSPARK_MAX_GAMMA];
        if (in) {
            A = __ldcg(&p.ws.acc[b]);
            fin = __ldcg(&p.ws.fin[b]);
            if (p.resid_keys) {
                rej = __ldcg(&p.ws.rej[b]);
                key = __ldcg(&p.ws.win[(size_t)b * kWinStride]);
            }
#pragma unroll
            for (int i = 0; i < DSPARK_MAX_GAMMA; ++i)
                if (i < gamma) tk[i] = __ldcg(&p.draft_tok[(size_t)b * gamma + i]);
        }
        __syncthreads();
        bool fb = false;
        if (in && p.resid_keys && (rej >= 0 || p.vs_full)) {
            p.ws.win[(size_t)b * kWinStride] = 0ull;   // cleared for the next draft
            if (key != 0ull) {
                fin = win_token(key);
                p.ws.fin[b] = fin;
            } else {
                fb = true;                              // no residual mass: draw from p below
                s_fb[atomicAdd(&s_nfb, 1)] = b;
                if (p.near_ties) atomicAdd(&p.near_ties[1], 1u);
            }
        }
        __syncthreads();
        for (int f = 0; f < s_nfb; ++f) {           // uniform loop; a bonus request draws on row gamma
            const int bb = s_fb[f];
            const int rb = __ldcg(&p.ws.rej[bb]);
            resid_fallback_draw<TT>(p.seed, p.step, p.req_base, gamma, p.V, p.inv_tau, p.ws.lse_rej[bb].x,
                                    p.target, bb, rb >= 0 ? rb : gamma, rb >= 0 ? 2u : 3u, &p.ws.fin[bb]);
        }
        if (fb) fin = __ldcg(&p.ws.fin[b]);          // written by this CTA before the draw's barrier
        // offsets: an exclusive prefix sum of A + 1 over the requests
        const int len = in ? A + 1 : 0;
        int incl = len;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, m);
            if (lane >= m) incl += y;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = s_warp[lane];
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, m);
                if (lane >= m) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int off = s_carry + (warp ? s_warp[warp - 1] : 0) + incl - len;
        if (in) {
#pragma unroll
            for (int i = 0; i < DSPARK_MAX_GAMMA; ++i)
                if (i < A) {
                    p.out_tok[off + i] = tk[i];
                    p.out_req[off + i] = b;
                    p.out_pos[off + i] = i;
                }
            p.out_tok[off + A] = fin;
            p.out_req[off + A] = b;
            p.out_pos[off + A] = A;
            p.out_off[b] = off;
            p.next_anchor[b] = fin;
        }
        __syncthreads();
        if (tid == 0) s_carry += s_warp[kCompactThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) {
        p.out_off[p.B] = s_carry;
        if (p.near_ties) atomicAdd(&p.near_ties[2], (unsigned)p.B);
    }
}

template <typename TT>
cudaError_t launch_verify_t(const VerifyParams& p, cudaStream_t s) {
    const size_t smem1 = 128 + vstream_smem_bytes(p.B);
    auto stream_grid = [&](long long items) {
        return (int)(items < 2LL * num_sms() ? items : 2LL * num_sms());
    };
    // The bonus draws ride in the log-sum-exp stream (kStreamAll) while its
    // fp32 rows keep it bound by HBM, which hides them.  A bf16 target halves
    // the bytes and leaves the draws exposed, full-prefix mode has no stream
    // before the accept walk, and the stored-logits path serves small steps:
    // there the draws run after the walk, for the requests that emit them.
    // Beside the draft (vs_full) the residual kernel draws them, the
    // tensor-core one or the stored-logits one (b1 step 143.9 -> 139.2 us
    // without the pass).
    const bool deferred = !p.vs_full && (p.zlog != nullptr || p.target_bf16 || p.tgt_slots > 0);
    const long long lse_items = (long long)p.B * p.gamma * p.ws.nseg;
    const long long bonus_items = (long long)p.B * p.ws.nseg;
    cudaError_t e0 = cudaSuccess;
    if (p.vs_full) {
        // the stream ran beside the draft: nothing to stream here
    } else if (!deferred) {
        e0 = cudaFuncSetAttribute(verify_stream_kernel<TT, kStreamAll>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem1);
        if (e0 != cudaSuccess) return e0;
        e0 = launch_dependent(verify_stream_kernel<TT, kStreamAll>, dim3(stream_grid(bonus_items + lse_items)),
                              dim3(kStreamThreads), smem1, s, p);
        if (e0 != cudaSuccess) return e0;
    } else if (p.tgt_slots == 0) {
        e0 = cudaFuncSetAttribute(verify_stream_kernel<TT, kStreamLse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem1);
        if (e0 != cudaSuccess) return e0;
        e0 = launch_dependent(verify_stream_kernel<TT, kStreamLse>, dim3(stream_grid(lse_items)), dim3(kStreamThreads),
                              smem1, s, p);
        if (e0 != cudaSuccess) return e0;
    }
    e0 = launch_dependent(verify_accept_kernel<TT>, dim3(p.B), dim3(32), 0, s, p);
    if (e0 != cudaSuccess) return e0;
    // the final token: the residual draw of the rejected requests (and, when
    // deferred, the bonus draw of the others), then the ragged layout
    auto finish = [&]() {
        if (deferred) {
            cudaError_t e = cudaFuncSetAttribute(verify_stream_kernel<TT, kStreamBonus>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
            if (e != cudaSuccess) return e;
            e = launch_dependent(verify_stream_kernel<TT, kStreamBonus>, dim3(stream_grid(bonus_items)),
                                 dim3(kStreamThreads), smem1, s, p);
            if (e != cudaSuccess) return e;
        }
        const cudaError_t e = launch_dependent(verify_compact_kernel<TT>, dim3(1), dim3(kCompactThreads), 0, s, p);
        return e != cudaSuccess ? e : cudaGetLastError();
    };
    const int nchunks = (p.B + kBC - 1) / kBC;
    const int ntiles = (p.V + kTV - 1) / kTV;
    int gx = (4 * num_sms()) / nchunks;
    gx = gx < 1 ? 1 : (gx > ntiles ? ntiles : gx);
    gx = gx > p.ws.parts ? p.ws.parts : gx;
    const size_t smem = sizeof(float) * ((size_t)kBC * p.r + (size_t)kBC * (kTV + 4));
    const dim3 g2(gx, nchunks);
    if (p.zlog) {
        // the draft's own logits: the rejected rows are read, not rebuilt
        auto kern = verify_residual_simt_kernel<float, float, TT, true>;
        const size_t smem_z = sizeof(float) * (size_t)kBC * (kTV + 4);
        kern<<<g2, kResThreads, smem_z, s>>>(p);
        return finish();
    }
    if (p.state && !resid_rows_supported(p)) return cudaErrorNotSupported;   // RNN rows: tensor-core path only
    if (p.state || resid_rows_supported(p)) {
        const cudaError_t e = launch_resid_rows(p, s);
        if (e != cudaSuccess) return e;
        VerifyParams pk = p;
        pk.resid_keys = 1;                       // the residual's draws are winner keys
        if (deferred) {
            cudaError_t e2 = cudaFuncSetAttribute(verify_stream_kernel<TT, kStreamBonus>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
            if (e2 != cudaSuccess) return e2;
            e2 = launch_dependent(verify_stream_kernel<TT, kStreamBonus>, dim3(stream_grid(bonus_items)),
                                  dim3(kStreamThreads), smem1, s, p);
            if (e2 != cudaSuccess) return e2;
        }
        const cudaError_t e3 = launch_dependent(verify_compact_kernel<TT>, dim3(1), dim3(kCompactThreads), 0, s, pk);
        return e3 != cudaSuccess ? e3 : cudaGetLastError();
    }
#define DSPARK_RES_LAUNCH(WT, UT)                                                                    \
    do {                                                                                             \
        auto kern = verify_residual_simt_kernel<WT, UT, TT>;                                         \
        if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        kern<<<g2, kResThreads, smem, s>>>(p);                                                       \
    } while (0)
    if (p.W_bf16) {
        if (p.U_bf16) DSPARK_RES_LAUNCH(uint16_t, uint16_t); else DSPARK_RES_LAUNCH(uint16_t, float);
    } else {
        if (p.U_bf16) DSPARK_RES_LAUNCH(float, uint16_t); else DSPARK_RES_LAUNCH(float, float);
    }
#undef DSPARK_RES_LAUNCH
    return finish();
}

}  // namespace

template <typename TT, int kCons>
static cudaError_t launch_side_t(const VerifyParams& v, cudaStream_t s) {
    const size_t smem = 128 + vstream_smem_bytes<kSideStages>(v.B);
    auto kern = verify_stream_side_kernel<TT, kCons>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, dim3(num_sms()), dim3((kCons + 1) * 32), smem, s, v);
}

// Measured (graph-replay steps, same outputs): two consumer warps at b64
// (296.6 -> 294.7 us), four at b256 (653.5 with two against 627.6 us) and at
// b1, whose draft leaves no room beside it, so the stream runs after it
// (142.8 against 145.5 us with two).
cudaError_t launch_target_stream_side(const VerifyParams& v, cudaStream_t s) {
    if (v.B > 1 && v.B <= 64) return v.target_bf16 ? launch_side_t<uint16_t, 2>(v, s) : launch_side_t<float, 2>(v, s);
    return v.target_bf16 ? launch_side_t<uint16_t, 4>(v, s) : launch_side_t<float, 4>(v, s);
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
    return p.target_bf16 ? launch_verify_t<uint16_t>(p, s) : launch_verify_t<float>(p, s);
}

}  // namespace dspark
