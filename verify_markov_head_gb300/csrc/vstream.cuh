// vstream.cuh -- the verify stream's work loop ("DSpark：半自回归生成与置信度调度的投机解码",
// section 形式化定义): online log-sum-exps of the walked target rows and the
// bonus Gumbel-max draws, shared by the standalone stream kernel (verify.cu)
// and the stream role of the draft rows kernel (draft_rows.cu).  One
// instance is 9 warps (8 consumers, 1 producer) with its own shared-memory
// ring; instances claim work items from one global counter in the workspace.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dspark {

constexpr int kStreamConsumers = 8;                        // consumer warps
static_assert(kStreamConsumers == kVerifySub, "one partial state per consumer warp");
constexpr int kStreamThreads = (kStreamConsumers + 1) * 32;  // + one producer warp
constexpr int kStreamStages = 3;
constexpr int kStreamChunk = 8192;                           // entries per bulk copy
constexpr int kStreamStageBytes = kStreamChunk * 4;          // fp32 chunk (bf16 uses half)
// Beside the draft, whose W2 and U tiles go through the same SM's bulk-copy
// engine, a chunk is copied in pieces of this many bytes: one 32 KB copy held
// the draft's copies back longer than four of 8 KB (b64 step 293.2 -> 290.2
// us, b256 635.7 -> 622.9 us; 4 KB pieces were slower again).  The standalone
// stream keeps one copy a chunk (b512 with pieces: 1322.9 -> 1330.6 us).
constexpr uint32_t kSidePiece = 8192;
constexpr int kPerThread = kStreamChunk / (32 * kStreamConsumers);   // 32 entries per consumer per chunk
constexpr long long kStreamDrainCycles = 200000000LL;        // ~0.1 s: bulk copies already issued landing
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStreamKCache = 2048;                          // verify lengths kept in shared memory up to this B (8 KB)

constexpr int kStreamAll = 0, kStreamLse = 1, kStreamBonus = 2;

// Shared memory of one instance: the ring, its barriers, the abort flag, the
// stage tags and (B <= kStreamKCache) the verify lengths; 128-byte aligned.
template <int kStages = kStreamStages>
__host__ __device__ constexpr size_t vstream_smem_bytes(int B) {
    return (size_t)kStages * kStreamStageBytes + 16 * kStages + 16 + sizeof(int2) * kStages +
           (B <= kStreamKCache ? sizeof(int) * (size_t)B : 0);
}

// Persistent streaming pass over target rows.  Two kinds of work item:
//   log-sum-exp item (b, i, seg): a kVerifySeg-entry slice of row i < K_b
//     (a walked row); items with i >= K_b are skipped;
//   bonus item (b, seg): a kVerifySeg-entry slice of row K_b, the Gumbel-max
//     draw (domain 3) of the token emitted when all K_b drafts are accepted.
// kMode selects them: kStreamAll takes the bonus items of every request
// first (they cost several times a plain item) and then the log-sum-exp
// items, so the draws hide under the streaming of the other rows;
// kStreamLse the log-sum-exp items alone; kStreamBonus, launched after the
// accept walk, only the bonus items of the requests whose walk rejected
// nothing (ws.rej[b] < 0).  CTAs take items from a global counter (dynamic
// claiming keeps their loads even).  A producer thread moves every
// 8192-entry chunk of its items into a 3-stage shared-memory ring with one
// bulk copy (evict-first) and tags the stage with the item; 8 consumer warps
// keep per item either their running log-sum-exp in base-2 units across the
// chunks (per chunk a max pass, one rescale, then exp2 of x*log2e/tau - m in
// four independent partial sums) or their Gumbel-max draw.  Each consumer
// warp writes its own partial per item; for the bonus rows the warp that
// completes a request's partials (an arrival ticket per request) merges them
// and writes the request's final token.  A stage tagged -1 ends the stream.
// kCons consumer warps (8, or 4 in the lean instance that runs beside the
// draft) and a ring of kStages stages: with 4 consumers each warp takes the
// entries of two of the 8 consumer slots of a chunk, keeps one running state
// for both, writes the empty state to the second slot's partial and counts
// for both slots in a bonus row's arrival ticket.
template <typename TT, int kMode, int kCons = kStreamConsumers, int kStages = kStreamStages,
          uint32_t kPiece = (uint32_t)kStreamStageBytes>
__device__ __forceinline__ void vstream_run(const VerifyParams& p, uint8_t* gbase, uint32_t base, int tid, int bar_id,
                                         bool first_instance, unsigned ninst) {
    constexpr bool kHasBonus = kMode != kStreamLse, kHasLse = kMode != kStreamBonus;
    static_assert(kStreamConsumers % kCons == 0, "consumer slots split evenly over the warps");
    constexpr int kVirt = kStreamConsumers / kCons;              // consumer slots per warp
    constexpr int kThr = (kCons + 1) * 32;                       // threads of the instance
    const uint32_t bar0 = base + kStages * kStreamStageBytes;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kStages + i); };
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + kStages * kStreamStageBytes + 16 * kStages);
    int2* s_meta = reinterpret_cast<int2*>(gbase + kStages * kStreamStageBytes + 16 * kStages + 16);
    // the verify lengths, read once (every item needs its request's K_b; a
    // global load per item would stall the producer between items)
    int* s_K = reinterpret_cast<int*>(s_meta + kStages);
    const bool k_cached = p.B <= kStreamKCache;

    const int gamma = p.gamma, V = p.V;
    const int nseg = p.ws.nseg;
    const long long wl = wait_limit_of(p.ws.wait_limit);   // bound of the waits on the other role
    const int nbonus = kHasBonus ? p.B * nseg : 0;           // bonus items come first
    // rows with log-sum-exp items: the walked rows, and in full-prefix mode
    // beside the draft also row K_b = gamma (its draw runs with the residual)
    const int lextra = p.vs_full ? 1 : 0;
    const bool row_merge = vs_row_merge(p);
    const int lrows = gamma + lextra;
    const int items = nbonus + (kHasLse ? p.B * lrows * nseg : 0);
    const int warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) { ptx::mbar_init(full(i), 1); ptx::mbar_init(empty(i), kCons); }
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    if (k_cached)
        for (int b = tid; b < p.B; b += kThr) s_K[b] = p.K ? p.K[b] : gamma;
    if (first_instance && p.K)
        for (int b = tid; b < p.B; b += kThr)
            if (p.K[b] < 0 || p.K[b] > gamma) raise_status(p.ws.status, kBadLength);
    ptx::named_barrier(bar_id, kThr);

    auto clampK = [&](int b) {
        const int Kb = k_cached ? s_K[b] : (p.K ? p.K[b] : gamma);
        return Kb < 0 ? 0 : (Kb > gamma ? gamma : Kb);
    };
    // item u -> (b, i, seg); returns whether the item has work
    auto decode = [&](int u, int& b, int& i, int& seg) {
        if (u < nbonus) {
            b = u / nseg;
            seg = u - b * nseg;
            i = clampK(b);
            return kMode != kStreamBonus || __ldcg(&p.ws.rej[b]) < 0;
        }
        const int v = u - nbonus, per = lrows * nseg;
        b = v / per;
        const int rest = v - b * per;
        i = rest / nseg;
        seg = rest - i * nseg;
        return i < clampK(b) + lextra;
    };

    if (warp == kCons) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = ptx::policy_evict_first();
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long nf = 0;                            // bulk copies issued
            for (;;) {
                const int u = (int)atomicAdd(&p.ws.vq[0], 1u);
                if (u >= items) break;
                int b, i, seg;
                if (!decode(u, b, i, seg)) continue;
                const int v_end = min(V, (seg + 1) * kVerifySeg);
                const TT* row = static_cast<const TT*>(p.target) + ((size_t)b * (gamma + 1) + i) * V;
                for (int v0 = seg * kVerifySeg; v0 < v_end; v0 += kStreamChunk) {
                    if (!(ok = ptx::mbar_wait_strict(empty(stage), ph ^ 1u, abort_flag, wl))) break;
                    s_meta[stage] = make_int2(u, v0);
                    const uint32_t bytes = (uint32_t)(min(kStreamChunk, v_end - v0) * (int)sizeof(TT));
                    ptx::mbar_arrive_expect_tx(full(stage), bytes);
                    for (uint32_t o = 0; o < bytes; o += kPiece)
                        ptx::bulk_load(base + (uint32_t)stage * kStreamStageBytes + o,
                                       reinterpret_cast<const char*>(row + v0) + o, min(kPiece, bytes - o),
                                       full(stage), pol);
                    ++nf;
                    if (++stage == kStages) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
            }
            // the end-of-stream tag
            if (ok && (ok = ptx::mbar_wait_strict(empty(stage), ph ^ 1u, abort_flag, wl))) {
                s_meta[stage] = make_int2(-1, 0);
                ptx::mbar_arrive(full(stage));
                ++nf;                                    // the tag completes a phase of its stage too
            }
            if (!ok) { raise_status(p.ws.status, kTimeout); *abort_flag = 1u; }
            // every copy issued lands before the instance leaves: the last fill of
            // each stage (complete already unless the consumers gave up)
            for (int i = 0; i < kStages; ++i)
                if (nf > i) {
                    const long long m = (nf - 1) - ((nf - 1 - i) % kStages);
                    ptx::mbar_wait_drain(full(i), (uint32_t)((m / kStages) & 1), kStreamDrainCycles);
                }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const float scale = p.inv_tau * kLog2e;          // x * log2(e) / tau
        int stage = 0;
        uint32_t ph = 0;
        int cur = -1, b = 0, i = 0, seg = 0;
        bool bonus = false;                              // the current item is a bonus item
        float m2 = -INFINITY;                            // running max of x*log2e/tau
        float s4[4] = {0.f, 0.f, 0.f, 0.f};              // sum of 2^(x*log2e/tau - m2), four chains
        float best = -INFINITY;
        int bidx = 0x7fffffff;
        // the finished item's partial, in natural-log units
        auto flush = [&]() {
            LseDraw st;
            st.m = m2 * kLn2;
            st.s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
            st.best = best;
            st.idx = bidx;
            if (m2 == -INFINITY) { st.m = -INFINITY; st.s = 0.f; }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) st = lsedraw_merge(st, shfl_xor(st, m));
            LseDraw* row_part = p.ws.verify_part + ((size_t)b * (gamma + 1) + i) * nseg * kVerifySub;
            if (lane == 0) {
                row_part[seg * kVerifySub + warp] = st;
#pragma unroll
                for (int h = 1; h < kVirt; ++h) row_part[seg * kVerifySub + warp + h * kCons] = lsedraw_empty();
            }
            if (kHasLse && !bonus && row_merge) {
                // beside the draft of one chunk of requests the stream has time to
                // spare: the warp that writes a row's last partial (an arrival
                // ticket per row) merges them into the row's log-sum-exp, so the
                // accept walk reads one value per row (above 64 requests the
                // longer stream has no such slack: b256 measured 630 -> 652 us)
                const int nsub = nseg * kVerifySub;
                uint32_t* tk = &p.ws.row_tickets[(size_t)b * (gamma + 1) + i];
                unsigned last = 0u;
                if (lane == 0) {
                    __threadfence();
                    last = atomicAdd(tk, (unsigned)kVirt) == (unsigned)(nsub - kVirt) ? 1u : 0u;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    LseDraw a = lsedraw_empty();
                    for (int sg = lane; sg < nsub; sg += 32) {
                        const float4 c = __ldcg(reinterpret_cast<const float4*>(row_part) + sg);
                        a = lsedraw_merge(a, LseDraw{c.x, c.y, c.z, __float_as_int(c.w)});
                    }
#pragma unroll
                    for (int m = 1; m < 32; m <<= 1) a = lsedraw_merge(a, shfl_xor(a, m));
                    if (lane == 0) {
                        p.ws.row_lse[(size_t)b * (gamma + 1) + i] = a.m + logf(a.s);
                        *tk = 0u;                        // zero again for the next launch
                    }
                }
            }
            if (kHasBonus && bonus) {
                // the warp that completes request b's partials merges them into its token
                const int nsub = nseg * kVerifySub;
                unsigned last = 0u;
                if (lane == 0) {
                    __threadfence();
                    last = atomicAdd(&p.ws.bonus_tickets[b], (unsigned)kVirt) == (unsigned)(nsub - kVirt) ? 1u : 0u;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    LseDraw a = lsedraw_empty();
                    for (int sg = lane; sg < nsub; sg += 32) {
                        const float4 c = __ldcg(reinterpret_cast<const float4*>(row_part) + sg);
                        a = lsedraw_merge(a, LseDraw{c.x, c.y, c.z, __float_as_int(c.w)});
                    }
#pragma unroll
                    for (int m = 1; m < 32; m <<= 1) a = lsedraw_merge(a, shfl_xor(a, m));
                    if (lane == 0) {
                        p.ws.fin[b] = a.idx;
                        p.ws.bonus_tickets[b] = 0u;      // zero again for the next launch
                    }
                }
            }
        };
        for (;;) {
            bool ok = ptx::mbar_wait_strict(full(stage), ph, abort_flag, wl);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {                                   // a consumer gave up: report it too
                if (lane == 0) raise_status(p.ws.status, kTimeout);
                *abort_flag = 1u;
                break;
            }
            const int2 meta = s_meta[stage];
            if (meta.x < 0) break;                       // end of stream
            if (meta.x != cur) {                         // a new item
                if (cur >= 0) flush();
                cur = meta.x;
                decode(cur, b, i, seg);
                bonus = cur < nbonus;
                m2 = -INFINITY;
                s4[0] = s4[1] = s4[2] = s4[3] = 0.f;
                best = -INFINITY;
                bidx = 0x7fffffff;
            }
            const int v0 = meta.y;
            const int v_end = min(V, (seg + 1) * kVerifySeg);
            const int n = min(kStreamChunk, v_end - v0);
            const TT* sbuf = reinterpret_cast<const TT*>(gbase + (size_t)stage * kStreamStageBytes);
            const int stage_now = stage;
            if (++stage == kStages) { stage = 0; ph ^= 1u; }
#pragma unroll 1
            for (int h = 0; h < kVirt; ++h) {
            const int vt = tid + h * 32 * kCons;          // the consumer slot's thread index
            float x[kPerThread];                          // raw target logits
#pragma unroll
            for (int j = 0; j < kPerThread / 4; ++j) {
                const int e0 = 4 * (vt + j * 32 * kStreamConsumers);
                const float4 x4 = (e0 < n) ? Vec4<TT>::load(sbuf + e0)
                                           : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                x[4 * j] = x4.x; x[4 * j + 1] = x4.y; x[4 * j + 2] = x4.z; x[4 * j + 3] = x4.w;
            }
            if (h == kVirt - 1) {
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(empty(stage_now));   // the chunk is in registers
            }
            float cm = x[0];
#pragma unroll
            for (int e = 1; e < kPerThread; ++e) cm = fmaxf(cm, x[e]);
            cm *= scale;                                  // scale > 0 keeps the maximum
            if (!bonus && cm > m2) {
                const float r = fast_exp2(m2 - cm);          // 0 when m2 = -inf
#pragma unroll
                for (int c = 0; c < 4; ++c) s4[c] *= r;
                m2 = cm;
            }
            if (!bonus && m2 > -INFINITY) {
                // two entries per packed multiply-add and add
                const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(-m2, -m2);
                float2 a01 = make_float2(s4[0], s4[1]), a23 = make_float2(s4[2], s4[3]);
#pragma unroll
                for (int e = 0; e < kPerThread; e += 4) {
                    const float2 y01 = __ffma2_rn(make_float2(x[e], x[e + 1]), sc2, nm2);
                    const float2 y23 = __ffma2_rn(make_float2(x[e + 2], x[e + 3]), sc2, nm2);
                    a01 = __fadd2_rn(a01, make_float2(fast_exp2(y01.x), fast_exp2(y01.y)));
                    a23 = __fadd2_rn(a23, make_float2(fast_exp2(y23.x), fast_exp2(y23.y)));
                }
                s4[0] = a01.x; s4[1] = a01.y; s4[2] = a23.x; s4[3] = a23.y;
            }
            if (kHasBonus && bonus) {
                // Gumbel-max as an exponential race against this thread's chunk
                // maximum cm: argmax x/tau + G = argmin E2 * 2^(cm - x*log2e/tau),
                // E2 = -log2 u (no outer logarithm, no divergent screen); the
                // chunk's winner goes back to a score for the running draw:
                //   x/tau + G = cm ln2 - ln(key ln2).
                const StreamRK rng(p.seed, p.step, 3u, (uint32_t)(p.req_base + b) * (uint32_t)(gamma + 1) + (uint32_t)i);
                float kbest = INFINITY;
                int kidx = 0x7fffffff;
#pragma unroll
                for (int j = 0; j < kPerThread / 4; ++j) {
                    const int e0 = 4 * (vt + j * 32 * kStreamConsumers);
                    if (e0 < n) {
                        const int v = v0 + e0;
                        const uint4 wq = rng.quad((uint32_t)v >> 2);
                        const uint32_t ws[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float key = exp2_variate_of(ws[e]) * fast_exp2(fmaf(-x[4 * j + e], scale, cm));
                            if (key < kbest) { kbest = key; kidx = v + e; }   // increasing v: lowest index on ties
                        }
                    }
                }
                if (kbest < INFINITY) {
                    const float sc = cm * kLn2 - logf(kbest * kLn2);
                    if (wins(sc, kidx, best, bidx)) { best = sc; bidx = kidx; }
                }
            }
            }
        }
        if (cur >= 0 && !*abort_flag) flush();
    }
    ptx::named_barrier(bar_id, kThr);
    // the last instance out clears the work counter for the next launch
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.ws.vq[1], 1u) == ninst - 1) {
            p.ws.vq[0] = 0u;
            p.ws.vq[1] = 0u;
            __threadfence();
        }
    }
}


}  // namespace dspark
