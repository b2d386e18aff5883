// draft_rows.cu -- Markov-head draft position on the tcgen05 tensor cores,
// requests on the TMEM lanes (any batch with bf16 weights, fp32 U and
// r a multiple of 64 up to 256).
//
// Per position k ("DSpark：半自回归生成与置信度调度的投机解码" sections 整体架构 and
// Markov Head; "拒绝盲猜与算力空转" section on the low-rank Markov head):
//   bias[b, v] = W1[x~_{k-1}(b)] . W2[:, v]      (rank r, bf16 in, fp32 accumulate)
//   z[b, v]    = (U[b, k-1, v] + bias[b, v]) / tau
//   x~_k       = argmax_v z + G,  lse_q = log sum exp z,  z_tok = z[x~_k]
//
// D[M = 128 rows, N = 128 vocabulary entries] = U tile + h * W2tile over K = r:
//   A = the gathered rows h = W1[x~_{k-1}] in TMEM (r bf16 per lane packed two
//       to a column, written by the epilogue warps with tcgen05.st once per
//       position; rows past the batch are zero),
//   B = a 128-entry slice of W2 read by TMA straight from the [r, V] row-major
//       tensor (MN-major, 128-byte swizzle), in 64-rank K-chunks,
//   D = fp32 in TMEM, 4 - RF buffers so the MMAs of later tiles overlap the
//       epilogue of a tile.  Before the MMAs D is loaded with the tile's U:
//       the U slices arrive by TMA (128 rows x 32 fp32, 128-byte swizzle) and
//       tcgen05.cp copies them into the accumulator, so the epilogue reads
//       U + bias in one tcgen05.ld and the U ring turns over as soon as the
//       copies have read it.
// A chunk of NC = 64 requests would leave TMEM lanes 64..127 (and the warps
// that read them) idle, so the 128 lanes hold RF = 128 / NC vocabulary tiles
// at once: the A operand of tile i is block diagonal, lanes [i*NC, (i+1)*NC)
// carry h and the others zeros, so one accumulator takes RF tiles through
// RF * r/64 K-chunk MMAs.  Each A operand takes 128 TMEM columns.
// With the request on the TMEM lane, every epilogue thread owns one request
// row and reads 32 consecutive vocabulary entries of it in one tcgen05.ld.
// Each thread folds z + Gumbel into its own running Gumbel-max + log-sum-exp
// state: no transposition, no per-tile cross-thread reduction.
//
// CTA = 19 warps: warps 0-15 epilogue (warp w reads TMEM lane quarter w % 4
// and the 32-column block w / 4 of each tile), warp 16 W2 producer (TMA),
// warp 17 TMEM owner and single-thread issuer of the U copies and the MMAs,
// warp 18 U producer (TMA).  Every mbarrier wait is bounded; on expiry the
// kernel raises the timeout bit, lets its copies land, frees TMEM and
// returns.  With one position per launch the partial states go to the
// workspace and the last CTA of a request chunk to arrive merges them
// (atomic ticket, no waiting).
//
// The same pipeline serves the residual draw of verification
// ("DSpark：半自回归生成与置信度调度的投机解码" section 形式化定义): for every
// request whose walk rejected draft j, h = W1[x~_{j-1}] and the epilogue forms
// q = softmax(z_j) and p = softmax(t_j / tau) from the passed log-normalisers,
// then draws argmax_v log(max(0, p - q)) + G (domain 2); the CTAs fold their
// draws into one 64-bit winner key per request and end, and the compaction
// launch behind them decodes the keys (drawing from p where p <= q
// everywhere left no key).  Each thread reads its own row of U and of the
// target logits (the rejected rows differ per request, so no common TMA box
// exists): D is h.W2 alone and no U slice ring is used.
//
// The first pass of a full-prefix verification (every draft checked against
// the target, section 形式化定义), the log-sum-exps of target rows
// 0..gamma-1 and the bonus draws of row gamma, either runs beside the draft
// or inside it.  kSide builds the plain draft for a lean stream kernel that
// shares its SMs (verify.cu): registers capped so that both fit on an SM,
// the largest shared-memory carve-out, and an early trigger that lets the
// stream start once every draft CTA is resident.  kTgt has the epilogue
// warps fold each tile's target block after their race.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "pdl.cuh"
#include "resid_tail.cuh"
#include "sm100_ptx.cuh"
#include "vstream.cuh"

namespace dspark {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kThreads = (kEpiWarps + 3) * 32;   // 608
constexpr int kProducerWarp = 16, kMmaWarp = 17, kUWarp = 18;
constexpr int kTN = 128;                          // vocabulary entries per tile
constexpr int kMaxStages = 12;                    // W2 K-chunk ring depth (barriers reserved)
// TMEM (512 columns): RF A operands of 128 columns, then 4 - RF accumulators
// of 128 columns (three at RF = 1, two at RF = 2).
constexpr int kMaxAcc = 3;
// W2 moves in K-chunks of kc ranks of one 128-entry tile (bf16), two 64-entry
// boxes per chunk.  The one-request form, bound by the ring's turnaround, takes
// kc = 128 where r allows (32 KB chunks: half the round trips per tile; measured
// 153.7 -> 149.3 us a b1 step); the race kernels keep kc = 64 (16 KB), which
// measured as fast or faster at 64 to 512 requests.
__host__ __device__ constexpr int w2_kc(int r, bool one_row) { return one_row && r % 128 == 0 ? 128 : 64; }
// Ring sizes: with the race in the epilogue five 16 KB chunks suffice (measured
// faster than nine at 64 and 512 requests); the one-request and residual forms
// take what shared memory allows.
constexpr int kRingBytesRace = 5 * 16 * 1024;
constexpr int kRingBytesMax = 12 * 16 * 1024;
// U slice ring (draft): slice n = 4 * tile + column block goes to slot
// n % kUSlots; the MMA warp alone reads the slots (copying them into TMEM),
// in fill order.
constexpr int kUSlots = 4;
constexpr int kTBufBytes = 32 * 128;              // target stream: one warp's 32 rows x 32 fp32 of a tile
constexpr int kZBufBytes = 32 * 128;              // logits store: one warp's 32 rows x 32 fp32 of a tile
constexpr int kUSlotsResid = 8;                   // residual: 16 warps x (4 KB U + 4 KB target) row staging
constexpr int kSmemBudget = 227 * 1024;
constexpr long long kWaitCycles = kDefaultWaitCycles;   // the MMA drain: ~2 s at 2 GHz
constexpr long long kDrainCycles = 200000000LL;   // ~0.1 s: copies already issued landing
// Margins of the exponential-race screens (relative on the running winner's
// variate, absolute on the candidate's bound): far above the rounding of the
// products and of the exact variates, so every entry the exact test would
// accept is passed to it.
constexpr float kRaceRel = 1.0000152587890625f;   // 1 + 2^-16
constexpr float kRaceSlack = 1.52587890625e-05f;  // 2^-16
// Margin on a winner key shared between the threads of one request row: it
// crosses two log2 / exp2 conversions and two additions of the winner's z2
// (kept below 2^10 in magnitude by the caller), each good to ~2^-21.
constexpr float kShareRel = 1.000244140625f;      // 1 + 2^-12
constexpr float kShareMaxZ2 = 1024.f;             // |z2| beyond which keys are not shared
// Floor of the screen threshold (per unit of t): an entry with t > 2^64 then
// always reaches the exact path, which moves the sum's reference before
// adding it; the floor only loosens the screen.
constexpr float kKhMin = 8.673617379884035e-19f;  // 2^-60

struct Layout {
    uint32_t b, a, u, t, z, merge, tmerge, bar, misc, total;
    int uslots, tslots, stages, kc;
    uint32_t stage_bytes;
};

constexpr int kSlotBytes = 128 * 128;             // one U slice: 128 rows x 32 fp32

// The A operands live in TMEM, so shared memory holds the W2 ring (whatever
// is left, up to kMaxStages K-chunks), the U slots (the residual mode uses
// that region as 16 per-warp 4 KB row-staging buffers), the fold buffers,
// the barriers and a few words.
__host__ __device__ inline Layout rows_layout(int NC, int r, bool resid, bool tgt = false, bool zst = false,
                                              bool one_row = false) {
    (void)NC;
    Layout L;
    L.kc = w2_kc(r, one_row);
    L.stage_bytes = (uint32_t)(kTN * L.kc * 2);
    L.uslots = resid ? kUSlotsResid : kUSlots;
    L.tslots = tgt ? kEpiWarps : 0;                            // one target buffer and barrier per epilogue warp
    const uint32_t tmerge_bytes = tgt ? 4u * 128u * 8u : 0u;   // target fold: [4 column blocks][128 rows] float2
    const uint32_t z_bytes = zst ? (uint32_t)(kEpiWarps * kZBufBytes) : 0u;   // logits store staging
    const uint32_t fixed = (uint32_t)(L.uslots * kSlotBytes + L.tslots * kTBufBytes) + z_bytes + 4u * 128u * 16u +
                           tmerge_bytes + 8u * (2 * kMaxStages + 2 * L.uslots + 2 * kMaxAcc + 2 + L.tslots) + 16u +
                           12u * 128u + 1024u + 64u;
    int st = (int)((kSmemBudget - (int)fixed) / L.stage_bytes);
    const int cap = (int)(((one_row || resid) ? kRingBytesMax : kRingBytesRace) / L.stage_bytes);
    L.stages = st > cap ? cap : st;
    L.b = 0;
    L.a = 0;
    L.u = L.b + (uint32_t)L.stages * L.stage_bytes;
    L.t = L.u + (uint32_t)(L.uslots * kSlotBytes);
    L.z = L.t + (uint32_t)(L.tslots * kTBufBytes);
    L.merge = L.z + z_bytes;
    L.tmerge = L.merge + 4u * 128u * 16u;
    L.bar = L.tmerge + tmerge_bytes;
    L.misc = L.bar + 8u * (2 * L.stages + 2 * L.uslots + 2 * kMaxAcc + 2 + L.tslots);
    L.misc = (L.misc + 15u) & ~15u;
    L.total = L.misc + 16u + 12u * 128u;   // s_tok, s_row and the shared winner keys, 128 words each
    return L;
}

struct RowsArgs {
    CUtensorMap w2map;   // bf16 [r][V], box {64 vocab, kc rank}, 128-byte swizzle
    CUtensorMap umap;    // fp32 [B][gamma][V], box {32 vocab, 1, NC requests}, 128-byte swizzle
    // target stream only: fp32 [B][gamma+1][V], box {32 vocab, 1, 32 requests}
    // (one epilogue warp's rows, 128-byte swizzle)
    CUtensorMap tmap;
    // logits store (draft with logits_out, requests-on-lanes race): fp32
    // [B][gamma][V], box {32 vocab, 1, 32 requests}, 128-byte swizzle
    CUtensorMap zmap;
    DraftParams p;
    int NC;              // request rows per CTA (32, 64 or 128)
    // residual mode only
    const void* target;  // [B][gamma+1][V]
    uint32_t* near_ties;
    // RNN head (kRnn only): the GRU steps run in the prologue and at the position boundaries
    GruParams gru;
};

// Registers a thread: 608 threads are 19 warps, at most 5 on each of the 4
// schedulers, whose register files hold 16384 each: 5 x 32 x 96 fit.  The
// draft that shares its SMs with the lean target stream keeps 88, which
// leaves a scheduler room for a stream warp of 72 (5 x 32 x 88 + 32 x 72
// = 16384).
constexpr int kMaxRegs = 96;
constexpr int kSideMaxRegs = 88;

// Target stream: adds 2^(x_j * sc - m) over the entries j < n of N columns
// of one row to its running base-2 log-sum-exp state (m, s).  The reference m
// is set from the first tile's maximum and moves only when a tile's sum would
// leave the safe range (an entry more than 64 above m: rare, the tile is then
// redone against its own maximum); entries far below m flush to zero, which
// leaves the sum unchanged in binary32.  kMask: entries j >= n lie past the
// vocabulary and count as -inf.
template <bool kMask, int N>
__device__ __forceinline__ void tgt_lse_add(const float (&x)[N], int n, float sc, float& m, float& s) {
    float xv[N];
#pragma unroll
    for (int j = 0; j < N; ++j) xv[j] = (!kMask || j < n) ? x[j] : -INFINITY;
    if (m == -INFINITY) {
        float cm = xv[0];
#pragma unroll
        for (int j = 1; j < N; ++j) cm = fmaxf(cm, xv[j]);
        m = cm * sc;                                 // sc > 0 keeps the maximum
        if (m == -INFINITY) return;
    }
    const float2 sc2 = make_float2(sc, sc);
    float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
    float2 nm = make_float2(-m, -m);
#pragma unroll
    for (int j = 0; j < N; j += 4) {
        const float2 d01 = __ffma2_rn(make_float2(xv[j], xv[j + 1]), sc2, nm);
        const float2 d23 = __ffma2_rn(make_float2(xv[j + 2], xv[j + 3]), sc2, nm);
        a01 = __fadd2_rn(a01, make_float2(fast_exp2(d01.x), fast_exp2(d01.y)));
        a23 = __fadd2_rn(a23, make_float2(fast_exp2(d23.x), fast_exp2(d23.y)));
    }
    float sum = (a01.x + a01.y) + (a23.x + a23.y);
    if (!(sum < 18446744073709551616.f)) {   // 2^64, or inf / NaN
        float cm = xv[0];
#pragma unroll
        for (int j = 1; j < N; ++j) cm = fmaxf(cm, xv[j]);
        cm *= sc;
        if (cm > m) {
            s *= fast_exp2(m - cm);
            m = cm;
        }
        sum = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) sum += fast_exp2(fmaf(xv[j], sc, -m));
    }
    s += sum;
}

// 16-byte load from a shared-memory address.
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

// (m, s) += (e.x, e.y) for base-2 log-sum-exp states (m = -inf: empty).
__device__ __forceinline__ void lse2_merge(float& m, float& s, const float2 e) {
    if (e.x == -INFINITY) return;
    if (m == -INFINITY) { m = e.x; s = e.y; return; }
    if (e.x > m) { s = s * fast_exp2(m - e.x) + e.y; m = e.x; }
    else s += e.y * fast_exp2(e.x - m);
}


// Bounded grid-wide barrier on a counter in global memory: every CTA adds 1,
// then waits until all `target` CTAs have.  The kernel is launched
// cooperatively, so all CTAs are resident.  Returns false on expiry or abort.
__device__ __forceinline__ bool grid_barrier(uint32_t* ctr, uint32_t target, const volatile uint32_t* abort,
                                             long long limit_cycles) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const long long t0 = clock64();
    for (;;) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) break;
        if (*abort) return false;
        if (clock64() - t0 > limit_cycles) return false;
        __nanosleep(32);
    }
    __threadfence();
    return true;
}

// A operands in TMEM.  A_i (i < RF, columns [128 i, 128 i + 128)) carries
// h = W1[x~] on the lanes of vocabulary tile i, rows [i NC, (i + 1) NC), and
// zeros on the other lanes: the block-diagonal operand that lets one
// accumulator take RF tiles.  A row is r bf16 packed two to a 32-bit column
// in rank order.  Epilogue warp (q, cb) writes lanes [32 q, 32 q + 32) and
// columns [32 cb, 32 cb + 32), ranks [64 cb, 64 cb + 64): the h slice of its
// lanes' requests into the A of their tile, and zeros into the other A
// operands when `zeros` is set (once per launch: later positions rewrite the
// h parts only).
__device__ __forceinline__ void store_a_slice(uint32_t tmem_base, int NC, int RF, int q, int cb, int lane,
                                              bool zeros, uint32_t (&v)[32]) {
    const int row = 32 * q + lane, ti = row / NC;
    const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * cb);
    // the 32 lanes of a warp belong to one tile (NC >= 32)
    ptx::tmem_st32(taddr + (uint32_t)(128 * ti), v);
    if (zeros) {
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = 0u;
        for (int i = 0; i < RF; ++i)
            if (i != ti) ptx::tmem_st32(taddr + (uint32_t)(128 * i), v);
    }
}

__device__ __forceinline__ void stage_a_tmem(uint32_t tmem_base, const uint16_t* W1, const int* s_tok, int NC,
                                             int RF, int r, int V, int q, int cb, int lane, bool zeros) {
    if (64 * cb >= r) return;                       // ranks past r are never read
    const int n = (32 * q + lane) % NC;
    uint32_t v[32];
    const int x = s_tok[n];
    if (x >= 0 && x < V) {                          // rows outside [0, V) stay zero
        const uint4* src = reinterpret_cast<const uint4*>(W1 + (size_t)x * r + (size_t)(64 * cb));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint4 w = src[u];
            v[4 * u] = w.x; v[4 * u + 1] = w.y; v[4 * u + 2] = w.z; v[4 * u + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = 0u;
    }
    store_a_slice(tmem_base, NC, RF, q, cb, lane, zeros, v);
}

// The same A operands for the RNN head: h is the request's fp32 state row
// st_base[pos][n] (pos < 0: the row's own position s_row[n]) rounded to
// bf16; rows whose token is invalid stay zero.
__device__ __forceinline__ void stage_a_state(uint32_t tmem_base, const float* st_base, size_t pos_stride,
                                              int pos, const int* s_row, const int* s_tok, int NC, int RF, int r,
                                              int V, int q, int cb, int lane, bool zeros) {
    if (64 * cb >= r) return;
    const int n = (32 * q + lane) % NC;
    uint32_t v[32];
    const int x = s_tok[n];
    if (x >= 0 && x < V) {
        const int ps = pos >= 0 ? pos : s_row[n];
        const float4* src =
            reinterpret_cast<const float4*>(st_base + (size_t)ps * pos_stride + (size_t)n * r + (size_t)(64 * cb));
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const float4 f = src[u];
            const __nv_bfloat162 lo = __floats2bfloat162_rn(f.x, f.y), hi = __floats2bfloat162_rn(f.z, f.w);
            v[2 * u] = *reinterpret_cast<const uint32_t*>(&lo);
            v[2 * u + 1] = *reinterpret_cast<const uint32_t*>(&hi);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = 0u;
    }
    store_a_slice(tmem_base, NC, RF, q, cb, lane, zeros, v);
}

// Winner key of a partial draw: larger best first, then the lower index, as
// in wins(); an unsigned 64-bit maximum over the keys picks the draw.  -0 is
// folded into +0, which wins() does not tell apart.
__device__ __forceinline__ unsigned long long win_key(const DrawLse& d) {
    const uint32_t bits = __float_as_uint(d.best == 0.f ? 0.f : d.best);
    const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)d.idx);
}

// One warp stages a 32-entry segment [v0, v0 + 32) of 32 rows (one per lane,
// row pointers in the lanes' `row`) into a shared buffer of 32 x (32 * sizeof(T))
// bytes: 16-byte asynchronous copies, a row's segment spread over consecutive
// lanes, rows of lanes outside `mask` skipped, entries past V zero-filled.
// The 16-byte chunk index is swizzled with the row (XOR with row % 8 for
// 128-byte rows, (row / 2) % 4 for 64-byte rows) so that a lane reading its
// own row meets no bank conflict.  The copies form one cp.async group; the
// caller waits for it and syncs the warp before reading.
template <typename T>
__device__ __forceinline__ void issue_rows(uint32_t buf, const T* row, unsigned mask, int v0, int V, int lane) {
    constexpr int kRowBytes = 32 * (int)sizeof(T);
    constexpr int kChunks = kRowBytes / 16;           // 8 (fp32) or 4 (bf16)
    constexpr int kRowsPerPass = 32 / kChunks;
    constexpr int kPerChunk = 16 / (int)sizeof(T);    // entries per chunk
#pragma unroll
    for (int j = 0; j < 32 / kRowsPerPass; ++j) {
        const int rr = j * kRowsPerPass + lane / kChunks, c = lane % kChunks;
        const T* src = reinterpret_cast<const T*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row), rr));
        if ((mask >> rr) & 1u) {
            const int vq = v0 + c * kPerChunk;
            const int swz = kChunks == 8 ? (rr & 7) : ((rr >> 1) & 3);
            const bool in = vq < V;
            ptx::cp_async_16(buf + (uint32_t)(rr * kRowBytes + ((c ^ swz) << 4)), in ? src + vq : src, in ? 16u : 0u);
        }
    }
    ptx::cp_async_commit();
}

__device__ __forceinline__ DrawLse drawlse_of(const float4 c) {
    DrawLse d;
    d.best = c.x; d.idx = __float_as_int(c.y); d.zb = c.z; d.lse = c.w;
    return d;
}

// The RNN head's GRU steps inside the persistent draft.  Step ks writes
// state[ks] = GRU(h, x) for every request, h = s0 and x = the anchor for
// ks = 0 (in the prologue), else h = state[ks - 1] and x = x~_ks, the draws
// of position ks (winner keys of index ks - 1).  This CTA takes the hidden
// units u = cta, cta + nctas, ... for every request, in two parts:
//   gh_compute: gh[b][g r + u] = W_hh[g r + u] . h_b + b_hh (gates g = r, z,
//     n) as soon as h is known, i.e. right after the previous step, while
//     the MMA already runs the next position.  An epilogue warp takes one
//     request at a time, lane l holding ranks [8 l, 8 l + 8) of h and of the
//     unit's three W_hh rows; the six partial sums of two units are summed
//     across the warp by recursive halving over 8 slots (9 shuffles), which
//     leaves slot s in lanes 4 s .. 4 s + 3.  For h = s0 one row serves
//     every request.
//   gate_step: once x is drawn, one thread per (unit, request) gathers the
//     three input projections P[x][g r + u] (a table computed once from E,
//     W_ih and b_ih), applies the gates and writes the new state.
// The step's critical path (draws known -> new state published) is thus a
// gather and the gate arithmetic.  Other CTAs' state rows are read through L2.
__device__ __forceinline__ float bf16f_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16f_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float dot8(const uint4 w, const float4 h0, const float4 h1, float a) {
    a = fmaf(bf16f_lo(w.x), h0.x, a); a = fmaf(bf16f_hi(w.x), h0.y, a);
    a = fmaf(bf16f_lo(w.y), h0.z, a); a = fmaf(bf16f_hi(w.y), h0.w, a);
    a = fmaf(bf16f_lo(w.z), h1.x, a); a = fmaf(bf16f_hi(w.z), h1.y, a);
    a = fmaf(bf16f_lo(w.w), h1.z, a); a = fmaf(bf16f_hi(w.w), h1.w, a);
    return a;
}

__device__ __forceinline__ void gh_compute(const GruParams& g, int ks_h, int cta, int nctas, int ewarp, int lane) {
    const int r = g.r;
    const float* hsrc = ks_h < 0 ? nullptr : g.state + (size_t)ks_h * g.B * r;
    const int B = hsrc ? g.B : 1;                 // s0: one row serves every request
    if (cta >= r || ewarp >= B) return;
    const unsigned full = 0xffffffffu;
    const int nu = (r - 1 - cta) / nctas + 1;
    const int e0 = 8 * lane;
    const bool act = e0 < r;
    const size_t gs = (size_t)r * r;
    for (int b = ewarp; b < B; b += kEpiWarps) {
        float4 h0 = make_float4(0.f, 0.f, 0.f, 0.f), h1 = h0;
        if (act) {
            const float* hr = hsrc ? hsrc + (size_t)b * r : g.s0;
            h0 = __ldcg(reinterpret_cast<const float4*>(hr + e0));
            h1 = __ldcg(reinterpret_cast<const float4*>(hr + e0 + 4));
        }
        for (int j0 = 0; j0 < nu; j0 += 2) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
            if (act) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (j0 + t >= nu) break;
                    const uint16_t* wh = g.W_hh + (size_t)(cta + (j0 + t) * nctas) * r + e0;
#pragma unroll
                    for (int gt = 0; gt < 3; ++gt)
                        v[3 * t + gt] = dot8(*reinterpret_cast<const uint4*>(wh + gt * gs), h0, h1, 0.f);
                }
            }
            // recursive halving: 8 slots -> 4 -> 2 -> 1, then the last two levels
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool up = lane & 16;
                const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
                v[i] = keep + __shfl_xor_sync(full, send, 16);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const bool up = lane & 8;
                const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
                v[i] = keep + __shfl_xor_sync(full, send, 8);
            }
            {
                const bool up = lane & 4;
                const float send = up ? v[0] : v[1], keep = up ? v[1] : v[0];
                v[0] = keep + __shfl_xor_sync(full, send, 4);
            }
            v[0] += __shfl_xor_sync(full, v[0], 2);
            v[0] += __shfl_xor_sync(full, v[0], 1);
            // slot s = 3 t + gate sits in lanes 4 s .. 4 s + 3
            const int slot = lane >> 2, t = slot / 3, gt = slot - 3 * t;
            if ((lane & 3) == 0 && slot < 6 && j0 + t < nu) {
                const int row = gt * r + cta + (j0 + t) * nctas;
                g.gh[(size_t)b * 3 * r + row] = v[0] + g.b_hh[row];
            }
        }
    }
}

__device__ __forceinline__ void gate_step(const GruParams& g, int ks, int cta, int nctas, int etid, int nthreads,
                                          const int* s_tok_all, const unsigned long long* win) {
    const int r = g.r, B = g.B;
    if (cta >= r) return;
    const float* hprev = ks == 0 ? nullptr : g.state + (size_t)(ks - 1) * B * r;
    float* hout = g.state + (size_t)ks * B * r;
    const int nu = (r - 1 - cta) / nctas + 1;
    for (int pr = etid; pr < nu * B; pr += nthreads) {
        const int ui = pr / B, b = pr - ui * B, u = cta + ui * nctas;
        const int x = ks == 0 ? g.anchor[b]
                              : (s_tok_all ? s_tok_all[b]
                                           : win_token(__ldcg(&win[((size_t)(ks - 1) * B + b) * kWinStride])));
        float gi0 = 0.f, gi1 = 0.f, gi2 = 0.f;
        if (x >= 0 && x < g.V) {
            const float* Pr = g.P + (size_t)x * 3 * r;
            gi0 = Pr[u]; gi1 = Pr[r + u]; gi2 = Pr[2 * r + u];
        }
        const float* ghr = g.gh + (size_t)(hprev ? b : 0) * 3 * r;
        const float hu = hprev ? __ldcg(hprev + (size_t)b * r + u) : g.s0[u];
        const float rg = 1.f / (1.f + expf(-(gi0 + ghr[u])));
        const float zg = 1.f / (1.f + expf(-(gi1 + ghr[r + u])));
        const float ng = tanhf(gi2 + rg * ghr[2 * r + u]);
        hout[(size_t)b * r + u] = (1.f - zg) * ng + zg * hu;
    }
}

// Positions k_first..k_last in one launch.  With more than one position the
// launch is cooperative: after each position every CTA writes its partial
// states and folds its draw of each request into a 64-bit atomic maximum
// (score, then lowest index), waits at a grid barrier, reads the winners of
// its requests (one load each), stages h = W1[x~_k] for the next position
// and releases the MMA issuer.  The log-sum-exp and the drawn logit need the
// full merge of the partials; the CTAs share it out by request and do it
// while the MMA starts the next position.  The TMA producer never stops at
// the boundaries: W2 and the next position's U do not depend on the drawn
// tokens.  Partial states alternate between two buffers, so a fast CTA
// never overwrites the ones a slow CTA still merges: the buffer of position
// k is written again at k + 2, after the grid barrier of k + 1, which no CTA
// reaches before its merges of k are done.
// 19 warps over 4 schedulers put 5 warps on three of them, whose 16384
// registers then allow 96 a thread.
// kOneRow (B = 1, the latency case): the chunk holds one request, so only
// lane 0 of the warps on its TMEM rows carries data.  Those warps spread each
// tile's 32 columns of that row over their lanes (one shuffle per column) and
// every lane races its own column; the lanes' partial states are merged at
// the end of the position.
// kTgt (full-prefix verification): position k also reduces target row k-1
// to log-sum-exp partials, the work of the verify stream on those rows.
// Every epilogue warp keeps its own 4 KB buffer: after its race on a tile
// it reads the tile's target block (its 32 request rows x 32 columns, lane =
// row, 128-byte swizzle), issues the TMA load of its next tile's block into
// the same buffer and folds the values into a running base-2 log-sum-exp
// per request row.  The load has a whole tile's race to land, and no warp
// waits on another's progress.  Nothing prefetches U or the target into L2:
// the extra L2 footprint evicts W2, whose re-reads from HBM cost more than
// the latency a prefetch hides.
template <bool kResid, typename TT, bool kRnn = false, bool kOneRow = false, bool kTgt = false, bool kSide = false>
__global__ void __maxnreg__(kSide ? kSideMaxRegs : kMaxRegs)
rows_kernel(const __grid_constant__ RowsArgs a, const int k_first, const int k_last) {
    static_assert(!(kTgt && (kResid || kRnn)), "the target stream belongs to the Markov draft");
    static_assert(!(kSide && (kResid || kRnn || kTgt)), "the stream beside the draft belongs to the plain Markov draft");
    // the draft race reads the accumulator a quad of columns at a time
    constexpr bool kQuadLoop = !kResid && !kOneRow;
    const DraftParams& p = a.p;
    const int NC = a.NC;
    const long long wl = wait_limit_of(p.ws.wait_limit);   // bound of the waits on other roles and CTAs
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int GX = (int)gridDim.x;
    // the draft's logits leave through a per-warp staging buffer and a tensor store
    const bool zst = kQuadLoop && !kTgt && p.logits_out != nullptr;
    const Layout L = rows_layout(NC, p.r, kResid, kTgt, zst, kOneRow);
    const int KC = L.kc, KCH = p.r / KC;
    const uint32_t sbytes = L.stage_bytes;
    const int RF = 128 / NC;                      // vocabulary tiles per accumulator
    const int US = L.uslots;
    const uint32_t slot_bytes = (uint32_t)kSlotBytes;
    const uint32_t blk = (uint32_t)NC * 128u;     // bytes of one U box (NC rows x 128 B)
    const bool persistent = k_last > k_first;
    const int nacc = 4 - RF;                      // accumulators after the RF A operands
    const uint32_t acc0 = 128u * (uint32_t)RF;    // TMEM column of accumulator 0

    const int kStages = L.stages;
    const uint32_t bar0 = base + L.bar;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto ufull = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto uempty = [&](int i) { return bar0 + 8u * (2 * kStages + US + i); };
    auto tfull = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * US + i); };
    auto tempty = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * US + kMaxAcc + i); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 2 * US + 2 * kMaxAcc);
    const uint32_t a_ready = bar0 + 8u * (2 * kStages + 2 * US + 2 * kMaxAcc + 1);
    auto tbar = [&](int w) { return bar0 + 8u * (2 * kStages + 2 * US + 2 * kMaxAcc + 2 + w); };   // kTgt
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L.misc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + L.misc + 4);
    volatile uint32_t* never = reinterpret_cast<volatile uint32_t*>(gbase + L.misc + 8);
    int* s_tok = reinterpret_cast<int*>(gbase + L.misc + 16);
    int* s_row = s_tok + 128;                       // residual mode: rejected row per request, or -1
    // draft: the best winner key found so far per request row by any of the
    // CTA's threads racing that row (order-preserving bits of log2 E2 - z2,
    // all ones = none yet), reset at every position
    uint32_t* s_key = reinterpret_cast<uint32_t*>(s_row + 128);
    DrawLse* s_merge = reinterpret_cast<DrawLse*>(gbase + L.merge);   // [4 column blocks][128 rows]

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int chunk = blockIdx.y, b_base = chunk * NC;
    const int nb = min(NC, p.B - b_base);
    const int V = p.V, gamma = p.gamma, r = p.r;
    const uint16_t* W1 = static_cast<const uint16_t*>(p.W1);
    const float* st_base = p.state ? p.state + (size_t)b_base * p.r : nullptr;   // RNN head rows of this chunk
    const uint32_t nctas = (uint32_t)GX * gridDim.y;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) { ptx::mbar_init(full(i), 1); ptx::mbar_init(empty(i), 1); }
        for (int i = 0; i < US; ++i) { ptx::mbar_init(ufull(i), 1); ptx::mbar_init(uempty(i), 1); }
        for (int i = 0; i < kMaxAcc; ++i) { ptx::mbar_init(tfull(i), 1); ptx::mbar_init(tempty(i), kEpiWarps); }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(a_ready, 1);
        if constexpr (kTgt)
            for (int w = 0; w < kEpiWarps; ++w) ptx::mbar_init(tbar(w), 1);
        *abort_flag = 0u;
        *never = 0u;
        ptx::fence_mbar_init();
    }
    if (tid == kProducerWarp * 32) ptx::prefetch_tmap(&a.w2map);
    if (tid == kUWarp * 32 && !kResid) {
        ptx::prefetch_tmap(&a.umap);
        if constexpr (kTgt) ptx::prefetch_tmap(&a.tmap);
    }
    if (kTgt && tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) *p.ws.tgt_token = p.tgt_token;
    if (warp == kMmaWarp) { ptx::tmem_alloc(base + L.misc, 512u); ptx::tmem_relinquish(); }
    // the target stream launched behind this draft runs on the SMs beside it;
    // the launch behind the residual draw (compaction) is scheduled early and
    // waits for it
    if ((kSide || kResid) && tid == 0) grid_launch_dependents();
    // the residual draw is launched as a programmatic dependent of the accept
    // walk: its set-up above overlaps the walk's tail, and it waits here before
    // reading the rejected rows and log-normalisers the walk writes
    if constexpr (kResid) {
        // W2 does not depend on the walk: the CTA's first super-tile of it goes
        // to L2 before the wait (two measured slower at b64, 297.0 against
        // 292.7 us a step: the launch starts during the walk, whose loads they
        // delay)
        if (tid == kProducerWarp * 32) {
            const int ntl = (V + kTN * RF - 1) / (kTN * RF);
            for (int t = blockIdx.x, n = 0; t < ntl && n < 1; t += GX, ++n)
                for (int i = 0; i < RF; ++i)
                    for (int j = 0; j < KCH; ++j) {
                        ptx::tma_prefetch_2d(&a.w2map, t * kTN * RF + i * kTN, j * KC);
                        ptx::tma_prefetch_2d(&a.w2map, t * kTN * RF + i * kTN + 64, j * KC);
                    }
        }
        grid_dependency_wait();
    }
    for (int n = tid; n < 128; n += kThreads) {
        int x = -1, prow = -1;
        if (n < nb) {
            const int b = b_base + n;
            if constexpr (kResid) {
                // both written by the accept walk: no load waits on another
                prow = __ldcg(&p.ws.rej[b]);
                x = __ldcg(&p.ws.rtok[b]);
                if (prow < 0) x = -1;
            } else {
                x = (k_first == 1) ? p.anchor[b] : p.draft_tok[(size_t)b * gamma + (k_first - 2)];
            }
            if (x >= V || (x < 0 && !kResid)) { raise_status(p.ws.status, kBadToken); x = -1; }
        }
        s_tok[n] = x;
        s_row[n] = prow;
        s_key[n] = 0xFFFFFFFFu;
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if constexpr (kRnn) {
        // RNN head: the GRU step of the first position (from s0 and the
        // anchors), shared out over the CTAs like the later ones
        if (warp < kEpiWarps) {
            __shared__ int s_pro_ok;
            const int cta_id = (int)(blockIdx.y * GX + blockIdx.x);
            gh_compute(a.gru, -1, cta_id, (int)nctas, warp, lane);
            ptx::named_barrier(1, 32 * kEpiWarps);
            gate_step(a.gru, 0, cta_id, (int)nctas, tid, 32 * kEpiWarps, nullptr, p.ws.win);
            ptx::named_barrier(1, 32 * kEpiWarps);
            if (tid == 0)
                s_pro_ok = grid_barrier(p.ws.gbar + kGbarGru + (kGridBarrierSlots - 1), nctas, abort_flag, wl);
            ptx::named_barrier(1, 32 * kEpiWarps);
            if (!s_pro_ok && tid == 0) {
                raise_timeout(p.ws.status, 10);
                *abort_flag = 1u;
            }
        }
    }
    if (warp < kEpiWarps) {                        // the A operands of the first position
        if constexpr (kResid) {
            // the first tile's rows of U and of the target, in flight during the
            // W1 gathers and the first MMAs (the tile loop issues the later ones)
            const int q0 = warp & 3, cb0 = warp >> 2, row0 = 32 * q0 + lane, nr0 = row0 % NC;
            if ((32 * q0) % NC < nb) {
                const bool bon0 = p.resid_bonus && nr0 < nb && s_row[nr0] < 0;
                const bool real0 = nr0 < nb && (s_row[nr0] >= 0 || bon0);
                const int tr = bon0 ? gamma : (real0 ? s_row[nr0] : 0), ur = bon0 ? 0 : tr, bq = b_base + nr0;
                const float* Ur = static_cast<const float*>(p.U) + ((size_t)bq * gamma + ur) * V;
                const TT* Tr = static_cast<const TT*>(a.target) + ((size_t)bq * (gamma + 1) + tr) * V;
                const unsigned m0 = __ballot_sync(0xffffffffu, real0);
                const uint32_t ub = base + L.u + (uint32_t)warp * 8192u;
                const int v00 = (int)blockIdx.x * kTN * RF + (row0 / NC) * kTN + 32 * cb0;
                issue_rows<float>(ub, Ur, m0, v00, V, lane);
                issue_rows<TT>(ub + 4096u, Tr, m0, v00, V, lane);
            }
        }
        if (st_base)
            stage_a_state(tmem_base, st_base, (size_t)p.B * r, kResid ? -1 : k_first - 1, s_row, s_tok, NC, RF, r,
                          V, warp & 3, warp >> 2, lane, true);
        else
            stage_a_tmem(tmem_base, W1, s_tok, NC, RF, r, V, warp & 3, warp >> 2, lane, true);
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const int ntiles = (V + kTN * RF - 1) / (kTN * RF);   // super-tiles of RF vocabulary tiles

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ W2 producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_last();
            int stage = 0, site = 0;
            uint32_t ph = 0;
            bool ok = true;
            long long nw = 0;                            // W2 chunks issued
            for (int k = k_first; k <= k_last && ok; ++k) {
                for (int t = blockIdx.x; t < ntiles && ok; t += GX) {
                    const int vs = t * kTN * RF;
                    for (int i = 0; i < RF && ok; ++i) {
                        for (int j = 0; j < KCH; ++j) {
                            if (!(ok = ptx::mbar_wait(empty(stage), ph ^ 1u, abort_flag, wl))) { site = 1; break; }
                            ptx::mbar_arrive_expect_tx(full(stage), sbytes);
                            const uint32_t dst = base + L.b + (uint32_t)stage * sbytes;
                            const int v0 = vs + i * kTN;
                            ptx::tma_load_2d(dst, &a.w2map, v0, j * KC, full(stage), pol_w);
                            ptx::tma_load_2d(dst + sbytes / 2, &a.w2map, v0 + 64, j * KC, full(stage), pol_w);
                            ++nw;
                            if (++stage == kStages) { stage = 0; ph ^= 1u; }
                        }
                    }
                }
            }
            if (!ok) { raise_timeout(p.ws.status, site); *abort_flag = 1u; }
            // every copy issued lands before the CTA leaves: wait for the last
            // fill of each stage (already complete on the normal path)
            for (int i = 0; i < kStages; ++i)
                if (nw > i) {
                    const long long m = (nw - 1) - ((nw - 1 - i) % kStages);
                    ptx::mbar_wait(full(i), (uint32_t)((m / kStages) & 1), never, kDrainCycles);
                }
        }
        __syncwarp();
    } else if (warp == kUWarp) {
        // ------------------------------------------------------------ U producer (draft)
        if (lane == 0 && !kResid) {
            const uint64_t pol_u = ptx::policy_evict_first();
            int site = 0;
            bool ok = true;
            int lt = 0;                                  // tiles issued, over all positions
            long long nu = 0;                            // U slices issued
            for (int k = k_first; k <= k_last && ok; ++k) {
                for (int t = blockIdx.x; t < ntiles && ok; t += GX, ++lt) {
                    const int vs = t * kTN * RF;
                    for (int c = 0; c < 4 && ok; ++c) {
                        const int n = lt * 4 + c, s = n % US;
                        const uint32_t par = (uint32_t)((n / US) & 1);
                        if (!(ok = ptx::mbar_wait(uempty(s), par ^ 1u, abort_flag, wl))) { site = 2; break; }
                        ptx::mbar_arrive_expect_tx(ufull(s), slot_bytes);
                        for (int i = 0; i < RF; ++i)      // rows [i*NC, (i+1)*NC) hold tile i's U slice
                            ptx::tma_load_3d(base + L.u + (uint32_t)s * slot_bytes + (uint32_t)i * blk, &a.umap,
                                             vs + i * kTN + 32 * c, k - 1, b_base, ufull(s), pol_u);
                        ++nu;
                    }
                }
            }
            if (!ok) { raise_timeout(p.ws.status, site); *abort_flag = 1u; }
            for (int i = 0; i < US; ++i)
                if (nu > i) {
                    const long long m = (nu - 1) - ((nu - 1 - i) % US);
                    ptx::mbar_wait(ufull(i), (uint32_t)((m / US) & 1), never, kDrainCycles);
                }

        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, kTN, /*A K-major*/ false, /*B MN-major*/ true);
            int stage = 0, acc = 0, site = 0, lt = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int k = k_first; k <= k_last && ok; ++k) {
                bool wait_a = k > k_first;   // h of this position is staged by the epilogue warps
                for (int t = blockIdx.x; t < ntiles && ok; t += GX, ++lt) {
                    if (!(ok = ptx::mbar_wait(tempty(acc), aph ^ 1u, abort_flag, wl))) { site = 4; break; }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc0 + (uint32_t)(acc * kTN);
                    if constexpr (!kResid) {
                        // the accumulator starts as the tile's U: four 32-column slices
                        // (128 rows x 128 B, 128-byte swizzle) copied 32 bytes a row at a
                        // time; the MMAs below then add h.W2 on top
                        for (int c = 0; c < 4 && ok; ++c) {
                            const int n = lt * 4 + c, s = n % US;
                            if (!(ok = ptx::mbar_wait(ufull(s), (uint32_t)((n / US) & 1), abort_flag, wl))) {
                                site = 9;
                                break;
                            }
                            ptx::tc_fence_after();
                            const uint32_t src = base + L.u + (uint32_t)s * slot_bytes;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                ptx::tmem_cp_128x256b(d_tmem + (uint32_t)(32 * c + 8 * j),
                                                      ptx::smem_desc_sw128(src + 32 * j, 16, 1024));
                            ptx::mma_commit(uempty(s));     // the slot is free once the copies have read it
                        }
                        if (!ok) break;
                    }
                    if (wait_a) {   // the first tile's U copies above do not need h
                        if (!(ok = ptx::mbar_wait(a_ready, (uint32_t)((k - k_first - 1) & 1), abort_flag, wl))) {
                            site = 3;
                            break;
                        }
                        ptx::tc_fence_after();
                        wait_a = false;
                    }
                    for (int i = 0; i < RF && ok; ++i) {
                        for (int j = 0; j < KCH; ++j) {
                            if (!(ok = ptx::mbar_wait(full(stage), ph, abort_flag, wl))) { site = 5; break; }
                            ptx::tc_fence_after();
                            const uint32_t b_addr = base + L.b + (uint32_t)stage * sbytes;
                            // A_i in TMEM: K-chunk j = KC/2 columns, 16 ranks = 8 columns
                            const uint32_t a_tmem = tmem_base + (uint32_t)(128 * i + (KC / 2) * j);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                if (kk == KC / 16) break;
                                // B: MN-major, the two 64-entry swizzle atoms half a stage
                                //    apart along N (LBO), 8-rank groups 1 KB apart along K
                                //    (SBO); 16 ranks = 2 KB.
                                const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 2048, sbytes / 2, 1024);
                                ptx::mma_f16_ts(d_tmem, a_tmem + (uint32_t)(8 * kk), bd, idesc,
                                                (!kResid || (i | j | kk) != 0) ? 1u : 0u);
                            }
                            ptx::mma_commit(empty(stage));
                            if (++stage == kStages) { stage = 0; ph ^= 1u; }
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(tfull(acc));
                    if (++acc == nacc) { acc = 0; aph ^= 1u; }
                }
            }
            if (!ok) { raise_timeout(p.ws.status, site); *abort_flag = 1u; }
            ptx::mma_commit(drain);                 // every MMA above completes before TMEM is freed
            ptx::mbar_wait(drain, 0u, never, kWaitCycles);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int etid = tid;                       // 0 .. 511
        const int q = warp & 3, cb = warp >> 2;     // lane quarter, 32-column block of the tile
        const int row = 32 * q + lane;              // TMEM lane
        const int ti = row / NC, nrow = row % NC;   // vocabulary tile of the super-tile, request row
        const bool active = (32 * q) % NC < nb;     // the warp's rows hold at least one request
        const int b = b_base + nrow;
        // residual mode: the rejected requests, and with resid_bonus the others
        // (their bonus draw from p on row gamma, with q taken as 0 and the
        // bonus noise, domain 3)
        const bool bon = kResid && p.resid_bonus && active && nrow < nb && s_row[nrow] < 0;
        const bool real = active && nrow < nb && (!kResid || s_row[nrow] >= 0 || bon);
        const float scale2 = p.inv_tau * 1.4426950408889634f;      // z -> z * log2(e)
        if constexpr (kRnn) {
            // W_hh . state[0] for the first boundary's GRU step, while the MMA
            // starts the first position
            if (k_first < k_last)
                gh_compute(a.gru, k_first - 1, (int)(blockIdx.y * GX + blockIdx.x), (int)nctas, warp, lane);
        }
        int acc = 0;
        uint32_t aph = 0;
        bool failed = false;
        // target stream (kTgt): this warp's buffer, its loads consumed, one in flight
        const uint32_t tbuf = base + L.t + (uint32_t)warp * (uint32_t)kTBufBytes;
        int ltile = 0;
        bool tinfl = false;
        auto tgt_issue = [&](int tn, int kn) {
            // rows (32 q) % NC .. + 31 of the chunk: TMEM lanes 32 q .. 32 q + 31
            ptx::fence_proxy_async_smem();          // the lanes' reads of the buffer come first
            ptx::mbar_arrive_expect_tx(tbar(warp), (uint32_t)kTBufBytes);
            ptx::tma_load_3d(tbuf, &a.tmap, tn * kTN * RF + ti * kTN + 32 * cb, kn - 1, b_base + (32 * q) % NC,
                             tbar(warp), ptx::policy_evict_first());
        };
        if (kTgt && active && lane == 0) tgt_issue(blockIdx.x, k_first);
        if (kTgt && active) tinfl = true;
        for (int k = k_first; k <= k_last && !failed; ++k) {
            // row of the target (and of U, except for a bonus draw, which reads U row 0 and scales q to 0)
            const int trow = kResid ? (bon ? gamma : (real ? s_row[nrow] : 0)) : (k - 1);
            const int urow = bon ? 0 : trow;
            const StreamRK rng(p.seed, p.step, kResid ? (bon ? 3u : 2u) : 0u,
                               (uint32_t)(p.req_base + b) * (uint32_t)(gamma + 1) + (uint32_t)trow);
            const size_t out_row = ((size_t)b * gamma + (k - 1)) * V;
            // kOneRow: every lane works on the chunk's one request
            const StreamRK rng1(p.seed, p.step, 0u, (uint32_t)(p.req_base + b_base) * (uint32_t)(gamma + 1) + (uint32_t)(k - 1));
            const size_t out_row1 = ((size_t)b_base * gamma + (k - 1)) * V;
            const float* Urow = static_cast<const float*>(p.U) + ((size_t)b * gamma + urow) * V;
            const TT* Trow = static_cast<const TT*>(a.target) + ((size_t)b * (gamma + 1) + trow) * V;
            float2 lse = make_float2(0.f, 0.f);
            if (kResid && real) lse = p.ws.lse_rej[b];
            const float lse_p2 = lse.x * 1.4426950408889634f, lse_q2 = lse.y * 1.4426950408889634f;
            // residual mode: E / r of the r-draw's winner, E / p of the p-draw's
            // (+inf: none yet), and the screens' thresholds
            float Kr = INFINITY, Krh = INFINITY;
            DrawLse st = drawlse_empty();            // idx, zb (u + bias of the winner)
            float osum = 0.f;                          // one-row form: sum of 2^(z2_v - rz2)
            float rz2 = -INFINITY, rE2 = INFINITY;     // winner's z*log2e and E2
            float rE2h = INFINITY;                     // rE2 * kRaceRel: the screen's threshold (one-row form)
            // draft form: the log-sum-exp as lsum = sum_v 2^(z2_v - ref2) against a
            // reference set by the data alone (the first quad's maximum, moved up
            // by >= 64 only when an entry exceeds it by that much), so the sum does
            // not depend on the race; the race as K2 = E2_best * 2^(ref2 - z2_best)
            // (v wins iff E2_v < K2 * t_v, t_v = 2^(z2_v - ref2)) and the screen's
            // threshold Kh on 1 - u per unit of t
            float ref2 = -INFINITY, lsum = 0.f, K2 = INFINITY;
            float Kh = INFINITY;
            Draw2 st2 = draw2_empty();
            float tm2 = -INFINITY, tsum = 0.f;         // target stream: this row's base-2 log-sum-exp state
            for (int t = blockIdx.x; t < ntiles; t += GX) {
                bool ok = ptx::mbar_wait(tfull(acc), aph, abort_flag, wl);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) { if (lane == 0 && !*abort_flag) raise_timeout(p.ws.status, 6); failed = true; break; }
                ptx::tc_fence_after();
                // this warp's 32 lanes x 32 columns of the accumulator
                const uint32_t acc_tile =
                    tmem_base + ((uint32_t)(32 * q) << 16) + acc0 + (uint32_t)(acc * kTN + 32 * cb);
                // the residual and one-request forms read the whole block at once and
                // free the accumulator; the draft race reads it a quad at a time and
                // frees it after the race
                auto release_acc = [&]() {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(tempty(acc));
                    if (++acc == nacc) { acc = 0; aph ^= 1u; }
                };
                float bias[32];              // residual: h.W2; one request: U + h.W2
                if constexpr (!kQuadLoop) {
                    if (active) {
                        ptx::tmem_ld32(acc_tile, bias);
                        ptx::tmem_wait_ld();
                    }
                    release_acc();
                }
                if (kResid && !active) continue;
                const int v0 = t * kTN * RF + ti * kTN + 32 * cb;
                if constexpr (kResid) {
                    // The rejected rows differ per request, so the warp stages its 32
                    // rows of U and of the target through two 4 KB shared buffers with
                    // asynchronous 16-byte copies (a row segment spread over
                    // consecutive lanes, all of them in flight at once, swizzled on the
                    // chunk index); each lane then reads its own row.  The U rows of
                    // the warp's next tile are fetched while this tile is computed.
                    const uint32_t ubuf = base + L.u + (uint32_t)warp * 8192u, tbuf = ubuf + 4096u;
                    uint8_t* wbuf = gbase + L.u + (size_t)warp * 8192 + 4096;      // target rows
                    const uint8_t* ubuf_g = gbase + L.u + (size_t)warp * 8192;
                    const unsigned real_mask = __ballot_sync(0xffffffffu, real);
                    float* z = bias;                           // z overwrites the bias in place
                    // (the first tile's rows were issued before the W1 gathers)
                    if (t != (int)blockIdx.x) issue_rows<TT>(tbuf, Trow, real_mask, v0, V, lane);
                    ptx::cp_async_wait_group<1>();             // this tile's U rows
                    __syncwarp();
                    if (real) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const float4 u4 = *reinterpret_cast<const float4*>(ubuf_g + lane * 128 + ((c ^ (lane & 7)) << 4));
                            z[4 * c] = u4.x + bias[4 * c];               // z * tau
                            z[4 * c + 1] = u4.y + bias[4 * c + 1];
                            z[4 * c + 2] = u4.z + bias[4 * c + 2];
                            z[4 * c + 3] = u4.w + bias[4 * c + 3];
                        }
                    }
                    __syncwarp();
                    const int tn = t + GX;
                    if (tn < ntiles) {
                        issue_rows<float>(ubuf, Urow, real_mask, tn * kTN * RF + ti * kTN + 32 * cb, V, lane);
                        ptx::cp_async_wait_group<1>();         // this tile's target rows
                    } else {
                        ptx::cp_async_wait_group<0>();
                    }
                    __syncwarp();
                    if (real) {
                        // The draw as an exponential race (argmax log w_v + G_v =
                        // argmin E_v / w_v, E = -ln u) on the residual law
                        // r = max(0, p - q).  A quad is screened with the bound
                        // E >= 1 - u (exact from the bits, no logarithm) against the
                        // running minimum, with margins above the rounding of the
                        // products and of E; quads that pass are re-run with the exact
                        // E, entries in increasing v (strict comparisons keep the lowest
                        // index on exact ties).  The fallback law p (no residual mass
                        // at all, which only rounding can produce) is drawn by the
                        // merging CTA, on the same E, when no CTA found a winner.
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int vq = v0 + 4 * c;
                            if (vq < V) {
                                float ts[4];
                                if constexpr (sizeof(TT) == 4) {
                                    const float4 t4 =
                                        *reinterpret_cast<const float4*>(wbuf + lane * 128 + ((c ^ (lane & 7)) << 4));
                                    ts[0] = t4.x; ts[1] = t4.y; ts[2] = t4.z; ts[3] = t4.w;
                                } else {
                                    const uint2 h4 = *reinterpret_cast<const uint2*>(
                                        wbuf + lane * 64 + (((c >> 1) ^ ((lane >> 1) & 3)) << 4) + ((c & 1) << 3));
                                    ts[0] = __uint_as_float(h4.x << 16); ts[1] = __uint_as_float(h4.x & 0xffff0000u);
                                    ts[2] = __uint_as_float(h4.y << 16); ts[3] = __uint_as_float(h4.y & 0xffff0000u);
                                }
                                const uint4 w = rng.quad((uint32_t)vq >> 2);
                                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                                float pv[4], rv[4];
                                bool cand = false;
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    pv[e] = fast_exp2(fmaf(ts[e], scale2, -lse_p2));
                                    rv[e] = pv[e] - fast_exp2(fmaf(z[4 * c + e], scale2, -lse_q2));
                                    const float wv = one_minus_uniform_of(ws[e]);
                                    cand |= rv[e] > 0.f && wv < fmaf(Krh, rv[e], kRaceSlack);
                                }
                                if (cand) {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float E = exp2_variate_of(ws[e]) * kLn2;
                                        if (rv[e] > 0.f && E < rv[e] * Kr) {
                                            Kr = __fdividef(E, rv[e]);
                                            Krh = fminf(Krh, Kr * kRaceRel);
                                            st2.idx_r = vq + e;
                                        }
                                    }
                                }
                            }
                            if ((c & 3) == 3 && Kr < INFINITY) {
                                // the key E / r needs no reference: share it with the row's
                                // other threads (the bits of positive floats order as the
                                // values) and screen against the best found so far
                                const uint32_t bo = min(atomicMin(&s_key[nrow], __float_as_uint(Kr)), __float_as_uint(Kr));
                                Krh = fminf(Krh, __uint_as_float(bo) * kRaceRel);
                            }
                        }
                    }
                    __syncwarp();
                } else if (kOneRow && active) {
                    // lane c takes column c of the row lane 0 loaded
                    float u = 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float x = __shfl_sync(0xffffffffu, bias[c], 0);
                        if (lane == c) u = x;
                    }
                    const int v = v0 + lane;
                    if (v < V) {
                        if (p.logits_out) p.logits_out[out_row1 + v] = u * p.inv_tau;
                        const uint4 w = rng1.quad((uint32_t)v >> 2);
                        const uint32_t wd = (v & 2) ? ((v & 1) ? w.w : w.z) : ((v & 1) ? w.y : w.x);
                        const float te = fast_exp2(fmaf(u, scale2, -rz2));
                        if (one_minus_uniform_of(wd) < fmaf(rE2h * kLn2, te, kRaceSlack)) {
                            const float E2 = exp2_variate_of(wd);
                            if (E2 < rE2 * te) {
                                osum = osum * fast_exp2(fmaf(-u, scale2, rz2)) + 1.f;
                                rz2 = u * scale2; rE2 = E2; rE2h = E2 * kRaceRel;
                                st.idx = v; st.zb = u;
                            } else {
                                osum += te;
                            }
                        } else {
                            osum += te;
                        }
                    }
                } else if (kQuadLoop) {
                    // The accumulator holds z*tau = U + h.W2 (it started as the tile's U).
                    // Exponential race in base-2 units: the winner minimises
                    // E2_v * 2^(-z2_v), z2 = z*log2e; with the winner's z2 as the
                    // log-sum-exp reference the race and the sum share one exp2:
                    //   t_v = 2^(z2_v - z2_best),  v wins iff E2_v < E2_best * t_v.
                    // Each quad is screened with the bound E2 = -log2(u) >=
                    // (1 - u) * log2e (no logarithm; 1 - u exact from the bits)
                    // against Kh, the smaller of this thread's winner key and the
                    // best key any thread of the CTA has found on this request row
                    // (shared every 16 entries): an entry that cannot beat a key
                    // already found cannot be the row's draw.  The margins of Kh
                    // and kRaceSlack cover the rounding.  Quads that pass are
                    // re-run entry by entry, the exact variate formed only for the
                    // entries that pass.  The quads are read from TMEM one at a
                    // time, the next one's load in flight during the current one,
                    // so the loop body exists once in the code.
                    const int nq = active ? min(8, (V - v0) >> 2) : 0;   // quads inside the vocabulary
                    // one quad of the race: us = z*tau of entries vq..vq+3, w their words
                    auto race_quad = [&](const float (&us)[4], int vq, const uint4 w) {
                        if (!zst && p.logits_out)
                            *reinterpret_cast<float4*>(p.logits_out + out_row + vq) = make_float4(
                                us[0] * p.inv_tau, us[1] * p.inv_tau, us[2] * p.inv_tau, us[3] * p.inv_tau);
                        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                        float t[4], wv[4];
                        bool cand = false;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            t[e] = fast_exp2(fmaf(us[e], scale2, -ref2));
                            wv[e] = one_minus_uniform_of(ws[e]);
                            cand |= wv[e] < fmaf(Kh, t[e], kRaceSlack);
                        }
                        const float lsum0 = lsum;
                        lsum += (t[0] + t[1]) + (t[2] + t[3]);
                        if (cand) {
                            // rare.  An entry more than 64 above the reference (and the
                            // first quad, ref2 = -inf) moves the reference to the quad's
                            // maximum first and takes the quad's sum again against it;
                            // otherwise the sum took the quad as the screened path does,
                            // so it depends on the data alone.
                            const float zm2 = fmaxf(fmaxf(us[0], us[1]), fmaxf(us[2], us[3])) * scale2;
                            if (zm2 > ref2 + 64.f) {
                                // t_v = 2^(z2_v - ref2) shrinks by rs = 2^(ref2 - zm2), so the
                                // sum takes rs and the keys compared against t (K2, Kh) grow by
                                // 1 / rs (+inf past the float range: every later candidate
                                // then beats the old winner, as it must)
                                float rs = 0.f;
                                if (ref2 > -INFINITY) {
                                    rs = fast_exp2(ref2 - zm2);
                                    const float up = fast_exp2(zm2 - ref2);
                                    K2 *= up;
                                    Kh = fmaxf(Kh * up, kKhMin);
                                }
                                ref2 = zm2;
#pragma unroll
                                for (int e = 0; e < 4; ++e) t[e] = fast_exp2(fmaf(us[e], scale2, -ref2));
                                lsum = lsum0 * rs + ((t[0] + t[1]) + (t[2] + t[3]));
                            }
                            // entries in increasing v (the strict comparison keeps the
                            // lowest index on exact ties); the exact variate only for the
                            // entries that pass the screen
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (wv[e] < fmaf(Kh, t[e], kRaceSlack)) {
                                    const float E2 = exp2_variate_of(ws[e]);
                                    if (E2 < K2 * t[e]) {
                                        K2 = E2 * fast_exp2(fmaf(-us[e], scale2, ref2));   // E2 / t_v
                                        Kh = fmaxf(fminf(Kh, K2 * (kRaceRel * kLn2)), kKhMin);
                                        rz2 = us[e] * scale2; rE2 = E2;
                                        st.idx = vq + e; st.zb = us[e];
                                    }
                                }
                            }
                        }
                    };
                    // two quads per step (their random words computed side by side),
                    // the next step's columns loading meanwhile.  After steps 1 and 3
                    // the thread shares its winner key with the CTA's other threads
                    // racing the same request row and takes the best found so far
                    // (an atomic minimum that returns the previous one).  The key read
                    // depends on timing, but only as a bound for the screen: the draw
                    // itself is exact and the sum never looks at the race.
                    // logits store: this warp's 32 rows x 32 columns of z go to its
                    // staging buffer (row = lane, 16-byte chunk c at c ^ (lane & 7), the
                    // 128-byte swizzle of the map), then out in one tensor store; the
                    // previous tile's store must have read the buffer first
                    const uint32_t zrow = base + L.z + (uint32_t)warp * (uint32_t)kZBufBytes + (uint32_t)lane * 128u;
                    if (zst && nq > 0) {
                        if (lane == 0) ptx::bulk_wait_read();
                        __syncwarp();
                    }
                    uint32_t nx[8];
                    if (nq > 0) ptx::tmem_ld8(acc_tile, nx);
#pragma unroll 1
                    for (int c = 0; c < nq; c += 2) {
                        ptx::tmem_wait_ld8(nx);
                        const float ua[4] = {__uint_as_float(nx[0]), __uint_as_float(nx[1]), __uint_as_float(nx[2]),
                                             __uint_as_float(nx[3])};
                        const float ub[4] = {__uint_as_float(nx[4]), __uint_as_float(nx[5]), __uint_as_float(nx[6]),
                                             __uint_as_float(nx[7])};
                        if (c + 2 < nq) ptx::tmem_ld8(acc_tile + (uint32_t)(4 * (c + 2)), nx);
                        if (zst) {
                            const float it = p.inv_tau;
                            ptx::sts_f4(zrow + ((uint32_t)(c ^ (lane & 7)) << 4),
                                        make_float4(ua[0] * it, ua[1] * it, ua[2] * it, ua[3] * it));
                            ptx::sts_f4(zrow + ((uint32_t)((c + 1) ^ (lane & 7)) << 4),
                                        make_float4(ub[0] * it, ub[1] * it, ub[2] * it, ub[3] * it));
                        }
                        if (real) {
                            const int vq = v0 + 4 * c;
                            const uint4 wa = rng.quad((uint32_t)vq >> 2);
                            const uint4 wb = rng.quad(((uint32_t)vq >> 2) + 1u);
                            race_quad(ua, vq, wa);
                            if (c + 1 < nq) race_quad(ub, vq + 4, wb);
                            if ((c & 3) == 2 && rE2 < INFINITY && fabsf(rz2) < kShareMaxZ2 &&
                                fabsf(ref2) < kShareMaxZ2) {
                                // key = log2(E2_best) - z2_best, as order-preserving bits
                                const float lk = fast_log2(rE2) - rz2;
                                const uint32_t kb = __float_as_uint(lk);
                                const uint32_t ko = (kb & 0x80000000u) ? ~kb : (kb | 0x80000000u);
                                const uint32_t bo = min(atomicMin(&s_key[nrow], ko), ko);
                                const float lb = __uint_as_float((bo & 0x80000000u) ? (bo & 0x7fffffffu) : ~bo);
                                // per unit of t; an exponent clamped at -100 only loosens
                                // the screen
                                Kh = fmaxf(fminf(Kh, fast_exp2(fmaxf(lb + ref2, -100.f)) * (kShareRel * kLn2)), kKhMin);
                            }
                        }
                        __syncwarp();          // the next TMEM load and wait are warp-collective
                    }
                    if (zst && nq > 0) {
                        // columns past V and rows past B are clipped by the store
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_3d(&a.zmap, zrow, v0, k - 1, b_base + (32 * q) % NC);
                            ptx::bulk_commit();
                        }
                    }
                    release_acc();
                }
                if constexpr (kTgt) {
                    // target row k-1 on this warp's 32 rows x 32 columns (after the
                    // race: the bias is dead by now), then the next tile's block into
                    // the same buffer
                    if (active) {
                        bool okt = ptx::mbar_wait(tbar(warp), (uint32_t)(ltile & 1), abort_flag, wl);
                        okt = __all_sync(0xffffffffu, okt);
                        if (!okt) { if (lane == 0 && !*abort_flag) raise_timeout(p.ws.status, 12); failed = true; break; }
                        tinfl = false;
                        ++ltile;
                        const uint32_t srow = tbuf + (uint32_t)lane * 128u;
                        const int nv = V - (t * kTN * RF + ti * kTN + 32 * cb);   // entries inside the vocabulary
#pragma unroll
                        for (int h = 0; h < 2; ++h) {           // two halves of 16 columns
                            float tv[16];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float4 v4 = lds_f4(srow + ((uint32_t)((4 * h + c) ^ (lane & 7)) << 4));
                                tv[4 * c] = v4.x; tv[4 * c + 1] = v4.y; tv[4 * c + 2] = v4.z; tv[4 * c + 3] = v4.w;
                            }
                            const int nh = nv - 16 * h;
                            if (nh >= 16) tgt_lse_add<false>(tv, 16, scale2, tm2, tsum);
                            else if (nh > 0) tgt_lse_add<true>(tv, nh, scale2, tm2, tsum);
                        }
                        __syncwarp();
                        int tn = t + GX, kn = k;
                        if (tn >= ntiles) { tn = blockIdx.x; ++kn; }
                        if (kn <= k_last) {
                            if (lane == 0) tgt_issue(tn, kn);
                            tinfl = true;
                        }
                    }
                }
            }
            // ---- this position's partial state per request: fold RF tiles x 4 column blocks
            if constexpr (kResid) {
                // back to scores: log w_v + G_v = -ln(E_v / w_v)
                st2.best_r = Kr < INFINITY ? -logf(Kr) : -INFINITY;
                st2.best_p = -INFINITY;                      // drawn by the merging CTA if needed
                reinterpret_cast<Draw2*>(s_merge)[cb * 128 + row] = st2;
            } else {
                // back to the Gumbel score in natural units: with E = E2 * ln 2 the
                // winner's score is z_best - ln E, and sum_v e^(z_v - score) = s * E
                DrawLse sn = drawlse_empty();
                if (rE2 < INFINITY) {
                    const float E = rE2 * kLn2;
                    sn.zb = st.zb * p.inv_tau;
                    sn.best = sn.zb - logf(E);
                    sn.idx = st.idx;
                }
                // log sum_v e^(z_v): the one-request form sums against its winner's
                // z2 (rz2 * ln2 = the winner's z), the draft form against ref2
                if constexpr (kOneRow) sn.lse = rE2 < INFINITY ? sn.zb + logf(osum) : -INFINITY;
                else sn.lse = lsum > 0.f ? ref2 * kLn2 + logf(lsum) : -INFINITY;
                if constexpr (kOneRow) {
                    // the lanes raced columns of the one request: merge them into lane 0's row
#pragma unroll
                    for (int m = 16; m > 0; m >>= 1) sn = drawlse_merge(sn, shfl_xor(sn, m));
                    if (lane != 0) sn = drawlse_empty();
                }
                s_merge[cb * 128 + row] = sn;
            }
            if constexpr (kTgt) reinterpret_cast<float2*>(gbase + L.tmerge)[cb * 128 + row] = make_float2(tm2, tsum);
            // one barrier publishes s_merge and makes a failure a group decision
            if (ptx::bar_red_or(1, 32 * kEpiWarps, failed)) { failed = true; *abort_flag = 1u; break; }
            // every thread is past its race: the next position starts with no shared keys
            if (etid < 128) s_key[etid] = 0xFFFFFFFFu;
            DrawLse* part_buf = p.ws.draft_part + (size_t)((k - 1) & 1) * p.B * p.ws.parts;
            if (etid < nb) {
                if constexpr (kResid) {
                    const Draw2* m2 = reinterpret_cast<const Draw2*>(s_merge);
                    Draw2 s2 = draw2_empty();
                    for (int i = 0; i < RF; ++i)
#pragma unroll
                        for (int c = 0; c < 4; ++c) s2 = draw2_merge(s2, m2[c * 128 + i * NC + etid]);
                    // the draw is decided by an atomic maximum over the CTAs (score,
                    // then lowest index), in the first winner-key line of the request
                    if ((s_row[etid] >= 0 || p.resid_bonus) && s2.best_r > -INFINITY) {
                        DrawLse dk = drawlse_empty();
                        dk.best = s2.best_r; dk.idx = s2.idx_r;
                        atomicMax(&p.ws.win[(size_t)(b_base + etid) * kWinStride], win_key(dk));
                    }
                } else {
                    DrawLse s1 = drawlse_empty();
                    for (int i = 0; i < RF; ++i)
#pragma unroll
                        for (int c = 0; c < 4; ++c) s1 = drawlse_merge(s1, s_merge[c * 128 + i * NC + etid]);
                    part_buf[(size_t)(b_base + etid) * p.ws.parts + blockIdx.x] = s1;
                    if constexpr (kTgt) {
                        // this CTA's log-sum-exp partial of target row k-1, in natural units
                        const float2* tmg = reinterpret_cast<const float2*>(gbase + L.tmerge);
                        float mm = -INFINITY, ss = 0.f;
                        for (int i = 0; i < RF; ++i)
#pragma unroll
                            for (int c = 0; c < 4; ++c) lse2_merge(mm, ss, tmg[c * 128 + i * NC + etid]);
                        LseDraw o = lsedraw_empty();
                        if (mm > -INFINITY) { o.m = mm * kLn2; o.s = ss; }
                        p.ws.tgt_part[((size_t)(b_base + etid) * gamma + (k - 1)) * kTgtSlots + blockIdx.x] = o;
                    }
                    // the draw itself is decided by an atomic maximum over the CTAs
                    if (persistent)
                        atomicMax(&p.ws.win[((size_t)(k - 1) * p.B + b_base + etid) * kWinStride], win_key(s1));
                }
                // one launch per position: the ticket merge below reads these; the
                // persistent loop orders them by the grid barrier's fence instead
                // (after the epilogue's barrier, the fence covers the whole CTA's writes)
                if (!persistent) __threadfence();
            }
            if (kResid || !persistent) break;
            // ---- grid barrier, then every CTA merges the partials of its own requests
            ptx::named_barrier(1, 32 * kEpiWarps);
            __shared__ int s_gb_ok;
            if (etid == 0) s_gb_ok = grid_barrier(p.ws.gbar + (k - k_first), nctas, abort_flag, wl) ? 1 : 0;
            ptx::named_barrier(1, 32 * kEpiWarps);
            if (!s_gb_ok) {
                if (etid == 0) raise_timeout(p.ws.status, 8);
                failed = true;
                *abort_flag = 1u;
                break;
            }
            // this position's draws: one load per request
            for (int n = etid; n < nb; n += 32 * kEpiWarps) {
                // no draw at all (every score NaN, say) leaves the empty index:
                // flagged, and the next position sees a zero row
                int x = win_token(__ldcg(&p.ws.win[((size_t)(k - 1) * p.B + b_base + n) * kWinStride]));
                if (x < 0 || x >= V) { raise_status(p.ws.status, kBadToken); x = -1; }
                s_tok[n] = x;
            }
            ptx::named_barrier(1, 32 * kEpiWarps);
            if (k < k_last) {
                // ---- h = W1[x~_k] into the A operands for the next position (the
                //      MMAs of this one are complete: the last commit released the
                //      final tile the warps just read)
                if constexpr (kRnn) {
                    // RNN head: the GRU step for every request, shared out by
                    // hidden unit over the CTAs, then a second grid barrier
                    gate_step(a.gru, k, (int)(blockIdx.y * GX + blockIdx.x), (int)nctas, etid,
                              32 * kEpiWarps, gridDim.y == 1 ? s_tok : nullptr, p.ws.win);
                    ptx::named_barrier(1, 32 * kEpiWarps);
                    if (etid == 0)
                        s_gb_ok = grid_barrier(p.ws.gbar + kGbarGru + (k - k_first), nctas, abort_flag, wl) ? 1 : 0;
                    ptx::named_barrier(1, 32 * kEpiWarps);
                    if (!s_gb_ok) {
                        if (etid == 0) raise_timeout(p.ws.status, 9);
                        failed = true;
                        *abort_flag = 1u;
                        break;
                    }
                    stage_a_state(tmem_base, st_base, (size_t)p.B * r, k, s_row, s_tok, NC, RF, r, V, q, cb, lane, false);
                } else {
                    stage_a_tmem(tmem_base, W1, s_tok, NC, RF, r, V, q, cb, lane, false);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::named_barrier(1, 32 * kEpiWarps);
                if (etid == 0) ptx::mbar_arrive(a_ready);
                if constexpr (kRnn) {
                    // W_hh . state[k] for the next boundary's GRU step, off its critical path
                    if (k + 1 < k_last)
                        gh_compute(a.gru, k, (int)(blockIdx.y * GX + blockIdx.x), (int)nctas, warp, lane);
                }
            }
            // ---- this position's outputs, while the MMA starts the next one: the
            //      CTAs share the requests, a warp folds one request's partials
            for (int n = blockIdx.x + warp * GX; n < nb; n += kEpiWarps * GX) {
                const float4* part = reinterpret_cast<const float4*>(part_buf + (size_t)(b_base + n) * p.ws.parts);
                DrawLse m = drawlse_empty();
                for (int i0 = lane; i0 < GX; i0 += 4 * 32) {
                    float4 c[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + 32 * u;
                        c[u] = i < GX ? __ldcg(part + i) : make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.f, -INFINITY);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) m = drawlse_merge(m, drawlse_of(c[u]));
                }
#pragma unroll
                for (int sh = 1; sh < 32; sh <<= 1) m = drawlse_merge(m, shfl_xor(m, sh));
                if (lane == 0) {
                    const size_t o = (size_t)(b_base + n) * gamma + (k - 1);
                    p.draft_tok[o] = m.idx;
                    p.lse_q[o] = m.lse;
                    p.z_tok[o] = m.zb;
                }
            }
            if (k == k_last) break;
        }
        if (failed) *abort_flag = 1u;
        // the logits stores have read their buffers before the CTA leaves
        if (zst && lane == 0) ptx::bulk_wait_all();
        // a target load still in flight (after a failure) lands before the CTA leaves
        if (kTgt && tinfl && lane == 0) ptx::mbar_wait(tbar(warp), (uint32_t)(ltile & 1), never, kDrainCycles);
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, 512u);
    }

    if (persistent) {
        // the last CTA out clears the barrier counters and the winner keys for
        // the next call (every CTA has read its winners before it got here)
        __shared__ int s_out_last;
        if (tid == 0) {
            __threadfence();
            s_out_last = atomicAdd(p.ws.gbar + kGbarExit, 1u) == nctas - 1;
        }
        __syncthreads();
        if (s_out_last) {
            __threadfence();
            for (int i = tid; i < p.gamma * p.B; i += kThreads) p.ws.win[(size_t)i * kWinStride] = 0ull;
            if (tid <= kGbarExit) p.ws.gbar[tid] = 0u;
            __threadfence();
        }
        return;
    }

    // residual draw: every CTA has folded its draws into the winner keys; the
    // compaction launch behind this one decodes them (and draws the fallback
    // law where a request found no residual mass)
    if constexpr (kResid) return;
    // single position: the last-arriving CTA of this request chunk merges the partial states
    uint32_t* ticket = &p.ws.tickets_draft[chunk];
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(ticket, 1u);
        s_last = (prev == (unsigned)GX - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // TM = 512 / NC consecutive threads per request, each folding every TM-th
    // partial with all loads of a batch in flight, then a shuffle merge
    const int k = k_first;
    const int TM = (32 * kEpiWarps) / NC;
    const int n = tid / TM, sub = tid - n * TM;
    const int nparts = GX;
    constexpr int kBatch = 5;
    if (tid < 32 * kEpiWarps) {
        const int bb = b_base + n;
        {
            DrawLse m = drawlse_empty();
            if (n < nb) {
                const float4* part = reinterpret_cast<const float4*>(
                    p.ws.draft_part + (size_t)((k - 1) & 1) * p.B * p.ws.parts + (size_t)bb * p.ws.parts);
                for (int i0 = sub; i0 < nparts; i0 += kBatch * TM) {
                    float4 c[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int i = i0 + u * TM;
                        c[u] = i < nparts ? __ldcg(part + i) : make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.f, -INFINITY);
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) m = drawlse_merge(m, drawlse_of(c[u]));
                }
            }
            for (int sh = 1; sh < TM; sh <<= 1) m = drawlse_merge(m, shfl_xor(m, sh));
            if (sub == 0 && n < nb) {
                const size_t o = (size_t)bb * gamma + (k - 1);
                p.draft_tok[o] = m.idx;
                p.lse_q[o] = m.lse;
                p.z_tok[o] = m.zb;
            }
        }
    }
    if (tid == 0) *ticket = 0u;
}

}  // namespace

void* tma_encoder() {
    static void* fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = f;
    }
    return fn;
}

bool rows_supported(const DraftParams& p) {
    return p.W_bf16 && !p.U_bf16 && p.B >= 1 && p.r % 64 == 0 && p.r <= 256 && p.V % 8 == 0 &&
           tma_encoder() != nullptr;
}

bool draft_rows_supported(const DraftParams& p) { return rows_supported(p); }

int draft_rows_grid_x(int B, int V, int parts) {
    const int NC = B <= 64 ? 64 : 128;
    const int nchunks = (B + NC - 1) / NC;
    const int ntiles = (V + kTN * (128 / NC) - 1) / (kTN * (128 / NC));
    int gx = num_sms() / nchunks;
    gx = gx < 1 ? 1 : gx;
    gx = gx > ntiles ? ntiles : gx;
    gx = gx > parts ? parts : gx;
    return gx;
}

bool cooperative_supported() {
    static int cached[64] = {0};     // 0 unknown, 1 yes, 2 no
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!cached[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev);
        cached[dev] = v ? 1 : 2;
    }
    return cached[dev] == 1;
}

static cudaError_t launch_rows(const DraftParams& p, int k_first, int k_last, bool resid, const void* target,
                               bool target_bf16, uint32_t* near_ties, cudaStream_t s,
                               const GruParams* gru = nullptr, bool side = false) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encoder());
    if (!enc) return cudaErrorNotSupported;
    RowsArgs a;
    a.p = p;
    a.NC = p.B <= 64 ? 64 : 128;           // RF = 2 or 1: RF = 4 would leave no TMEM for accumulators
    a.target = target;
    a.near_ties = near_ties;
    if (gru) a.gru = *gru;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.r};
        const cuuint64_t strides[1] = {(cuuint64_t)p.V * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)w2_kc(p.r, !resid && !gru && p.B == 1)};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&a.w2map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.W2), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.gamma, (cuuint64_t)p.B};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 4, (cuuint64_t)p.gamma * p.V * 4};
        const cuuint32_t box[3] = {32, 1, (cuuint32_t)a.NC};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&a.umap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(p.U), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // the target stream (Markov draft only): target [B][gamma+1][V] fp32, one
    // epilogue warp's block
    const bool tgt = !resid && !gru && !side && p.target != nullptr;
    if (tgt) {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)(p.gamma + 1), (cuuint64_t)p.B};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 4, (cuuint64_t)(p.gamma + 1) * p.V * 4};
        const cuuint32_t es[3] = {1, 1, 1};
        const cuuint32_t box[3] = {32, 1, 32};
        if (enc(&a.tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.target), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // the logits leave by tensor stores (the requests-on-lanes race without the
    // target stream; the one-request form stores its lanes' columns directly)
    const bool zst = !resid && !tgt && (gru != nullptr || p.B > 1) && p.logits_out != nullptr;
    if (zst) {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.gamma, (cuuint64_t)p.B};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 4, (cuuint64_t)p.gamma * p.V * 4};
        const cuuint32_t box[3] = {32, 1, 32};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&a.zmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.logits_out, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const Layout L = rows_layout(a.NC, p.r, resid, tgt, zst, !resid && !gru && p.B == 1);
    const size_t smem = L.total + 1024;
    auto kern = resid ? (target_bf16 ? rows_kernel<true, uint16_t> : rows_kernel<true, float>)
                : gru ? rows_kernel<false, float, true>
                : tgt ? (p.B == 1 ? rows_kernel<false, float, false, true, true> : rows_kernel<false, float, false, false, true>)
                : side ? (p.B == 1 ? rows_kernel<false, float, false, true, false, true>
                                   : rows_kernel<false, float, false, false, false, true>)
                       : (p.B == 1 ? rows_kernel<false, float, false, true> : rows_kernel<false, float>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the target stream beside the draft needs the rest of the SM's shared
    // memory: configure the largest shared-memory carve-out
    if (side) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    const int nchunks = (p.B + a.NC - 1) / a.NC;
    const int gx = draft_rows_grid_x(p.B, p.V, p.ws.parts);
    if (tgt && gx > kTgtSlots) return cudaErrorInvalidConfiguration;
    if (side && (k_last == k_first || (int)(gx * nchunks) > num_sms())) return cudaErrorInvalidConfiguration;
    const dim3 grid(gx, nchunks);
    if (k_last > k_first) {
        // every CTA waits for all others between positions: they must be co-resident
        void* args[] = {&a, const_cast<int*>(&k_first), const_cast<int*>(&k_last)};
        return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), grid, dim3(kThreads), args, smem, s);
    }
    if (resid) return launch_dependent(kern, grid, dim3(kThreads), smem, s, a, k_first, k_last);
    kern<<<grid, kThreads, smem, s>>>(a, k_first, k_last);
    return cudaGetLastError();
}

cudaError_t launch_draft_rows(const DraftParams& p, int k_first, int k_last, cudaStream_t s) {
    return launch_rows(p, k_first, k_last, false, nullptr, false, nullptr, s);
}

// All gamma positions of the draft.  bf16 weights with fp32 U run the
// tensor-core rows kernel: one cooperative launch for the gamma positions,
// or one launch per position where the device lacks cooperative launch (and
// for gamma = 1); any other combination runs the CUDA-core kernel, one
// launch per position.
cudaError_t launch_draft(const DraftParams& p, cudaStream_t s) {
    const bool rows = rows_supported(p);
    if (rows && p.gamma > 1 && cooperative_supported()) return launch_draft_rows(p, 1, p.gamma, s);
    for (int k = 1; k <= p.gamma; ++k) {
        const cudaError_t e = rows ? launch_draft_rows(p, k, k, s) : launch_draft_simt(p, k, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool draft_target_supported(const DraftParams& p) {
    return rows_supported(p) && p.target != nullptr && draft_rows_grid_x(p.B, p.V, p.ws.parts) <= kTgtSlots;
}

// Several positions in one cooperative launch (one draft CTA per SM): the
// verify stream runs beside the draft, on the same SMs.
bool draft_target_vs(const DraftParams& p) {
    return rows_supported(p) && p.target != nullptr && p.gamma > 1 && cooperative_supported() &&
           draft_rows_grid_x(p.B, p.V, p.ws.parts) * ((p.B + (p.B <= 64 ? 64 : 128) - 1) / (p.B <= 64 ? 64 : 128)) <=
               num_sms();
}

// The Markov draft with the target stream: the lean stream kernel beside the
// draft when draft_target_vs holds; otherwise the epilogue warps reduce the
// target rows themselves, in one cooperative launch for the gamma positions
// or one launch per position (the rows kernel merges a single position's
// partials itself).
cudaError_t launch_draft_target(const DraftParams& p, cudaStream_t s) {
    if (draft_target_vs(p)) {
        // the plain draft, then the lean target stream on the SMs beside it
        DraftParams q = p;
        q.target = nullptr;
        cudaError_t e = launch_rows(q, 1, p.gamma, false, nullptr, false, nullptr, s, nullptr, true);
        if (e != cudaSuccess) return e;
        VerifyParams v;
        v.vs_full = 1;                              // rows 0..gamma: the bonus row too
        v.target = p.target; v.target_bf16 = p.target_bf16;
        v.U = p.U; v.U_bf16 = p.U_bf16; v.W1 = p.W1; v.W2 = p.W2; v.W_bf16 = p.W_bf16;
        v.anchor = p.anchor; v.draft_tok = p.draft_tok; v.lse_q = p.lse_q; v.z_tok = p.z_tok; v.K = nullptr;
        v.B = p.B; v.gamma = p.gamma; v.V = p.V; v.r = p.r; v.req_base = p.req_base;
        v.inv_tau = p.inv_tau; v.seed = p.seed; v.step = p.step;
        v.accepted = nullptr; v.out_tok = nullptr; v.out_req = nullptr; v.out_pos = nullptr;
        v.out_off = nullptr; v.next_anchor = nullptr; v.p_tok = nullptr; v.near_ties = nullptr;
        v.ws = p.ws;
        v.tgt_token = p.tgt_token;
        return launch_target_stream_side(v, s);
    }
    if (!draft_target_supported(p)) return cudaErrorNotSupported;
    if (p.gamma > 1 && cooperative_supported()) return launch_rows(p, 1, p.gamma, false, nullptr, false, nullptr, s);
    for (int k = 1; k <= p.gamma; ++k) {
        const cudaError_t e = launch_rows(p, k, k, false, nullptr, false, nullptr, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// The RNN head's draft in one cooperative launch: positions k_first..k_last,
// the GRU step for position k + 1 run inside the kernel after position k's
// draws (state[k_first - 1] must be ready).
cudaError_t launch_draft_rows_rnn(const DraftParams& p, const GruParams& g, int k_first, int k_last,
                                  cudaStream_t s) {
    return launch_rows(p, k_first, k_last, false, nullptr, false, nullptr, s, &g);
}

bool resid_rows_supported(const VerifyParams& v) {
    DraftParams p = draft_view(v);
    return rows_supported(p);
}

cudaError_t launch_resid_rows(const VerifyParams& v, cudaStream_t s) {
    return launch_rows(draft_view(v), 1, 1, true, v.target, v.target_bf16 != 0, v.near_ties, s);
}

}  // namespace dspark
