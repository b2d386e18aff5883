// sts_fit.cu -- sequential temperature scaling (STS): the per-position
// temperature fit ("DSpark：半自回归生成与置信度调度的投机解码", section
// 校准问题：原始置信度不可靠; "DeepSeek-AI与北京大学联手破局", section 四).
//
// One launch per draft position k, left to right.  For every candidate
// temperature T_g of the grid, the expected calibration error of the prefix-k
// survival
//     a_n(T_g) = prod_{i<k} sigma(s_{n,i} / T_i) * sigma(s_{n,k} / T_g)
// against the labels y_n = [acc_len_n >= k], over M equal-width bins of [0, 1]:
//     ECE(T_g) = (1/N) sum_m | sum_{n in bin m} (y_n - a_n) |.
// The earlier T_i are the grid values the earlier launches chose.
//
// Work split.  CTA (slice, chunk) takes a contiguous slice of the samples and
// a chunk of 32*CPL candidates.  Lane l of every warp owns the chunk's
// candidates l, l+32, ..., so each (bin, candidate) accumulator in shared
// memory belongs to one lane of one warp: plain read-modify-write, no
// atomics, and the bank is the lane.  A warp takes 32 samples at a time:
// their score rows and labels arrive by cp.async one batch ahead, lane j
// forms sample j's 1 / (M * prod_{i<k} sigma) and M * label, and every lane
// then evaluates its candidates on each of the 32 samples.  One evaluation
// is a 2^x, a fused multiply-add and a reciprocal for M * a, the bin by
// round-to-integer arithmetic and one shared-memory read-modify-write.  The
// 2^x, the reciprocal and the two shared-memory accesses all go through the
// SM's shared memory-and-special-function issue path, which bounds the
// kernel (up to 20 warps per SM hide the latency of the rest).
//
// Bin decisions are taken in binary32: with the 2^x and reciprocal errors of
// the hardware approximations (about 2^-22 and 2^-23 relative) the computed
// M * a_n stays within about M * k * 6e-7 of the exact value, so a sample
// whose exact M * a_n lies that close to an integer may fall in the
// neighbouring bin.  The float64 oracle decides bins exactly; tests flag such
// samples as near-ties.
//
// Sums.  Per warp in binary32 (fixed sample order), per CTA over the warps in
// a fixed order, then rounded to fixed point (2^-24 units of M * (y - a)) and
// added into a global int64 accumulator [gamma][M][G]: integer addition makes
// the totals independent of the order in which CTAs arrive, so equal
// candidates (equal grid values, or scores of 0) produce equal totals.  The
// last CTA of the launch (arrival ticket) turns the totals into ECE values
// and picks the candidate with the smallest sum of |bin totals|, the lowest
// grid index on ties.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRound = 12582912.f;      // 1.5 * 2^23: x + kRound rounds 0 <= x < 2^22 to an integer
constexpr int kRoundBits = 0x4B400000;    // bit pattern of kRound
constexpr float kFix = 16777216.f;        // 2^24, fixed-point scale of the global totals
constexpr int kMaxWarps = 20;
constexpr size_t kSmemBudget = 220 * 1024;

__device__ __forceinline__ float fast_rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// sigmoid(s / T) = 1 / (1 + 2^(s * c)) with c = -log2(e) / T.
__device__ __forceinline__ float sigmoid_c(float s, float c) { return fast_rcp(1.f + fast_exp2(s * c)); }

__device__ __forceinline__ bool less_key(unsigned long long a, int ia, unsigned long long b, int ib) {
    return a < b || (a == b && ia < ib);
}

// 4-byte asynchronous copy global -> shared.
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Shared memory of one warp: staged samples, two buffers of raw score rows
// and labels (the batch being evaluated and the next one, in flight), and
// the warp's bin sums with one spare row for M * a rounding up to M.  The
// size is a multiple of 16 bytes, so every warp's region is float4-aligned.
__host__ __device__ __forceinline__ size_t warp_smem_bytes(int gamma, int M, int Gc) {
    return 32 * sizeof(float4) + 2 * 32 * (size_t)gamma * sizeof(float) + 2 * 32 * sizeof(int) +
           (size_t)(M + 1) * Gc * sizeof(float);
}

// Copy the score rows and labels of samples [b, b + cnt) into a raw buffer.
__device__ __forceinline__ void prefetch_batch(const StsFitParams& p, long long b, int cnt, float* raw, int* lab,
                                               int lane) {
    const float* src = p.score + b * p.gamma;
    const int nf = cnt * p.gamma;
    for (int i = lane; i < nf; i += 32) cp_async_4(raw + i, src + i);
    if (lane < cnt) cp_async_4(lab + lane, p.acc_len + b + lane);
    cp_async_commit();
}

// One staged sample against the lane's CPL candidates: the bin row offset
// and M * (y - a) of each.  v = (s_k, 1 / (M * prefix), M * label).
template <int CPL>
__device__ __forceinline__ void eval_sample(const float4 v, const float (&cg)[CPL], int (&addr)[CPL],
                                            float (&d)[CPL]) {
    constexpr int Gc = 32 * CPL;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const float e = fast_exp2(v.x * cg[c]);          // exp(-s_k / T)
        const float u = fast_rcp(fmaf(v.y, e, v.y));     // M * a = M * prefix / (1 + e)
        const float t = u + kRound;                      // 0 <= u <= M (1 + 2^-20)
        const float r = t - kRound;                      // u rounded to the nearest integer
        const int bin = (__float_as_int(t) - kRoundBits) - (u < r ? 1 : 0);   // floor(u)
        addr[c] = bin * Gc + 32 * c;
        d[c] = v.z - u;
    }
}

// Add the evaluations into the lane's bin sums.  The CPL addresses are
// distinct (different columns): load all, then store all.
template <int CPL>
__device__ __forceinline__ void add_sample(float* acc, const int (&addr)[CPL], const float (&d)[CPL]) {
    float old[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) old[c] = acc[addr[c]];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[addr[c]] = old[c] + d[c];
}

template <int CPL>
__global__ void __launch_bounds__(kMaxWarps * 32, 1)
sts_eval_kernel(StsFitParams p, int k, long long per_cta) {
    constexpr int Gc = 32 * CPL;
    extern __shared__ float4 smem4[];
    __shared__ float c_prev[DSPARK_MAX_GAMMA];
    __shared__ unsigned s_last;
    __shared__ unsigned long long s_best[kMaxWarps];
    __shared__ int s_bidx[kMaxWarps];

    const int nw = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int M = p.M, gamma = p.gamma;
    // [nw] x { stage[32] float4 | raw[2][32 * gamma] | lab[2][32] | acc[M + 1][Gc] }
    const size_t wbytes = warp_smem_bytes(gamma, M, Gc);
    char* wbase = reinterpret_cast<char*>(smem4) + (size_t)warp * wbytes;
    float4* st = reinterpret_cast<float4*>(wbase);
    float* raw = reinterpret_cast<float*>(wbase + 32 * sizeof(float4));
    int* lab = reinterpret_cast<int*>(raw + 2 * 32 * gamma);
    float* accw = reinterpret_cast<float*>(lab + 2 * 32);
    for (int i = lane; i < (M + 1) * Gc; i += 32) accw[i] = 0.f;
    if (threadIdx.x < k - 1) c_prev[threadIdx.x] = -kLog2e / p.T_out[threadIdx.x];

    const int g0 = blockIdx.y * Gc;
    float cg[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int g = g0 + lane + 32 * c;
        float T = 1.f;
        if (g < p.G) {
            T = p.grid[g];
            if (!(T > 0.f && T < INFINITY)) {
                if (blockIdx.x == 0) raise_status(p.status, kBadInput);
                T = 1.f;
            }
        }
        cg[c] = -kLog2e / T;
    }

    const long long n0 = (long long)blockIdx.x * per_cta;
    const long long n1 = min((long long)p.N, n0 + per_cta);
    const float fM = (float)M;
    float* acc = accw + lane;
    const long long stride = 32LL * nw;
    long long b = n0 + 32LL * warp;
    if (b < n1) prefetch_batch(p, b, (int)min(32LL, n1 - b), raw, lab, lane);
    __syncthreads();   // c_prev

    for (int buf = 0; b < n1; b += stride, buf ^= 1) {
        const int cnt = (int)min(32LL, n1 - b);
        const long long bn = b + stride;
        if (bn < n1) {
            prefetch_batch(p, bn, (int)min(32LL, n1 - bn), raw + (buf ^ 1) * 32 * gamma, lab + (buf ^ 1) * 32,
                           lane);
            cp_async_wait_group<1>();
        } else {
            cp_async_wait_group<0>();
        }
        __syncwarp();
        float4 q = make_float4(0.f, 3.402823466e38f, 0.f, 0.f);
        if (lane < cnt) {
            const float* s = raw + buf * 32 * gamma + lane * gamma;
            float PM = fM;
            bool finite = true;
            for (int i = 0; i < k - 1; ++i) {
                const float z = s[i];
                finite &= fabsf(z) < INFINITY;
                PM *= sigmoid_c(z, c_prev[i]);
            }
            const float zk = s[k - 1];
            finite &= fabsf(zk) < INFINITY;
            if (finite) q = make_float4(zk, fminf(fast_rcp(PM), 3.402823466e38f),
                                        lab[buf * 32 + lane] >= k ? fM : 0.f, 0.f);
            else raise_status(p.status, kBadInput);
        }
        st[lane] = q;
        __syncwarp();
        int j = 0;
        for (; j + 1 < cnt; j += 2) {
            int a0[CPL], a1[CPL];
            float d0[CPL], d1[CPL];
            eval_sample<CPL>(st[j], cg, a0, d0);
            eval_sample<CPL>(st[j + 1], cg, a1, d1);
            add_sample<CPL>(acc, a0, d0);
            add_sample<CPL>(acc, a1, d1);
        }
        if (j < cnt) {
            int a0[CPL];
            float d0[CPL];
            eval_sample<CPL>(st[j], cg, a0, d0);
            add_sample<CPL>(acc, a0, d0);
        }
        __syncwarp();
    }
    __syncthreads();

    // CTA totals (warps in a fixed order; the spare row joins row M-1) into
    // the global fixed-point accumulator.
    long long* gacc = p.acc + (size_t)(k - 1) * M * p.G;
    for (int i = threadIdx.x; i < M * Gc; i += blockDim.x) {
        const int m = i / Gc, col = i - m * Gc;   // column lane + 32c holds candidate g0 + column
        const int g = g0 + col;
        if (g >= p.G) continue;
        float sum = 0.f;
        for (int w = 0; w < nw; ++w) {
            const float* aw = reinterpret_cast<const float*>(reinterpret_cast<const char*>(smem4) + (size_t)w * wbytes +
                                                             32 * sizeof(float4) + 2 * 32 * gamma * sizeof(float) +
                                                             2 * 32 * sizeof(int));
            sum += aw[m * Gc + col];
            if (m == M - 1) sum += aw[M * Gc + col];
        }
        const long long fx = __float2ll_rn(sum * kFix);
        if (fx) atomicAdd(reinterpret_cast<unsigned long long*>(gacc + (size_t)m * p.G + g), (unsigned long long)fx);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(p.tickets + (k - 1), 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // Last CTA: ECE of every candidate and the argmin.
    const double norm = 1.0 / ((double)kFix * (double)p.N * (double)M);
    unsigned long long best = ~0ull;
    int bidx = 0x7fffffff;
    for (int g = threadIdx.x; g < p.G; g += blockDim.x) {
        unsigned long long tot = 0;
        for (int m = 0; m < M; ++m) {
            const long long v = (long long)__ldcg(reinterpret_cast<const unsigned long long*>(gacc + (size_t)m * p.G + g));
            tot += (unsigned long long)(v < 0 ? -v : v);
        }
        p.ece_out[(size_t)(k - 1) * p.G + g] = (double)tot * norm;
        if (less_key(tot, g, best, bidx)) { best = tot; bidx = g; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (less_key(ob, oi, best, bidx)) { best = ob; bidx = oi; }
    }
    if (lane == 0) { s_best[warp] = best; s_bidx[warp] = bidx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < nw; ++w)
            if (less_key(s_best[w], s_bidx[w], best, bidx)) { best = s_best[w]; bidx = s_bidx[w]; }
        p.idx_out[k - 1] = bidx;
        p.T_out[k - 1] = p.grid[bidx];
    }
}

template <int CPL>
cudaError_t launch_cpl(const StsFitParams& p, cudaStream_t s) {
    constexpr int Gc = 32 * CPL;
    const size_t per_warp = warp_smem_bytes(p.gamma, p.M, Gc);
    int nw = (int)(kSmemBudget / per_warp);
    nw = nw > kMaxWarps ? kMaxWarps : (nw < 1 ? 1 : nw);
    const size_t smem = per_warp * nw;
    cudaError_t e = cudaFuncSetAttribute(sts_eval_kernel<CPL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sts_eval_kernel<CPL>, nw * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int nchunk = (p.G + Gc - 1) / Gc;
    const long long want = ((long long)num_sms() * per_sm + nchunk - 1) / nchunk;
    const long long max_slices = ((long long)p.N + 31) / 32;
    long long slices = want < max_slices ? want : max_slices;
    if (slices < 1) slices = 1;
    // Samples per CTA: a multiple of 32 * warps when a slice is that large,
    // so every warp of a full CTA gets the same number of batches.
    const long long quantum = (long long)p.N >= slices * 32LL * nw ? 32LL * nw : 32;
    long long per_cta = ((long long)p.N + slices - 1) / slices;
    per_cta = (per_cta + quantum - 1) / quantum * quantum;
    slices = ((long long)p.N + per_cta - 1) / per_cta;
    const dim3 grid((unsigned)slices, (unsigned)nchunk);
    for (int k = 1; k <= p.gamma; ++k) {
        sts_eval_kernel<CPL><<<grid, nw * 32, smem, s>>>(p, k, per_cta);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_sts_fit(const StsFitParams& p, cudaStream_t s) {
    if (p.G > 64) return launch_cpl<4>(p, s);
    if (p.G > 32) return launch_cpl<2>(p, s);
    return launch_cpl<1>(p, s);
}

}  // namespace dspark
