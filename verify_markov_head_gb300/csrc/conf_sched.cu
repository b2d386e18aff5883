// conf_sched.cu -- confidence head + sequential temperature scaling + prefix
// survival, and the hardware-aware greedy prefix scheduler.
//
// confidence_kernel: one CTA per (draft position k, request).
//   s_k = w_c . [h_k ; emb(x~_{k-1})] + b_c  (float4 loads, block sum); the
//   last CTA of a request forms
//   conf_cal = sigmoid(s_k / T_k), log_surv = running sum of log conf_cal
//   ("DSpark：半自回归生成与置信度调度的投机解码" sections 置信度头 and 校准问题;
//    "DeepSeek-AI与北京大学联手破局" section 四).  logit(sigmoid(s)) = s, so the
//   calibrated confidence is formed from s directly.
//
// schedule_kernel: one CTA of 1024 threads ("DSpark：半自回归生成与置信度调度的投机解码"
//   section 硬件感知前缀调度器; "DeepSeek-AI与北京大学联手破局" sections 四, 五).
//   Keys are the order-preserving bit patterns of log a, complemented so an
//   ascending sort gives descending survival; a stable LSD radix sort (8
//   passes of 4 bits) keeps the (b, j) order of equal keys.  The survival
//   prefix sums and Theta(n) = (R + sum) * SPS(R + n) are formed in fp64 by a
//   block scan; the admitted count is a block min-reduction (synchronous: the
//   first n with Theta(n+1) <= Theta(n)) or a block argmax (asynchronous).
#include "common.cuh"
#include "internal.h"
#include "pdl.cuh"

namespace dspark {
namespace {

constexpr int kConfThreads = 256;

// One CTA per (position k, request b): s_k = w_c . [h_k ; emb(x~_{k-1})] + b_c
// as a block reduction with the loads of a thread in flight together; the
// last CTA of a request to finish (atomic ticket) turns the gamma scores into
// calibrated confidences and the running log-survival.
template <typename ET>
__global__ void __launch_bounds__(kConfThreads) confidence_kernel(const ConfParams p) {
    grid_dependency_wait();
    const int k = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gamma = p.gamma, d = p.d, e = p.e;
    __shared__ float s_red[kConfThreads / 32];
    int x = (k == 0) ? p.anchor[b] : p.draft_tok[(size_t)b * gamma + (k - 1)];
    if (x < 0 || x >= p.V) {
        if (tid == 0) raise_status(p.status, kBadToken);
        x = -1;
    }
    const float* hk = p.h + ((size_t)b * gamma + k) * d;
    const ET* ek = static_cast<const ET*>(p.emb) + (size_t)(x < 0 ? 0 : x) * e;
    float acc = 0.f;
    if ((d % 4) == 0 && (e % 4) == 0) {
#pragma unroll 4
        for (int i = 4 * tid; i < d; i += 4 * kConfThreads) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(p.w_c + i));
            const float4 hv = __ldcs(reinterpret_cast<const float4*>(hk + i));
            acc = fmaf(w.x, hv.x, fmaf(w.y, hv.y, fmaf(w.z, hv.z, fmaf(w.w, hv.w, acc))));
        }
        if (x >= 0) {
#pragma unroll 4
            for (int i = 4 * tid; i < e; i += 4 * kConfThreads) {
                const float4 w = __ldg(reinterpret_cast<const float4*>(p.w_c + d + i));
                const float4 ev = Vec4<ET>::load(ek + i);
                acc = fmaf(w.x, ev.x, fmaf(w.y, ev.y, fmaf(w.z, ev.z, fmaf(w.w, ev.w, acc))));
            }
        }
    } else {
        for (int i = tid; i < d; i += kConfThreads) acc = fmaf(p.w_c[i], hk[i], acc);
        if (x >= 0)
            for (int i = tid; i < e; i += kConfThreads) acc = fmaf(p.w_c[d + i], to_f32(ek[i]), acc);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) s_red[warp] = acc;
    __syncthreads();
    if (tid != 0) return;
    float sk = p.b_c;
    for (int w = 0; w < kConfThreads / 32; ++w) sk += s_red[w];
    p.score[(size_t)b * gamma + k] = sk;
    __threadfence();
    if (atomicAdd(&p.tickets[b], 1u) != (unsigned)(gamma - 1)) return;
    __threadfence();
    float run = 0.f;
    for (int i = 0; i < gamma; ++i) {
        const float xi = __ldcg(&p.score[(size_t)b * gamma + i]) / p.T[i];
        // sigmoid and its log, stable for either sign of x
        const float en = expf(-fabsf(xi));
        const float c = (xi >= 0.f) ? 1.f / (1.f + en) : en / (1.f + en);
        const float logc = (xi >= 0.f) ? -log1pf(en) : xi - log1pf(en);
        run += logc;
        const size_t o = (size_t)b * gamma + i;
        p.conf_cal[o] = c;
        p.log_surv[o] = run;
    }
    p.tickets[b] = 0u;
}

// ----------------------------------------------------------------- scheduler
constexpr int kST = 1024;                       // threads
constexpr int kIPT = DSPARK_MAX_SCHED_ITEMS / kST;   // items per thread (4)
constexpr int kDigits = 16;

__device__ __forceinline__ uint32_t desc_key(float f) {
    uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);   // -0 and +0 compare equal
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // ascending bits = ascending float
    return ~u;                                          // ascending bits = descending float
}

struct SchedSmem {
    uint32_t key[2][DSPARK_MAX_SCHED_ITEMS];
    uint16_t val[2][DSPARK_MAX_SCHED_ITEMS];
    int cnt[kDigits * kST];
    double dscan[kST / 32];
    int iscan[kST / 32];
    int kcount[DSPARK_MAX_SCHED_ITEMS];
    int red_i[kST / 32];
    double red_d[kST / 32];
};

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix.
__device__ int block_exscan_int(int x, int* wsum, int& total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int incl = x;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, m);
        if (lane >= m) incl += y;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, m);
            if (lane >= m) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    total = wsum[31];
    return (warp ? wsum[warp - 1] : 0) + incl - x;
}

__device__ double block_exscan_double(double x, double* wsum, double& total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    double incl = x;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, m);
        if (lane >= m) incl += y;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double w = wsum[lane];
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, w, m);
            if (lane >= m) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    total = wsum[31];
    return (warp ? wsum[warp - 1] : 0.0) + incl - x;
}

// Stable sort of the n candidates of `ls` by descending survival; the result
// order (candidate ids b*gamma + j-1) ends in S.val[0][0..n).
__device__ void sort_candidates(SchedSmem& S, const float* ls, int n) {
    const int tid = threadIdx.x;
    for (int i = tid; i < n; i += kST) { S.key[0][i] = desc_key(ls[i]); S.val[0][i] = (uint16_t)i; }
    __syncthreads();
    int cur = 0;
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 4 * pass;
        int c[kDigits];
#pragma unroll
        for (int dg = 0; dg < kDigits; ++dg) c[dg] = 0;
        const int i0 = tid * kIPT;
#pragma unroll
        for (int j = 0; j < kIPT; ++j)
            if (i0 + j < n) c[(S.key[cur][i0 + j] >> shift) & 15u]++;
#pragma unroll
        for (int dg = 0; dg < kDigits; ++dg) S.cnt[dg * kST + tid] = c[dg];
        __syncthreads();
        // exclusive scan over (digit-major, thread-minor): 16 entries per thread
        int local[kDigits];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < kDigits; ++j) { local[j] = sum; sum += S.cnt[tid * kDigits + j]; }
        int total;
        const int base = block_exscan_int(sum, S.iscan, total);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kDigits; ++j) S.cnt[tid * kDigits + j] = base + local[j];
        __syncthreads();
        int pos[kDigits];
#pragma unroll
        for (int dg = 0; dg < kDigits; ++dg) pos[dg] = S.cnt[dg * kST + tid];
#pragma unroll
        for (int j = 0; j < kIPT; ++j) {
            if (i0 + j < n) {
                const uint32_t kk = S.key[cur][i0 + j];
                const int dg = (kk >> shift) & 15u;
                const int o = pos[dg]++;
                S.key[cur ^ 1][o] = kk;
                S.val[cur ^ 1][o] = S.val[cur][i0 + j];
            }
        }
        __syncthreads();
        cur ^= 1;
    }
    // 8 passes: the result is back in buffer 0
}

// Theta(m) for the sorted list in S.val[0]: thread tid owns m = tid*kIPT + 1 .. +kIPT
// (m = 0 is R * SPS(R)).  Writes theta[j] for its items; returns via arrays.
__device__ void theta_items(SchedSmem& S, const float* ls, const float* sps, int n, int B,
                            double th[kIPT]) {
    const int tid = threadIdx.x;
    const int i0 = tid * kIPT;
    double a[kIPT];
    double sum = 0.0;
#pragma unroll
    for (int j = 0; j < kIPT; ++j) {
        a[j] = (i0 + j < n) ? (double)expf(ls[S.val[0][i0 + j]]) : 0.0;
        sum += a[j];
    }
    double total;
    double run = (double)B + block_exscan_double(sum, S.dscan, total);
#pragma unroll
    for (int j = 0; j < kIPT; ++j) {
        run += a[j];
        th[j] = (i0 + j < n) ? run * (double)sps[B + i0 + j] : -INFINITY;   // Theta(i0 + j + 1)
    }
}

__global__ void __launch_bounds__(kST) schedule_kernel(const SchedParams p) {
    grid_dependency_wait();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SchedSmem& S = *reinterpret_cast<SchedSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int B = p.B, gamma = p.gamma, n = B * gamma;
    const double theta0 = (double)B * (double)p.sps[B - 1];

    if (p.mode == DSPARK_SCHED_OFF) {       // every request verifies its whole block
        for (int b = tid; b < B; b += kST) p.K[b] = gamma;
        if (tid == 0) { *p.n_total = n; *p.theta = 0.f; }
        return;
    }
    int admit = 0;
    if (p.mode == DSPARK_SCHED_ASYNC) {
        const float* src = p.log_surv_hist ? p.log_surv_hist : p.log_surv;
        sort_candidates(S, src, n);
        double th[kIPT];
        theta_items(S, src, p.sps, n, B, th);
        // first argmax over m = 0..n of Theta_hist(m)
        double bv = (tid == 0) ? theta0 : -INFINITY;
        int bi = 0;
#pragma unroll
        for (int j = 0; j < kIPT; ++j)
            if (th[j] > bv) { bv = th[j]; bi = tid * kIPT + j + 1; }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            const double ov = __shfl_xor_sync(0xffffffffu, bv, m);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, m);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { S.red_d[warp] = bv; S.red_i[warp] = bi; }
        __syncthreads();
        if (tid == 0) {
            double v = S.red_d[0]; int i = S.red_i[0];
            for (int w = 1; w < kST / 32; ++w)
                if (S.red_d[w] > v || (S.red_d[w] == v && S.red_i[w] < i)) { v = S.red_d[w]; i = S.red_i[w]; }
            S.red_i[0] = i;
        }
        __syncthreads();
        admit = S.red_i[0];
        __syncthreads();
    }

    sort_candidates(S, p.log_surv, n);
    double th[kIPT];
    theta_items(S, p.log_surv, p.sps, n, B, th);
    if (p.mode == DSPARK_SCHED_SYNC) {
        // first m in [0, n) with Theta(m+1) <= Theta(m); Theta(m) of item i is
        // th of item i-1, held by the same or the previous thread
        const double prev_last = __shfl_up_sync(0xffffffffu, th[kIPT - 1], 1);
        __syncthreads();
        if (lane == 31) S.red_d[warp] = th[kIPT - 1];
        __syncthreads();
        double before = (tid == 0) ? theta0 : (lane ? prev_last : S.red_d[warp - 1]);
        int stop = n;
#pragma unroll
        for (int j = 0; j < kIPT; ++j) {
            const int m = tid * kIPT + j;   // candidate m+1 raises Theta(m) -> th[j]?
            if (m < n && stop == n && !(th[j] > before)) stop = m;
            before = th[j];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) stop = min(stop, __shfl_xor_sync(0xffffffffu, stop, m));
        __syncthreads();
        if (lane == 0) S.red_i[warp] = stop;
        __syncthreads();
        if (tid == 0) {
            int v = S.red_i[0];
            for (int w = 1; w < kST / 32; ++w) v = min(v, S.red_i[w]);
            S.red_i[0] = v;
        }
        __syncthreads();
        admit = S.red_i[0];
    } else if (p.mode == DSPARK_SCHED_OFF) {
        admit = n;
    }
    __syncthreads();
    // K_b = admitted candidates of request b (a prefix of its block)
    for (int b = tid; b < B; b += kST) S.kcount[b] = 0;
    __syncthreads();
    if (p.mode == DSPARK_SCHED_OFF) {
        for (int b = tid; b < B; b += kST) S.kcount[b] = gamma;
    } else {
        for (int i = tid; i < admit; i += kST) atomicAdd(&S.kcount[S.val[0][i] / gamma], 1);
    }
    __syncthreads();
    for (int b = tid; b < B; b += kST) p.K[b] = S.kcount[b];
    // Theta at the admitted count: Theta(admit) = th of item admit-1 (or theta0)
    if (tid == 0 && (admit == 0 || p.mode == DSPARK_SCHED_OFF)) {
        *p.n_total = admit;
        *p.theta = (p.mode == DSPARK_SCHED_OFF) ? 0.f : (float)theta0;
    }
    if (p.mode != DSPARK_SCHED_OFF && admit > 0) {
        const int owner = (admit - 1) / kIPT;
        if (tid == owner) {
            const int j = (admit - 1) - owner * kIPT;
            double v = th[0];
#pragma unroll
            for (int q = 1; q < kIPT; ++q) if (q == j) v = th[q];
            *p.n_total = admit;
            *p.theta = (float)v;
        }
    }
}

}  // namespace

cudaError_t launch_confidence(const ConfParams& p, cudaStream_t s) {
    const dim3 grid(p.gamma, p.B);
    const cudaError_t e = p.emb_bf16 ? launch_dependent(confidence_kernel<uint16_t>, grid, dim3(kConfThreads), 0, s, p)
                                     : launch_dependent(confidence_kernel<float>, grid, dim3(kConfThreads), 0, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_schedule(const SchedParams& p, cudaStream_t s) {
    const size_t smem = sizeof(SchedSmem);
    cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    const cudaError_t e = launch_dependent(schedule_kernel, dim3(1), dim3(kST), smem, s, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
