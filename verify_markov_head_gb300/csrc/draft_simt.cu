// draft_simt.cu -- Markov-head draft position on CUDA cores (fp32 weights and
// shapes the tensor-core path does not take).
//
// One launch per draft position k.  A CTA owns a chunk of kBC requests and a
// strided set of 128-entry vocabulary tiles:
//   1. gathers h = W1[x~_{k-1}] for its requests into shared memory,
//   2. per tile, forms the bias h . W2[:, v] with fp32 FMAs, adds U_k and
//      scales by 1/tau (the draft logits z, "DSpark：半自回归生成与置信度调度的投机解码"
//      section 整体架构 and section Markov Head),
//   3. transposes the tile through shared memory so each thread walks 8
//      consecutive entries of one request, and folds them into a running
//      Gumbel-max + log-sum-exp state (DrawLse),
//   4. writes one partial state per (request, CTA); the last CTA of the chunk
//      to arrive (atomic ticket, no waiting) merges the partials into
//      x~_k, lse_q and z(x~_k).
#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kTV = 128;       // vocabulary entries per tile
constexpr int kBC = kChunk;    // requests per CTA chunk
constexpr int kThreads = 256;

template <typename WT, typename UT>
__global__ void __launch_bounds__(kThreads)
draft_simt_kernel(const DraftParams p, const int k) {
    extern __shared__ __align__(16) float smem[];
    float* sh = smem;                               // [kBC][r]
    float* tile = smem + kBC * p.r;                 // [kBC][kTV + 4]
    constexpr int kLd = kTV + 4;

    const int tid = threadIdx.x;
    const int chunk = blockIdx.y;
    const int b0 = chunk * kBC;
    const int nb = min(kBC, p.B - b0);
    const int V = p.V, r = p.r, gamma = p.gamma;
    const WT* W1 = static_cast<const WT*>(p.W1);
    const WT* W2 = static_cast<const WT*>(p.W2);
    const UT* U = static_cast<const UT*>(p.U);

    // 1. h rows of the chunk (zero for padding rows and invalid tokens)
    for (int i = tid; i < kBC * r; i += kThreads) {
        const int bl = i / r, rho = i - bl * r;
        float v = 0.f;
        if (bl < nb) {
            const int b = b0 + bl;
            const int x = (k == 1) ? p.anchor[b] : p.draft_tok[(size_t)b * gamma + (k - 2)];
            if (x >= 0 && x < V) v = to_f32(W1[(size_t)x * r + rho]);
            else if (rho == 0) raise_status(p.ws.status, kBadToken);
        }
        sh[i] = v;
    }
    __syncthreads();

    const int v_local = tid % kTV, bh = tid / kTV;        // bias mapping: 8 requests per thread
    const int bl_e = tid / 16, seg = tid % 16;              // epilogue mapping: 8 entries per thread
    const int ntiles = (V + kTV - 1) / kTV;
    // running draw (best, idx, zb) and sum s = sum exp(z - best) of this thread's entries
    DrawLse st = drawlse_empty();
    float ssum = 0.f;
    const uint32_t prow = (uint32_t)(p.req_base + b0 + bl_e) * (uint32_t)(gamma + 1) + (uint32_t)(k - 1);
    const Stream rng(p.seed, p.step, 0u, prow);

    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int v0 = t * kTV;
        const int v = v0 + v_local;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        if (v < V) {
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
            float z = -INFINITY;
            if (bl < nb && v < V) {
                const size_t off = ((size_t)(b0 + bl) * gamma + (k - 1)) * V + v;
                z = (to_f32(U[off]) + acc[j]) * p.inv_tau;
                if (p.logits_out) p.logits_out[off] = z;
            }
            tile[bl * kLd + v_local] = z;
        }
        __syncthreads();
        if (bl_e < nb) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int vl = seg * 8 + q * 4;
                const int vq = v0 + vl;
                if (vq < V) {
                    const uint4 w = rng.quad((uint32_t)vq >> 2);
                    const float4 z4 = *reinterpret_cast<const float4*>(tile + bl_e * kLd + vl);
                    const float zs[4] = {z4.x, z4.y, z4.z, z4.w};
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float sc = zs[e] + gumbel_of(ws[e]);
                        const int idx = vq + e;
                        if (st.best == -INFINITY) {
                            st.best = sc; st.idx = idx; st.zb = zs[e];
                            ssum = __expf(zs[e] - sc);
                        } else if (wins(sc, idx, st.best, st.idx)) {
                            ssum = ssum * __expf(st.best - sc) + __expf(zs[e] - sc);
                            st.best = sc; st.idx = idx; st.zb = zs[e];
                        } else {
                            ssum += __expf(zs[e] - st.best);
                        }
                    }
                }
            }
        }
        __syncthreads();
    }

    st.lse = ssum > 0.f ? st.best + logf(ssum) : -INFINITY;
    // 16 threads share a request: butterfly over lanes xor 1..8
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) st = drawlse_merge(st, shfl_xor(st, m));
    if (seg == 0 && bl_e < nb) p.ws.draft_part[(size_t)(b0 + bl_e) * p.ws.parts + blockIdx.x] = st;

    // 4. last-arriving CTA of this chunk merges the partials
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(&p.ws.tickets_draft[chunk], 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int warp = tid / 32, lane = tid % 32;
    for (int bl = warp; bl < nb; bl += kThreads / 32) {
        const int b = b0 + bl;
        const DrawLse* part = p.ws.draft_part + (size_t)b * p.ws.parts;
        DrawLse a = drawlse_empty();
        for (int i = lane; i < (int)gridDim.x; i += 32) {
            DrawLse c;
            c.best = __ldcg(&part[i].best); c.idx = __ldcg(&part[i].idx);
            c.zb = __ldcg(&part[i].zb); c.lse = __ldcg(&part[i].lse);
            a = drawlse_merge(a, c);
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) a = drawlse_merge(a, shfl_xor(a, m));
        if (lane == 0) {
            const size_t o = (size_t)b * gamma + (k - 1);
            p.draft_tok[o] = a.idx;
            p.lse_q[o] = a.lse;
            p.z_tok[o] = a.zb;
        }
    }
    if (tid == 0) p.ws.tickets_draft[chunk] = 0u;
}

}  // namespace

cudaError_t launch_draft_simt(const DraftParams& p, int k, cudaStream_t s) {
    const int nchunks = (p.B + kBC - 1) / kBC;
    const int ntiles = (p.V + kTV - 1) / kTV;
    int gx = (4 * num_sms()) / nchunks;
    gx = gx < 1 ? 1 : gx;
    gx = gx > ntiles ? ntiles : gx;
    gx = gx > p.ws.parts ? p.ws.parts : gx;
    const dim3 grid(gx, nchunks);
    const size_t smem = sizeof(float) * ((size_t)kBC * p.r + (size_t)kBC * (kTV + 4));
    if (p.W_bf16) {
        auto kern = p.U_bf16 ? draft_simt_kernel<uint16_t, uint16_t> : draft_simt_kernel<uint16_t, float>;
        if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, s>>>(p, k);
    } else {
        auto kern = p.U_bf16 ? draft_simt_kernel<float, uint16_t> : draft_simt_kernel<float, float>;
        if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, s>>>(p, k);
    }
    return cudaGetLastError();
}

}  // namespace dspark
