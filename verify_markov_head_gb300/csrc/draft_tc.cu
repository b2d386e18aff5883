// draft_tc.cu -- Markov-head draft position on the tcgen05 tensor cores.
//
// Per position k ("DSpark：半自回归生成与置信度调度的投机解码" sections 整体架构 and
// Markov Head; "拒绝盲猜与算力空转" section on the low-rank Markov head):
//   bias[b, v] = W1[x~_{k-1}(b)] . W2[:, v]      (rank r, bf16 in, fp32 accumulate)
//   z[b, v]    = (U[b, k-1, v] + bias[b, v]) / tau
//   x~_k       = argmax_v z + G,  lse_q = log sum exp z,  z_tok = z[x~_k]
//
// The contraction runs swap-AB: M = 128 vocabulary entries per tile (the W2
// tile is the A operand, MN-major, loaded by TMA straight from the [r, V]
// row-major W2 with 128-byte swizzle), N = NC requests (the gathered W1 rows,
// K-major, staged once per CTA), K = r.  The fp32 accumulator lives in TMEM
// (two buffers, so the MMA of tile t+1 overlaps the epilogue of tile t) and
// never reaches global memory.
//
// A persistent CTA of 6 warps walks a strided set of vocabulary tiles:
//   warp 0     TMA producer: W2 K-chunks (evict-last, so W2 can stay in L2
//              across the gamma launches) and U row blocks (evict-first)
//   warp 1     TMEM owner and single-thread MMA issuer (tcgen05.mma, commit
//              to mbarriers)
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one vocabulary row
//              per thread), z = (U + bias)/tau written into the staged U tile,
//              then a transposed pass (one request row per thread group,
//              consecutive entries per thread, one Philox call per 4 entries)
//              that folds z + Gumbel into a running Gumbel-max + log-sum-exp
//              state per request.
// Partial states go to the workspace; the last CTA of a request chunk to
// arrive (atomic ticket, no waiting) merges them.  Every mbarrier wait is
// bounded: on expiry the kernel raises the timeout bit of the status word,
// lets its async copies land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace dspark {
namespace {

constexpr int kStages = 4;          // W2 K-chunk ring (16 KB each)
constexpr int kUStages = 4;         // U row-block ring
constexpr int kABytes = 128 * 64 * 2;   // one K-chunk of the A tile: 128 vocab x 64 rank, bf16
constexpr int kThreads = 192;
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz

template <int NC>
struct Cfg {
    static constexpr int SC = NC < 32 ? NC : 32;    // epilogue sub-chunk: requests per pass
    static constexpr int NSUB = NC / SC;
    static constexpr int TPR = 128 / SC;            // epilogue threads per request row
    static constexpr int VPT = 128 / TPR;           // entries per thread per pass
    static constexpr int NQ = VPT / 4;              // float4 quads per thread per pass
    static constexpr int TMEM_COLS = 2 * NC < 32 ? 32 : 2 * NC;
    static constexpr int U_BYTES = SC * 128 * 4;
};

struct Layout {
    uint32_t a, b, u, st, bar, misc, total;
};

__host__ __device__ inline Layout tc_layout(int NC, int SC, int r) {
    Layout L;
    L.a = 0;
    L.b = L.a + kStages * kABytes;
    L.u = L.b + (uint32_t)(r / 64) * (uint32_t)NC * 128u;
    L.st = L.u + (uint32_t)kUStages * (uint32_t)SC * 512u;      // per-thread running states
    L.bar = L.st + 128u * (uint32_t)(NC / SC) * 16u;
    L.misc = L.bar + 8u * (2 * kStages + 2 * kUStages + 5);
    L.misc = (L.misc + 15u) & ~15u;
    L.total = L.misc + 16u + 4u * (uint32_t)NC;
    return L;
}

struct TcArgs {
    CUtensorMap w2map;   // bf16 [r][V], box {64 vocab, 64 rank}, 128-byte swizzle
    CUtensorMap umap;    // fp32 [B][gamma][V], box {128 vocab, 1, SC requests}
    DraftParams p;
};

template <int NC>
__global__ void __launch_bounds__(kThreads, 1)
draft_tc_kernel(const __grid_constant__ TcArgs a, const int k) {
    using C = Cfg<NC>;
    const DraftParams& p = a.p;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const Layout L = tc_layout(NC, C::SC, p.r);
    const int KCH = p.r / 64;

    const uint32_t bar0 = base + L.bar;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kStages + i); };
    auto ufull = [&](int i) { return bar0 + 8u * (2 * kStages + i); };
    auto uempty = [&](int i) { return bar0 + 8u * (2 * kStages + kUStages + i); };
    auto tfull = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kUStages + i); };
    auto tempty = [&](int i) { return bar0 + 8u * (2 * kStages + 2 * kUStages + 2 + i); };
    const uint32_t drain = bar0 + 8u * (2 * kStages + 2 * kUStages + 4);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L.misc);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + L.misc + 4);
    volatile uint32_t* never = reinterpret_cast<volatile uint32_t*>(gbase + L.misc + 8);
    int* s_tok = reinterpret_cast<int*>(gbase + L.misc + 16);

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int chunk = blockIdx.y, b_base = chunk * NC;
    const int nb = min(NC, p.B - b_base);
    const int V = p.V, gamma = p.gamma, r = p.r;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) { ptx::mbar_init(full(i), 1); ptx::mbar_init(empty(i), 1); }
        for (int i = 0; i < kUStages; ++i) { ptx::mbar_init(ufull(i), 1); ptx::mbar_init(uempty(i), 1); }
        for (int i = 0; i < 2; ++i) { ptx::mbar_init(tfull(i), 1); ptx::mbar_init(tempty(i), 128); }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0u;
        *never = 0u;
        ptx::fence_mbar_init();
    }
    if (tid == 32) { ptx::prefetch_tmap(&a.w2map); ptx::prefetch_tmap(&a.umap); }
    if (warp == 1) { ptx::tmem_alloc(base + L.misc, C::TMEM_COLS); ptx::tmem_relinquish(); }
    for (int n = tid; n < NC; n += kThreads) {
        int x = -1;
        if (n < nb) {
            const int b = b_base + n;
            x = (k == 1) ? p.anchor[b] : p.draft_tok[(size_t)b * gamma + (k - 2)];
            if (x < 0 || x >= V) { raise_status(p.ws.status, kBadToken); x = -1; }
        }
        s_tok[n] = x;
    }
    __syncthreads();
    // h = W1[x~_{k-1}] rows -> B operand, K-major, 128-byte swizzle:
    // K-chunk j (64 ranks) is a [NC rows][128 B] block; 16-byte unit u of row n
    // sits at unit u ^ (n mod 8).
    {
        const uint16_t* W1 = static_cast<const uint16_t*>(p.W1);
        const int units = r / 8;
        for (int idx = tid; idx < NC * units; idx += kThreads) {
            const int n = idx / units, u16 = idx - n * units;
            const int j = u16 >> 3, u = u16 & 7;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            const int x = s_tok[n];
            if (x >= 0) val = *reinterpret_cast<const uint4*>(W1 + (size_t)x * r + (size_t)u16 * 8);
            uint8_t* dst = gbase + L.b + (size_t)j * (NC * 128) + (size_t)n * 128 + ((u ^ (n & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = val;
        }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int ntiles = (V + 127) / 128;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = ptx::policy_evict_last(), pol_u = ptx::policy_evict_first();
            int stage = 0, us = 0;
            uint32_t ph = 0, uph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int v0 = t * 128;
                for (int j = 0; j < KCH; ++j) {
                    if (!(ok = ptx::mbar_wait(empty(stage), ph ^ 1u, abort_flag, kWaitCycles))) break;
                    ptx::mbar_arrive_expect_tx(full(stage), kABytes);
                    const uint32_t dst = base + L.a + (uint32_t)stage * kABytes;
                    ptx::tma_load_2d(dst, &a.w2map, v0, j * 64, full(stage), pol_w);
                    ptx::tma_load_2d(dst + kABytes / 2, &a.w2map, v0 + 64, j * 64, full(stage), pol_w);
                    if (++stage == kStages) { stage = 0; ph ^= 1u; }
                }
                for (int c = 0; c < C::NSUB && ok; ++c) {
                    if (!(ok = ptx::mbar_wait(uempty(us), uph ^ 1u, abort_flag, kWaitCycles))) break;
                    ptx::mbar_arrive_expect_tx(ufull(us), C::U_BYTES);
                    ptx::tma_load_3d(base + L.u + (uint32_t)us * C::U_BYTES, &a.umap, v0, k - 1,
                                     b_base + c * C::SC, ufull(us), pol_u);
                    if (++us == kUStages) { us = 0; uph ^= 1u; }
                }
            }
            if (!ok) { raise_status(p.ws.status, kTimeout); *abort_flag = 1u; }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, NC, /*A MN-major*/ true, /*B K-major*/ false);
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                if (!(ok = ptx::mbar_wait(tempty(acc), aph ^ 1u, abort_flag, kWaitCycles))) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NC);
                for (int j = 0; j < KCH; ++j) {
                    if (!(ok = ptx::mbar_wait(full(stage), ph, abort_flag, kWaitCycles))) break;
                    ptx::tc_fence_after();
                    const uint32_t a_addr = base + L.a + (uint32_t)stage * kABytes;
                    const uint32_t b_addr = base + L.b + (uint32_t)j * (NC * 128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // A: MN-major, 64-entry swizzle atoms 8 KB apart along M (LBO),
                        //    8-rank groups 1 KB apart along K (SBO); 16 ranks = 2 KB per step.
                        const uint64_t ad = ptx::smem_desc_sw128(a_addr + kk * 2048, 8192, 1024);
                        // B: K-major rows of 128 B, 8-row groups 1 KB apart (SBO); 16 ranks = 32 B.
                        const uint64_t bd = ptx::smem_desc_sw128(b_addr + kk * 32, 16, 1024);
                        ptx::mma_f16(d_tmem, ad, bd, idesc, (j | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(empty(stage));
                    if (++stage == kStages) { stage = 0; ph ^= 1u; }
                }
                if (!ok) break;
                ptx::mma_commit(tfull(acc));
                if (++acc == 2) { acc = 0; aph ^= 1u; }
            }
            if (!ok) { raise_status(p.ws.status, kTimeout); *abort_flag = 1u; }
            // every MMA issued above completes before TMEM is released
            ptx::mma_commit(drain);
            ptx::mbar_wait(drain, 0u, never, kWaitCycles);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int etid = tid - 64;
        const int q = warp & 3;
        const int v_row = 32 * q + lane;             // TMEM lane = vocabulary row of the tile
        const int b_loc = etid / C::TPR, seg = etid % C::TPR;
        // running state of this thread for sub-chunk c: sst[c * 128 + etid]
        DrawLse* sst = reinterpret_cast<DrawLse*>(gbase + L.st);
        for (int c = 0; c < C::NSUB; ++c) sst[c * 128 + etid] = drawlse_empty();
        int acc = 0, us = 0;
        uint32_t aph = 0, uph = 0;
        bool failed = false;
        for (int t = blockIdx.x; t < ntiles && !failed; t += gridDim.x) {
            const int v0 = t * 128;
            bool ok = ptx::mbar_wait(tfull(acc), aph, abort_flag, kWaitCycles);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) ptx::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < C::NSUB; ++c) {
                float bias[C::SC];
                if (ok) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * NC + c * C::SC);
                    if constexpr (C::SC == 32) ptx::tmem_ld32(taddr, bias);
                    else ptx::tmem_ld16(taddr, bias);
                    ptx::tmem_wait_ld();
                }
                if (c == C::NSUB - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(tempty(acc));
                }
                const bool uok = ok && ptx::mbar_wait(ufull(us), uph, abort_flag, kWaitCycles);
                float* sU = reinterpret_cast<float*>(gbase + L.u + (size_t)us * C::U_BYTES);
                if (uok) {
                    const int v = v0 + v_row;
#pragma unroll
                    for (int j = 0; j < C::SC; ++j) {
                        const float z = (sU[j * 128 + v_row] + bias[j]) * p.inv_tau;
                        sU[j * 128 + v_row] = z;
                        const int b = b_base + c * C::SC + j;
                        if (p.logits_out && b < p.B && v < V)
                            p.logits_out[((size_t)b * gamma + (k - 1)) * V + v] = z;
                    }
                }
                if (ptx::bar_red_or(1, 128, !uok)) { failed = true; break; }
                // transposed pass: request row b_loc, entries seg*VPT .. +VPT
                const int b = b_base + c * C::SC + b_loc;
                if (b < p.B) {
                    const Stream rng(p.seed, p.step, 0u,
                                     (uint32_t)(p.req_base + b) * (uint32_t)(gamma + 1) + (uint32_t)(k - 1));
                    DrawLse s = sst[c * 128 + etid];
#pragma unroll 2
                    for (int qi = 0; qi < C::NQ; ++qi) {
                        const int qq = (C::SC == 32) ? ((qi + lane) & 7) : ((qi + (lane >> 1)) & 3);
                        const int vl = seg * C::VPT + 4 * qq;
                        const int vq = v0 + vl;
                        if (vq < V) {
                            const float4 z4 = *reinterpret_cast<const float4*>(sU + b_loc * 128 + vl);
                            const uint4 w = rng.quad((uint32_t)vq >> 2);
                            const float zs[4] = {z4.x, z4.y, z4.z, z4.w};
                            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float sc = zs[e] + gumbel_of(ws[e]);
                                const int idx = vq + e;
                                if (s.best == -INFINITY) {
                                    s.best = sc; s.idx = idx; s.zb = zs[e]; s.s = __expf(zs[e] - sc);
                                } else if (wins(sc, idx, s.best, s.idx)) {
                                    s.s = s.s * __expf(s.best - sc) + __expf(zs[e] - sc);
                                    s.best = sc; s.idx = idx; s.zb = zs[e];
                                } else {
                                    s.s += __expf(zs[e] - s.best);
                                }
                            }
                        }
                    }
                    sst[c * 128 + etid] = s;
                }
                ptx::fence_proxy_async_smem();   // generic accesses to this U slot precede the next TMA write
                ptx::named_barrier(1, 128);
                if (etid == 0) ptx::mbar_arrive(uempty(us));
                if (++us == kUStages) { us = 0; uph ^= 1u; }
            }
            if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
        if (failed) *abort_flag = 1u;
        // fold the TPR threads of each request row, publish one partial per (request, CTA)
        for (int c = 0; c < C::NSUB; ++c) {
            DrawLse s = sst[c * 128 + etid];
#pragma unroll
            for (int m = 1; m < C::TPR; m <<= 1) s = drawlse_merge(s, shfl_xor(s, m));
            const int b = b_base + c * C::SC + b_loc;
            if (seg == 0 && b < p.B) p.ws.draft_part[(size_t)b * p.ws.parts + blockIdx.x] = s;
        }
    }

    if (*abort_flag) {
        // let any copy still in flight land before the shared memory is released
        for (int i = 0; i < 64; ++i) __nanosleep(1000);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::TMEM_COLS);
    }

    // last-arriving CTA of this request chunk merges the partial states
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
    for (int n = warp; n < nb; n += kThreads / 32) {
        const int b = b_base + n;
        const DrawLse* part = p.ws.draft_part + (size_t)b * p.ws.parts;
        DrawLse acc = drawlse_empty();
        for (int i = lane; i < (int)gridDim.x; i += 32) {
            DrawLse c;
            c.best = __ldcg(&part[i].best); c.idx = __ldcg(&part[i].idx);
            c.zb = __ldcg(&part[i].zb); c.s = __ldcg(&part[i].s);
            acc = drawlse_merge(acc, c);
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) acc = drawlse_merge(acc, shfl_xor(acc, m));
        if (lane == 0) {
            const size_t o = (size_t)b * gamma + (k - 1);
            p.draft_tok[o] = acc.idx;
            p.lse_q[o] = acc.best + logf(acc.s);
            p.z_tok[o] = acc.zb;
        }
    }
    if (tid == 0) p.ws.tickets_draft[chunk] = 0u;
}

int pick_nc(int B, int r) {
    int nc = 16;
    while (nc < B && nc < 256) nc *= 2;
    while ((r / 64) * nc * 128 > 64 * 1024) nc /= 2;    // keep the B operand within 64 KB
    return nc;
}

template <int NC>
cudaError_t launch_nc(const DraftParams& p, int k, cudaStream_t s) {
    using C = Cfg<NC>;
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encoder());
    if (!enc) return cudaErrorNotSupported;
    TcArgs a;
    a.p = p;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)p.V, (cuuint64_t)p.r};
        const cuuint64_t strides[1] = {(cuuint64_t)p.V * 2};
        const cuuint32_t box[2] = {64, 64};
        const cuuint32_t es[2] = {1, 1};
        if (enc(&a.w2map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.W2), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.gamma, (cuuint64_t)p.B};
        const cuuint64_t strides[2] = {(cuuint64_t)p.V * 4, (cuuint64_t)p.gamma * p.V * 4};
        const cuuint32_t box[3] = {128, 1, (cuuint32_t)C::SC};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&a.umap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(p.U), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const Layout L = tc_layout(NC, C::SC, p.r);
    const size_t smem = L.total + 1024;
    // the opt-in limit covers static + dynamic shared memory, so request exactly what this launch needs
    cudaError_t e = cudaFuncSetAttribute(draft_tc_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int nchunks = (p.B + NC - 1) / NC;
    const int ntiles = (p.V + 127) / 128;
    int gx = num_sms() / nchunks;
    gx = gx < 1 ? 1 : gx;
    gx = gx > ntiles ? ntiles : gx;
    gx = gx > p.ws.parts ? p.ws.parts : gx;
    draft_tc_kernel<NC><<<dim3(gx, nchunks), kThreads, smem, s>>>(a, k);
    return cudaGetLastError();
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

bool draft_tc_supported(const DraftParams& p) {
    if (!p.W_bf16 || p.U_bf16) return false;
    if (p.r % 64 != 0 || p.r > 512 || p.V % 8 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(p.W2) & 15) || (reinterpret_cast<uintptr_t>(p.U) & 15)) return false;
    if (tma_encoder() == nullptr) return false;
    if (getenv("DSPARK_DRAFT_SIMT")) return false;
    return true;
}

cudaError_t launch_draft_tc(const DraftParams& p, int k, cudaStream_t s) {
    if (draft_rows_supported(p) && !getenv("DSPARK_DRAFT_VOCAB_LANES")) return launch_draft_rows(p, k, k, s);
    switch (pick_nc(p.B, p.r)) {
        case 16: return launch_nc<16>(p, k, s);
        case 32: return launch_nc<32>(p, k, s);
        case 64: return launch_nc<64>(p, k, s);
        case 128: return launch_nc<128>(p, k, s);
        default: return launch_nc<256>(p, k, s);
    }
}

// All gamma positions of the draft.  The requests-on-lanes tensor-core kernel
// runs them in one cooperative launch when the device supports it; otherwise
// one launch per position.
cudaError_t launch_draft(const DraftParams& p, cudaStream_t s) {
    const bool tc = draft_tc_supported(p);
    if (tc && draft_rows_supported(p) && !getenv("DSPARK_DRAFT_VOCAB_LANES") && p.gamma > 1 &&
        cooperative_supported() && !getenv("DSPARK_DRAFT_PER_POSITION"))
        return launch_draft_rows(p, 1, p.gamma, s);
    for (int k = 1; k <= p.gamma; ++k) {
        const cudaError_t e = tc ? launch_draft_tc(p, k, s) : launch_draft_simt(p, k, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
