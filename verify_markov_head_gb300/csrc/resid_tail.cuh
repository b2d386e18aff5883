// The end of a residual draw (lossless verification, the first rejected
// draft: a token from max(0, p - q), renormalised; all drafts accepted: the
// bonus token from p of the next row), after the tensor-core residual launch
// has folded every CTA's draw into one 64-bit winner key per request.
//
// Sources (cited by page title and section):
//   "DSpark：半自回归生成与置信度调度的投机解码" §形式化定义 (accept with
//     min(1, p/q); on rejection sample from the normalised residual);
//   "DeepSeek-AI与北京大学联手破局" §四 (lossless verification).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dspark {

// The token of a winner key (the low word holds the complemented index).
__device__ __forceinline__ int win_token(unsigned long long key) {
    return (int)(0xFFFFFFFFu - (uint32_t)key);
}

// A request whose residual draw has no winner key at all (the residual
// max(0, p - q) had no mass, which only rounding produces) is marked with this
// final token until the fallback draw below replaces it.
constexpr int32_t kFallbackPending = (int32_t)0x80000000;

// The fallback law p for request bb: the draw from p on row urow of the target
// with the residual's noise (domain 2; for a bonus draw, row gamma with the
// bonus noise, domain 3), by the whole CTA over the row, lowest index on ties;
// lse_p (natural units) normalises the row.  The token goes to *fin.  Kept out
// of line so that its registers do not weigh on the caller.
template <typename TT>
__device__ __noinline__ void resid_fallback_draw(uint64_t seed, uint64_t step, int req_base, int gamma, int V,
                                                 float inv_tau, float lse_p, const void* target, int bb, int urow,
                                                 uint32_t domain, int32_t* fin) {
    __shared__ float s_fkey[32];
    __shared__ int s_fidx[32];
    const int tid = (int)threadIdx.x, lane = tid % 32, warp = tid / 32, nwarps = (int)blockDim.x / 32;
    const float scale2 = inv_tau * 1.4426950408889634f;
    const StreamRK rng(seed, step, domain, (uint32_t)(req_base + bb) * (uint32_t)(gamma + 1) + (uint32_t)urow);
    const TT* trow = static_cast<const TT*>(target) + ((size_t)bb * (gamma + 1) + urow) * V;
    const float lse_p2 = lse_p * 1.4426950408889634f;
    float key = INFINITY;
    int idx = 0x7fffffff;
    for (int qd = tid; qd < V / 4; qd += (int)blockDim.x) {
        const uint4 w = rng.quad((uint32_t)qd);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float pv = fast_exp2(fmaf(to_f32(trow[4 * qd + e]), scale2, -lse_p2));
            const float E = exp2_variate_of(ws[e]) * kLn2;
            if (pv > 0.f && E < key * pv) { key = E / pv; idx = 4 * qd + e; }
        }
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        const float ok = __shfl_xor_sync(0xffffffffu, key, sh);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, sh);
        if (ok < key || (ok == key && oi < idx)) { key = ok; idx = oi; }
    }
    if (lane == 0) { s_fkey[warp] = key; s_fidx[warp] = idx; }
    __syncthreads();
    if (tid == 0) {
        for (int w2 = 1; w2 < nwarps; ++w2)
            if (s_fkey[w2] < key || (s_fkey[w2] == key && s_fidx[w2] < idx)) { key = s_fkey[w2]; idx = s_fidx[w2]; }
        *fin = idx;
    }
    __syncthreads();
}

}  // namespace dspark
