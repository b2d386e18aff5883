// rnn.cu -- the RNN draft head ("DSpark：半自回归生成与置信度调度的投机解码",
// section RNN Head：长程依赖; "DeepSeek-AI与北京大学联手破局", section 三).
//
// The RNN head replaces the Markov head's row W1[x~_{k-1}] by a recurrent
// state that has seen every token of the block so far:
//     s_k = GRU(s_{k-1}, E[x~_{k-1}]),  s_0 learned,  x~_0 the anchor,
//     B_k = bf16(s_k) . W2,
// with the standard GRU cell (gate rows stacked r, z, n):
//     r  = sigma(W_ir x + b_ir + W_hr h + b_hr)
//     z  = sigma(W_iz x + b_iz + W_hz h + b_hz)
//     n  = tanh(W_in x + b_in + r * (W_hn h + b_hn))
//     h' = (1 - z) * n + z * h.
// The draft rows kernel stages its A operands from state[k-1] instead of W1
// rows.  In the cooperative draft launch the kernel runs every GRU step
// itself: the first in its prologue, the others at its position boundaries
// (each CTA a slice of the hidden units, then a grid barrier).  Without
// cooperative launch, each position is a gru_kernel launch (below) followed
// by a single-position draft launch.
//
// gru_kernel: the two [B x r] x [r x 3r] products per position are small
// (6 B r^2 multiply-adds, 25 M at B = 64, r = 256) and latency-bound, so they
// run on the CUDA cores.  A CTA takes 32 hidden units (one per lane) for 8
// requests (one per warp).  The K dimension goes in chunks of 64: the 6 weight
// rows of the CTA's units (W_ih and W_hh, three gates each) are staged in
// shared memory with a one-word pad per row, so lane j reading its row meets
// no bank conflict, and the chunk of x = E[x~] and h of each request is
// staged as fp32 and read as a broadcast.
#include <cuda_runtime.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kUnits = 32;     // hidden units per CTA (one per lane)
constexpr int kReqs = 8;       // requests per CTA (one per warp)
constexpr int kKc = 64;        // K chunk
constexpr int kRowWords = kKc / 2 + 1;   // a staged weight row: 32 bf16 pairs and one pad word

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kReqs * 32)
gru_kernel(const GruParams g, const int k) {
    __shared__ uint32_t Ws[6][kUnits][kRowWords];   // gate rows of W_ih (0..2) and W_hh (3..5)
    __shared__ float xs[kReqs][kKc];
    __shared__ float hs[kReqs][kKc];
    __shared__ int s_x[kReqs];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = g.r, B = g.B;
    const int j0 = blockIdx.x * kUnits;
    const int b0 = blockIdx.y * kReqs;
    const int j = j0 + lane, b = b0 + warp;
    const float* hprev = (k == 1) ? nullptr : g.state + (size_t)(k - 2) * B * r;

    if (threadIdx.x < kReqs) {
        const int bb = b0 + threadIdx.x;
        int x = -1;
        if (bb < B) {
            x = (k == 1) ? g.anchor[bb] : g.draft_tok[(size_t)bb * g.gamma + (k - 2)];
            if (x < 0 || x >= g.V) { raise_status(g.status, kBadToken); x = -1; }   // zero input row
        }
        s_x[threadIdx.x] = x;
    }

    float acc[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int kc = 0; kc < r; kc += kKc) {
        __syncthreads();   // s_x ready / the previous chunk fully read
        // weight rows: 6 gates x 32 units x 32 words, 16-byte loads
        for (int i = threadIdx.x; i < 6 * kUnits * (kKc / 8); i += blockDim.x) {
            const int seg = i % (kKc / 8), row = i / (kKc / 8), gate = row / kUnits, u = row % kUnits;
            const uint16_t* Wm = gate < 3 ? g.W_ih : g.W_hh;
            const int grow = (gate % 3) * r + j0 + u;
            const uint4 w = *reinterpret_cast<const uint4*>(Wm + (size_t)grow * r + kc + 8 * seg);
            uint32_t* dst = &Ws[gate][u][4 * seg];
            dst[0] = w.x; dst[1] = w.y; dst[2] = w.z; dst[3] = w.w;
        }
        // x and h chunks of the CTA's requests
        for (int i = threadIdx.x; i < kReqs * kKc; i += blockDim.x) {
            const int q = i / kKc, c = i % kKc, bb = b0 + q;
            float xv = 0.f, hv = 0.f;
            if (bb < B) {
                const int x = s_x[q];
                if (x >= 0) xv = __uint_as_float((uint32_t)g.E[(size_t)x * r + kc + c] << 16);
                hv = hprev ? hprev[(size_t)bb * r + kc + c] : g.s0[kc + c];
            }
            xs[q][c] = xv;
            hs[q][c] = hv;
        }
        __syncthreads();
#pragma unroll 4
        for (int c2 = 0; c2 < kKc / 2; ++c2) {
            const float x0 = xs[warp][2 * c2], x1 = xs[warp][2 * c2 + 1];
            const float h0 = hs[warp][2 * c2], h1 = hs[warp][2 * c2 + 1];
#pragma unroll
            for (int gt = 0; gt < 3; ++gt) {
                const uint32_t wi = Ws[gt][lane][c2], wh = Ws[3 + gt][lane][c2];
                acc[gt] = fmaf(bf16_lo(wi), x0, fmaf(bf16_hi(wi), x1, acc[gt]));
                acc[3 + gt] = fmaf(bf16_lo(wh), h0, fmaf(bf16_hi(wh), h1, acc[3 + gt]));
            }
        }
    }
    if (b >= B || j >= r) return;
    const float gi_r = acc[0] + g.b_ih[j], gi_z = acc[1] + g.b_ih[r + j], gi_n = acc[2] + g.b_ih[2 * r + j];
    const float gh_r = acc[3] + g.b_hh[j], gh_z = acc[4] + g.b_hh[r + j], gh_n = acc[5] + g.b_hh[2 * r + j];
    const float rg = 1.f / (1.f + expf(-(gi_r + gh_r)));
    const float zg = 1.f / (1.f + expf(-(gi_z + gh_z)));
    const float ng = tanhf(gi_n + rg * gh_n);
    const float hj = hprev ? hprev[(size_t)b * r + j] : g.s0[j];
    g.state[((size_t)(k - 1) * B + b) * r + j] = (1.f - zg) * ng + zg * hj;
}

}  // namespace

cudaError_t launch_gru(const GruParams& g, int k, cudaStream_t s) {
    const dim3 grid((unsigned)((g.r + kUnits - 1) / kUnits), (unsigned)((g.B + kReqs - 1) / kReqs));
    gru_kernel<<<grid, kReqs * 32, 0, s>>>(g, k);
    return cudaGetLastError();
}

// The draft loop with the RNN head: one cooperative draft launch that runs
// the GRU steps itself; without cooperative launch, a GRU launch and a
// single-position draft launch per position.
cudaError_t launch_draft_rnn(const DraftParams& p, const GruParams& g, cudaStream_t s) {
    if (p.gamma > 1 && cooperative_supported() && !getenv("DSPARK_DRAFT_PER_POSITION"))
        return launch_draft_rows_rnn(p, g, 1, p.gamma, s);
    for (int k = 1; k <= p.gamma; ++k) {
        cudaError_t e = launch_gru(g, k, s);
        if (e != cudaSuccess) return e;
        e = launch_draft_rows(p, k, k, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
