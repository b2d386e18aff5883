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
// The input x is an embedding row, so its projection W_ih x + b_ih depends on
// the token alone: rnn_input_table_kernel (below) computes it once for every
// token, P[v] = W_ih E[v] + b_ih ([V][3r] fp32), and a GRU step then gathers
// three entries of P where it would take three dot products.
//
// The draft rows kernel stages its A operands from state[k-1] instead of W1
// rows.  In the cooperative draft launch the kernel runs every GRU step
// itself: the first in its prologue, the others at its position boundaries
// (each CTA a slice of the hidden units, then a grid barrier).  Without
// cooperative launch, each position is a gru_kernel launch (below) followed
// by a single-position draft launch.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// P[v][j] = sum_i E[v][i] W_ih[j][i] + b_ih[j] for v < V, j < 3r: a
// [V x r] x [r x 3r] product, run once per set of weights (30 GFLOP at
// V = 151936, r = 256).  Tiles of 64 tokens x 64 outputs, K in chunks of 32
// staged in shared memory as fp32 (rows padded by one word), 16 x 16 threads
// with 4 x 4 outputs each.
constexpr int kTT = 64, kTK = 32;

__global__ void __launch_bounds__(256)
rnn_input_table_kernel(const uint16_t* __restrict__ E, const uint16_t* __restrict__ W_ih,
                       const float* __restrict__ b_ih, int V, int r, float* __restrict__ P) {
    __shared__ float Es[kTT][kTK + 1];
    __shared__ float Ws[kTT][kTK + 1];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int v0 = blockIdx.y * kTT, j0 = blockIdx.x * kTT, J = 3 * r;
    float acc[4][4] = {};
    for (int kc = 0; kc < r; kc += kTK) {
        __syncthreads();
        for (int i = threadIdx.x; i < kTT * kTK; i += 256) {
            const int row = i / kTK, c = i % kTK;
            const int v = v0 + row, j = j0 + row;
            Es[row][c] = v < V ? __uint_as_float((uint32_t)E[(size_t)v * r + kc + c] << 16) : 0.f;
            Ws[row][c] = j < J ? __uint_as_float((uint32_t)W_ih[(size_t)j * r + kc + c] << 16) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < kTK; ++c) {
            float e[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { e[i] = Es[ty + 16 * i][c]; w[i] = Ws[tx + 16 * i][c]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][q] = fmaf(e[i], w[q], acc[i][q]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int v = v0 + ty + 16 * i;
        if (v >= V) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = j0 + tx + 16 * q;
            if (j < J) P[(size_t)v * J + j] = acc[i][q] + b_ih[j];
        }
    }
}

// One GRU step for every request, the launch form of the step (used without
// cooperative launch): state[k-1] = GRU(h, x~_{k-1}), h = state[k-2] (s0 for
// k = 1).  The hidden side W_hh h is a [B x r] x [r x 3r] product: a CTA
// takes 32 hidden units (one per lane) for 8 requests (one per warp), K in
// chunks of 64 with the three W_hh rows of each unit staged in shared memory
// (one pad word per row, so lane j reading its row meets no bank conflict)
// and the chunk of each request's h staged as fp32 and read as a broadcast.
// The input side is three entries of P.
constexpr int kUnits = 32;     // hidden units per CTA (one per lane)
constexpr int kReqs = 8;       // requests per CTA (one per warp)
constexpr int kKc = 64;        // K chunk
constexpr int kRowWords = kKc / 2 + 1;   // a staged weight row: 32 bf16 pairs and one pad word

__global__ void __launch_bounds__(kReqs * 32)
gru_kernel(const GruParams g, const int k) {
    __shared__ uint32_t Ws[3][kUnits][kRowWords];
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
            if (x < 0 || x >= g.V) { raise_status(g.status, kBadToken); x = -1; }   // no input projection
        }
        s_x[threadIdx.x] = x;
    }

    float acc[3] = {0.f, 0.f, 0.f};
    for (int kc = 0; kc < r; kc += kKc) {
        __syncthreads();   // s_x ready / the previous chunk fully read
        for (int i = threadIdx.x; i < 3 * kUnits * (kKc / 8); i += blockDim.x) {
            const int seg = i % (kKc / 8), row = i / (kKc / 8), gate = row / kUnits, u = row % kUnits;
            const uint4 w = *reinterpret_cast<const uint4*>(g.W_hh + (size_t)(gate * r + j0 + u) * r + kc + 8 * seg);
            uint32_t* dst = &Ws[gate][u][4 * seg];
            dst[0] = w.x; dst[1] = w.y; dst[2] = w.z; dst[3] = w.w;
        }
        for (int i = threadIdx.x; i < kReqs * kKc; i += blockDim.x) {
            const int q = i / kKc, c = i % kKc, bb = b0 + q;
            float hv = 0.f;
            if (bb < B) hv = hprev ? hprev[(size_t)bb * r + kc + c] : g.s0[kc + c];
            hs[q][c] = hv;
        }
        __syncthreads();
#pragma unroll 4
        for (int c2 = 0; c2 < kKc / 2; ++c2) {
            const float h0 = hs[warp][2 * c2], h1 = hs[warp][2 * c2 + 1];
#pragma unroll
            for (int gt = 0; gt < 3; ++gt) {
                const uint32_t wh = Ws[gt][lane][c2];
                acc[gt] = fmaf(bf16_lo(wh), h0, fmaf(bf16_hi(wh), h1, acc[gt]));
            }
        }
    }
    if (b >= B || j >= r) return;
    const int x = s_x[warp];
    float gi[3] = {0.f, 0.f, 0.f};
    if (x >= 0) {
        const float* Pr = g.P + (size_t)x * 3 * r;
        gi[0] = Pr[j]; gi[1] = Pr[r + j]; gi[2] = Pr[2 * r + j];
    }
    const float rg = 1.f / (1.f + expf(-(gi[0] + acc[0] + g.b_hh[j])));
    const float zg = 1.f / (1.f + expf(-(gi[1] + acc[1] + g.b_hh[r + j])));
    const float ng = tanhf(gi[2] + rg * (acc[2] + g.b_hh[2 * r + j]));
    const float hj = hprev ? hprev[(size_t)b * r + j] : g.s0[j];
    g.state[((size_t)(k - 1) * B + b) * r + j] = (1.f - zg) * ng + zg * hj;
}

}  // namespace

cudaError_t launch_rnn_input_table(const uint16_t* E, const uint16_t* W_ih, const float* b_ih, int V, int r,
                                   float* P, cudaStream_t s) {
    const dim3 grid((unsigned)((3 * r + kTT - 1) / kTT), (unsigned)((V + kTT - 1) / kTT));
    rnn_input_table_kernel<<<grid, 256, 0, s>>>(E, W_ih, b_ih, V, r, P);
    return cudaGetLastError();
}

cudaError_t launch_gru(const GruParams& g, int k, cudaStream_t s) {
    const dim3 grid((unsigned)((g.r + kUnits - 1) / kUnits), (unsigned)((g.B + kReqs - 1) / kReqs));
    gru_kernel<<<grid, kReqs * 32, 0, s>>>(g, k);
    return cudaGetLastError();
}

// The draft loop with the RNN head: one cooperative draft launch that runs
// the GRU steps itself; without cooperative launch, a GRU launch and a
// single-position draft launch per position.
cudaError_t launch_draft_rnn(const DraftParams& p, const GruParams& g, cudaStream_t s) {
    if (p.gamma > 1 && cooperative_supported()) return launch_draft_rows_rnn(p, g, 1, p.gamma, s);
    for (int k = 1; k <= p.gamma; ++k) {
        cudaError_t e = launch_gru(g, k, s);
        if (e != cudaSuccess) return e;
        e = launch_draft_rows(p, k, k, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dspark
