// diag.cu -- the random streams as seen by the kernels, for tests and diagnostics.
#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

__global__ void gumbel_stream_kernel(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, int n,
                                     float* g_out, float* u_out) {
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * q >= n) return;
    const uint4 w = Stream(seed, step, domain, row).quad((uint32_t)q);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int v = 4 * q + e;
        if (v < n) {
            if (g_out) g_out[v] = gumbel_of(ws[e]);
            if (u_out) u_out[v] = uniform_of(ws[e]);
        }
    }
}

}  // namespace

cudaError_t launch_gumbel_stream(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row, int n, float* g,
                                 float* u, cudaStream_t s) {
    const int quads = (n + 3) / 4;
    gumbel_stream_kernel<<<(quads + 255) / 256, 256, 0, s>>>(seed, step, domain, row, n, g, u);
    return cudaGetLastError();
}

}  // namespace dspark
