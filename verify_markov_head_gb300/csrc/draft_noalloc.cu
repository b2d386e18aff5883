// draft_noalloc.cu -- the draft loop for callers that cannot allocate device
// memory.
//
// dspark_draft_markov needs a caller-provided workspace.  Some callers have
// no way to obtain one at the point where they draft: code embedded in a host
// framework that owns every device allocation, real-time loops that must not
// take an allocator's locks or its implicit device synchronisation, or
// environments that forbid allocation after start-up.  This entry point runs
// the same draft kernels with their scratch (status word, arrival counters,
// per-CTA partial states) in a fixed array that lives in the library's own
// device data segment.  Every GPU that loads the library holds the array
// until the process exits.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

// Fixed scratch: 8 MiB + 64 KiB covers the draft's status word, counters
// and two buffers of partial states for B * min(1024, ceil(V/128)) <= 262144
// (for example B = 256 with V up to 131072, or B = 64 at any V).
constexpr size_t kStaticScratchBytes = (size_t)8 * 1024 * 1024 + 64 * 1024;
static __device__ __align__(256) unsigned char g_draft_scratch[kStaticScratchBytes];

// The array's device address on each device, looked up once with that
// device current.  In host code the symbol is only a stand-in for the device
// object, so the kernels must be handed this address, never the symbol.
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

cudaError_t scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_draft_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" dspark_status dspark_draft_markov_noalloc(
    const void* U, dspark_dtype U_t, const void* W1, const void* W2, dspark_dtype W_t,
    const int32_t* anchor, int B, int gamma, int V, int r, int req_base, float tau,
    uint64_t seed, uint64_t step, int32_t* draft_tok, float* lse_q, float* z_tok, float* logits_out,
    void* stream) {
    if (B < 1 || B > 1000000 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 8 || (V % 8) != 0 || r < 1 ||
        r > 1024 || !(tau > 0.f) || req_base < 0)
        return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;
    if ((U_t != DSPARK_F32 && U_t != DSPARK_BF16) || (W_t != DSPARK_F32 && W_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    if (!U || !W1 || !W2 || !anchor || !draft_tok || !lse_q || !z_tok) return DSPARK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(U) | reinterpret_cast<uintptr_t>(W1) | reinterpret_cast<uintptr_t>(W2)) & 15)
        return DSPARK_ERR_INVALID;
    // the draft kernels touch the workspace up to the end of their partial states
    const WsLayout L = ws_layout(B, gamma, V);
    if (L.verify_part > kStaticScratchBytes) {
        fprintf(stderr,
                "dspark_draft_markov_noalloc: B=%d, V=%d need %zu bytes of scratch but the fixed array holds %zu; "
                "use dspark_draft_markov with a workspace\n",
                B, V, (size_t)L.verify_part, kStaticScratchBytes);
        return DSPARK_ERR_UNSUPPORTED;
    }
    void* ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) {
        fprintf(stderr, "dspark_draft_markov_noalloc: scratch lookup failed: %s\n", cudaGetErrorString(e));
        return DSPARK_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left.  The status word and
    // the arrival counters must start at zero; the partial states are fully
    // rewritten by every launch.
    e = cudaMemsetAsync(ws, 0, L.draft_part, s);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;

    DraftParams p;
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = W1; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau;
    p.seed = seed; p.step = step;
    p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.logits_out = logits_out;
    p.ws = ws_ptrs(ws, B, gamma, V);
    e = launch_draft(p, s);
    if (e != cudaSuccess) {
        fprintf(stderr, "dspark_draft_markov_noalloc: launch failed: %s\n", cudaGetErrorString(e));
        return DSPARK_ERR_CUDA;
    }
    return DSPARK_OK;
}
