// draft_noalloc.cu -- the draft loop for callers that cannot allocate device
// memory.
//
// dspark_draft_markov needs a caller-provided workspace.  Some callers have
// no way to obtain one at the point where they draft: code embedded in a host
// framework that owns every device allocation, real-time loops that must not
// take an allocator's locks or its implicit device synchronisation, or
// environments that forbid allocation after start-up.  This entry point runs
// the same draft kernels with their scratch (status word, arrival counters,
// grid-barrier counters, winner keys, per-CTA partial states) in a fixed
// array that lives in the library's own device data segment.  Every GPU that
// loads the library holds the array until the process exits.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

// The array covers the draft's workspace prefix (ws_draft_prefix: status
// word, tickets, barrier counters, winner keys, stream counters and the two
// buffers of partial states) for every call with B <= kNoallocMaxB and
// gamma <= DSPARK_MAX_GAMMA, at any V: the partial states per request are
// capped at kMaxParts whatever the vocabulary.  8.5 MiB + 1 KiB.
constexpr int kNoallocMaxB = 256;
constexpr size_t kStaticScratchBytes = ws_draft_prefix(kNoallocMaxB, DSPARK_MAX_GAMMA, kMaxParts).end;
static_assert(kStaticScratchBytes == (size_t)8 * 1024 * 1024 + 512 * 1024 + 1024,
              "fixed scratch size changed: update the limit stated in dspark.h");
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
    // the checks of dspark_draft_markov, workspace aside
    if (!sizes_ok(B, gamma, V, r) || !(tau > 0.f) || req_base < 0) return DSPARK_ERR_INVALID;
    if ((double)(req_base + (double)B) * (gamma + 1) >= 4294967295.0) return DSPARK_ERR_INVALID;
    if ((U_t != DSPARK_F32 && U_t != DSPARK_BF16) || (W_t != DSPARK_F32 && W_t != DSPARK_BF16))
        return DSPARK_ERR_UNSUPPORTED;
    if (!is_device_ptr(U) || !is_device_ptr(W1) || !is_device_ptr(W2) || !is_device_ptr(anchor) ||
        !is_device_ptr(draft_tok) || !is_device_ptr(lse_q) || !is_device_ptr(z_tok))
        return DSPARK_ERR_INVALID;
    if (logits_out && (!is_device_ptr(logits_out) || (reinterpret_cast<uintptr_t>(logits_out) & 15)))
        return DSPARK_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(U) | reinterpret_cast<uintptr_t>(W1) | reinterpret_cast<uintptr_t>(W2)) & 15)
        return DSPARK_ERR_INVALID;
    // the draft kernels touch the workspace up to the end of their partial states
    const size_t need = ws_draft_prefix(B, gamma, ws_layout(B, gamma, V).parts).end;
    if (B > kNoallocMaxB || need > kStaticScratchBytes) {
        fprintf(stderr,
                "dspark_draft_markov_noalloc: B=%d (at most %d), gamma=%d, V=%d need %zu bytes of scratch; the "
                "fixed array holds %zu; use dspark_draft_markov with a workspace\n",
                B, kNoallocMaxB, gamma, V, need, kStaticScratchBytes);
        return DSPARK_ERR_UNSUPPORTED;
    }
    void* ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) {
        fprintf(stderr, "dspark_draft_markov_noalloc: scratch lookup failed: %s\n", cudaGetErrorString(e));
        return DSPARK_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left.  The counters must
    // start at zero; the partial states are fully rewritten by every launch.
    // The status word is left alone: dspark_noalloc_sync_status reads and
    // clears it.
    const WsDraftPrefix P = ws_draft_prefix(B, gamma, ws_layout(B, gamma, V).parts);
    e = cudaMemsetAsync(static_cast<char*>(ws) + P.tickets, 0, P.draft_part - P.tickets, s);
    if (e != cudaSuccess) return launch_status(e);

    DraftParams p;
    p.U = U; p.U_bf16 = (U_t == DSPARK_BF16);
    p.W1 = W1; p.W2 = W2; p.W_bf16 = (W_t == DSPARK_BF16);
    p.anchor = anchor;
    p.B = B; p.gamma = gamma; p.V = V; p.r = r; p.req_base = req_base;
    p.inv_tau = 1.f / tau;
    p.seed = seed; p.step = step;
    p.draft_tok = draft_tok; p.lse_q = lse_q; p.z_tok = z_tok; p.logits_out = logits_out;
    p.ws = ws_ptrs(ws, B, gamma, V);
    return launch_status(launch_draft(p, s));
}

// The status word of the fixed array, as dspark_sync_status reads a
// workspace's: synchronise `stream`, read the word, clear it.
extern "C" dspark_status dspark_noalloc_sync_status(void* stream, uint32_t* bits) {
    void* ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) {
        fprintf(stderr, "dspark_noalloc_sync_status: scratch lookup failed: %s\n", cudaGetErrorString(e));
        return DSPARK_ERR_CUDA;
    }
    return read_status_word(ws, static_cast<cudaStream_t>(stream), bits);
}
