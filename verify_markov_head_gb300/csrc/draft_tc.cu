// draft_tc.cu -- Markov-head draft position on the tcgen05 tensor cores.
#include "common.cuh"
#include "internal.h"

namespace dspark {

bool draft_tc_supported(const DraftParams& p) { (void)p; return false; }

cudaError_t launch_draft_tc(const DraftParams& p, int k, cudaStream_t s) {
    (void)p; (void)k; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace dspark
