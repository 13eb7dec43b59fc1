// tcgen05 tensor-core kernel for the chunkwise gated delta rule (bf16).
#include "gdn_internal.h"

bool gdn_tc_supported(const GdnArgs &) { return false; }

cudaError_t gdn_launch_tc(const GdnArgs &, cudaStream_t, int *launches)
{
    *launches = 0;
    return cudaErrorNotSupported;
}
