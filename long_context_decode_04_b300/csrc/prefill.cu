// prefill.cu -- fused causal prefill on the tensor cores (tcgen05 / TMEM).
#include "common.cuh"
#include "internal.h"

namespace ta {

cudaError_t launch_prefill_causal(const void *, const void *, const void *, void *, float *, int, int, int, int,
                                  int, float, int32_t *, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace ta
