// TMA + tcgen05/TMEM attention forward (d in {64, 128}).
#include "attn_internal.h"

namespace attn {

cudaError_t launch_tcgen05(const FwdParams &, cudaStream_t, unsigned int *)
{
    return cudaErrorNotSupported;
}

} // namespace attn
