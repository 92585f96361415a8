// Instantiation of the attention forward kernel: head dim 128, bf16 I/O.
#include "sdp_fwd_kernel.cuh"
#include "sdp_launch.h"

namespace sdp {

cudaError_t launch_d128_bf16(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &o,
                             const KernelParams &p, int grid, cudaStream_t stream)
{
    return launch_sdp_fwd<128, true>(q, k, v, o, p, grid, stream);
}

}  // namespace sdp
