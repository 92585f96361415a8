// Instantiation of the attention forward kernel: head dim 256, fp16 I/O.
#include "sdp_fwd_kernel.cuh"
#include "sdp_launch.h"

namespace sdp {

cudaError_t launch_d256_fp16(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &o,
                             const KernelParams &p, int grid, cudaStream_t stream)
{
    return launch_sdp_fwd<256, false>(q, k, v, o, p, grid, stream);
}

}  // namespace sdp
