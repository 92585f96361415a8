// Instantiation of the attention forward kernels: head dim 256, fp16 I/O.
#include "sdp_fwd_pair_persist.cuh"
#include "sdp_fwd_persist.cuh"
#include "sdp_launch.h"

namespace sdp {

cudaError_t launch_d256_fp16(const LaunchMaps &m, const KernelParams &p, int grid, cudaStream_t stream)
{
    if (use_pair(p, grid, 256)) {
        if (use_persistent(p, grid))
            return launch_sdp_fwd_pair_persistent<256, false>(m.q, m.k_half, m.v, p, grid, stream);
        return launch_sdp_fwd_pair<256, false>(m.q, m.k_half, m.v, m.o, p, grid, stream);
    }
    if (use_persist(p, grid))
        return launch_sdp_fwd_persist<256, false>(m.q, m.k, m.v, p, grid, stream);
    return launch_sdp_fwd<256, false>(m.q, m.k, m.v, m.o, p, grid, stream);
}

}  // namespace sdp
