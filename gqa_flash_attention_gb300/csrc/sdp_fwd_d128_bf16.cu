// Instantiation of the attention forward kernels: head dim 128, bf16 I/O.
#include "sdp_fwd_pair2.cuh"
#include "sdp_fwd_persist.cuh"
#include "sdp_launch.h"

namespace sdp {

cudaError_t launch_d128_bf16(const LaunchMaps &m, const KernelParams &p, int grid, cudaStream_t stream)
{
    if (!(p.debug_flags & DEBUG_PAIR_D128) && use_pair2(p, grid))
        return launch_sdp_fwd_pair2<true>(m.q, m.k32, m.v, m.o, p, stream);
    if (use_pair(p, grid, 128))
        return launch_sdp_fwd_pair<128, true>(m.q, m.k_half, m.v, m.o, p, grid, stream);
    if (use_persist(p, grid))
        return launch_sdp_fwd_persist<128, true>(m.q, m.k, m.v, p, grid, stream);
    return launch_sdp_fwd<128, true>(m.q, m.k, m.v, m.o, p, grid, stream);
}

}  // namespace sdp
