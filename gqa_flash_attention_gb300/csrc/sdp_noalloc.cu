// sdp_fwd_noalloc: the attention forward for callers that cannot allocate
// device memory.
//
// sdp_fwd allocates a 4-byte status word on each device the first time it
// runs there. Some callers cannot allow that: code that runs inside a memory
// pool or arena that owns every device byte of the process, plugins whose
// host forbids allocations outside its own allocator, and setups where an
// allocation would synchronise the device at a point the caller cannot
// afford. This entry point needs no allocation: the only scratch the kernel
// uses, its status word, lives in the file-scope device array below, which is
// part of the library image (every GPU that loads the library holds these 256
// bytes until the process exits).
//
// The launch is sdp_fwd's own (sdp::forward_with: the same checks, head
// packing, kernel choice, wait limit and debug flags); only where its status
// word lives differs. sdp_fwd_noalloc_status reads that word back.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "sdp.h"
#include "sdp_launch.h"

namespace {

// Scratch shared by every sdp_fwd_noalloc call in the process. Word 0 is the
// kernel's status word, then the claim counters of the persistent single-CTA
// kernel (the same layout as sdp_fwd's per-device status region).
constexpr unsigned kScratchWords = SDP_NOALLOC_SCRATCH_BYTES / sizeof(unsigned int);
constexpr unsigned kStatusWordsPerCall = 1;
static_assert(1 + sdp::CLAIM_SLOTS <= kScratchWords, "scratch array too small for the status region");

static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;

std::mutex g_mu;
unsigned int *g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// Status source of sdp::forward_with for this entry point. The first call on a
// device (with that device current) looks up the device address of the scratch
// array, whose name in host code is only a stand-in; every call then clears the
// status word on `stream`, ahead of its kernel.
int scratch_status(int dev, unsigned int **status, cudaStream_t stream)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SDP_ERR_UNSUPPORTED;
    unsigned int *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_scratch_ptr[dev] == nullptr) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
                return SDP_ERR_CUDA;
            g_scratch_ptr[dev] = static_cast<unsigned int *>(addr);
        }
        ptr = g_scratch_ptr[dev];
    }
    if (cudaMemsetAsync(ptr, 0, kStatusWordsPerCall * sizeof(unsigned int), stream) != cudaSuccess)
        return SDP_ERR_CUDA;
    *status = ptr;
    return SDP_OK;
}

}  // namespace

namespace sdp {

void noalloc_forget()
{
    std::lock_guard<std::mutex> lk(g_mu);
    for (unsigned int *&p : g_scratch_ptr)
        p = nullptr;
}

}  // namespace sdp

extern "C" int sdp_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                               int Hkv, int Sq, int Skv, int D, float scale, int dtype, void *stream)
{
    // A launch needs one status word of the array whatever the problem size.
    if (kStatusWordsPerCall * sizeof(unsigned int) > SDP_NOALLOC_SCRATCH_BYTES)
        return SDP_ERR_OVERFLOW;
    return sdp::forward_with(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, 0, scratch_status, stream);
}

extern "C" int sdp_fwd_noalloc_status(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SDP_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_noalloc_scratch, sizeof(word), 0, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SDP_ERR_CUDA;
    if (word == 0)
        return SDP_OK;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice) != cudaSuccess)
        return SDP_ERR_CUDA;
    return sdp::status_code_of(word);
}
