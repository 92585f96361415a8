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
// The kernel is the same sdp_fwd_kernel; only where its status word lives and
// how it is set up differ. Nothing in this file is used by sdp_fwd.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "sdp.h"
#include "sdp_launch.h"

namespace {

// Scratch shared by every sdp_fwd_noalloc call in the process. Word 0 is the
// kernel's status word; the rest is headroom up to the stated maximum.
constexpr unsigned kScratchWords = SDP_NOALLOC_SCRATCH_BYTES / sizeof(unsigned int);
constexpr unsigned kStatusWordsPerCall = 1;
static_assert(kStatusWordsPerCall <= kScratchWords, "scratch array too small for one call");

static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
constexpr unsigned long long kTimeoutNs = 2000ull * 1000000ull;  // 2 s per wait, as sdp_fwd's default

std::mutex g_mu;
unsigned int *g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device
int g_cc_ok[kMaxDevices] = {};                   // 0 unknown, 1 sm_103, -1 other

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device set-up, done by the first call on each device with that device
// current: check the architecture and look up the device address of the
// scratch array (its name in host code is only a stand-in).
int setup_device(int dev, unsigned int **scratch)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SDP_ERR_CUDA;
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_cc_ok[dev] != 1)
        return SDP_ERR_UNSUPPORTED;
    if (g_scratch_ptr[dev] == nullptr) {
        unsigned int *ptr = nullptr;
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return SDP_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return SDP_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *scratch = g_scratch_ptr[dev];
    return SDP_OK;
}

// Same view as sdp_fwd uses: [planes, rows, D], box 64 x 128 x 1, 128-byte swizzle.
int encode(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long planes,
           unsigned box_rows = 128)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = g_encode(map, dtype == SDP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                          3, const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SDP_OK : SDP_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int sdp_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                               int Hkv, int Sq, int Skv, int D, float scale, int dtype, void *stream)
{
    if (dtype != SDP_FP16 && dtype != SDP_BF16)
        return SDP_ERR_UNSUPPORTED;
    if (D != 128 && D != 256)
        return SDP_ERR_UNSUPPORTED;
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr)
        return SDP_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || Hq % Hkv != 0)
        return SDP_ERR_INVALID_ARG;
    if (!std::isfinite(scale))
        return SDP_ERR_INVALID_ARG;
    if (o == q || o == k || o == v)
        return SDP_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
        return SDP_ERR_ALIGNMENT;
    const long long n_qtiles = (static_cast<long long>(Sq) + 127) / 128;
    const long long n_kvtiles = (static_cast<long long>(Skv) + 127) / 128;
    const long long planes_q = static_cast<long long>(B) * Hq;
    const long long planes_kv = static_cast<long long>(B) * Hkv;
    const long long units = planes_q * n_qtiles;
    if (planes_q > INT32_MAX || planes_kv > INT32_MAX || units > INT32_MAX)
        return SDP_ERR_OVERFLOW;
    // Scratch this launch needs: one status word, for any problem size.
    if (kStatusWordsPerCall * sizeof(unsigned int) > SDP_NOALLOC_SCRATCH_BYTES)
        return SDP_ERR_OVERFLOW;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return SDP_ERR_CUDA;
    unsigned int *scratch = nullptr;
    int rc = setup_device(dev, &scratch);
    if (rc != SDP_OK)
        return rc;

    sdp::LaunchMaps maps;
    if (encode(&maps.q, q, dtype, D, Sq, planes_q) != SDP_OK || encode(&maps.k, k, dtype, D, Skv, planes_kv) != SDP_OK ||
        encode(&maps.k_half, k, dtype, D, Skv, planes_kv, 64) != SDP_OK ||
        encode(&maps.v, v, dtype, D, Skv, planes_kv) != SDP_OK || encode(&maps.o, o, dtype, D, Sq, planes_q) != SDP_OK)
        return SDP_ERR_CUDA;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The status word must start at zero; it keeps whatever the previous call left.
    if (cudaMemsetAsync(scratch, 0, kStatusWordsPerCall * sizeof(unsigned int), st) != cudaSuccess)
        return SDP_ERR_CUDA;

    sdp::KernelParams p{};
    p.lse = lse;
    p.status = scratch;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = Sq;
    p.Skv = Skv;
    p.n_qtiles = static_cast<int>(n_qtiles);
    p.n_kvtiles = static_cast<int>(n_kvtiles);
    p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.timeout_ns = kTimeoutNs;
    p.debug_flags = 0;
    p.causal = 0;
    p.kv_splits = 1;
    p.tiles_per_split = static_cast<int>(n_kvtiles);
    p.planes_q = static_cast<int>(planes_q);

    const int grid = static_cast<int>(units);
    cudaError_t e;
    if (D == 128)
        e = dtype == SDP_BF16 ? sdp::launch_d128_bf16(maps, p, grid, st) : sdp::launch_d128_fp16(maps, p, grid, st);
    else
        e = dtype == SDP_BF16 ? sdp::launch_d256_bf16(maps, p, grid, st) : sdp::launch_d256_fp16(maps, p, grid, st);
    return e == cudaSuccess ? SDP_OK : SDP_ERR_CUDA;
}
