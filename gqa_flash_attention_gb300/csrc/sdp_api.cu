// C ABI of libsdp.so (declared in include/sdp.h): argument validation, TMA
// tensor-map encoding, the per-device status word, and dispatch to the
// kernel instantiation for (head dim, dtype).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sdp.h"
#include "sdp_launch.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned kDefaultTimeoutMs = 2000;

std::mutex g_mu;
unsigned int *g_status[kMaxDevices] = {};
int g_cc_checked[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
std::atomic<int> g_last_cuda_error{0};
std::atomic<unsigned> g_timeout_ms{kDefaultTimeoutMs};
std::atomic<int> g_debug_flags{0};
std::atomic<unsigned> g_last_detail{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e)
{
    g_last_cuda_error.store(static_cast<int>(e));
    return SDP_ERR_CUDA;
}

EncodeTiledFn encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

// Status word of `dev`, allocated (and zeroed) on first use.
int device_state(int dev, unsigned int **status)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_checked[dev] == 0) {
        int major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess)
            return cuda_fail(e);
        g_cc_checked[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_cc_checked[dev] != 1)
        return SDP_ERR_UNSUPPORTED;
    if (g_status[dev] == nullptr) {
        unsigned int *p = nullptr;
        cudaError_t e = cudaMalloc(&p, sizeof(unsigned int));
        if (e == cudaSuccess)
            e = cudaMemset(p, 0, sizeof(unsigned int));
        if (e != cudaSuccess) {
            if (p)
                cudaFree(p);
            return cuda_fail(e);
        }
        g_status[dev] = p;
    }
    *status = g_status[dev];
    return SDP_OK;
}

// 3-D map over a [planes, rows, D] 16-bit tensor; box = 64 columns x box_rows rows
// x 1 plane with 128-byte swizzle. Rows past `rows` read as zero and are not written.
int encode_map(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long planes,
               unsigned box_rows = 128)
{
    EncodeTiledFn enc = encoder();
    if (enc == nullptr)
        return cuda_fail(cudaErrorNotSupported);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = enc(map, dtype == SDP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return cuda_fail(cudaErrorInvalidValue);
    return SDP_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace {

int forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
            int Skv, int D, float scale, int dtype, int causal, void *stream)
{
    // ---- validation: no CUDA call happens before all of it passes
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

    // ---- device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    unsigned int *status = nullptr;
    int rc = device_state(dev, &status);
    if (rc != SDP_OK)
        return rc;

    sdp::LaunchMaps maps;
    if ((rc = encode_map(&maps.q, q, dtype, D, Sq, planes_q)) != SDP_OK ||
        (rc = encode_map(&maps.k, k, dtype, D, Skv, planes_kv)) != SDP_OK ||
        (rc = encode_map(&maps.k_half, k, dtype, D, Skv, planes_kv, 64)) != SDP_OK ||
        (rc = encode_map(&maps.v, v, dtype, D, Skv, planes_kv)) != SDP_OK ||
        (rc = encode_map(&maps.o, o, dtype, D, Sq, planes_q)) != SDP_OK)
        return rc;

    sdp::KernelParams p{};
    p.lse = lse;
    p.status = status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = Sq;
    p.Skv = Skv;
    p.n_qtiles = static_cast<int>(n_qtiles);
    p.n_kvtiles = static_cast<int>(n_kvtiles);
    p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // scale * log2(e)
    p.timeout_ns = static_cast<unsigned long long>(g_timeout_ms.load()) * 1000000ull;
    p.debug_flags = g_debug_flags.load();
    p.causal = causal ? 1 : 0;

    const int grid = static_cast<int>(units);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 128)
        e = dtype == SDP_BF16 ? sdp::launch_d128_bf16(maps, p, grid, st) : sdp::launch_d128_fp16(maps, p, grid, st);
    else
        e = dtype == SDP_BF16 ? sdp::launch_d256_bf16(maps, p, grid, st) : sdp::launch_d256_fp16(maps, p, grid, st);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDP_OK;
}

}  // namespace

extern "C" {

int sdp_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
            int Skv, int D, float scale, int dtype, void *stream)
{
    return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, 0, stream);
}

int sdp_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                   int Skv, int D, float scale, int dtype, void *stream)
{
    return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, 1, stream);
}

int sdp_poll_status(void *stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e);
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess)
        return cuda_fail(e);
    unsigned int *status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (dev >= 0 && dev < kMaxDevices)
            status = g_status[dev];
    }
    if (status == nullptr)
        return SDP_OK;
    unsigned int word = 0;
    if ((e = cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e);
    if (word == 0)
        return SDP_OK;
    g_last_detail.store(word);
    if ((e = cudaMemset(status, 0, sizeof(unsigned int))) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaDeviceSynchronize()) != cudaSuccess)
        return cuda_fail(e);
    return SDP_ERR_DEVICE_TIMEOUT;
}

unsigned int sdp_last_status_detail(void) { return g_last_detail.load(); }

unsigned int sdp_set_wait_timeout_ms(unsigned int ms) { return g_timeout_ms.exchange(ms == 0 ? kDefaultTimeoutMs : ms); }

int sdp_set_debug_flags(int flags) { return g_debug_flags.exchange(flags); }

int sdp_last_cuda_error(void) { return g_last_cuda_error.load(); }

const char *sdp_strerror(int code)
{
    switch (code) {
    case SDP_OK:
        return "ok";
    case SDP_ERR_INVALID_ARG:
        return "invalid argument (null pointer, non-positive size, Hq not a multiple of Hkv, non-finite scale, "
               "or o aliasing an input)";
    case SDP_ERR_UNSUPPORTED:
        return "unsupported (head dim must be 128 or 256, dtype fp16 or bf16, device sm_103)";
    case SDP_ERR_ALIGNMENT:
        return "misaligned pointer (q, k, v, o need 16 bytes; lse needs 4)";
    case SDP_ERR_OVERFLOW:
        return "problem too large for 32-bit tile and plane counters";
    case SDP_ERR_CUDA:
        return "CUDA call failed (see sdp_last_cuda_error)";
    case SDP_ERR_DEVICE_TIMEOUT:
        return "a kernel wait timed out; its output tile was not written";
    default:
        return "unknown status code";
    }
}

int sdp_version(void) { return 102; }

void sdp_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (int d = 0; d < kMaxDevices; ++d) {
        if (g_status[d] != nullptr) {
            if (cudaSetDevice(d) == cudaSuccess)
                cudaFree(g_status[d]);
            g_status[d] = nullptr;
        }
    }
    if (have_cur)
        cudaSetDevice(cur);
}

}  // extern "C"
