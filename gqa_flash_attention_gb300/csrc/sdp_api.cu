// C ABI of libsdp.so (declared in include/sdp.h): argument validation, TMA
// tensor-map encoding, the per-device status word, and dispatch to the
// kernel instantiation for (head dim, dtype).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>
#include <unordered_map>

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
// Claim counters of the persistent single-CTA kernel (after each device's status word): one
// per stream, found by the stream's unique id, so that only launches ordered on one stream
// share a counter (each zeroes it in stream order before its kernel). g_claim_mu is held
// across the reset and the launch, so two host threads on one stream cannot interleave them.
std::mutex g_claim_mu;
std::unordered_map<unsigned long long, int> g_claim_slot;

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

// Facts of device `dev` that every launch needs, looked up once per device:
// whether it is an sm_103 part, and its SM count.
int g_sms[kMaxDevices] = {};

int device_info_locked(int dev, int *sms)
{
    if (g_cc_checked[dev] == 0) {
        int major = 0, minor = 0, n = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return cuda_fail(e);
        g_sms[dev] = n;
        g_cc_checked[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    if (g_cc_checked[dev] != 1)
        return SDP_ERR_UNSUPPORTED;
    *sms = g_sms[dev];
    return SDP_OK;
}

int device_info(int dev, int *sms)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    return device_info_locked(dev, sms);
}

// Status word of `dev`, allocated (and zeroed) on first use.
int device_state(int dev, unsigned int **status, cudaStream_t)
{
    if (dev < 0 || dev >= kMaxDevices)
        return SDP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    int sms = 0;
    int rc = device_info_locked(dev, &sms);
    if (rc != SDP_OK)
        return rc;
    if (g_status[dev] == nullptr) {
        // the status word, then the claim counters of the persistent single-CTA kernel
        const size_t bytes = (1 + sdp::CLAIM_SLOTS) * sizeof(unsigned int);
        unsigned int *p = nullptr;
        cudaError_t e = cudaMalloc(&p, bytes);
        if (e == cudaSuccess)
            e = cudaMemset(p, 0, bytes);
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
// The encoder is a driver entry point and needs a current context. A host thread that has
// made no runtime call yet has none (the runtime binds the device's primary context to a
// thread lazily, on its first call that needs it), so on CUDA_ERROR_INVALID_CONTEXT the
// current device's primary context is bound (cudaSetDevice) and the encode retried once.
template <class Encode>
CUresult encode_in_context(Encode &&encode)
{
    CUresult r = encode();
    if (r == CUDA_ERROR_INVALID_CONTEXT) {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess)
            r = encode();
    }
    return r;
}

int encode_map_uncached(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long planes,
                        unsigned box_rows)
{
    EncodeTiledFn enc = encoder();
    if (enc == nullptr)
        return cuda_fail(cudaErrorNotSupported);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(planes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = encode_in_context([&] {
        return enc(map, dtype == SDP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    });
    if (r != CUDA_SUCCESS)
        return cuda_fail(cudaErrorInvalidValue);
    return SDP_OK;
}

// 3-D map over a (token, head, dim) 16-bit tensor [rows, heads, D], in the
// same (column, row, plane) coordinate order as encode_map: plane = head, with
// a row stride of heads * D elements and a plane stride of D.
int encode_map_thd_uncached(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long heads,
                            unsigned box_rows)
{
    EncodeTiledFn enc = encoder();
    if (enc == nullptr)
        return cuda_fail(cudaErrorNotSupported);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(heads) * D * 2, static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    const CUresult r = encode_in_context([&] {
        return enc(map, dtype == SDP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void *>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    });
    if (r != CUDA_SUCCESS)
        return cuda_fail(cudaErrorInvalidValue);
    return SDP_OK;
}

// Encoded maps are a pure function of (address, dtype, D, rows, planes, box
// rows, layout), so repeated calls on the same buffers reuse them instead of
// re-encoding (a few microseconds of host time per map): a small table,
// replaced round robin, under its own lock.
struct MapKey {
    const void *base;
    int dtype, D;
    long long rows, planes;
    unsigned box_rows;
    bool thd;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && dtype == o.dtype && D == o.D && rows == o.rows && planes == o.planes &&
               box_rows == o.box_rows && thd == o.thd;
    }
};
constexpr int kMapCacheSize = 64;
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool valid;
};
std::mutex g_map_mu;
MapEntry g_map_cache[kMapCacheSize] = {};
int g_map_next = 0;

int encode_cached(CUtensorMap *map, const MapKey &key)
{
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (const MapEntry &e : g_map_cache)
            if (e.valid && e.key == key) {
                *map = e.map;
                return SDP_OK;
            }
    }
    const int rc = key.thd ? encode_map_thd_uncached(map, key.base, key.dtype, key.D, key.rows, key.planes, key.box_rows)
                           : encode_map_uncached(map, key.base, key.dtype, key.D, key.rows, key.planes, key.box_rows);
    if (rc != SDP_OK)
        return rc;
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_map_cache[g_map_next] = MapEntry{key, *map, true};
    g_map_next = (g_map_next + 1) % kMapCacheSize;
    return SDP_OK;
}

int encode_map(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long planes,
               unsigned box_rows = 128)
{
    return encode_cached(map, MapKey{base, dtype, D, rows, planes, box_rows, false});
}

int encode_map_thd(CUtensorMap *map, const void *base, int dtype, int D, long long rows, long long heads,
                   unsigned box_rows = 128)
{
    return encode_cached(map, MapKey{base, dtype, D, rows, heads, box_rows, true});
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace {

constexpr int kDebugNoPack = 4;  // host-side test hook: never pack the query heads of a group
// Host-side test hook: variable-length launches cover n_qtiles tiles for every sequence
// instead of the compact list of the tiles that exist.
constexpr int kDebugFullVarlenGrid = 32;
// Sequences per batch up to which variable-length launches use the compact list. Each CTA
// finds its tile by scanning the offsets, 32 sequences per step: one pass (stopping at its
// sequence) without the causal mask; with it, one pass and a binary search over tile
// levels on counts held in registers. These limits keep that under a microsecond or so.
constexpr int kCompactMaxSeqs = 512;
constexpr int kCompactMaxSeqsCausal = sdp::VARLEN_LEVEL_MAX_SEQS;

int validate(const void *q, const void *k, const void *v, const void *o, const float *lse, int B, int Hq, int Hkv,
             int Sq, int Skv, int D, float scale, int dtype)
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
    return SDP_OK;
}

// The launch shape of one call. Without causal masking, the G query heads of
// a KV group are packed into one head of G * Sq rows when Sq is not a
// multiple of the 128-row query tile: Q[b, g*G + hi, i] sits at row
// hi * Sq + i of plane (b, g) of the same buffer, so this is only a different
// view (O and LSE likewise), and every packed row still reads KV plane (b, g).
// It fills the tiles that small Sq (decode: Sq = 1) leaves mostly empty.
struct Shape {
    int Hq, G, Sq;  // after packing
    long long n_qtiles, n_kvtiles, planes_q, planes_kv, units;
    int splits, tiles_per_split;
};

int shape_of(int B, int Hq, int Hkv, int Sq, int Skv, int causal, Shape *sh)
{
    const int G = Hq / Hkv;
    const bool pack = !causal && G > 1 && Sq % 128 != 0 && static_cast<long long>(G) * Sq <= INT32_MAX &&
                      !(g_debug_flags.load() & kDebugNoPack);
    sh->Hq = pack ? Hkv : Hq;
    sh->G = pack ? 1 : G;
    sh->Sq = pack ? G * Sq : Sq;
    sh->n_qtiles = (static_cast<long long>(sh->Sq) + 127) / 128;
    sh->n_kvtiles = (static_cast<long long>(Skv) + 127) / 128;
    sh->planes_q = static_cast<long long>(B) * sh->Hq;
    sh->planes_kv = static_cast<long long>(B) * Hkv;
    sh->units = sh->planes_q * sh->n_qtiles;
    sh->splits = 1;
    sh->tiles_per_split = static_cast<int>(sh->n_kvtiles > INT32_MAX ? INT32_MAX : sh->n_kvtiles);
    if (sh->planes_q > INT32_MAX || sh->planes_kv > INT32_MAX || sh->units > INT32_MAX)
        return SDP_ERR_OVERFLOW;
    return SDP_OK;
}

// Split count for a split-KV call: `requested` (0 = as many as fit the SMs in
// one wave: one CTA per SM, so a second, mostly empty wave would add a whole
// run's time), clamped to [1, KV tiles], then evened out so that every split
// reads the same number of tiles except a shorter last one.
int set_splits(Shape *sh, int requested, int sms)
{
    long long s = requested;
    if (s <= 0)
        s = sh->units >= sms ? 1 : sms / sh->units;
    s = s < 1 ? 1 : (s > sh->n_kvtiles ? sh->n_kvtiles : s);
    const long long tps = (sh->n_kvtiles + s - 1) / s;
    s = (sh->n_kvtiles + tps - 1) / tps;
    if (s * sh->planes_q > INT32_MAX || s * sh->units > INT32_MAX)
        return SDP_ERR_OVERFLOW;
    sh->splits = static_cast<int>(s);
    sh->tiles_per_split = static_cast<int>(tps);
    return SDP_OK;
}

long long align256(long long x) { return (x + 255) & ~255LL; }

// Workspace of a split-KV call: partial O [splits, B*Hq*Sq, D] (I/O dtype),
// then partial LSE [splits, B*Hq*Sq] fp32 at the next 256-byte boundary.
long long workspace_bytes(const Shape &sh, int D)
{
    if (sh.splits <= 1)
        return 0;
    const long long rows = sh.planes_q * sh.Sq;
    return align256(sh.splits * rows * D * 2) + sh.splits * rows * 4;
}

// Claim counter index of stream `st`, or -1 (then no persistent single-CTA launch): the
// stream is capturing (a graph may be replayed on any stream, beside eager launches that
// use the same counter), its id cannot be read, or every counter has a stream. The caller
// holds g_claim_mu.
int claim_slot_locked(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    if (cs != cudaStreamCaptureStatusNone)
        return -1;
    unsigned long long id = 0;
    if (cudaStreamGetId(st, &id) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    const auto it = g_claim_slot.find(id);
    if (it != g_claim_slot.end())
        return it->second;
    if (g_claim_slot.size() >= static_cast<size_t>(sdp::CLAIM_SLOTS))
        return -1;
    const int slot = static_cast<int>(g_claim_slot.size());
    g_claim_slot.emplace(id, slot);
    return slot;
}

// Encode the maps and launch the kernel for `sh`. O / LSE go to `o` / `lse`
// ([splits * planes_q, Sq, D] and [splits * planes_q, Sq] when splits > 1).
int launch(const Shape &sh, const void *q, const void *k, const void *v, void *o, float *lse, int Hkv, int Skv,
           int D, float scale, int dtype, int causal, unsigned int *status, int sms, cudaStream_t st)
{
    sdp::LaunchMaps maps;
    int rc;
    const long long out_planes = sh.planes_q * sh.splits;
    if ((rc = encode_map(&maps.q, q, dtype, D, sh.Sq, sh.planes_q)) != SDP_OK ||
        (rc = encode_map(&maps.k, k, dtype, D, Skv, sh.planes_kv)) != SDP_OK ||
        (rc = encode_map(&maps.k_half, k, dtype, D, Skv, sh.planes_kv, 64)) != SDP_OK ||
        (rc = encode_map(&maps.v, v, dtype, D, Skv, sh.planes_kv)) != SDP_OK ||
        (rc = encode_map(&maps.o, o, dtype, D, sh.Sq, out_planes)) != SDP_OK)
        return rc;
    if (D == 128 && (rc = encode_map(&maps.k32, k, dtype, D, Skv, sh.planes_kv, 32)) != SDP_OK)
        return rc;

    sdp::KernelParams p{};
    p.lse = lse;
    p.status = status;
    p.Hq = sh.Hq;
    p.Hkv = Hkv;
    p.G = sh.G;
    p.Sq = sh.Sq;
    p.Skv = Skv;
    p.n_qtiles = static_cast<int>(sh.n_qtiles);
    p.n_kvtiles = static_cast<int>(sh.n_kvtiles);
    p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // scale * log2(e)
    p.timeout_ns = static_cast<unsigned long long>(g_timeout_ms.load()) * 1000000ull;
    p.debug_flags = g_debug_flags.load();
    p.causal = causal ? 1 : 0;
    p.kv_splits = sh.splits;
    p.tiles_per_split = sh.tiles_per_split;
    p.planes_q = static_cast<int>(sh.planes_q);
    p.o = o;  // [planes, Sq, D]: the persistent kernels write O rows directly
    p.num_sms = sms;

    const int grid = static_cast<int>(sh.units * sh.splits);
    // A claim counter for launches that may run persistent on single CTAs (dense, unsplit,
    // unmasked, more units than SMs), held with the lock until the launch is enqueued.
    std::unique_lock<std::mutex> claim_lk(g_claim_mu, std::defer_lock);
    if (!causal && sh.splits == 1 && grid > sms) {
        claim_lk.lock();
        const int slot = claim_slot_locked(st);
        if (slot >= 0)
            p.claim = status + 1 + slot;
        else
            claim_lk.unlock();
    }
    cudaError_t e;
    if (D == 128)
        e = dtype == SDP_BF16 ? sdp::launch_d128_bf16(maps, p, grid, st) : sdp::launch_d128_fp16(maps, p, grid, st);
    else
        e = dtype == SDP_BF16 ? sdp::launch_d256_bf16(maps, p, grid, st) : sdp::launch_d256_fp16(maps, p, grid, st);
    return e == cudaSuccess ? SDP_OK : cuda_fail(e);
}

int forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
            int Skv, int D, float scale, int dtype, int causal, void *stream)
{
    return sdp::forward_with(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, causal, device_state, stream);
}

// Shape of a split-KV call on the current device (validation of the sizes only).
int splitkv_shape(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype, int n_splits, Shape *sh, int *dev)
{
    if (dtype != SDP_FP16 && dtype != SDP_BF16)
        return SDP_ERR_UNSUPPORTED;
    if (D != 128 && D != 256)
        return SDP_ERR_UNSUPPORTED;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || Hq % Hkv != 0 || n_splits < 0)
        return SDP_ERR_INVALID_ARG;
    int rc = shape_of(B, Hq, Hkv, Sq, Skv, 0, sh);
    if (rc != SDP_OK)
        return rc;
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    int sms = 0;
    if ((rc = device_info(*dev, &sms)) != SDP_OK)
        return rc;
    return set_splits(sh, n_splits, sms);
}

}  // namespace

namespace sdp {

int forward_with(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                 int Skv, int D, float scale, int dtype, int causal, StatusSource status_of, void *stream)
{
    // validation: no CUDA call happens before all of it passes
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype);
    if (rc != SDP_OK)
        return rc;
    Shape sh;
    if ((rc = shape_of(B, Hq, Hkv, Sq, Skv, causal, &sh)) != SDP_OK)
        return rc;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    int sms = 0;
    if ((rc = device_info(dev, &sms)) != SDP_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int *status = nullptr;
    if ((rc = status_of(dev, &status, st)) != SDP_OK)
        return rc;
    return launch(sh, q, k, v, o, lse, Hkv, Skv, D, scale, dtype, causal, status, sms, st);
}

int status_code_of(unsigned int word)
{
    g_last_detail.store(word);
    return (word & 0xffu) == 7u ? SDP_ERR_BAD_SEQLENS : SDP_ERR_DEVICE_TIMEOUT;
}

}  // namespace sdp

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

int sdp_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, const int *cu_seqlens_q,
                   const int *cu_seqlens_k, int nseq, int Hq, int Hkv, int total_q, int total_k, int max_seqlen_q,
                   int D, float scale, int dtype, int causal, void *stream)
{
    if (dtype != SDP_FP16 && dtype != SDP_BF16)
        return SDP_ERR_UNSUPPORTED;
    if (D != 128 && D != 256)
        return SDP_ERR_UNSUPPORTED;
    if (nseq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0)
        return SDP_ERR_INVALID_ARG;
    if (total_q == 0)
        return SDP_OK;  // no query rows (empty tensors may have null pointers): nothing to compute
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || cu_seqlens_q == nullptr ||
        cu_seqlens_k == nullptr || max_seqlen_q == 0)
        return SDP_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || o == q || o == k || o == v)
        return SDP_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
        return SDP_ERR_ALIGNMENT;
    const long long n_qtiles = (static_cast<long long>(max_seqlen_q) + 127) / 128;
    const long long n_kvtiles = (static_cast<long long>(total_k) + 127) / 128;
    const long long units = static_cast<long long>(nseq) * Hq * n_qtiles;
    if (units > INT32_MAX)
        return SDP_ERR_OVERFLOW;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    int sms = 0;
    int rc = device_info(dev, &sms);
    if (rc != SDP_OK)
        return rc;
    unsigned int *status = nullptr;
    if ((rc = device_state(dev, &status, static_cast<cudaStream_t>(stream))) != SDP_OK)
        return rc;
    // A batch without keys still gets valid maps (one row); no load is issued then.
    const long long kv_rows = total_k > 0 ? total_k : 1;
    sdp::LaunchMaps maps;
    if ((rc = encode_map_thd(&maps.q, q, dtype, D, total_q, Hq)) != SDP_OK ||
        (rc = encode_map_thd(&maps.k, k, dtype, D, kv_rows, Hkv)) != SDP_OK ||
        (rc = encode_map_thd(&maps.k_half, k, dtype, D, kv_rows, Hkv, 64)) != SDP_OK ||
        (rc = encode_map_thd(&maps.v, v, dtype, D, kv_rows, Hkv)) != SDP_OK ||
        (rc = encode_map_thd(&maps.o, o, dtype, D, total_q, Hq)) != SDP_OK)
        return rc;

    sdp::KernelParams p{};
    p.lse = lse;
    p.status = status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Sq = total_q;
    p.Skv = total_k;
    p.n_qtiles = static_cast<int>(n_qtiles);
    p.n_kvtiles = static_cast<int>(n_kvtiles);
    p.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // scale * log2(e)
    p.timeout_ns = static_cast<unsigned long long>(g_timeout_ms.load()) * 1000000ull;
    p.debug_flags = g_debug_flags.load();
    p.causal = causal ? 1 : 0;
    p.kv_splits = 1;
    p.tiles_per_split = static_cast<int>(n_kvtiles > 0 ? n_kvtiles : 1);
    p.planes_q = Hq;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.o = o;
    p.o_row_stride = static_cast<long long>(Hq) * D;
    p.num_sms = sms;
    // Valid sequences hold at most total_q rows in all, so the tiles that exist number at
    // most (total_q + 127 * nseq) / 128: the compact grid has that many slots per head.
    p.nseq = nseq;
    const long long slots = std::min(static_cast<long long>(nseq) * n_qtiles,
                                     (static_cast<long long>(total_q) + 127LL * nseq) / 128);
    const bool compact = nseq <= (causal ? kCompactMaxSeqsCausal : kCompactMaxSeqs) &&
                         !(p.debug_flags & kDebugFullVarlenGrid);
    p.n_tiles = compact ? static_cast<int>(slots) : 0;

    const int grid = static_cast<int>(compact ? slots * Hq : units);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (D == 128)
        e = dtype == SDP_BF16 ? sdp::launch_d128_bf16(maps, p, grid, st) : sdp::launch_d128_fp16(maps, p, grid, st);
    else
        e = dtype == SDP_BF16 ? sdp::launch_d256_bf16(maps, p, grid, st) : sdp::launch_d256_fp16(maps, p, grid, st);
    return e == cudaSuccess ? SDP_OK : cuda_fail(e);
}

long long sdp_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype, int n_splits)
{
    Shape sh;
    int dev = 0;
    const int rc = splitkv_shape(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits, &sh, &dev);
    return rc != SDP_OK ? rc : workspace_bytes(sh, D);
}

int sdp_fwd_splitkv_count(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype, int n_splits)
{
    Shape sh;
    int dev = 0;
    const int rc = splitkv_shape(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits, &sh, &dev);
    return rc != SDP_OK ? rc : sh.splits;
}

int sdp_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                    int Skv, int D, float scale, int dtype, int n_splits, void *workspace,
                    unsigned long long workspace_bytes_given, void *stream)
{
    int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype);
    if (rc != SDP_OK)
        return rc;
    if (n_splits < 0)
        return SDP_ERR_INVALID_ARG;
    Shape sh;
    int dev = 0;
    if ((rc = splitkv_shape(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits, &sh, &dev)) != SDP_OK)
        return rc;
    const long long need = workspace_bytes(sh, D);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes_given < static_cast<unsigned long long>(need))
            return SDP_ERR_INVALID_ARG;
        if (!aligned(workspace, 16))
            return SDP_ERR_ALIGNMENT;
        const char *w0 = static_cast<const char *>(workspace);
        const char *w1 = w0 + need;
        for (const void *x : {q, k, v, static_cast<const void *>(o)})
            if (static_cast<const char *>(x) >= w0 && static_cast<const char *>(x) < w1)
                return SDP_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int *status = nullptr;
    if ((rc = device_state(dev, &status, st)) != SDP_OK)
        return rc;
    int sms = 0;
    if ((rc = device_info(dev, &sms)) != SDP_OK)
        return rc;
    if (sh.splits == 1)
        return launch(sh, q, k, v, o, lse, Hkv, Skv, D, scale, dtype, 0, status, sms, st);
    const long long rows = sh.planes_q * sh.Sq;
    char *ws_o = static_cast<char *>(workspace);
    float *ws_lse = reinterpret_cast<float *>(ws_o + align256(sh.splits * rows * D * 2));
    if ((rc = launch(sh, q, k, v, ws_o, ws_lse, Hkv, Skv, D, scale, dtype, 0, status, sms, st)) != SDP_OK)
        return rc;
    return sdp_merge(ws_o, ws_lse, sh.splits, rows, D, dtype, o, lse, stream);
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
    if ((e = cudaMemset(status, 0, sizeof(unsigned int))) != cudaSuccess)
        return cuda_fail(e);
    if ((e = cudaDeviceSynchronize()) != cudaSuccess)
        return cuda_fail(e);
    return sdp::status_code_of(word);
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
    case SDP_ERR_BAD_SEQLENS:
        return "variable-length batch: sequence offsets out of range, decreasing, or longer than max_seqlen_q; "
               "those sequences were not written";
    default:
        return "unknown status code";
    }
}

int sdp_version(void) { return 107; }

void sdp_shutdown(void)
{
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        for (MapEntry &e : g_map_cache)
            e.valid = false;
    }
    sdp::noalloc_forget();
    {
        std::lock_guard<std::mutex> lk(g_claim_mu);
        g_claim_slot.clear();
    }
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
