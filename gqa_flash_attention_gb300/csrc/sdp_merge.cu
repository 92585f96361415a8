// sdp_merge: combine partial attention results computed over disjoint key
// sets into the result over their union -- the state exchange of ring /
// context-parallel attention ("SyclKittens" summary, section I.2: after each
// ring step the partial output and online-softmax state are merged).
//
// For row r and parts p:  LSE = ln sum_p exp(LSE_p),  O = sum_p exp(LSE_p - LSE) O_p.
//
// Memory-bound: one warp per row; lane l owns D/32 consecutive columns and
// reads them from every part with one 8- or 16-byte load, so each part's row
// is one coalesced 256- or 512-byte read. The per-part weights come from a
// warp reduction over the part log-sum-exps. Accumulation is fp32; the output
// is rounded to the I/O type (round to nearest even).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "sdp.h"

namespace {

constexpr int kWarpsPerBlock = 4;

// With up to NP parts (a template bound of 8, 16 or 32; 0 for none) every load
// of a row (the part rows and lane p's part LSE) is issued at once: the split-KV
// merge of a decode step has few rows and is bound by that one round trip (about
// 0.8 us to L2 on this GPU, so a row read in five trips costs four times as
// much). The bound sizes the row's register array, so a caller picks the
// smallest one that holds its P: an HBM-bound merge of many rows then keeps its
// occupancy. Beyond the bound, the part LSEs are read once (lane p holds part
// p's while P <= 32) and the part rows MAX_IN_FLIGHT at a time. The arithmetic
// does not depend on the bound.
constexpr int MAX_IN_FLIGHT = 8;

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u)
{
    if constexpr (BF16) {
        __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
        return __bfloat1622float2(v);
    } else {
        __half2 v = *reinterpret_cast<__half2 *>(&u);
        return __half22float2(v);
    }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

// W 32-bit words (2*W elements) per lane: W = D / 64.
template <int D, bool BF16>
__device__ __forceinline__ void accumulate(float *acc, const uint32_t *words, float w)
{
#pragma unroll
    for (int i = 0; i < D / 64; ++i) {
        const float2 f = unpack2<BF16>(words[i]);
        acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
    }
}

template <int D, bool BF16>
__device__ __forceinline__ void store_row(uint16_t *o, float *lse, long long r, int lane, const float *acc,
                                          float lse_r)
{
    constexpr int W = D / 64;
    using Vec = typename std::conditional<W == 4, uint4, uint2>::type;
    Vec out;
    uint32_t *ow = reinterpret_cast<uint32_t *>(&out);
#pragma unroll
    for (int i = 0; i < W; ++i)
        ow[i] = pack2<BF16>(acc[2 * i], acc[2 * i + 1]);
    reinterpret_cast<Vec *>(o)[r * 32 + lane] = out;
    if (lse != nullptr && lane == 0)
        lse[r] = lse_r;
}

// Row r of P parts ([P, rows, D] 16-bit O and [P, rows] fp32 LSE) into o / lse;
// called by all 32 lanes of a warp.
template <int D, bool BF16, int NP>
__device__ __forceinline__ void merge_row(const uint16_t *__restrict__ o_parts, const float *__restrict__ lse_parts,
                                          int P, long long rows, long long r, int lane, uint16_t *__restrict__ o,
                                          float *__restrict__ lse)
{
    constexpr int W = D / 64;  // 2 (8-byte loads) at D=128, 4 (16-byte loads) at D=256
    using Vec = typename std::conditional<W == 4, uint4, uint2>::type;
    const Vec *src = reinterpret_cast<const Vec *>(o_parts) + r * 32 + lane;
    const long long part_stride = rows * 32;  // in Vec units
    float acc[2 * W];
#pragma unroll
    for (int i = 0; i < 2 * W; ++i)
        acc[i] = 0.f;

    if constexpr (NP > 0) {
        if (P <= NP) {
            Vec v[NP];
#pragma unroll
            for (int u = 0; u < NP; ++u)
                if (u < P)
                    v[u] = __ldg(src + static_cast<long long>(u) * part_stride);
            const float l = lane < P ? __ldg(lse_parts + static_cast<long long>(lane) * rows + r) : -INFINITY;
            float m = l;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            const float e = lane < P ? expf(l - m) : 0.f;
            float sum = e;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, off);
            const float w_l = e / sum;
#pragma unroll
            for (int u = 0; u < NP; ++u) {
                const float w = __shfl_sync(0xffffffffu, w_l, u);
                if (u < P)
                    accumulate<D, BF16>(acc, reinterpret_cast<const uint32_t *>(&v[u]), w);
            }
            store_row<D, BF16>(o, lse, r, lane, acc, m + logf(sum));
            return;
        }
    }

    // Row log-sum-exp over the parts: max, then sum of exp relative to it.
    // The first 32 part LSEs stay in a register (lane p: part p).
    const float l0 = lane < P ? __ldg(lse_parts + static_cast<long long>(lane) * rows + r) : -INFINITY;
    float m = l0;
    for (int p = lane + 32; p < P; p += 32)
        m = fmaxf(m, __ldg(lse_parts + static_cast<long long>(p) * rows + r));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float e0 = lane < P ? expf(l0 - m) : 0.f;
    float sum = e0;
    for (int p = lane + 32; p < P; p += 32)
        sum += expf(__ldg(lse_parts + static_cast<long long>(p) * rows + r) - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lse_r = m + logf(sum);
    const float inv_sum = 1.f / sum;

    for (int p0 = 0; p0 < P; p0 += 32) {
        // weight of part p0 + lane, broadcast below
        const int pl = p0 + lane;
        const float w_l = p0 == 0 ? e0 * inv_sum
                                  : (pl < P ? expf(__ldg(lse_parts + static_cast<long long>(pl) * rows + r) - lse_r)
                                            : 0.f);
        const int pend = min(32, P - p0);
        for (int q = 0; q < pend; q += MAX_IN_FLIGHT) {
            Vec v[MAX_IN_FLIGHT];
#pragma unroll
            for (int u = 0; u < MAX_IN_FLIGHT; ++u)
                if (q + u < pend)
                    v[u] = __ldg(src + static_cast<long long>(p0 + q + u) * part_stride);
#pragma unroll
            for (int u = 0; u < MAX_IN_FLIGHT; ++u) {
                const float w = __shfl_sync(0xffffffffu, w_l, (q + u) & 31);
                if (q + u < pend)
                    accumulate<D, BF16>(acc, reinterpret_cast<const uint32_t *>(&v[u]), w);
            }
        }
    }
    store_row<D, BF16>(o, lse, r, lane, acc, lse_r);
}

// One instantiation per all-in-flight bound NP (8, 16, 32; 0: none), so that each
// has the registers (and occupancy) of its own row array.
template <int D, bool BF16, int NP>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    merge_kernel(const uint16_t *__restrict__ o_parts, const float *__restrict__ lse_parts, int P, long long rows,
                 uint16_t *__restrict__ o, float *__restrict__ lse)
{
    const long long r = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (r >= rows)
        return;
    merge_row<D, BF16, NP>(o_parts, lse_parts, P, rows, r, threadIdx.x & 31, o, lse);
}

template <int D, bool BF16>
cudaError_t launch(const void *o_parts, const float *lse_parts, int P, long long rows, void *o, float *lse,
                   cudaStream_t st)
{
    const unsigned blocks = static_cast<unsigned>((rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
    const auto *op = static_cast<const uint16_t *>(o_parts);
    auto *out = static_cast<uint16_t *>(o);
    if (P <= 8)
        merge_kernel<D, BF16, 8><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(op, lse_parts, P, rows, out, lse);
    else if (P <= 16)
        merge_kernel<D, BF16, 16><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(op, lse_parts, P, rows, out, lse);
    else if (P <= 32)
        merge_kernel<D, BF16, 32><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(op, lse_parts, P, rows, out, lse);
    else
        merge_kernel<D, BF16, 0><<<blocks, 32 * kWarpsPerBlock, 0, st>>>(op, lse_parts, P, rows, out, lse);
    return cudaGetLastError();
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int sdp_merge(const void *o_parts, const float *lse_parts, int nparts, long long rows, int D, int dtype,
                         void *o, float *lse, void *stream)
{
    if (dtype != SDP_FP16 && dtype != SDP_BF16)
        return SDP_ERR_UNSUPPORTED;
    if (D != 128 && D != 256)
        return SDP_ERR_UNSUPPORTED;
    if (o_parts == nullptr || lse_parts == nullptr || o == nullptr || nparts <= 0 || rows <= 0)
        return SDP_ERR_INVALID_ARG;
    if (o == o_parts)
        return SDP_ERR_INVALID_ARG;
    if (!aligned(o_parts, 16) || !aligned(o, 16) || !aligned(lse_parts, 4) || !aligned(lse, 4))
        return SDP_ERR_ALIGNMENT;
    if ((rows + kWarpsPerBlock - 1) / kWarpsPerBlock > 0x7fffffffLL)
        return SDP_ERR_OVERFLOW;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (D == 128)
        e = dtype == SDP_BF16 ? launch<128, true>(o_parts, lse_parts, nparts, rows, o, lse, st)
                              : launch<128, false>(o_parts, lse_parts, nparts, rows, o, lse, st);
    else
        e = dtype == SDP_BF16 ? launch<256, true>(o_parts, lse_parts, nparts, rows, o, lse, st)
                              : launch<256, false>(o_parts, lse_parts, nparts, rows, o, lse, st);
    return e == cudaSuccess ? SDP_OK : SDP_ERR_CUDA;
}
