// Internal interface between the C ABI (sdp_api.cu) and the per-instantiation
// kernel translation units. Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace sdp {

// Arguments of one launch beyond the four tensor maps.
struct KernelParams {
    float *lse;            // [B, Hq, Sq] fp32, or nullptr
    unsigned int *status;  // device status word (0 = fine)
    int Hq, Hkv, G, Sq, Skv;
    int n_qtiles, n_kvtiles;
    float c;  // scale * log2(e): scores in base-2 units
    unsigned long long timeout_ns;
    int debug_flags;
    int causal;  // row i sees keys 0..i only
    // Split-KV launches: the grid is kv_splits copies of the unit grid, split s
    // reading KV tiles [s * tiles_per_split, +tiles_per_split) and writing its
    // partial O / LSE to output plane s * planes_q + (b, h). 1 / n_kvtiles otherwise.
    int kv_splits, tiles_per_split, planes_q;
    // Variable-length batches (cu_q != nullptr): sequence b owns Q/O rows
    // [cu_q[b], cu_q[b+1]) and K/V rows [cu_k[b], cu_k[b+1]) of tensors laid out
    // (token, head, dim); the planes are heads, Sq / Skv hold the token totals,
    // LSE is [Hq, total_q], and n_qtiles covers the longest sequence. A tile
    // that ends past its sequence is written row by row through `o`, element
    // (token t, head h) at o + t * o_row_stride + h * D.
    const int *cu_q, *cu_k;
    void *o;
    long long o_row_stride;
    // Compact unit list of a variable-length batch (n_tiles > 0): n_tiles list
    // slots per query head, at least the number of query tiles that exist
    // (sum over the nseq sequences of ceil(rows / 128)); slots past the last
    // real tile return at once. 0: the grid covers n_qtiles tiles per sequence.
    int nseq, n_tiles;
    // Host-side facts of the launching device (not read by the kernels): its
    // SM count, cached per device so that a launch makes no attribute query.
    int num_sms;
    // Units of the launch (the per-unit grid: one CTA per unit); set by the
    // persistent launchers, whose grids are smaller.
    int units;
    // A counter for the persistent single-CTA kernel's unit claims: one word of the
    // launching device's status region (the status word, then CLAIM_SLOTS counters),
    // the launching stream's own, so that only launches ordered on one stream share
    // it; zeroed in stream order by the launcher that uses it. Null (no persistent
    // single-CTA launch) under stream capture or when every counter has a stream.
    unsigned int *claim;
};

// Claim counters after the status word of each device's status region.
constexpr int CLAIM_SLOTS = 1024;

// Heads per block of the dense causal single-CTA unit order: query tiles go longest
// first across the heads of a block of ceil(CAUSAL_LANES / G) KV groups.
constexpr int CAUSAL_LANES = 4;

// Sequences per batch up to which causal variable-length launches use the compact
// unit list (its level-order search holds two sequences per lane in registers).
constexpr int VARLEN_LEVEL_MAX_SEQS = 64;

// Tensor maps of one launch: Q, K, V, O with 128-row boxes, K with 64-row
// boxes (half a KV tile) for the CTA-pair kernel, and (dense launches at head
// dim 128) K with 32-row boxes for the two-tile CTA-pair kernel.
struct LaunchMaps {
    CUtensorMap q, k, k_half, k32, v, o;
};

// Launches the CTA-pair kernel when consecutive units pair up within one
// (batch, KV head) and DEBUG_SINGLE_CTA is not set, else the single-CTA kernel.
#define SDP_DECLARE_LAUNCH(NAME) cudaError_t NAME(const LaunchMaps &m, const KernelParams &p, int grid, cudaStream_t stream);

SDP_DECLARE_LAUNCH(launch_d128_fp16)
SDP_DECLARE_LAUNCH(launch_d128_bf16)
SDP_DECLARE_LAUNCH(launch_d256_fp16)
SDP_DECLARE_LAUNCH(launch_d256_bf16)

#undef SDP_DECLARE_LAUNCH

// Where a launch's status word comes from: called for the current device `dev`
// once every argument check has passed, it returns the word's device address
// (zeroed, or zeroed in stream order before the kernel) or a status code.
using StatusSource = int (*)(int dev, unsigned int **status, cudaStream_t stream);

// The dense forward of sdp_fwd / sdp_fwd_causal: validation, the launch shape
// (head packing), tensor maps and the kernel launch, with the status word from
// `status_of`. Nothing is launched and `status_of` is not called when a check
// fails.
int forward_with(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq, int Hkv, int Sq,
                 int Skv, int D, float scale, int dtype, int causal, StatusSource status_of, void *stream);

// Records `word` as the status detail that sdp_last_status_detail() returns and
// maps it to its status code (SDP_ERR_BAD_SEQLENS or SDP_ERR_DEVICE_TIMEOUT).
int status_code_of(unsigned int word);

// Forgets the per-device addresses that sdp_fwd_noalloc looked up (called by
// sdp_shutdown, after which a reset device may hold the array elsewhere).
void noalloc_forget();

// Sets the cudaFuncAttributeMaxDynamicSharedMemorySize of a kernel once per
// device (`done` is that kernel's bit mask of devices already set).
template <typename Kernel>
cudaError_t set_smem_once(Kernel kern, int bytes, unsigned long long &done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (__atomic_load_n(&done, __ATOMIC_ACQUIRE) & bit))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0)
        __atomic_fetch_or(&done, bit, __ATOMIC_RELEASE);
    return e;
}

}  // namespace sdp
