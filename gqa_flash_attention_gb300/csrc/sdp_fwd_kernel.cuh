// Fused grouped-query attention forward for sm_103a (GB300).
//
// One CTA computes one unit = (batch b, query head h, 128 query rows). It
// streams the 128-key tiles of KV head g = h / (Hq/Hkv) once, keeping the
// online-softmax state (row maximum m, row sum l) in fp32 registers and the
// output accumulator O in tensor memory ("xe2-sdp-hd256" page, section
// "HD=256 Architecture Differences": single pass over KV chunks of 128 with a
// 128-row Q tile held on chip; "xe2-sdp-bf16" page, section "Data flow
// diagram": 16-bit operands into the contractions, fp32 softmax, output
// rounded to the input type at the very end).
//
// Warp roles (256 threads):
//   warps 0-3  softmax, lazy O rescale, epilogue. Thread t owns query row t,
//              which is TMEM lane t (warp w may only touch lanes 32w..32w+31).
//   warp 4     TMA producer: Q once, then K/V chunks through a ring of
//              32 KB shared-memory slots (full/empty mbarriers).
//   warp 5     TMEM owner and issuer of S_j = Q K_j^T (SMEM x SMEM -> TMEM fp32).
//   warp 6     issuer of O += P_j V_j (P from TMEM, V from SMEM).
//   warp 7     idle.
// The tensor queue is shallow, so a single issuing thread that waits on a
// barrier leaves the pipe idle; with two issuers one's waits are filled by
// the other's MMAs. The two MMA streams are ordered only where they share
// tensor memory: S_j overwrites the buffer that held P_{j-NSBUF}, so its
// issuer first waits for PV_{j-NSBUF} to complete.
//
// S has NSBUF tensor-memory buffers (2 at D=256, 3 at D=128), so the scores of
// the next tiles are computed while the softmax of tile j runs; P_j overwrites
// the first 64 columns of S_j's buffer as packed 16-bit pairs.
//
// Every mbarrier wait is bounded: after the timeout the waiting thread
// records a status code, raises a CTA-wide abort flag, and every role leaves
// its loop, drains what it has in flight, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"
#include "sdp_launch.h"

namespace sdp {

enum : uint32_t {
    SITE_Q_FULL = 1,
    SITE_SLOT_EMPTY = 2,
    SITE_SLOT_FULL = 3,
    SITE_S_FULL = 4,
    SITE_P_FULL = 5,
    SITE_O_DONE = 6,
    SITE_SEQLENS = 7,  // variable-length batch: sequence offsets out of range or not increasing
};

constexpr int DEBUG_NO_LOADS = 1;
constexpr int DEBUG_SINGLE_CTA = 2;  // never use the CTA-pair kernel
constexpr int DEBUG_PAIR_D128 = 8;   // use the CTA-pair kernel at D=128 too, where it qualifies
constexpr int DEBUG_NO_PERSIST = 16; // one unit per CTA pair even where the persistent form applies
constexpr int NUM_THREADS = 256;
constexpr int O_DONE_RING = 4;  // PV completion barriers, used round robin

template <int D>
struct Layout {
    static constexpr int BM = 128;                        // query rows per unit
    static constexpr int BN = 128;                        // keys per KV tile
    static constexpr int BOX_COLS = 64;                   // one 128-byte swizzle row of 16-bit values
    static constexpr int BOX_BYTES = 128 * BOX_COLS * 2;  // 16 KB: 128 rows x 64 columns
    static constexpr int CHUNK_BYTES = 2 * BOX_BYTES;     // 32 KB: 128 rows x 128 columns
    static constexpr int CHUNKS_PER_TILE = D / 128;       // ring chunks per K (or V) tile
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int NSLOTS = (SMEM_LIMIT - 2048 - Q_BYTES) / CHUNK_BYTES;
    static constexpr int NSBUF = (D == 128) ? 3 : 2;      // S/P buffers in tensor memory
    static constexpr int NBARS = 1 + 2 * NSLOTS + 2 * NSBUF + O_DONE_RING + 2;
    static constexpr int BAR_OFF = Q_BYTES + NSLOTS * CHUNK_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;  // barriers, then slack to align the base to 1 KB
    static constexpr int TM_O = 0;                           // O accumulator: columns [0, D)
    static constexpr int TM_S = D;                           // S/P buffer b: columns [D + 128b, D + 128b + 128)
    static constexpr int TMEM_COLS = 512;
    static_assert(D == 128 || D == 256, "head dim");
    static_assert(NSLOTS >= 2, "ring");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(D + NSBUF * BN <= TMEM_COLS, "tensor memory");
    static_assert(8 * NBARS + 8 <= 256, "barrier area");
    static_assert(O_DONE_RING >= NSBUF + 1, "PV completion ring must outrun the S buffers");
    // An issuer waiting on the chunk at load position P reads slot P % NSLOTS by
    // parity, which is only sound if the chunk at P - NSLOTS has landed. The
    // S issuer waits for K_t before PV_{t-NSBUF}, having seen PV_{t-NSBUF-1}
    // complete and every earlier K land, so only V_{t-NSBUF} .. V_{t-2} may be
    // in flight. The PV issuer waits for V_j having seen S_{j-1} complete (one
    // chunk per tile: before P_j is ready) or S_j (two: after), and every
    // earlier V, so only K_j and K_{j+1} (resp. K_{j+1}) may be in flight. With
    // one chunk per tile and NSBUF <= 3, or two chunks and NSBUF = 2, each of
    // those sits 1 to 3 positions before the waited chunk, never NSLOTS >= 4.
    static_assert(NSLOTS >= 4 && (CHUNKS_PER_TILE == 1 ? NSBUF <= 3 : NSBUF == 2), "ring parity soundness");
};

// Lazy rescale threshold in base-2 units: the running maximum is only moved
// when a tile's maximum exceeds it by more than this, so P <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr float LN2 = 0.6931471805599453f;

struct WaitCtx {
    volatile int *abort_flag;
    unsigned int *status;
    unsigned long long timeout_ns;
};

// Slow path of wait_bounded: poll until the phase completes, the CTA aborts,
// or the timeout passes (then raise the abort flag and record `site` and the
// CTA index in the status word).
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              unsigned int *status, unsigned long long timeout_ns, uint32_t site)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((it & 15u) == 0) {
            if (*abort_flag)
                return false;
            if (ptx::globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1;
                const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
                atomicCAS(status, 0u, site | (cta << 8));
                return false;
            }
        }
    }
}

// Bounded wait for the phase of `bar` with parity `parity`; false if the CTA
// is aborting or the wait ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx &cx, uint32_t site)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    return wait_slow(bar, parity, cx.abort_flag, cx.status, cx.timeout_ns, site);
}

// Bounded wait that ignores the abort flag: used only to drain copies and MMAs
// this thread issued itself, which always complete.
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > timeout_ns)
            return false;
    }
    return true;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Epilogue read-out of one accumulator row: O's D fp32 columns leave tensor memory GROUP
// chunks of 32 at a time behind one wait (one load latency per group instead of per chunk;
// the softmax arrays are dead here, so the 32 * GROUP values fit in registers), are scaled
// by 1/l and rounded to 16 bits, and each chunk's 16 packed words go to emit(chunk, words).
template <int D, bool BF16, int GROUP, typename Emit>
__device__ __forceinline__ void drain_o_row(uint32_t t_o, float inv_l, Emit &&emit)
{
    static_assert((D / 32) % GROUP == 0, "chunk groups");
#pragma unroll 1
    for (int c0 = 0; c0 < D / 32; c0 += GROUP) {
        uint32_t o[GROUP][32];
#pragma unroll
        for (int g = 0; g < GROUP; ++g)
            ptx::tmem_ld32(t_o + 32 * (c0 + g), o[g]);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < GROUP; ++g) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack2<BF16>(__uint_as_float(o[g][2 * i]) * inv_l, __uint_as_float(o[g][2 * i + 1]) * inv_l);
            emit(c0 + g, pk);
        }
    }
}

// Geometry of one unit's sequence: where its Q/O rows and K/V rows start in
// the (token) row coordinate, and how many of each it has. Without a
// variable-length batch it is the whole plane.
struct SeqGeom {
    int q_row0, kv_row0, sq, skv;
    bool ok;
};

__device__ __forceinline__ SeqGeom seq_geom(const KernelParams &p, int b)
{
    if (p.cu_q == nullptr)
        return SeqGeom{0, 0, p.Sq, p.Skv, true};
    const int q0 = __ldg(p.cu_q + b), q1 = __ldg(p.cu_q + b + 1);
    const int k0 = __ldg(p.cu_k + b), k1 = __ldg(p.cu_k + b + 1);
    const bool ok = 0 <= q0 && q0 <= q1 && q1 <= p.Sq && 0 <= k0 && k0 <= k1 && k1 <= p.Skv &&
                    q1 - q0 <= p.n_qtiles * 128;
    return SeqGeom{q0, k0, q1 - q0, k1 - k0, ok};
}

// What the compact unit list of a variable-length batch reads (by value, so the
// scan below takes no pointer to the kernel's parameters).
struct VarlenScan {
    const int *cu_q, *cu_k;
    int nseq, n_qtiles, Sq, Skv;
};
struct TileRef {
    int b, qt;
    bool found, any_bad;
};

// Query tiles of sequence idx: ceil(rows / 128), or 0 for an index past the
// batch or a sequence whose offsets fail seq_geom's checks (then `bad` is set).
__device__ __forceinline__ int varlen_tiles(const VarlenScan &v, int idx, bool &bad)
{
    bad = false;
    if (idx >= v.nseq)
        return 0;
    const int q0 = __ldg(v.cu_q + idx), q1 = __ldg(v.cu_q + idx + 1);
    const int k0 = __ldg(v.cu_k + idx), k1 = __ldg(v.cu_k + idx + 1);
    const bool ok = 0 <= q0 && q0 <= q1 && q1 <= v.Sq && 0 <= k0 && k0 <= k1 && k1 <= v.Skv &&
                    q1 - q0 <= v.n_qtiles * 128;
    bad = !ok;
    return ok ? (q1 - q0 + 127) / 128 : 0;
}

// The compact unit list of a variable-length batch (p.n_tiles > 0) holds only
// the query tiles that exist, sum over sequences of ceil(rows / 128), instead of
// the longest sequence's tile count for every sequence. Entry t of the list, in
// sequence order then tile order, or (by_level, causal launches) in descending
// tile index then sequence order, so that the units that read the most KV tiles
// start first. Computed by every warp on its own (lanes take 32 sequences at a
// time; no shared memory, no barrier); `found` is false past the last real
// tile. any_bad reports a sequence with invalid offsets among those scanned:
// all of them when scan_all or by_level, else those up to the one found.
static __device__ __noinline__ TileRef varlen_tile(const VarlenScan v, int t, bool by_level, bool scan_all)
{
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    TileRef r{0, 0, false, false};
    if (!by_level) {
        int acc = 0;  // tiles of the sequences before this group of 32
        for (int base = 0; base < v.nseq; base += 32) {
            bool bad;
            const int nb = varlen_tiles(v, base + lane, bad);
            r.any_bad |= __any_sync(FULL, bad);
            int incl = nb;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int x = __shfl_up_sync(FULL, incl, d);
                if (lane >= d)
                    incl += x;
            }
            const int excl = incl - nb;
            const unsigned hit = __ballot_sync(FULL, acc + excl <= t && t < acc + incl);
            if (hit != 0u) {
                const int src = __ffs(hit) - 1;
                r.b = base + src;
                r.qt = t - acc - __shfl_sync(FULL, excl, src);
                r.found = true;
            }
            acc += __shfl_sync(FULL, incl, 31);
            if (r.found && !scan_all)
                break;
        }
        return r;
    }
    // Level order, for at most VARLEN_LEVEL_MAX_SEQS = 64 sequences (the host's limit for
    // it): two tile counts per lane, held in registers. Tiles with index >= q number
    // C(q) = sum_b max(0, n_b - q); entry t lies on the level q with C(q + 1) <= t < C(q).
    static_assert(VARLEN_LEVEL_MAX_SEQS <= 64, "two sequences per lane");
    bool bad0, bad1;
    const int n0 = varlen_tiles(v, lane, bad0);
    const int n1 = varlen_tiles(v, lane + 32, bad1);
    r.any_bad = __any_sync(FULL, bad0 || bad1);
    auto count_from = [&](int q) -> int {
        int s = max(0, n0 - q) + max(0, n1 - q);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            s += __shfl_xor_sync(FULL, s, d);
        return s;
    };
    if (t >= count_from(0))
        return r;
    int lo = 0, hi = v.n_qtiles - 1;  // the largest q with C(q) > t
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (count_from(mid) > t)
            lo = mid;
        else
            hi = mid - 1;
    }
    int rank = t - count_from(lo + 1);  // among the sequences with more than lo tiles
    unsigned m = __ballot_sync(FULL, n0 > lo);
    const unsigned m1 = __ballot_sync(FULL, n1 > lo);
    int base = 0;
    if (rank >= __popc(m)) {
        rank -= __popc(m);
        m = m1;
        base = 32;
    }
    for (int i = 0; i < rank; ++i)
        m &= m - 1u;
    r.b = base + __ffs(m) - 1;
    r.qt = lo;
    r.found = true;
    return r;
}

// Slot u (head-in-group index already taken out) of a compact variable-length
// launch, n_tiles slots per KV head. Without the causal mask a KV head's tiles
// run sequence by sequence (their K/V stay in L2); with it, in level order
// across the KV heads. Block 0 scans every sequence and reports invalid offsets.
// Returns the unit index that the full grid gives the same (sequence, tile, KV
// head), so that one decode serves both grids, or -1 for a slot past the last
// real tile (both CTAs of a pair get the same answer).
__device__ __forceinline__ int varlen_compact_unit(const KernelParams &p, int u)
{
    int t, g;
    if (p.causal) {
        g = u % p.Hkv;
        t = u / p.Hkv;
    } else {
        t = u % p.n_tiles;
        g = u / p.n_tiles;
    }
    const TileRef r = varlen_tile(VarlenScan{p.cu_q, p.cu_k, p.nseq, p.n_qtiles, p.Sq, p.Skv}, t, p.causal != 0,
                                  blockIdx.x == 0);
    if (r.any_bad && blockIdx.x == 0 && threadIdx.x == 0)
        atomicCAS(p.status, 0u, static_cast<unsigned>(SITE_SEQLENS));
    if (!r.found)
        return -1;
    const int bg = r.b * p.Hkv + g;
    return p.causal ? (p.n_qtiles - 1 - r.qt) * (p.nseq * p.Hkv) + bg : bg * p.n_qtiles + r.qt;
}

// Dense causal launches: query tile qt and (batch, KV head) bg of unit u (head-in-group
// index already taken out; n_bg = B * Hkv). A unit does qt + 1 tiles. Blocks of W
// consecutive KV groups (at least CAUSAL_LANES heads), longest tiles first inside a block
// across its groups: the grid's last units are short ones of several heads rather than one
// head's whole range of lengths, and the units in flight read at most a block's K/V.
__device__ __forceinline__ void causal_block_unit(const KernelParams &p, int u, int n_bg, int &qt, int &bg)
{
    const int W = min(n_bg, (CAUSAL_LANES + p.G - 1) / p.G);
    const int blk = u / (W * p.n_qtiles);
    const int r = u - blk * W * p.n_qtiles;
    const int wsz = min(W, n_bg - blk * W);
    qt = p.n_qtiles - 1 - r / wsz;
    bg = blk * W + r % wsz;
}

// Position of a chunk in the load order K_0, then for j = 0..n-1: K_{j+1} (if
// any), V_j. Tiles are CPT chunks long; the producer and both issuers derive
// ring slot = pos % NSLOTS and phase = (pos / NSLOTS) & 1 from it. Every
// chunk's consumption depends only on chunks earlier in this order, so the
// producer's in-order refill cannot deadlock.
template <int CPT>
__device__ __forceinline__ int pos_k(int t)
{
    return t == 0 ? 0 : CPT * (2 * t - 1);
}
template <int CPT>
__device__ __forceinline__ int pos_v(int j, int n)
{
    return j == n - 1 ? CPT * (2 * j + 1) : CPT * (2 * j + 2);
}

// VARLEN: launched for variable-length batches (p.cu_q != nullptr); only that
// instantiation carries the compact unit list's decode.
template <int D, bool BF16, bool VARLEN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    sdp_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const KernelParams p)
{
    using L = Layout<D>;
    constexpr int NS = L::NSLOTS;
    constexpr int NB = L::NSBUF;
    constexpr int CPT = L::CHUNKS_PER_TILE;
    constexpr uint32_t IDESC_S = ptx::idesc_f16_f32acc(128, L::BN, BF16, false);  // Q (K-major) x K (K-major)
    constexpr uint32_t IDESC_PV = ptx::idesc_f16_f32acc(128, 128, BF16, true);    // P (TMEM) x V (N-major)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t s_q = sbase;  // Q tile; reused as the O staging tile in the epilogue
    const uint32_t s_ring = sbase + L::Q_BYTES;
    const uint32_t bar0 = sbase + L::BAR_OFF;
    const uint32_t q_full = bar0;
    const uint32_t slot_full0 = bar0 + 8u;
    const uint32_t slot_empty0 = bar0 + 8u * (1 + NS);
    const uint32_t s_full0 = bar0 + 8u * (1 + 2 * NS);
    const uint32_t p_full0 = bar0 + 8u * (1 + 2 * NS + NB);
    const uint32_t o_done0 = bar0 + 8u * (1 + 2 * NS + 2 * NB);
    const uint32_t final0 = bar0 + 8u * (1 + 2 * NS + 2 * NB + O_DONE_RING);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Unit order: head-in-group fastest, then query tile, then (batch, KV head),
    // so CTAs resident together read the same K/V tiles from L2 (dense causal
    // launches: query tile outside a block of KV groups, below).
    int u = blockIdx.x;
    // KV split (split-KV launches): the outermost unit coordinate.
    const int units_per_split = static_cast<int>(gridDim.x) / p.kv_splits;
    const int split = u / units_per_split;
    u -= split * units_per_split;
    const int hi = u % p.G;
    u /= p.G;
    if constexpr (VARLEN) {
        if (p.n_tiles > 0 && (u = varlen_compact_unit(p, u)) < 0)
            return;  // a slot past the last query tile
    }
    int qt, bg;  // query tile; b * Hkv + g
    if (p.cu_q != nullptr && p.causal) {
        // Causal variable-length batch: query tile outermost, highest first. A unit of tile qt
        // reads qt + 1 KV tiles whatever its sequence, so the costliest units start first.
        // (Without the mask a unit's cost is its sequence's key count, unrelated to qt: the
        // group-major order stays.)
        const int n_bg = VARLEN ? p.nseq * p.Hkv : units_per_split / (p.G * p.n_qtiles);
        qt = p.n_qtiles - 1 - u / n_bg;
        bg = u % n_bg;
    } else if (p.causal) {
        causal_block_unit(p, u, units_per_split / (p.G * p.n_qtiles), qt, bg);
    } else {
        qt = u % p.n_qtiles;
        bg = u / p.n_qtiles;
    }
    const int b = bg / p.Hkv;
    const int g = bg - b * p.Hkv;
    const bool varlen = p.cu_q != nullptr;
    // (b, h) plane of Q, O and LSE and (b, g) plane of K and V; heads h and g
    // in a variable-length batch, whose sequences are runs of rows.
    const int z_q = varlen ? g * p.G + hi : b * p.Hq + g * p.G + hi;
    const int z_kv = varlen ? g : bg;
    const int q0 = qt * L::BM;  // first query row of the unit within its sequence
    const SeqGeom sg = seq_geom(p, b);
    if (!sg.ok) {
        if (threadIdx.x == 0) {
            const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
            atomicCAS(p.status, 0u, SITE_SEQLENS | (cta << 8));
        }
        return;
    }
    if (q0 >= sg.sq)
        return;  // a tile past the end of a shorter sequence: nothing to do
    const int n_kv = (sg.skv + L::BN - 1) / L::BN;
    // Tiles this unit reads: all of them, or (causal) those holding keys <= its last row.
    const int t0 = split * p.tiles_per_split;  // first KV tile of this unit
    const int n = p.causal ? min(n_kv, qt + 1) : min(n_kv - t0, p.tiles_per_split);
    const int z_out = split * p.planes_q + z_q;  // output plane of O and LSE
    const int q_row = sg.q_row0 + q0;            // row coordinate of the tile in Q and O
    if (n <= 0) {
        // A sequence without keys: its rows attend to nothing, O = 0 and LSE = -inf.
        const int rows = min(L::BM, sg.sq - q0);
        for (int i = threadIdx.x; i < rows * (D / 8); i += NUM_THREADS) {
            const int r = i / (D / 8), c8 = i % (D / 8);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) +
                                                   static_cast<size_t>(q_row + r) * p.o_row_stride +
                                                   static_cast<size_t>(z_q) * D) + c8;
            *dst = make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.lse != nullptr)
            for (int r = threadIdx.x; r < rows; r += NUM_THREADS)
                p.lse[static_cast<size_t>(z_out) * p.Sq + q_row + r] = -INFINITY;
        return;
    }
    // A variable-length tile that ends past its sequence is stored row by row.
    const bool direct_store = varlen && q0 + L::BM > sg.sq;

    // The first DRAM reads (the Q tile, K_0 and V_0, the producer's first copies, same boxes) start
    // now, into L2, so that their latency overlaps barrier set-up and the tensor-memory allocation.
    if (warp == 4 && lane == 0 && !(p.debug_flags & DEBUG_NO_LOADS)) {
        const int y = sg.kv_row0 + t0 * L::BN;
#pragma unroll
        for (int c = 0; c < D / L::BOX_COLS; ++c) {
            ptx::tma_prefetch_3d(&tm_q, c * L::BOX_COLS, q_row, z_q);
            ptx::tma_prefetch_3d(&tm_k, c * L::BOX_COLS, y, z_kv);
            ptx::tma_prefetch_3d(&tm_v, c * L::BOX_COLS, y, z_kv);
        }
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(slot_full0 + 8u * s, 1);
            ptx::mbar_init(slot_empty0 + 8u * s, 1);
        }
        for (int i = 0; i < NB; ++i) {
            ptx::mbar_init(s_full0 + 8u * i, 1);
            ptx::mbar_init(p_full0 + 8u * i, 128);
        }
        for (int i = 0; i < O_DONE_RING; ++i)
            ptx::mbar_init(o_done0 + 8u * i, 1);
        ptx::mbar_init(final0, 1);
        ptx::mbar_init(final0 + 8u, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx cx{abort_flag, p.status, p.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        {  // whole warp; one elected lane issues
            int slot = 0;
            uint32_t ph = 0, armed_mask = 0, armed_par = 0;
            bool q_armed = false;
            if (!(p.debug_flags & DEBUG_NO_LOADS)) {
                ptx::mbar_arrive_expect_tx_w(q_full, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / L::BOX_COLS; ++c)
                    ptx::tma_load_3d_w(s_q + c * L::BOX_BYTES, &tm_q, q_full, c * L::BOX_COLS, q_row, z_q);
                q_armed = true;
                auto load_tile = [&](const CUtensorMap *map, int j) -> bool {
#pragma unroll
                    for (int ch = 0; ch < CPT; ++ch) {
                        const uint32_t full = slot_full0 + 8u * slot;
                        const bool ok = wait_bounded(slot_empty0 + 8u * slot, ph ^ 1u, cx, SITE_SLOT_EMPTY);
                        if (!__all_sync(0xffffffffu, ok))
                            return false;
                        ptx::mbar_arrive_expect_tx_w(full, L::CHUNK_BYTES);
                        const uint32_t dst = s_ring + slot * L::CHUNK_BYTES;
                        const int y = sg.kv_row0 + (t0 + j) * L::BN;
                        ptx::tma_load_3d_w(dst, map, full, ch * 128, y, z_kv);
                        ptx::tma_load_3d_w(dst + L::BOX_BYTES, map, full, ch * 128 + L::BOX_COLS, y, z_kv);
                        armed_mask |= 1u << slot;
                        armed_par = (armed_par & ~(1u << slot)) | (ph << slot);
                        if (++slot == NS) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                    return true;
                };
                bool ok = load_tile(&tm_k, 0);
                for (int j = 0; ok && j < n; ++j) {
                    if (j + 1 < n)
                        ok = load_tile(&tm_k, j + 1);
                    if (ok)
                        ok = load_tile(&tm_v, j);
                }
            }
            // Every copy this thread issued lands before the CTA may exit.
            if (q_armed)
                wait_drain(q_full, 0, p.timeout_ns);
            for (int s = 0; s < NS; ++s)
                if (armed_mask & (1u << s))
                    wait_drain(slot_full0 + 8u * s, (armed_par >> s) & 1u, p.timeout_ns);
        }
    } else if (warp == 5) {
        // ------------------------------------------- S = Q K^T issuer (1 thread)
        {  // whole warp; one elected lane issues
            const uint64_t dq = ptx::smem_desc_sw128(s_q, 16, 1024);
            const uint64_t dk = ptx::smem_desc_sw128(s_ring, 16, 1024);
            bool issued = false;
            bool ok = __all_sync(0xffffffffu, wait_bounded(q_full, 0, cx, SITE_Q_FULL));
            for (int t = 0; ok && t < n; ++t) {
                const int p0 = pos_k<CPT>(t);
                // K_t has usually landed long before PV_{t-NB} completes, so its
                // slots are waited for first, off the PV_{t-NB} -> S_t path.
#pragma unroll
                for (int ch = 0; ch < CPT; ++ch) {
                    const int pos = p0 + ch;
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * (pos % NS), (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                        break;
                }
                if (!ok)
                    break;
                if (t >= NB) {  // buffer t % NB held P_{t-NB}: PV_{t-NB} must have read it
                    const int pv = t - NB;
                    ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx,
                                                              SITE_O_DONE));
                    if (!ok)
                        break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + L::TM_S + (t % NB) * L::BN;
#pragma unroll
                for (int ch = 0; ch < CPT; ++ch) {
                    const int pos = p0 + ch;
                    const int slot = pos % NS;
                    const uint64_t kslot = dk + static_cast<uint64_t>((slot * L::CHUNK_BYTES) >> 4);
                    const uint64_t qch = dq + static_cast<uint64_t>((2 * ch * L::BOX_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = ((kk >> 2) * L::BOX_BYTES + (kk & 3) * 32) >> 4;
                        ptx::mma_ss_w(d_tmem, qch + off, kslot + off, IDESC_S, (ch | kk) != 0);
                    }
                    issued = true;
                    ptx::mma_commit_w(slot_empty0 + 8u * slot);
                }
                ptx::mma_commit_w(s_full0 + 8u * (t % NB));
            }
            if (issued) {  // all of this thread's MMAs complete before TMEM is freed
                ptx::mma_commit_w(final0);
                wait_drain(final0, 0, p.timeout_ns);
            }
        }
    } else if (warp == 6) {
        // ------------------------------------------ O += P V issuer (1 thread)
        {  // whole warp; one elected lane issues
            const uint64_t dv = ptx::smem_desc_sw128(s_ring, L::BOX_BYTES, 1024);
            bool issued = false;
            bool ok = true;
            for (int j = 0; ok && j < n; ++j) {
                const int buf = j % NB;
                const int p0 = pos_v<CPT>(j, n);
                // With one ring chunk per tile, V_j has usually landed before P_j is
                // ready, so its slot is waited for first, off the P_j -> PV_j path.
                // (With two, the chunk NSLOTS before V_j's first can belong to K_j,
                // which only P_j being ready shows to have landed: that order stays.)
                if constexpr (CPT == 1) {
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * (p0 % NS), (p0 / NS) & 1, cx, SITE_SLOT_FULL))))
                        break;
                }
                if (!(ok = __all_sync(0xffffffffu, wait_bounded(p_full0 + 8u * buf, (j / NB) & 1, cx, SITE_P_FULL))))
                    break;
                ptx::tc_fence_after();
                const uint32_t a_tmem = tmem + L::TM_S + buf * L::BN;
#pragma unroll
                for (int ch = 0; ch < CPT; ++ch) {
                    const int pos = p0 + ch;
                    const int slot = pos % NS;
                    if constexpr (CPT != 1) {
                        if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                            break;
                        ptx::tc_fence_after();
                    }
                    const uint64_t vslot = dv + static_cast<uint64_t>((slot * L::CHUNK_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        ptx::mma_ts_w(tmem + L::TM_O + ch * 128, a_tmem + kk * 8, vslot + ((kk * 2048) >> 4), IDESC_PV,
                                    (j > 0) || (kk > 0));
                    issued = true;
                    ptx::mma_commit_w(slot_empty0 + 8u * slot);
                }
                if (!ok)
                    break;
                ptx::mma_commit_w(o_done0 + 8u * (j % O_DONE_RING));
            }
            if (issued) {
                ptx::mma_commit_w(final0 + 8u);
                wait_drain(final0 + 8u, 0, p.timeout_ns);
            }
        }
    } else if (warp < 4) {
        // --------------------------------------- softmax / correction / epilogue
        const int row = threadIdx.x;  // query row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t t_s = tmem + lane_off + L::TM_S;
        const uint32_t t_o = tmem + lane_off + L::TM_O;
        const float c = p.c;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        bool s_seen = false;  // S_j's barrier was seen complete while tile j-1 ended

        for (int j = 0; j < n; ++j) {
            const int buf = j % NB;
            if (!__all_sync(0xffffffffu, s_seen)) {
                ok = wait_bounded(s_full0 + 8u * buf, (j / NB) & 1, cx, SITE_S_FULL);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
            }
            ptx::tc_fence_after();
            const uint32_t ts = t_s + buf * L::BN;
            uint32_t sr[128];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                ptx::tmem_ld32(ts + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * q]));
            ptx::tmem_wait_ld();
            float s[128];
#pragma unroll
            for (int i = 0; i < 128; ++i)
                s[i] = __uint_as_float(sr[i]);

            // keys of this tile the row sees (>= 1): all < Skv, and (causal) <= the row itself
            const int valid = (p.causal ? min(sg.skv, q0 + row + 1) : sg.skv) - (t0 + j) * L::BN;  // >= 1
            // Only a tile holding a key this row must not see (the ragged last tile,
            // a causal diagonal) takes the masked path; the others run without any
            // per-element test (a warp-uniform branch, not predication).
            const bool tail = __any_sync(0xffffffffu, valid < L::BN);
            if (tail) {
#pragma unroll
                for (int i = 1; i < 128; ++i)
                    if (i >= valid)
                        s[i] = s[0];  // neutral for the max; weights zeroed below
            }
            // Row extreme of the raw scores (maximum of s * c: of s when c >= 0, else
            // its minimum), four three-input chains.
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
            if (c >= 0.f) {
#pragma unroll
                for (int i = 4; i < 124; i += 8) {
                    mx0 = ptx::max3(mx0, s[i], s[i + 1]);
                    mx1 = ptx::max3(mx1, s[i + 2], s[i + 3]);
                    mx2 = ptx::max3(mx2, s[i + 4], s[i + 5]);
                    mx3 = ptx::max3(mx3, s[i + 6], s[i + 7]);
                }
                mx0 = ptx::max3(mx0, s[124], s[125]);
                mx1 = ptx::max3(mx1, s[126], s[127]);
                mx0 = ptx::max3(mx0, mx1, fmaxf(mx2, mx3));
            } else {
#pragma unroll
                for (int i = 4; i < 124; i += 8) {
                    mx0 = ptx::min3(mx0, s[i], s[i + 1]);
                    mx1 = ptx::min3(mx1, s[i + 2], s[i + 3]);
                    mx2 = ptx::min3(mx2, s[i + 4], s[i + 5]);
                    mx3 = ptx::min3(mx3, s[i + 6], s[i + 7]);
                }
                mx0 = ptx::min3(mx0, s[124], s[125]);
                mx1 = ptx::min3(mx1, s[126], s[127]);
                mx0 = ptx::min3(mx0, mx1, fminf(mx2, mx3));
            }
            const float m_tile = mx0 * c;  // this tile's row maximum of s * scale * log2(e)
            const float m_new = (j == 0 || m_tile > m_used + RESCALE_THRESHOLD) ? m_tile : m_used;
            const float alpha = (j == 0 || m_new == m_used) ? 1.f : ptx::ex2(m_used - m_new);
            const float neg_m = -m_new;

            // p = 2^(s * c - m), two elements per f32x2 instruction for the scaling
            // and the running sums (each lane rounds exactly as fmaf / + would).
            uint32_t pk[64];
            const uint64_t c2 = ptx::f2_pack(c, c), negm2 = ptx::f2_pack(neg_m, neg_m);
            uint64_t sum01 = ptx::f2_pack(0.f, 0.f), sum23 = sum01;
            auto exp_tile = [&](auto masked) {
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    float x0, x1, x2, x3;
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[2 * i], s[2 * i + 1]), c2, negm2), x0, x1);
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[2 * i + 2], s[2 * i + 3]), c2, negm2), x2, x3);
                    float p0 = ptx::ex2(x0);
                    float p1 = ptx::ex2(x1);
                    float p2 = ptx::ex2(x2);
                    float p3 = ptx::ex2(x3);
                    if constexpr (decltype(masked)::value) {
                        p0 = (2 * i < valid) ? p0 : 0.f;
                        p1 = (2 * i + 1 < valid) ? p1 : 0.f;
                        p2 = (2 * i + 2 < valid) ? p2 : 0.f;
                        p3 = (2 * i + 3 < valid) ? p3 : 0.f;
                    }
                    sum01 = ptx::f2_add(sum01, ptx::f2_pack(p0, p1));
                    sum23 = ptx::f2_add(sum23, ptx::f2_pack(p2, p3));
                    pk[i] = pack2<BF16>(p0, p1);
                    pk[i + 1] = pack2<BF16>(p2, p3);
                }
            };
            if (tail)
                exp_tile(std::true_type{});
            else
                exp_tile(std::false_type{});
            // Poll S_{j+1}'s barrier now, so the answer returns while P_j is stored
            // and handed off (no parity aliasing: S_j complete implies
            // S_{j+1-NSBUF} complete, and S_{j+1+NSBUF} waits for P_{j+1}).
            s_seen = j + 1 < n && ptx::mbar_test_wait(s_full0 + 8u * ((j + 1) % NB), ((j + 1) / NB) & 1);
            float sum0, sum1, sum2, sum3;
            ptx::f2_unpack(sum01, sum0, sum1);
            ptx::f2_unpack(sum23, sum2, sum3);
            ptx::tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            ptx::tmem_st32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            ptx::tmem_wait_st();
            const float tile_sum = (sum0 + sum1) + (sum2 + sum3);
            l = (j == 0) ? tile_sum : fmaf(l, alpha, tile_sum);

            // Rescale O only in warps where some row's maximum moved; only they
            // wait for PV_{j-1}. The skipped waits cannot alias: S_j completing
            // implies PV_{j-NSBUF} completed, so the barrier that holds PV_{j-1}
            // is at most one phase away (O_DONE_RING >= NSBUF + 1).
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const int pv = j - 1;
                ok = wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx, SITE_O_DONE);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
                ptx::tc_fence_after();
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    ptx::tmem_ld32(t_o + 32 * cc, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    ptx::tmem_st32(t_o + 32 * cc, o);
                }
                ptx::tmem_wait_st();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(p_full0 + 8u * buf);
            m_used = m_new;
        }

        // ------------------------------------------------------------ epilogue
        ptx::named_bar_sync(1, 128);
        ok = ok && !*abort_flag;
        if (ok) {
            const int pv = n - 1;
            ok = wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx, SITE_O_DONE);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            ptx::tc_fence_after();
            drain_o_row<D, BF16, 4>(t_o, 1.f / l, [&](int cc, const uint32_t (&pk)[16]) {
                if (direct_store) {
                    // the rows of this sequence only, 64 bytes per row per step
                    if (q0 + row < sg.sq) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) +
                                                               static_cast<size_t>(q_row + row) * p.o_row_stride +
                                                               static_cast<size_t>(z_q) * D + 32 * cc);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                    return;
                }
                // 32 columns = four 16-byte units of row `row` in box cc/2, 128-byte swizzled.
                const uint32_t row_addr = s_q + (cc >> 1) * L::BOX_BYTES + row * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint32_t unit = static_cast<uint32_t>((cc & 1) * 4 + v);
                    st_shared_v4(row_addr + ((unit ^ static_cast<uint32_t>(row & 7)) << 4), pk[4 * v], pk[4 * v + 1],
                                 pk[4 * v + 2], pk[4 * v + 3]);
                }
            });
            if (p.lse != nullptr && q0 + row < sg.sq)
                p.lse[static_cast<size_t>(z_out) * p.Sq + q_row + row] = (m_used + ptx::lg2(l)) * LN2;
            ptx::fence_proxy_async_smem();
        }
        ptx::named_bar_sync(1, 128);
        if (threadIdx.x == 0 && !*abort_flag && !direct_store) {
#pragma unroll
            for (int c2 = 0; c2 < D / L::BOX_COLS; ++c2)
                ptx::tma_store_3d(&tm_o, s_q + c2 * L::BOX_BYTES, c2 * L::BOX_COLS, q_row, z_out);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read_all();
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// Host-side launcher, one instantiation per (head dim, dtype).
template <int D, bool BF16>
cudaError_t launch_sdp_fwd(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const CUtensorMap &o,
                           const KernelParams &p, int grid, cudaStream_t stream)
{
    static unsigned long long set_dense = 0, set_varlen = 0;
    const bool vl = p.cu_q != nullptr;
    auto kern = vl ? sdp_fwd_kernel<D, BF16, true> : sdp_fwd_kernel<D, BF16, false>;
    cudaError_t e = set_smem_once(kern, Layout<D>::SMEM_BYTES, vl ? set_varlen : set_dense);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, NUM_THREADS, Layout<D>::SMEM_BYTES, stream>>>(q, k, v, o, p);
    return cudaGetLastError();
}

}  // namespace sdp
