// Grouped-query attention forward on a CTA pair (cta_group::2), sm_103a.
//
// Same method and roles as sdp_fwd_kernel (see sdp_fwd_kernel.cuh), but two
// CTAs on two SMs form a cluster and share every K/V tile: each CTA keeps its
// own unit (128 query rows, its S/P buffers and its O accumulator in its own
// tensor memory) while the tensor cores of both SMs run one M=256 MMA per
// k-step, issued by the leader CTA's (rank 0) two issuer warps.
//
//   S = Q K^T  : M=256 (128 rows per CTA), N=128 keys; CTA r holds keys
//                [64r, 64r+64) of the tile (half of B, K-major).
//   O += P V   : M=256, N=D; P from each CTA's own TMEM; CTA r holds the
//                value columns [rD/2, rD/2 + D/2) of the tile (half of B,
//                N-major).
//
// Each SM therefore receives half of every K and V tile from L2: at D=256 the
// single-CTA kernel is bound by that stream (about 43 B/clk per SM), which this
// halves; the leader also issues half as many MMA instructions per FLOP. (At
// D=128 the single-CTA kernel measured as fast or faster and is the default.)
//
// Cross-CTA protocol (barriers live in each CTA at the same offsets):
//   q_full, slot_full : armed by the leader's producer for both halves; both
//                       CTAs' TMA loads complete on the leader's barrier.
//   slot_empty, s_full, o_done : arrived by the leader's MMA commits,
//                       multicast to both CTAs.
//   p_part, p_full    : in the leader; one arrival per softmax warp of both
//                       CTAs (the peer's arrive remotely) per part of P_j.
//                       P_j is handed over in P_PARTS parts of consecutive
//                       keys (p_part for all but the last, p_full for the
//                       last), and the PV issuer runs each part's K steps as
//                       soon as it arrives: the S_j -> softmax_j -> PV_j ->
//                       S_{j+NSBUF} chain that bounds this kernel then keeps
//                       only the last part's MMAs after the softmax ends.
// Both CTAs must belong to the same (batch, KV head) and, in a variable-length
// batch, the same sequence and query tile: the launcher only pairs units when
// each (batch, KV head) has an even number of units (query tiles x query heads
// per group; an even group size for causal and variable-length launches);
// otherwise it runs the single-CTA kernel.
#pragma once

#include "sdp_fwd_kernel.cuh"

namespace sdp {

template <int D>
struct PairLayout {
    static constexpr int BM = 128;                       // query rows per CTA
    static constexpr int BN = 128;                       // keys per KV tile (both CTAs)
    static constexpr int Q_BOX_BYTES = 128 * 128;        // 128 rows x 64 columns
    static constexpr int K_BOX_BYTES = 64 * 128;         // 64 keys x 64 columns
    static constexpr int V_BOX_BYTES = 128 * 128;        // 128 keys x 64 columns
    static constexpr int HALF_BYTES = 64 * D * 2;        // half a K tile = half a V tile
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int BAR_AREA = 512;
    static constexpr int NSLOTS = (SMEM_LIMIT - BAR_AREA - 1024 - Q_BYTES) / HALF_BYTES;
    static constexpr int NSBUF = (D == 128) ? 3 : 2;
    static constexpr int P_ARRIVALS = 8;                 // 4 softmax warps in each CTA
    // P_j is handed over in parts of 128 / P_PARTS keys. Each part costs a hand-off
    // (fence, warp sync, one arrival per warp, remote from the peer): at D=256 the
    // S -> softmax -> PV chain bounds the kernel and parts shorten it; at D=128 the
    // softmax is the bound and the hand-offs only lengthen it (one part, -25 % with four).
    static constexpr int P_PARTS = (D == 256) ? 4 : 1;
    static_assert(P_PARTS == 1 || P_PARTS == 2 || P_PARTS == 4, "P hand-off parts");
    static constexpr int NBARS = 1 + 2 * NSLOTS + (1 + P_PARTS) * NSBUF + O_DONE_RING + 2;
    static constexpr int BAR_OFF = Q_BYTES + NSLOTS * HALF_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + BAR_AREA + 1024;
    static constexpr int TM_O = 0;
    static constexpr int TM_S = D;
    static constexpr int TMEM_COLS = 512;
    static_assert(D == 128 || D == 256, "head dim");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(D + NSBUF * BN <= TMEM_COLS, "tensor memory");
    static_assert(8 * NBARS + 8 <= BAR_AREA, "barrier area");
    static_assert(O_DONE_RING >= NSBUF + 1, "PV completion ring must outrun the S buffers");
    // Same parity-soundness argument as the single-CTA ring, with one slot per
    // half tile (so CHUNKS_PER_TILE = 1).
    static_assert(NSLOTS >= 4 && NSBUF <= 3, "ring parity soundness");
};

// Slow path for a wait whose phase is completed by arrivals from the peer CTA.
static __device__ __noinline__ bool wait_slow_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                                      unsigned int *status, unsigned long long timeout_ns,
                                                      uint32_t site)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait_cluster(bar, parity))
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

__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const WaitCtx &cx, uint32_t site)
{
    if (ptx::mbar_try_wait_cluster(bar, parity))
        return true;
    return wait_slow_cluster(bar, parity, cx.abort_flag, cx.status, cx.timeout_ns, site);
}

template <int D, bool BF16, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    sdp_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const KernelParams p)
{
    using L = PairLayout<D>;
    constexpr int NS = L::NSLOTS;
    constexpr int NB = L::NSBUF;
    constexpr uint32_t IDESC_S = ptx::idesc_f16_f32acc(256, L::BN, BF16, false);  // Q x K half, both K-major
    constexpr uint32_t IDESC_PV = ptx::idesc_f16_f32acc(256, D, BF16, true);      // P (TMEM) x V half (N-major)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t s_q = sbase;
    const uint32_t s_ring = sbase + L::Q_BYTES;
    const uint32_t bar0 = sbase + L::BAR_OFF;
    const uint32_t q_full = bar0;
    const uint32_t slot_full0 = bar0 + 8u;
    const uint32_t slot_empty0 = bar0 + 8u * (1 + NS);
    const uint32_t s_full0 = bar0 + 8u * (1 + 2 * NS);
    const uint32_t p_full0 = bar0 + 8u * (1 + 2 * NS + NB);
    const uint32_t o_done0 = bar0 + 8u * (1 + 2 * NS + 2 * NB);
    const uint32_t final0 = bar0 + 8u * (1 + 2 * NS + 2 * NB + O_DONE_RING);
    // part q < P_PARTS - 1 of P_j is in tensor memory: p_part0 + 8 * (NB * q + buf); the last part is p_full
    const uint32_t p_part0 = final0 + 16u;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank == 0);

    int u = blockIdx.x;
    // KV split (split-KV launches): the outermost unit coordinate.
    const int units_per_split = static_cast<int>(gridDim.x) / p.kv_splits;
    const int split = u / units_per_split;
    u -= split * units_per_split;
    const int hi = u % p.G;
    u /= p.G;
    if constexpr (VARLEN) {
        if (p.n_tiles > 0 && (u = varlen_compact_unit(p, u)) < 0)
            return;  // both CTAs of the pair: the same slot past the last query tile
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
    } else {
        // Causal units do qt + 1 tiles: start the longest ones first.
        qt = p.causal ? p.n_qtiles - 1 - (u % p.n_qtiles) : (u % p.n_qtiles);
        bg = u / p.n_qtiles;
    }
    const int b = bg / p.Hkv;
    const int g = bg - b * p.Hkv;
    const bool varlen = p.cu_q != nullptr;
    const int z_q = varlen ? g * p.G + hi : b * p.Hq + g * p.G + hi;
    const int z_kv = varlen ? g : bg;
    const int q0 = qt * L::BM;
    // Sequence geometry and the early exits are the same in both CTAs of a pair:
    // a pair is two heads of one group on the same query tile of one sequence.
    const SeqGeom sg = seq_geom(p, b);
    if (!sg.ok) {
        if (threadIdx.x == 0) {
            const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
            atomicCAS(p.status, 0u, SITE_SEQLENS | (cta << 8));
        }
        return;
    }
    if (q0 >= sg.sq)
        return;
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

    // This CTA's first DRAM reads (its Q tile, its half of K_0 and of V_0: the producer's first copies,
    // same boxes) start now, into L2, so that their latency overlaps barrier set-up, the tensor-memory
    // allocation and the cluster barrier.
    if (warp == 4 && lane == 0 && !(p.debug_flags & DEBUG_NO_LOADS)) {
        const int y = sg.kv_row0 + t0 * L::BN;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            ptx::tma_prefetch_3d(&tm_q, c * 64, q_row, z_q);
            ptx::tma_prefetch_3d(&tm_k, c * 64, y + 64 * static_cast<int>(rank), z_kv);
        }
#pragma unroll
        for (int c = 0; c < D / 128; ++c)
            ptx::tma_prefetch_3d(&tm_v, static_cast<int>(rank) * (D / 2) + c * 64, y, z_kv);
    }

    if (threadIdx.x == 0) {
        ptx::mbar_init(q_full, 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(slot_full0 + 8u * s, 1);
            ptx::mbar_init(slot_empty0 + 8u * s, 1);
        }
        for (int i = 0; i < NB; ++i) {
            ptx::mbar_init(s_full0 + 8u * i, 1);
            ptx::mbar_init(p_full0 + 8u * i, L::P_ARRIVALS);
            for (int q = 0; q + 1 < L::P_PARTS; ++q)
                ptx::mbar_init(p_part0 + 8u * (NB * q + i), L::P_ARRIVALS);
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
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    // Barriers of both CTAs are initialised before either CTA signals the other.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx cx{abort_flag, p.status, p.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------- TMA producer (both CTAs)
        if (!(p.debug_flags & DEBUG_NO_LOADS)) {  // whole warp; one elected lane issues
            const uint32_t q_full_l = ptx::map_to_rank(q_full, 0);
            if (leader)
                ptx::mbar_arrive_expect_tx_w(q_full, 2 * L::Q_BYTES);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                ptx::tma_load_3d_pair_w(s_q + c * L::Q_BOX_BYTES, &tm_q, q_full_l, c * 64, q_row, z_q);
            int slot = 0;
            uint32_t ph = 0;
            auto next_slot = [&](uint32_t &full_l, uint32_t &dst) -> bool {
                const bool ok = wait_bounded(slot_empty0 + 8u * slot, ph ^ 1u, cx, SITE_SLOT_EMPTY);
                if (!__all_sync(0xffffffffu, ok))
                    return false;
                if (leader)
                    ptx::mbar_arrive_expect_tx_w(slot_full0 + 8u * slot, 2 * L::HALF_BYTES);
                full_l = ptx::map_to_rank(slot_full0 + 8u * slot, 0);
                dst = s_ring + slot * L::HALF_BYTES;
                if (++slot == NS) {
                    slot = 0;
                    ph ^= 1u;
                }
                return true;
            };
            auto load_k = [&](int j) -> bool {  // keys [j*128 + 64*rank, +64), all D columns
                uint32_t full_l, dst;
                if (!next_slot(full_l, dst))
                    return false;
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d_pair_w(dst + c * L::K_BOX_BYTES, &tm_k, full_l, c * 64,
                                          sg.kv_row0 + (t0 + j) * L::BN + 64 * static_cast<int>(rank), z_kv);
                return true;
            };
            auto load_v = [&](int j) -> bool {  // keys [j*128, +128), columns [rank*D/2, +D/2)
                uint32_t full_l, dst;
                if (!next_slot(full_l, dst))
                    return false;
#pragma unroll
                for (int c = 0; c < D / 128; ++c)
                    ptx::tma_load_3d_pair_w(dst + c * L::V_BOX_BYTES, &tm_v, full_l,
                                          static_cast<int>(rank) * (D / 2) + c * 64, sg.kv_row0 + (t0 + j) * L::BN,
                                          z_kv);
                return true;
            };
            bool ok = load_k(0);
            for (int j = 0; ok && j < n; ++j) {
                if (j + 1 < n)
                    ok = load_k(j + 1);
                if (ok)
                    ok = load_v(j);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------- S = Q K^T issuer (leader, 1 thread)
        if (leader) {  // whole warp; one elected lane issues
            const uint64_t dq = ptx::smem_desc_sw128(s_q, 16, 1024);
            const uint64_t dk = ptx::smem_desc_sw128(s_ring, 16, 1024);
            bool issued = false;
            bool ok = __all_sync(0xffffffffu, wait_bounded(q_full, 0, cx, SITE_Q_FULL));
            for (int t = 0; ok && t < n; ++t) {
                // K_t first (it has usually landed), then PV_{t-NB}: the slot wait
                // stays off the PV_{t-NB} -> S_t path.
                const int pos = pos_k<1>(t);
                const int slot = pos % NS;
                if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                    break;
                if (t >= NB) {
                    const int pv = t - NB;
                    ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx,
                                                              SITE_O_DONE));
                    if (!ok)
                        break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + L::TM_S + (t % NB) * L::BN;
                const uint64_t kslot = dk + static_cast<uint64_t>((slot * L::HALF_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t box = kk >> 2, off = (kk & 3) * 32;
                    ptx::mma_ss_pair_w(d_tmem, dq + ((box * L::Q_BOX_BYTES + off) >> 4),
                                     kslot + ((box * L::K_BOX_BYTES + off) >> 4), IDESC_S, kk != 0);
                }
                issued = true;
                ptx::mma_commit_pair_w(slot_empty0 + 8u * slot);
                ptx::mma_commit_pair_w(s_full0 + 8u * (t % NB));
            }
            if (issued) {
                ptx::mma_commit_pair_w(final0);
                wait_drain(final0, 0, p.timeout_ns);
            }
        }
    } else if (warp == 6) {
        // ------------------------------------ O += P V issuer (leader, 1 thread)
        if (leader) {  // whole warp; one elected lane issues
            const uint64_t dv = ptx::smem_desc_sw128(s_ring, L::V_BOX_BYTES, 1024);
            bool issued = false;
            bool ok = true;
            for (int j = 0; ok && j < n; ++j) {
                const int buf = j % NB;
                // V_j first (it has usually landed), then P_j: the slot wait stays
                // off the P_j -> PV_j path.
                const int pos = pos_v<1>(j, n);
                const int slot = pos % NS;
                if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                    break;
                const uint32_t a_tmem = tmem + L::TM_S + buf * L::BN;
                const uint64_t vslot = dv + static_cast<uint64_t>((slot * L::HALF_BYTES) >> 4);
                // each part of P_j's keys (8 / P_PARTS K steps) as soon as it is in tensor memory
#pragma unroll
                for (int h = 0; h < L::P_PARTS; ++h) {
                    const uint32_t bar = h + 1 < L::P_PARTS ? p_part0 + 8u * (NB * h + buf) : p_full0 + 8u * buf;
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar, (j / NB) & 1, cx, SITE_P_FULL))))
                        break;
                    ptx::tc_fence_after();
                    constexpr int KS = 8 / L::P_PARTS;
#pragma unroll
                    for (int kk = KS * h; kk < KS * h + KS; ++kk)
                        ptx::mma_ts_pair_w(tmem + L::TM_O, a_tmem + kk * 8, vslot + ((kk * 2048) >> 4), IDESC_PV,
                                         (j > 0) || (kk > 0));
                    issued = true;
                }
                if (!ok)
                    break;
                ptx::mma_commit_pair_w(slot_empty0 + 8u * slot);
                ptx::mma_commit_pair_w(o_done0 + 8u * (j % O_DONE_RING));
            }
            if (issued) {
                ptx::mma_commit_pair_w(final0 + 8u);
                wait_drain(final0 + 8u, 0, p.timeout_ns);
            }
        }
    } else if (warp < 4) {
        // --------------------------------------- softmax / correction / epilogue
        const int row = threadIdx.x;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t t_s = tmem + lane_off + L::TM_S;
        const uint32_t t_o = tmem + lane_off + L::TM_O;
        const float c = p.c;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;

        for (int j = 0; j < n; ++j) {
            const int buf = j % NB;
            ok = wait_bounded(s_full0 + 8u * buf, (j / NB) & 1, cx, SITE_S_FULL);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
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
            const int valid = (p.causal ? min(sg.skv, q0 + row + 1) : sg.skv) - (t0 + j) * L::BN;
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
            const float m_tile = mx0 * c;
            const float m_new = (j == 0 || m_tile > m_used + RESCALE_THRESHOLD) ? m_tile : m_used;
            const float alpha = (j == 0 || m_new == m_used) ? 1.f : ptx::ex2(m_used - m_new);
            const float neg_m = -m_new;

            // p = 2^(s * c - m), two elements per f32x2 instruction for the scaling
            // and the running sums (each lane rounds exactly as fmaf / + would).
            // P_j is handed over in P_PARTS parts of consecutive keys, so PV_j's first
            // MMAs start while the softmax computes the later parts.
            constexpr int PW = 64 / L::P_PARTS;  // packed 16-bit pairs (32-bit words) per part
            uint32_t pk[64];
            const uint64_t c2 = ptx::f2_pack(c, c), negm2 = ptx::f2_pack(neg_m, neg_m);
            uint64_t sum01 = ptx::f2_pack(0.f, 0.f), sum23 = sum01;
            auto exp_part = [&](auto masked, auto part) {
                constexpr int Q = decltype(part)::value;
#pragma unroll
                for (int i = PW * Q; i < PW * Q + PW; i += 2) {
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
            // exponentials of one part, stored to its columns of S_j's buffer
            auto compute_part = [&](auto part) {
                constexpr int Q = decltype(part)::value;
                if (tail)
                    exp_part(std::true_type{}, part);
                else
                    exp_part(std::false_type{}, part);
                if constexpr (PW == 16) {
                    ptx::tmem_st16(ts + 16 * Q, *reinterpret_cast<uint32_t(*)[16]>(&pk[16 * Q]));
                } else {
#pragma unroll
                    for (int w = 0; w < PW; w += 32)
                        ptx::tmem_st32(ts + PW * Q + w, *reinterpret_cast<uint32_t(*)[32]>(&pk[PW * Q + w]));
                }
                ptx::tmem_wait_st();
            };
            // One arrival per warp on the leader's barrier, after every lane's TMEM writes.
            auto hand_over = [&](uint32_t bar) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        ptx::mbar_arrive(bar);
                    else
                        ptx::mbar_arrive_cluster(ptx::map_to_rank(bar, 0));
                }
            };
            auto part_bar = [&](int q) { return q + 1 < L::P_PARTS ? p_part0 + 8u * (NB * q + buf) : p_full0 + 8u * buf; };
            compute_part(std::integral_constant<int, 0>{});

            // Same lazy-rescale rule and aliasing argument as the single-CTA kernel:
            // S_j completing implies PV_{j-NSBUF} completed. O is rescaled before the
            // first part of P_j is handed over (PV_j starts accumulating then).
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
            hand_over(part_bar(0));
            if constexpr (L::P_PARTS >= 2) {
                compute_part(std::integral_constant<int, 1>{});
                hand_over(part_bar(1));
            }
            if constexpr (L::P_PARTS == 4) {
                compute_part(std::integral_constant<int, 2>{});
                hand_over(part_bar(2));
                compute_part(std::integral_constant<int, 3>{});
                hand_over(part_bar(3));
            }
            float sum0, sum1, sum2, sum3;
            ptx::f2_unpack(sum01, sum0, sum1);
            ptx::f2_unpack(sum23, sum2, sum3);
            const float tile_sum = (sum0 + sum1) + (sum2 + sum3);
            l = (j == 0) ? tile_sum : fmaf(l, alpha, tile_sum);
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
            // o_done of the last PV implies every S MMA (which read both CTAs' Q) completed,
            // so the Q tile can be reused as the O staging tile.
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
                const uint32_t row_addr = s_q + (cc >> 1) * L::Q_BOX_BYTES + row * 128;
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
            for (int c2 = 0; c2 < D / 64; ++c2)
                ptx::tma_store_3d(&tm_o, s_q + c2 * L::Q_BOX_BYTES, c2 * 64, q_row, z_out);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read_all();
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    // After an abort, loads this CTA issued may still be landing (their
    // completions are counted in the leader); give them time before the pair exits.
    if (*abort_flag) {
        for (int i = 0; i < 100; ++i)
            ptx::nanosleep_ns(1000);
    }
    // Neither CTA leaves while the other may still signal its barriers or read
    // its shared or tensor memory.
    ptx::cluster_sync();
    if (warp == 5) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, L::TMEM_COLS);
    }
}

// Units 2c and 2c+1 share (batch, KV head) exactly when the units of one
// (batch, KV head), query tiles x heads per group, are even in number.
// Causal units of one pair must also share the query tile (same tile count):
// with the head-in-group index fastest that holds when G is even.
inline bool use_pair(const KernelParams &p, int grid, int D)
{
    if (p.debug_flags & DEBUG_SINGLE_CTA)
        return false;
    // At D=128 the single-CTA kernel measured as fast or faster (GQA with 4 heads per group: +5 %;
    // MHA: within 2 %): a 128-key tile there is half the tensor work of D=256, the softmax takes
    // the larger share, and the pair's halved K/V traffic per SM buys little.
    if (D == 128 && !(p.debug_flags & DEBUG_PAIR_D128))
        return false;
    // Variable-length batches pair two heads of one group on the same tile (G even), so both CTAs
    // of a pair always see the same sequence and leave together.
    if (p.cu_q != nullptr && (p.G % 2) != 0)
        return false;
    if (p.causal && (p.G % 2) != 0)
        return false;
    return ((p.n_qtiles * p.G) % 2 == 0) && (grid % 2 == 0);
}

template <int D, bool BF16>
cudaError_t launch_sdp_fwd_pair(const CUtensorMap &q, const CUtensorMap &k_half, const CUtensorMap &v,
                                const CUtensorMap &o, const KernelParams &p, int grid, cudaStream_t stream)
{
    static unsigned long long set_dense = 0, set_varlen = 0;
    const bool vl = p.cu_q != nullptr;
    auto kern = vl ? sdp_fwd_pair_kernel<D, BF16, true> : sdp_fwd_pair_kernel<D, BF16, false>;
    cudaError_t e = set_smem_once(kern, PairLayout<D>::SMEM_BYTES, vl ? set_varlen : set_dense);
    if (e != cudaSuccess)
        return e;
    kern<<<grid, NUM_THREADS, PairLayout<D>::SMEM_BYTES, stream>>>(q, k_half, v, o, p);
    return cudaGetLastError();
}

}  // namespace sdp
