// Grouped-query attention forward at head dim 128: two query tiles per CTA on a
// CTA pair (cta_group::2), sm_103a.
//
// At D=128 a 128-key tile is 1024 tensor cycles per SM, and the one-warp-per-
// sub-partition softmax of the single-CTA kernel needs more than that per tile
// (row maximum, 128 exponentials, P store and hand-off per row). Here every CTA
// holds two 128-row query tiles, A and B, each with its own softmax warpgroup,
// so two independent softmax warps share each sub-partition, and the pair of
// CTAs splits every K/V tile (each SM receives and feeds half of it).
//
// Softmax warps 0-3 own tile A's rows, warps 4-7 tile B's (warp w reads TMEM
// lanes 32 (w mod 4) + [0, 32)); warp 8 loads (TMA), warp 9 issues tile A's
// MMAs and owns the tensor memory, warp 10 issues tile B's (leader CTA only),
// warp 11 idles (twelve warps: three per sub-partition, 168 registers each).
//
// Keys are taken in steps of 64 (half a 128-key tile), so that each tile gets
// two score buffers in the 512 tensor-memory columns:
//   [0,128) O_A   [128,256) O_B   [256,320) S_A0  [320,384) S_A1
//   [384,448) S_B0  [448,512) S_B1
// S_X(s) = Q_X K_s^T (M=256 over both CTAs, N=64 keys) goes to buffer s mod 2.
// The softmax of step s loads S(s+1) into registers before it stores P(s), and
// stores P(s) (64 keys as 16-bit pairs, 32 columns) into the upper half of
// buffer (s+1) mod 2, whose scores it has just read; only the last step's P
// goes to the lower half of its own buffer. Buffer s mod 2 is then free as soon
// as step s's scores are in registers, except for P(s-1) in its upper half, so
// S(s+2) waits only for PV(s-1) (and, for S(2), for P(0)). The chain
// S -> softmax -> PV -> S spans three steps instead of one, and the two tiles'
// MMAs fill each other's gaps on the tensor pipe.
//
// K is loaded so that each CTA holds, per 128-key tile, keys 32r + [0, 32) of
// each 64-key half (r = CTA rank): one N=64 MMA reads the half's keys from both
// CTAs. V is split by columns as in the one-tile pair kernel.
//
// Serves dense, non-causal launches at D=128 (not variable-length batches)
// whose (batch, KV head) groups hold an even number of two-tile units and that
// fill at least one wave of CTAs. The online softmax runs over 64-key steps, so the
// result rounds differently from the 128-key kernels (same function, within the
// same tolerances), and the lazy rescale threshold applies per step.
#pragma once

#include "sdp_fwd_pair.cuh"

namespace sdp {

constexpr int DEBUG_NO_PAIR2 = 64;      // never the two-tile pair kernel at D=128
constexpr int DEBUG_FORCE_PAIR2 = 128;  // the two-tile pair kernel wherever its units pair, even below one wave
// Whether dense D=128 launches that fill a wave take this kernel by default. Off while
// it measures slower than the single-CTA kernel on the D=128 workloads in alternating runs
// (-4.7 % on 4 heads per group at 8192 keys, -1.2 % on MHA at 16384); flag 128 selects it.
constexpr bool PAIR2_BY_DEFAULT = false;

struct Pair2Layout {
    static constexpr int D = 128;
    static constexpr int BM = 128;                    // query rows per tile (two tiles per CTA)
    static constexpr int BN = 128;                    // keys per K/V tile (both CTAs)
    static constexpr int STEP = 64;                   // keys per softmax step
    static constexpr int THREADS = 384;               // 8 softmax warps, producer, two issuers, one idle
    static constexpr int Q_BOX_BYTES = 128 * 128;     // 128 rows x 64 columns
    static constexpr int QT_BYTES = BM * D * 2;       // one query tile
    static constexpr int K_BOX_BYTES = 64 * 128;      // this CTA's 64 keys of a tile x 64 columns
    static constexpr int K_HALF_OFF = 32 * 128;       // rows of the tile's second 64-key half
    static constexpr int HALF_BYTES = 64 * D * 2;     // this CTA's half of a K tile = half of a V tile
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int BAR_AREA = 512;
    static constexpr int NSLOTS = (SMEM_LIMIT - BAR_AREA - 1024 - 2 * QT_BYTES) / HALF_BYTES;
    static constexpr int P_ARRIVALS = 8;              // 4 softmax warps of a tile in each CTA
    static constexpr int PV_RING = 4;                 // PV completion barriers per tile
    // q_full[2], slot_full[NS], slot_empty[NS], s_full[2][2], p_full[2][2], p_last[2],
    // o_done[2][PV_RING], final[2]
    static constexpr int NBARS = 2 + 2 * NSLOTS + 4 + 4 + 2 + 2 * PV_RING + 2;
    static constexpr int BAR_OFF = 2 * QT_BYTES + NSLOTS * HALF_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFF + BAR_AREA + 1024;
    static constexpr int TM_O = 0;                    // O_X at TM_O + 128 X
    static constexpr int TM_S = 256;                  // S_X buffer b at TM_S + 128 X + 64 b
    static constexpr int TMEM_COLS = 512;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
    static_assert(8 * NBARS + 8 <= BAR_AREA, "barrier area");
    // Each issuer waits for every K and V chunk in the order 0, 2, 1, 3, 4, 5, ...
    // (K_0, V_0, K_1, K_2, V_1, ...): when it waits for position P it has already seen
    // every position up to P - 2 land, so the chunk NSLOTS before P has landed and
    // the slot's parity cannot alias.
    static_assert(NSLOTS >= 3, "ring parity soundness");
};

__device__ __forceinline__ uint32_t pair2_s_col(int x, int b) { return Pair2Layout::TM_S + 128u * x + 64u * b; }

// Tensor-memory column of P(s) of tile x: the upper half of the next buffer,
// or, for the last step, the lower half of its own.
__device__ __forceinline__ uint32_t pair2_p_col(int x, int s, int n)
{
    return s + 1 < n ? pair2_s_col(x, (s + 1) & 1) + 32u : pair2_s_col(x, s & 1);
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Pair2Layout::THREADS, 1)
    sdp_fwd_pair2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k32,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const KernelParams p)
{
    using L = Pair2Layout;
    constexpr int D = L::D;
    constexpr int NS = L::NSLOTS;
    constexpr int RING = L::PV_RING;
    constexpr uint32_t IDESC_S = ptx::idesc_f16_f32acc(256, L::STEP, BF16, false);  // Q x K step, both K-major
    constexpr uint32_t IDESC_PV = ptx::idesc_f16_f32acc(256, D, BF16, true);        // P (TMEM) x V half (N-major)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t s_q0 = sbase;  // Q_A, then Q_B; each reused as its tile's O staging
    const uint32_t s_ring = sbase + 2 * L::QT_BYTES;
    const uint32_t bar0 = sbase + L::BAR_OFF;
    const uint32_t q_full0 = bar0;                         // + 8 x
    const uint32_t slot_full0 = bar0 + 16u;
    const uint32_t slot_empty0 = slot_full0 + 8u * NS;
    const uint32_t s_full0 = slot_empty0 + 8u * NS;        // + 8 (2 x + b)
    const uint32_t p_full0 = s_full0 + 32u;                // + 8 (2 x + b): P of steps before the last
    const uint32_t p_last0 = p_full0 + 32u;                // + 8 x: P of the last step
    const uint32_t o_done0 = p_last0 + 16u;                // + 8 (RING x + s % RING)
    const uint32_t final0 = o_done0 + 8u * (2 * RING);     // + 8 x: issuer x drained
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * L::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank == 0);

    // Unit = (batch, query head, pair of 128-row query tiles): head-in-group fastest,
    // then the tile pair, then (batch, KV head); the KV split (split-KV launches) is
    // the outermost coordinate. Both CTAs of a cluster share (batch, KV head) and split.
    int u = blockIdx.x;
    const int units_per_split = static_cast<int>(gridDim.x) / p.kv_splits;
    const int split = u / units_per_split;
    u -= split * units_per_split;
    const int hi = u % p.G;
    u /= p.G;
    const int n_qpairs = (p.n_qtiles + 1) / 2;
    const int qp = u % n_qpairs;
    const int bg = u / n_qpairs;
    const int b = bg / p.Hkv;
    const int g = bg - b * p.Hkv;
    const int z_q = b * p.Hq + g * p.G + hi;
    const int z_kv = bg;
    const int q0 = qp * 2 * L::BM;  // first row of tile A; tile B starts 128 rows later
    const int t0 = split * p.tiles_per_split;
    const int n_tiles = min(p.n_kvtiles - t0, p.tiles_per_split);    // K/V tiles this unit reads (>= 1)
    const int keys = min(p.Skv - t0 * L::BN, n_tiles * L::BN);      // keys this unit reads
    const int n = (keys + L::STEP - 1) / L::STEP;                    // 64-key steps
    const int z_out = split * p.planes_q + z_q;

    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            ptx::mbar_init(q_full0 + 8u * x, 1);
            ptx::mbar_init(p_last0 + 8u * x, L::P_ARRIVALS);
            ptx::mbar_init(final0 + 8u * x, 1);
            for (int bb = 0; bb < 2; ++bb) {
                ptx::mbar_init(s_full0 + 8u * (2 * x + bb), 1);
                ptx::mbar_init(p_full0 + 8u * (2 * x + bb), L::P_ARRIVALS);
            }
            for (int i = 0; i < RING; ++i)
                ptx::mbar_init(o_done0 + 8u * (RING * x + i), 1);
        }
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(slot_full0 + 8u * s, 1);
            ptx::mbar_init(slot_empty0 + 8u * s, 2);  // one commit from each tile's issuer
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 8 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k32);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
    }
    if (warp == 9) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    // Barriers of both CTAs are initialised before either CTA signals the other.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx cx{abort_flag, p.status, p.timeout_ns};

    if (warp == 8) {
        // ------------------------------------------------- TMA producer (both CTAs)
        if (!(p.debug_flags & DEBUG_NO_LOADS)) {  // whole warp; one elected lane issues
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (leader)
                    ptx::mbar_arrive_expect_tx_w(q_full0 + 8u * x, 2 * L::QT_BYTES);
                const uint32_t qf_l = ptx::map_to_rank(q_full0 + 8u * x, 0);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d_pair_w(s_q0 + x * L::QT_BYTES + c * L::Q_BOX_BYTES, &tm_q, qf_l, c * 64,
                                            q0 + x * L::BM, z_q);
            }
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
            // K tile j: keys 64 h + 32 rank + [0, 32) of each half h, all D columns
            auto load_k = [&](int j) -> bool {
                uint32_t full_l, dst;
                if (!next_slot(full_l, dst))
                    return false;
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        ptx::tma_load_3d_pair_w(dst + c * L::K_BOX_BYTES + h * L::K_HALF_OFF, &tm_k32, full_l, c * 64,
                                                (t0 + j) * L::BN + 64 * h + 32 * static_cast<int>(rank), z_kv);
                return true;
            };
            // V tile j: all 128 keys, columns [64 rank, 64 rank + 64)
            auto load_v = [&](int j) -> bool {
                uint32_t full_l, dst;
                if (!next_slot(full_l, dst))
                    return false;
                ptx::tma_load_3d_pair_w(dst, &tm_v, full_l, static_cast<int>(rank) * 64, (t0 + j) * L::BN, z_kv);
                return true;
            };
            bool ok = load_k(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles)
                    ok = load_k(j + 1);
                if (ok)
                    ok = load_v(j);
            }
        }
    } else if (warp == 9 || warp == 10) {
        // ----------------------------- MMA issuer of tile x (leader; whole warp, one lane issues)
        const int x = warp - 9;
        if (leader) {
            const uint64_t dq = ptx::smem_desc_sw128(s_q0 + x * L::QT_BYTES, 16, 1024);
            const uint64_t dk = ptx::smem_desc_sw128(s_ring, 16, 1024);
            const uint64_t dv = ptx::smem_desc_sw128(s_ring, L::HALF_BYTES, 1024);
            bool issued = false;
            // Ring slots are waited for ahead of use, while the issuer would otherwise wait for
            // the next P: a barrier round trip costs ~200 cycles under tensor load even when the
            // chunk has landed, and here it stays off the P -> PV -> S chain. Slots are waited in
            // the order K_0, V_0, K_1, K_2, V_1, K_3, V_2, ...: positions 0, 2, 1, 3, 4, 5, 6, ...
            auto wait_slot = [&](int pos) -> bool {
                return __all_sync(0xffffffffu,
                                  wait_bounded(slot_full0 + 8u * (pos % NS), (pos / NS) & 1, cx, SITE_SLOT_FULL));
            };
            // S_x(t): buffer t mod 2; K tile t / 2 (its slot waited for), this half's 32 keys in each CTA.
            auto issue_s = [&](int t) {
                const int j = t >> 1, h = t & 1;
                const int slot = pos_k<1>(j) % NS;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + pair2_s_col(x, t & 1);
                const uint64_t kslot = dk + static_cast<uint64_t>((slot * L::HALF_BYTES + h * L::K_HALF_OFF) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t box = kk >> 2, off = (kk & 3) * 32;
                    ptx::mma_ss_pair_w(d_tmem, dq + ((box * L::Q_BOX_BYTES + off) >> 4),
                                       kslot + ((box * L::K_BOX_BYTES + off) >> 4), IDESC_S, kk != 0);
                }
                issued = true;
                ptx::mma_commit_pair_w(s_full0 + 8u * (2 * x + (t & 1)));
                if (h == 1 || t == n - 1)
                    ptx::mma_commit_pair_w(slot_empty0 + 8u * slot);  // this tile's last read of K_j
            };
            // O_x += P_x(s) V: V tile s / 2 (its slot waited for), keys 64 (s mod 2) + [0, 64) in K steps of 16.
            auto issue_pv = [&](int s) -> bool {
                const int j = s >> 1, h = s & 1;
                const int slot = pos_v<1>(j, n_tiles) % NS;
                const uint32_t pbar = s + 1 < n ? p_full0 + 8u * (2 * x + (s & 1)) : p_last0 + 8u * x;
                const uint32_t ppar = s + 1 < n ? static_cast<uint32_t>((s >> 1) & 1) : 0u;
                if (!__all_sync(0xffffffffu, wait_bounded(pbar, ppar, cx, SITE_P_FULL)))
                    return false;
                ptx::tc_fence_after();
                const uint32_t a_tmem = tmem + pair2_p_col(x, s, n);
                const uint64_t vslot = dv + static_cast<uint64_t>((slot * L::HALF_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < L::STEP / 16; ++kk)
                    ptx::mma_ts_pair_w(tmem + L::TM_O + 128u * x, a_tmem + kk * 8,
                                       vslot + ((((4 * h + kk) * 2048)) >> 4), IDESC_PV, (s > 0) || (kk > 0));
                issued = true;
                ptx::mma_commit_pair_w(o_done0 + 8u * (RING * x + s % RING));
                if (h == 1 || s == n - 1)
                    ptx::mma_commit_pair_w(slot_empty0 + 8u * slot);  // this tile's last read of V_j
                return true;
            };
            bool ok = __all_sync(0xffffffffu, wait_bounded(q_full0 + 8u * x, 0, cx, SITE_Q_FULL)) && wait_slot(0);
            if (ok) {
                issue_s(0);
                if (n > 1)
                    issue_s(1);
                ok = wait_slot(pos_v<1>(0, n_tiles)) && (n <= 2 || wait_slot(pos_k<1>(1)));  // V_0; K_1 for S(2), S(3)
            }
            for (int s = 0; ok && s < n; ++s) {
                if (!(ok = issue_pv(s)))
                    break;
                // S(2) overwrites S(0)'s buffer, whose scores the softmax read before P(0).
                if (s == 0 && n > 2)
                    issue_s(2);
                // S(s+3) overwrites buffer (s+1) mod 2: S(s+1) (read before P(s) was stored)
                // and P(s) in its upper half, which PV(s) must have consumed.
                if (s + 3 < n) {
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (RING * x + s % RING),
                                                                    (s / RING) & 1, cx, SITE_O_DONE))))
                        break;
                    issue_s(s + 3);
                }
                // the slots of the next PV and the S after it, while P(s+1) is being computed
                if (s + 1 < n && ((s + 1) & 1) == 0 && !(ok = wait_slot(pos_v<1>((s + 1) >> 1, n_tiles))))
                    break;
                if (s + 4 < n && ((s + 4) & 1) == 0 && !(ok = wait_slot(pos_k<1>((s + 4) >> 1))))
                    break;
            }
            if (issued) {  // all of this thread's MMAs complete before TMEM is freed
                ptx::mma_commit_pair_w(final0 + 8u * x);
                wait_drain(final0 + 8u * x, 0, p.timeout_ns);
            }
        }
    } else if (warp < 8) {
        // ---------------------------- softmax / correction / epilogue of tile x (warps 0-7)
        const int x = warp >> 2;
        const int w4 = warp & 3;
        const int row = w4 * 32 + lane;  // row within tile x = TMEM lane
        const uint32_t t_base = tmem + (static_cast<uint32_t>(w4 * 32) << 16);
        const uint32_t t_o = t_base + L::TM_O + 128u * x;
        const float c = p.c;
        float m_used = -INFINITY, l = 0.f;
        float sc[L::STEP];  // scores of the current step
        auto load_scores = [&](int s) -> bool {
            const bool ok = __all_sync(0xffffffffu, wait_bounded(s_full0 + 8u * (2 * x + (s & 1)), (s >> 1) & 1, cx,
                                                                 SITE_S_FULL));
            if (!ok)
                return false;
            ptx::tc_fence_after();
            uint32_t sr[L::STEP];
            const uint32_t ts = t_base + pair2_s_col(x, s & 1);
            ptx::tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
            ptx::tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < L::STEP; ++i)
                sc[i] = __uint_as_float(sr[i]);
            return true;
        };
        bool ok = load_scores(0);
        for (int s = 0; ok && s < n; ++s) {
            // keys of this step (the same for every row: no causal mask here)
            const int valid = keys - s * L::STEP;
            const bool tail = valid < L::STEP;
            if (tail) {
#pragma unroll
                for (int i = 1; i < L::STEP; ++i)
                    if (i >= valid)
                        sc[i] = sc[0];  // neutral for the max; weights zeroed below
            }
            // Row extreme of the raw scores (maximum of s * c: of s when c >= 0, else its minimum).
            float mx0 = sc[0], mx1 = sc[1], mx2 = sc[2], mx3 = sc[3];
            if (c >= 0.f) {
#pragma unroll
                for (int i = 4; i < 60; i += 8) {
                    mx0 = ptx::max3(mx0, sc[i], sc[i + 1]);
                    mx1 = ptx::max3(mx1, sc[i + 2], sc[i + 3]);
                    mx2 = ptx::max3(mx2, sc[i + 4], sc[i + 5]);
                    mx3 = ptx::max3(mx3, sc[i + 6], sc[i + 7]);
                }
                mx0 = ptx::max3(mx0, sc[60], sc[61]);
                mx1 = ptx::max3(mx1, sc[62], sc[63]);
                mx0 = ptx::max3(mx0, mx1, fmaxf(mx2, mx3));
            } else {
#pragma unroll
                for (int i = 4; i < 60; i += 8) {
                    mx0 = ptx::min3(mx0, sc[i], sc[i + 1]);
                    mx1 = ptx::min3(mx1, sc[i + 2], sc[i + 3]);
                    mx2 = ptx::min3(mx2, sc[i + 4], sc[i + 5]);
                    mx3 = ptx::min3(mx3, sc[i + 6], sc[i + 7]);
                }
                mx0 = ptx::min3(mx0, sc[60], sc[61]);
                mx1 = ptx::min3(mx1, sc[62], sc[63]);
                mx0 = ptx::min3(mx0, mx1, fminf(mx2, mx3));
            }
            const float m_tile = mx0 * c;
            const float m_new = (s == 0 || m_tile > m_used + RESCALE_THRESHOLD) ? m_tile : m_used;
            const float alpha = (s == 0 || m_new == m_used) ? 1.f : ptx::ex2(m_used - m_new);
            const float neg_m = -m_new;

            // p = 2^(s * c - m): scaling and running sums two elements per f32x2 instruction
            uint32_t pk[L::STEP / 2];
            const uint64_t c2 = ptx::f2_pack(c, c), negm2 = ptx::f2_pack(neg_m, neg_m);
            uint64_t sum01 = ptx::f2_pack(0.f, 0.f), sum23 = sum01;
            auto exp_step = [&](auto masked) {
#pragma unroll
                for (int i = 0; i < L::STEP / 2; i += 2) {
                    float x0, x1, x2, x3;
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sc[2 * i], sc[2 * i + 1]), c2, negm2), x0, x1);
                    ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sc[2 * i + 2], sc[2 * i + 3]), c2, negm2), x2, x3);
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
                exp_step(std::true_type{});
            else
                exp_step(std::false_type{});

            // The next step's scores come out of buffer (s+1) mod 2 before P(s) goes into its upper half.
            if (s + 1 < n && !(ok = load_scores(s + 1)))
                break;
            ptx::tmem_st32(t_base + pair2_p_col(x, s, n), *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            ptx::tmem_wait_st();
            // O_x is rescaled before P(s) is handed over (PV(s) accumulates on it), after P(s)
            // is stored (fewer registers live); only
            // warps where some row's maximum moved wait for PV(s-1). Aliasing: S(s) being
            // complete implies PV(s-3) completed, and PV(s+1) cannot start before P(s+1).
            if (s > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const int pv = s - 1;
                ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (RING * x + pv % RING), (pv / RING) & 1, cx,
                                                          SITE_O_DONE));
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
            // one arrival per warp on the leader's barrier, after every lane's tensor-memory writes
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                const uint32_t bar = s + 1 < n ? p_full0 + 8u * (2 * x + (s & 1)) : p_last0 + 8u * x;
                if (leader)
                    ptx::mbar_arrive(bar);
                else
                    ptx::mbar_arrive_cluster(ptx::map_to_rank(bar, 0));
            }
            float sum0, sum1, sum2, sum3;
            ptx::f2_unpack(sum01, sum0, sum1);
            ptx::f2_unpack(sum23, sum2, sum3);
            const float step_sum = (sum0 + sum1) + (sum2 + sum3);
            l = (s == 0) ? step_sum : fmaf(l, alpha, step_sum);
            m_used = m_new;
        }

        // ------------------------------------------------------------ epilogue of tile x
        const int tile_row0 = q0 + x * L::BM;  // first row of tile x in its plane
        const uint32_t s_stage = s_q0 + x * L::QT_BYTES;
        ptx::named_bar_sync(1 + x, 128);
        ok = ok && !*abort_flag;
        if (ok) {
            const int pv = n - 1;
            ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (RING * x + pv % RING), (pv / RING) & 1, cx,
                                                      SITE_O_DONE));
        }
        if (ok) {
            // PV_x(n-1) complete implies every S_x MMA (which read both CTAs' Q_x) completed,
            // so Q_x's shared memory can hold the O staging tile.
            ptx::tc_fence_after();
            // two chunks per wait: 384 threads leave at most 168 registers a thread
            drain_o_row<D, BF16, 2>(t_o, 1.f / l, [&](int cc, const uint32_t (&pk)[16]) {
                // 32 columns = four 16-byte units of row `row` in box cc/2, 128-byte swizzled
                const uint32_t row_addr = s_stage + (cc >> 1) * L::Q_BOX_BYTES + row * 128;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint32_t unit = static_cast<uint32_t>((cc & 1) * 4 + v);
                    st_shared_v4(row_addr + ((unit ^ static_cast<uint32_t>(row & 7)) << 4), pk[4 * v], pk[4 * v + 1],
                                 pk[4 * v + 2], pk[4 * v + 3]);
                }
            });
            if (p.lse != nullptr && tile_row0 + row < p.Sq)
                p.lse[static_cast<size_t>(z_out) * p.Sq + tile_row0 + row] = (m_used + ptx::lg2(l)) * LN2;
            ptx::fence_proxy_async_smem();
        }
        ptx::named_bar_sync(1 + x, 128);
        // one thread per tile stores it (rows past Sq are clipped; a tile wholly past Sq is skipped)
        if (w4 == 0 && lane == 0 && !*abort_flag && tile_row0 < p.Sq) {
#pragma unroll
            for (int c2 = 0; c2 < D / 64; ++c2)
                ptx::tma_store_3d(&tm_o, s_stage + c2 * L::Q_BOX_BYTES, c2 * 64, tile_row0, z_out);
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
    if (warp == 9) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, L::TMEM_COLS);
    }
}

// The two-tile pair kernel serves dense, non-causal launches at D=128 (not variable-
// length batches) whose clusters pair two-tile units of one (batch, KV head) and
// split (their count per split even) and that give at least one CTA per SM.
inline bool use_pair2(const KernelParams &p, int grid)
{
    if (p.debug_flags & (DEBUG_SINGLE_CTA | DEBUG_NO_PAIR2))
        return false;
    if (p.causal || p.cu_q != nullptr || p.num_sms <= 0)
        return false;
    const long long n_qpairs = (p.n_qtiles + 1) / 2;
    const long long per_split = static_cast<long long>(p.planes_q) * n_qpairs;
    const bool forced = (p.debug_flags & DEBUG_FORCE_PAIR2) != 0;
    if (!forced && !PAIR2_BY_DEFAULT)
        return false;
    const bool fills = per_split * p.kv_splits >= p.num_sms || forced;
    return (n_qpairs * p.G) % 2 == 0 && fills &&
           static_cast<long long>(grid) == static_cast<long long>(p.planes_q) * p.n_qtiles * p.kv_splits;
}

template <bool BF16>
cudaError_t launch_sdp_fwd_pair2(const CUtensorMap &q, const CUtensorMap &k32, const CUtensorMap &v,
                                 const CUtensorMap &o, const KernelParams &p, cudaStream_t stream)
{
    static unsigned long long set = 0;
    auto kern = sdp_fwd_pair2_kernel<BF16>;
    cudaError_t e = set_smem_once(kern, Pair2Layout::SMEM_BYTES, set);
    if (e != cudaSuccess)
        return e;
    const long long grid = static_cast<long long>(p.planes_q) * ((p.n_qtiles + 1) / 2) * p.kv_splits;
    kern<<<static_cast<unsigned>(grid), Pair2Layout::THREADS, Pair2Layout::SMEM_BYTES, stream>>>(q, k32, v, o, p);
    return cudaGetLastError();
}

}  // namespace sdp
