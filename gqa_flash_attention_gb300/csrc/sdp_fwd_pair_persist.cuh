// Persistent form of the CTA-pair kernel, for unsplit launches: one cluster
// per SM pair loops over unit pairs. Without the causal mask every unit
// reads all KV tiles and cluster c takes unit pairs c, c + C, c + 2C, ...
// (C clusters). With it, unit pairs run longest first (query tile descending,
// then batch and KV head, then the heads of a group) and round r of the walk
// assigns its C pairs in forward order when r is even and in reverse order when
// r is odd, so that the few tiles by which consecutive pairs shrink within a
// round even out over the rounds: every cluster ends within about one round's
// length difference of the others, with no scheduler state on the device.
//
// The per-tile protocol is the pair kernel's (see sdp_fwd_pair.cuh); what
// changes is that nothing is set up or torn down per unit, and the next unit
// starts while the current one ends:
//   - every tile and ring counter is global across a cluster's units (barrier
//     phases carry over; K/V ring positions continue, so the ring's parity
//     argument holds across unit boundaries with NSLOTS >= 4);
//   - q_free (the S issuer's commit after a unit's last S MMA, multicast)
//     lets the producer load the next unit's Q while the current unit's last
//     softmax, PVs and epilogue run, and the S issuer then computes the next
//     unit's first scores;
//   - o_free (one arrival per softmax warp of both CTAs once the epilogue has
//     read O out of tensor memory) lets the PV issuer start the next unit's
//     first PV, which overwrites O;
//   - O is written from registers straight to global memory (Q's shared
//     memory is the next unit's, so it cannot stage O).
#pragma once

#include "sdp_fwd_pair.cuh"

namespace sdp {

template <int D, bool BF16, bool VARLEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    sdp_fwd_pair_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                   const __grid_constant__ CUtensorMap tm_v, const KernelParams p)
{
    using L = PairLayout<D>;
    constexpr int NS = L::NSLOTS;
    constexpr int NB = L::NSBUF;
    constexpr int NBARS = L::NBARS + 2;  // + q_free, o_free
    static_assert(8 * NBARS + 8 <= L::BAR_AREA, "barrier area");
    constexpr uint32_t IDESC_S = ptx::idesc_f16_f32acc(256, L::BN, BF16, false);
    constexpr uint32_t IDESC_PV = ptx::idesc_f16_f32acc(256, D, BF16, true);

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
    const uint32_t p_part0 = final0 + 16u;
    const uint32_t q_free = p_part0 + 8u * (NB * (L::P_PARTS - 1));  // this unit's S MMAs read Q for the last time
    const uint32_t o_free = q_free + 8u;                             // (leader) the epilogue has read O
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::BAR_OFF + 8 * NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank == 0);

    // Unit pairs: without the causal mask as in the pair kernel (head-in-group
    // fastest, then query tile, then (batch, KV head)); with it, query tile
    // descending outermost, then (batch, KV head), then head-in-group, so that the
    // walk below takes them longest first (a causal unit of query tile qt reads
    // qt + 1 KV tiles). Variable-length batches take the units of the per-unit
    // grid in the same order, from the compact list of tiles that exist when the
    // launch has one (sequence order without the mask, level order with it); the
    // walk alternates direction there too, since sequences differ in length. Both
    // units of a pair share the query tile (the group size is even), the
    // sequence and so the tile count.
    const int n_pairs = p.units / 2;
    const int n_clusters = static_cast<int>(gridDim.x) / 2;
    const int cid = static_cast<int>(blockIdx.x) / 2;
    // Causal launches with few query heads per KV head (below 8) walk items of two
    // units of one head each: query tiles qt and n_qtiles - 1 - qt, n_qtiles + 1 KV
    // tiles together, so every item costs the same and a static walk balances; items
    // are ordered (batch, KV head) outermost, so the units in flight share their K/V
    // in L2 (taken longest first across KV heads instead, units in flight would read
    // as many different K/V as there are units: MHA causal ran 30 % slower that way).
    // Causal launches with 8 or more query heads per KV head, where the units of one
    // query tile already share each K/V many times over, and causal variable-length
    // batches, take their units longest first (query tile descending outermost; level
    // order), walked in alternating directions per round; the rest walk units c,
    // c + C, c + 2C, ...
    const bool items = p.causal != 0 && !VARLEN && p.G < 8;
    const bool snake = p.causal != 0 && !items;
    const int n_qpair = (p.n_qtiles + 1) / 2;                       // items per head (group)
    const int n_items = items ? p.planes_q / 2 * n_qpair : 0;  // pairs of heads of a group x items per head
    int n_it;
    if (items) {
        n_it = cid < n_items ? 2 * ((n_items - cid + n_clusters - 1) / n_clusters) : 0;
    } else if (!snake) {
        n_it = cid < n_pairs ? (n_pairs - cid + n_clusters - 1) / n_clusters : 0;
    } else {
        const int full = n_pairs / n_clusters, rem = n_pairs % n_clusters;
        const bool in_last = rem > 0 && ((full & 1) == 0 ? cid < rem : cid >= n_clusters - rem);
        n_it = full + (in_last ? 1 : 0);
    }
    // A unit's geometry: Q/O plane and K/V plane, its first query row within its
    // sequence (q0) and in the row coordinate of Q and O (q_row), the first K/V
    // row, the sequence's rows and keys, and the KV tiles it reads. n = 0: nothing
    // to compute (a slot past the last tile, or (zero) a sequence without keys,
    // whose rows get O = 0 and LSE = -inf, or (bad) invalid sequence offsets).
    struct Unit {
        int z_q, z_kv, q0, q_row, kv_row0, sq, skv, n;
        bool zero, bad;
    };
    auto unit_of = [&](int it) {
        Unit r{};
        int hi, qt, bg;
        if (items) {
            // item (batch x KV head, pair of query tiles, heads): first the longer unit, then its complement
            int i = (it >> 1) * n_clusters + cid;
            hi = 2 * (i % (p.G / 2)) + static_cast<int>(rank);
            i /= p.G / 2;
            const int pp = i % n_qpair;
            bg = i / n_qpair;
            qt = (it & 1) == 0 ? p.n_qtiles - 1 - pp : pp;
            if ((it & 1) == 1 && pp == p.n_qtiles - 1 - pp)
                return r;  // the middle query tile of an odd count forms an item alone
        } else {
            const int pos = (snake && (it & 1)) ? n_clusters - 1 - cid : cid;
            int u = 2 * (it * n_clusters + pos) + static_cast<int>(rank);
            hi = u % p.G;
            u /= p.G;
            if constexpr (VARLEN) {
                if (p.n_tiles > 0 && (u = varlen_compact_unit(p, u)) < 0)
                    return r;  // a slot past the last query tile
            }
            if (p.causal) {
                const int n_bg = VARLEN ? p.nseq * p.Hkv : p.planes_q / p.G;  // sequences (batch) x KV heads
                bg = u % n_bg;
                qt = p.n_qtiles - 1 - u / n_bg;
            } else {
                qt = u % p.n_qtiles;
                bg = u / p.n_qtiles;
            }
        }
        const int b = bg / p.Hkv;
        const int g = bg - b * p.Hkv;
        r.z_q = VARLEN ? g * p.G + hi : b * p.Hq + g * p.G + hi;
        r.z_kv = VARLEN ? g : bg;
        r.q0 = qt * L::BM;
        const SeqGeom sg = seq_geom(p, b);
        if (!sg.ok) {
            r.bad = true;
            return r;
        }
        if (r.q0 >= sg.sq)
            return r;  // a tile past the end of a shorter sequence
        r.q_row = sg.q_row0 + r.q0;
        r.kv_row0 = sg.kv_row0;
        r.sq = sg.sq;
        r.skv = sg.skv;
        const int n_kv = (sg.skv + L::BN - 1) / L::BN;
        r.n = p.causal ? min(n_kv, qt + 1) : n_kv;
        r.zero = r.n == 0;
        return r;
    };
    if (n_it == 0)
        return;  // uniform across the cluster: both CTAs have the same cid

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
        ptx::mbar_init(q_free, 1);
        ptx::mbar_init(o_free, L::P_ARRIVALS);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 5) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), L::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const WaitCtx cx{abort_flag, p.status, p.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------- TMA producer (both CTAs)
        if (!(p.debug_flags & DEBUG_NO_LOADS)) {  // whole warp; one elected lane issues
            const uint32_t q_full_l = ptx::map_to_rank(q_full, 0);
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
            bool ok = true;
            for (int it = 0, k = 0; ok && it < n_it; ++it) {  // k: units with work so far
                const Unit un = unit_of(it);
                if (un.n == 0)
                    continue;
                auto load_k = [&](int j) -> bool {  // keys [j*128 + 64*rank, +64), all D columns
                    uint32_t full_l, dst;
                    if (!next_slot(full_l, dst))
                        return false;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        ptx::tma_load_3d_pair_w(dst + c * L::K_BOX_BYTES, &tm_k, full_l, c * 64,
                                              un.kv_row0 + j * L::BN + 64 * static_cast<int>(rank), un.z_kv);
                    return true;
                };
                auto load_v = [&](int j) -> bool {  // keys [j*128, +128), columns [rank*D/2, +D/2)
                    uint32_t full_l, dst;
                    if (!next_slot(full_l, dst))
                        return false;
#pragma unroll
                    for (int c = 0; c < D / 128; ++c)
                        ptx::tma_load_3d_pair_w(dst + c * L::V_BOX_BYTES, &tm_v, full_l,
                                              static_cast<int>(rank) * (D / 2) + c * 64, un.kv_row0 + j * L::BN,
                                              un.z_kv);
                    return true;
                };
                // Q of this unit once the previous unit's last S MMA has read its Q
                if (k > 0 && !(ok = __all_sync(0xffffffffu, wait_bounded(q_free, (k - 1) & 1, cx, SITE_Q_FULL))))
                    break;
                ++k;
                if (leader)
                    ptx::mbar_arrive_expect_tx_w(q_full, 2 * L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_3d_pair_w(s_q + c * L::Q_BOX_BYTES, &tm_q, q_full_l, c * 64, un.q_row, un.z_q);
                const int n = un.n;
                ok = load_k(0);
                for (int j = 0; ok && j < n; ++j) {
                    if (j + 1 < n)
                        ok = load_k(j + 1);
                    if (ok)
                        ok = load_v(j);
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------- S = Q K^T issuer (leader, 1 thread)
        if (leader) {  // whole warp; one elected lane issues
            const uint64_t dq = ptx::smem_desc_sw128(s_q, 16, 1024);
            const uint64_t dk = ptx::smem_desc_sw128(s_ring, 16, 1024);
            bool issued = false;
            bool ok = true;
            int g0 = 0, pos0 = 0;  // tiles and ring chunks of the earlier units
            for (int it = 0, k = 0; ok && it < n_it; ++it) {
                const int n = unit_of(it).n;
                if (n == 0)
                    continue;
                if (!(ok = __all_sync(0xffffffffu, wait_bounded(q_full, k & 1, cx, SITE_Q_FULL))))
                    break;
                ++k;
                for (int t = 0; ok && t < n; ++t) {
                    const int gt = g0 + t;
                    const int pos = pos0 + pos_k<1>(t);
                    const int slot = pos % NS;
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                        break;
                    if (gt >= NB) {  // buffer gt % NB held P of tile gt - NB: its PV must have read it
                        const int pv = gt - NB;
                        if (!(ok = __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (pv % O_DONE_RING),
                                                                        (pv / O_DONE_RING) & 1, cx, SITE_O_DONE))))
                            break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem + L::TM_S + (gt % NB) * L::BN;
                    const uint64_t kslot = dk + static_cast<uint64_t>((slot * L::HALF_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t box = kk >> 2, off = (kk & 3) * 32;
                        ptx::mma_ss_pair_w(d_tmem, dq + ((box * L::Q_BOX_BYTES + off) >> 4),
                                         kslot + ((box * L::K_BOX_BYTES + off) >> 4), IDESC_S, kk != 0);
                    }
                    issued = true;
                    ptx::mma_commit_pair_w(slot_empty0 + 8u * slot);
                    ptx::mma_commit_pair_w(s_full0 + 8u * (gt % NB));
                }
                if (!ok)
                    break;
                ptx::mma_commit_pair_w(q_free);  // both CTAs may load the next unit's Q
                g0 += n;
                pos0 += 2 * n;
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
            int g0 = 0, pos0 = 0;
            for (int it = 0, k = 0; ok && it < n_it; ++it) {
                const int n = unit_of(it).n;
                if (n == 0)
                    continue;
                for (int j = 0; ok && j < n; ++j) {
                    const int gj = g0 + j;
                    const int buf = gj % NB;
                    // V_j first (it has usually landed), then P_j: the slot wait stays
                    // off the P_j -> PV_j path.
                    const int pos = pos0 + pos_v<1>(j, n);
                    const int slot = pos % NS;
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx, SITE_SLOT_FULL))))
                        break;
                    // a unit's first PV overwrites O: the previous unit's epilogue must have read it
                    if (j == 0 && k > 0 &&
                        !(ok = __all_sync(0xffffffffu, wait_bounded_cluster(o_free, (k - 1) & 1, cx, SITE_O_DONE))))
                        break;
                    const uint32_t a_tmem = tmem + L::TM_S + buf * L::BN;
                    const uint64_t vslot = dv + static_cast<uint64_t>((slot * L::HALF_BYTES) >> 4);
#pragma unroll
                    for (int h = 0; h < L::P_PARTS; ++h) {
                        const uint32_t bar = h + 1 < L::P_PARTS ? p_part0 + 8u * (NB * h + buf) : p_full0 + 8u * buf;
                        if (!(ok = __all_sync(0xffffffffu, wait_bounded(bar, (gj / NB) & 1, cx, SITE_P_FULL))))
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
                    ptx::mma_commit_pair_w(o_done0 + 8u * (gj % O_DONE_RING));
                }
                g0 += n;
                pos0 += 2 * n;
                ++k;
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
        bool ok = true;
        // One arrival per warp on the leader's barrier, after every lane's TMEM accesses.
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
        // Row `row` of a unit's O: [planes, Sq, D], or (variable-length batch) token-major
        // [total_q, Hq, D]; LSE is [planes, Sq] or [Hq, total_q].
        auto o_row = [&](const Unit &un) {
            const size_t off = VARLEN ? static_cast<size_t>(un.q_row + row) * p.o_row_stride + static_cast<size_t>(un.z_q) * D
                                      : (static_cast<size_t>(un.z_q) * p.Sq + un.q0 + row) * D;
            return reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) + off);
        };
        int g0 = 0;
        for (int it = 0; ok && it < n_it; ++it) {
            const Unit un = unit_of(it);
            const int n = un.n;
            if (n == 0) {
                if (un.bad && threadIdx.x == 0) {
                    const uint32_t cta = blockIdx.x < 0xFFFFFFu ? blockIdx.x : 0xFFFFFFu;
                    atomicCAS(p.status, 0u, SITE_SEQLENS | (cta << 8));
                }
                if (un.zero && un.q0 + row < un.sq) {
                    // a sequence without keys: its rows attend to nothing, O = 0 and LSE = -inf
                    uint4 *dst = o_row(un);
#pragma unroll 1
                    for (int c8 = 0; c8 < D / 8; ++c8)
                        dst[c8] = make_uint4(0u, 0u, 0u, 0u);
                    if (p.lse != nullptr)
                        p.lse[static_cast<size_t>(un.z_q) * p.Sq + un.q_row + row] = -INFINITY;
                }
                continue;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int gj = g0 + j;
                const int buf = gj % NB;
                ok = wait_bounded(s_full0 + 8u * buf, (gj / NB) & 1, cx, SITE_S_FULL);
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

                // keys of this tile the row sees (>= 1): all < Skv, and (causal) <= the row
                // itself; only the ragged last tile or a causal diagonal takes the masked path
                const int valid = (p.causal ? min(un.skv, un.q0 + row + 1) : un.skv) - j * L::BN;
                const bool tail = __any_sync(0xffffffffu, valid < L::BN);
                if (tail) {
#pragma unroll
                    for (int i = 1; i < 128; ++i)
                        if (i >= valid)
                            s[i] = s[0];  // neutral for the max; weights zeroed below
                }
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

                constexpr int PW = 64 / L::P_PARTS;
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
                auto part_bar = [&](int q) { return q + 1 < L::P_PARTS ? p_part0 + 8u * (NB * q + buf) : p_full0 + 8u * buf; };
                compute_part(std::integral_constant<int, 0>{});
                // lazy rescale (tile gj-1's PV complete; S_gj complete implies PV_{gj-NSBUF} complete)
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    const int pv = gj - 1;
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
            if (!ok)
                break;

            // ------------------------------------------------------- epilogue
            // O of this unit once its last PV is done; written row by row to global
            // memory (rows past Sq are not written), then O's tensor memory is
            // released to the next unit's first PV.
            {
                const int pv = g0 + n - 1;
                ok = wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx, SITE_O_DONE);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
            }
            ptx::tc_fence_after();
            const bool row_ok = un.q0 + row < un.sq;
            uint4 *dst = o_row(un);
            // One chunk per wait and O released after the stores: the next unit's S MMAs run
            // meanwhile, and four-chunk loads with an earlier release measured 6 % slower here.
            drain_o_row<D, BF16, 1>(t_o, 1.f / l, [&](int cc, const uint32_t (&pk)[16]) {
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[4 * cc + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            });
            hand_over(o_free);
            if (p.lse != nullptr && row_ok)
                p.lse[static_cast<size_t>(un.z_q) * p.Sq + un.q_row + row] = (m_used + ptx::lg2(l)) * LN2;
            g0 += n;
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

// Host-side launcher: one cluster per SM pair (at most one per unit pair).
template <int D, bool BF16>
cudaError_t launch_sdp_fwd_pair_persistent(const CUtensorMap &q, const CUtensorMap &k_half, const CUtensorMap &v,
                                           const KernelParams &p, int grid, cudaStream_t stream)
{
    static unsigned long long set_dense = 0, set_varlen = 0;
    const bool vl = p.cu_q != nullptr;
    auto kern = vl ? sdp_fwd_pair_persistent_kernel<D, BF16, true> : sdp_fwd_pair_persistent_kernel<D, BF16, false>;
    cudaError_t e = set_smem_once(kern, PairLayout<D>::SMEM_BYTES, vl ? set_varlen : set_dense);
    if (e != cudaSuccess)
        return e;
    KernelParams pp = p;
    pp.units = grid;  // the units the per-unit kernel would run as CTAs
    const int sms = p.num_sms;
    const int clusters = grid / 2 < sms / 2 ? grid / 2 : sms / 2;
    kern<<<2 * clusters, NUM_THREADS, PairLayout<D>::SMEM_BYTES, stream>>>(q, k_half, v, pp);
    return cudaGetLastError();
}

// The persistent form serves unsplit launches with more units than SMs
// (otherwise each cluster would run one unit pair anyway): dense ones, causal or
// not, and causal variable-length batches. (Without the causal mask a
// variable-length batch measured the same either way, -0.6 to 0 %, so it keeps
// the per-unit kernel.)
inline bool use_persistent(const KernelParams &p, int grid)
{
    if (p.debug_flags & DEBUG_NO_PERSIST)
        return false;
    return p.kv_splits == 1 && p.o != nullptr && p.num_sms > 0 && grid > p.num_sms &&
           (p.cu_q == nullptr || p.causal);
}

}  // namespace sdp
