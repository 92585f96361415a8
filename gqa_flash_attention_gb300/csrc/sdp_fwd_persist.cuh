// Persistent form of the single-CTA kernel (see sdp_fwd_kernel.cuh), for dense
// launches (no variable-length batch, no split-KV; the launcher keeps causal
// launches on the per-unit grid) with more units than SMs:
// one CTA per SM runs unit after unit, with no set-up or tear-down between
// them, and the next unit starts while the current one ends.
//
// Units are claimed in launch order: CTA c first takes unit c, then each CTA
// takes gridDim + atomicAdd(counter, 1) once the loads of its current unit are
// issued, shortly before it is free (the counter is zeroed in stream order
// before the launch). A static walk (c, c + C, ...)
// lets CTAs drift apart over the rounds, so the units in flight spread over
// more KV heads than L2 holds; claiming in order keeps them a window of
// consecutive units, as the hardware's block scheduler does for the per-unit
// grid.
//
// The producer warp claims the units and announces each to the other roles
// through a ring of ANN shared-memory entries (unit id + mbarrier). A role
// reads unit k's announcement at most NSBUF + QB units after it was written
// (the producer announces unit k once unit k - QB's S MMAs are done, each S MMA
// of a tile waits for the PV NSBUF tiles back, each unit has at least one
// tile), so the ring is never overwritten early and each entry's mbarrier
// parity is unambiguous.
//
// As in the persistent CTA-pair kernel, every tile and ring counter is global
// across a CTA's units. At D=128 there are two query tiles in shared memory
// (the ring keeps five slots), so the next unit's Q loads while the current
// unit runs and its first scores follow the current unit's last without a
// wait; at D=256 one (Q loads once the unit before's last S MMA has read it).
// q_free[b] (the S issuer's commit after a unit's last S MMA) frees query tile
// b for the unit QB later; o_free (one arrival per softmax warp once the
// epilogue has read O out of tensor memory) lets the PV issuer start the next
// unit's first PV, which overwrites O. O is written from registers straight to
// global memory (the query tiles hold the next units' Q, so they cannot stage O).
#pragma once

#include "sdp_fwd_kernel.cuh"

namespace sdp {

template <int D>
struct PersistLayout {
    using L = Layout<D>;
    static constexpr int BAR_AREA = 512;
    // Query tiles in shared memory: two at D=128 (the next unit's Q loads while this unit runs),
    // one at D=256 (two would leave too few ring slots).
    static constexpr int QB = D == 128 ? 2 : 1;
    static constexpr int NSLOTS = (L::SMEM_LIMIT - BAR_AREA - 1024 - QB * L::Q_BYTES) / L::CHUNK_BYTES;
    static constexpr int ANN = 8;  // unit announcements (ring entries)
    // q_full[QB], slot_full[NS], slot_empty[NS], s_full[NB], p_full[NB], o_done[ring], final[2],
    // q_free[QB], o_free, ann[ANN]
    static constexpr int NBARS = QB + 2 * NSLOTS + 2 * L::NSBUF + O_DONE_RING + 2 + QB + 1 + ANN;
    static constexpr int BAR_OFF = QB * L::Q_BYTES + NSLOTS * L::CHUNK_BYTES;
    static constexpr int IDS_OFF = BAR_OFF + 8 * NBARS;  // ANN ints: announced unit ids (-1: no more)
    static constexpr int HOLDER_OFF = IDS_OFF + 4 * ANN;  // TMEM address, then the abort flag
    static constexpr int SMEM_BYTES = BAR_OFF + BAR_AREA + 1024;
    static_assert(HOLDER_OFF + 8 <= BAR_OFF + BAR_AREA, "barrier area");
    static_assert(SMEM_BYTES <= L::SMEM_LIMIT, "shared memory");
    // The producer announces unit k once unit k - QB's S MMAs are done; a role is then at most
    // NSBUF + QB units behind.
    static_assert(ANN >= L::NSBUF + QB + 2, "announcement ring depth");
    // Ring parity across units (global load positions; checked by enumerating every sequence
    // of unit lengths up to six units of up to four tiles): the S issuer may wait for its K slot
    // before PV_{t-NSBUF} only with one chunk per tile and six slots (the V chunks it cannot yet
    // know have landed lie at most 5 positions back); otherwise it waits for PV_{t-NSBUF} first
    // (at most 3 back, for one or two chunks per tile), and the PV issuer waits for P_j before
    // its V chunks when a tile is two chunks.
    static constexpr bool S_SLOT_FIRST = L::CHUNKS_PER_TILE == 1 && NSLOTS >= 6 && L::NSBUF <= 3;
    static_assert(S_SLOT_FIRST || (NSLOTS >= 4 && L::NSBUF <= 3), "ring parity soundness across units");
};

template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    sdp_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const KernelParams p)
{
    using L = Layout<D>;
    using PL = PersistLayout<D>;
    constexpr int NS = PL::NSLOTS;
    constexpr int NB = L::NSBUF;
    constexpr int CPT = L::CHUNKS_PER_TILE;
    constexpr int ANN = PL::ANN;
    constexpr uint32_t IDESC_S = ptx::idesc_f16_f32acc(128, L::BN, BF16, false);
    constexpr uint32_t IDESC_PV = ptx::idesc_f16_f32acc(128, 128, BF16, true);

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    constexpr int QB = PL::QB;
    const uint32_t s_q0 = sbase;  // query tile b at s_q0 + b * Q_BYTES
    const uint32_t s_ring = sbase + QB * L::Q_BYTES;
    const uint32_t bar0 = sbase + PL::BAR_OFF;
    const uint32_t q_full0 = bar0;  // + 8 b
    const uint32_t slot_full0 = bar0 + 8u * QB;
    const uint32_t slot_empty0 = slot_full0 + 8u * NS;
    const uint32_t s_full0 = slot_empty0 + 8u * NS;
    const uint32_t p_full0 = s_full0 + 8u * NB;
    const uint32_t o_done0 = p_full0 + 8u * NB;
    const uint32_t final0 = o_done0 + 8u * O_DONE_RING;
    const uint32_t q_free0 = final0 + 16u;  // + 8 b: unit k's S MMAs, the last to read query tile k % QB, are done
    const uint32_t o_free = q_free0 + 8u * QB;
    const uint32_t ann0 = o_free + 8u;  // + 8 (k % ANN)
    volatile int *ids = reinterpret_cast<volatile int *>(smem + PL::IDS_OFF);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + PL::HOLDER_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // A unit's geometry (dense: one plane of Sq rows per query head, Skv keys per KV head):
    // query head plane, KV plane, first query row, KV tiles read.
    struct Unit {
        int z_q, z_kv, q0, n;
    };
    auto unit_of = [&](int u) {
        Unit r;
        const int hi = u % p.G;
        u /= p.G;
        // Causal launches do not run this kernel (use_persist); the causal order here is the one
        // its causal measurements used. Decoding the per-unit grid's blocked causal order here
        // took 219 registers instead of 217 and ran 0.6-1.0 % slower on the dense launches.
        const int qt = p.causal ? p.n_qtiles - 1 - (u % p.n_qtiles) : (u % p.n_qtiles);
        const int bg = u / p.n_qtiles;  // b * Hkv + g
        const int b = bg / p.Hkv;
        const int g = bg - b * p.Hkv;
        r.z_q = b * p.Hq + g * p.G + hi;
        r.z_kv = bg;
        r.q0 = qt * L::BM;
        const int n_kv = (p.Skv + L::BN - 1) / L::BN;
        r.n = p.causal ? min(n_kv, qt + 1) : n_kv;
        return r;
    };

    // The first unit's Q tile and first K/V tiles start their DRAM reads now, into L2.
    if (warp == 4 && lane == 0 && !(p.debug_flags & DEBUG_NO_LOADS)) {
        const Unit un = unit_of(static_cast<int>(blockIdx.x));
#pragma unroll
        for (int c = 0; c < D / L::BOX_COLS; ++c) {
            ptx::tma_prefetch_3d(&tm_q, c * L::BOX_COLS, un.q0, un.z_q);
            ptx::tma_prefetch_3d(&tm_k, c * L::BOX_COLS, 0, un.z_kv);
            ptx::tma_prefetch_3d(&tm_v, c * L::BOX_COLS, 0, un.z_kv);
        }
    }

    if (threadIdx.x == 0) {
        for (int b = 0; b < QB; ++b) {
            ptx::mbar_init(q_full0 + 8u * b, 1);
            ptx::mbar_init(q_free0 + 8u * b, 1);
        }
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
        ptx::mbar_init(o_free, 4);  // one arrival per softmax warp
        for (int i = 0; i < ANN; ++i)
            ptx::mbar_init(ann0 + 8u * i, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
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
    // Unit k's announcement: wait for its entry, then read the id (-1: no more units).
    auto announced = [&](int k, int &u) -> bool {
        const bool ok = __all_sync(0xffffffffu, wait_bounded(ann0 + 8u * (k % ANN), (k / ANN) & 1, cx, SITE_Q_FULL));
        u = ids[k % ANN];
        return ok;
    };

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (!(p.debug_flags & DEBUG_NO_LOADS)) {  // whole warp; one elected lane issues
            int slot = 0;
            uint32_t ph = 0;
            bool ok = true;
            int u = static_cast<int>(blockIdx.x);
            for (int k = 0; ok; ++k) {
                // Unit k - QB's S MMAs, the last to read query tile k % QB, are done, so that tile and
                // announcement entry k % ANN (read by every role NSBUF + QB units ago at most) are free.
                const int b = k % QB;
                if (k >= QB && !(ok = __all_sync(0xffffffffu, wait_bounded(q_free0 + 8u * b, ((k - QB) / QB) & 1, cx,
                                                                            SITE_Q_FULL))))
                    break;
                const bool done = u >= p.units;
                if (lane == 0) {
                    ids[k % ANN] = done ? -1 : u;
                    ptx::mbar_arrive(ann0 + 8u * (k % ANN));  // release: the id before the arrival
                }
                __syncwarp();
                if (done)
                    break;
                const Unit un = unit_of(u);
                ptx::mbar_arrive_expect_tx_w(q_full0 + 8u * b, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / L::BOX_COLS; ++c)
                    ptx::tma_load_3d_w(s_q0 + b * L::Q_BYTES + c * L::BOX_BYTES, &tm_q, q_full0 + 8u * b, c * L::BOX_COLS,
                                       un.q0, un.z_q);
                auto load_tile = [&](const CUtensorMap *map, int j) -> bool {
#pragma unroll
                    for (int ch = 0; ch < CPT; ++ch) {
                        const uint32_t full = slot_full0 + 8u * slot;
                        const bool w = wait_bounded(slot_empty0 + 8u * slot, ph ^ 1u, cx, SITE_SLOT_EMPTY);
                        if (!__all_sync(0xffffffffu, w))
                            return false;
                        ptx::mbar_arrive_expect_tx_w(full, L::CHUNK_BYTES);
                        const uint32_t dst = s_ring + slot * L::CHUNK_BYTES;
                        const int y = j * L::BN;
                        ptx::tma_load_3d_w(dst, map, full, ch * 128, y, un.z_kv);
                        ptx::tma_load_3d_w(dst + L::BOX_BYTES, map, full, ch * 128 + L::BOX_COLS, y, un.z_kv);
                        if (++slot == NS) {
                            slot = 0;
                            ph ^= 1u;
                        }
                    }
                    return true;
                };
                const int n = un.n;
                ok = load_tile(&tm_k, 0);
                for (int j = 0; ok && j < n; ++j) {
                    if (j + 1 < n)
                        ok = load_tile(&tm_k, j + 1);
                    if (ok)
                        ok = load_tile(&tm_v, j);
                }
                // The next unit is claimed only now, with this unit's loads issued (the ring keeps the
                // producer a few tiles ahead of the MMAs): a CTA takes a unit when it is about to be
                // free, as the block scheduler hands out the per-unit grid. Claiming a whole unit ahead
                // left long causal units queued behind busy CTAs at the end (-12 % on causal MHA).
                int next = 0;
                if (lane == 0)
                    next = static_cast<int>(gridDim.x) + static_cast<int>(atomicAdd(p.claim, 1u));
                u = __shfl_sync(0xffffffffu, next, 0);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------- S = Q K^T issuer (1 thread)
        {  // whole warp; one elected lane issues
            const uint64_t dk = ptx::smem_desc_sw128(s_ring, 16, 1024);
            bool issued = false;
            bool ok = true;
            int g0 = 0, pos0 = 0;  // tiles and ring chunks of the earlier units
            for (int k = 0; ok; ++k) {
                int u;
                if (!(ok = announced(k, u)) || u < 0)
                    break;
                const int n = unit_of(u).n;
                const int b = k % QB;
                const uint64_t dq = ptx::smem_desc_sw128(s_q0 + b * L::Q_BYTES, 16, 1024);
                if (!(ok = __all_sync(0xffffffffu, wait_bounded(q_full0 + 8u * b, (k / QB) & 1, cx, SITE_Q_FULL))))
                    break;
                for (int t = 0; ok && t < n; ++t) {
                    const int gt = g0 + t;
                    const int p0 = pos0 + pos_k<CPT>(t);
                    // buffer gt % NB held P of tile gt - NB: its PV must have read it
                    auto pv_done = [&]() -> bool {
                        if (gt < NB)
                            return true;
                        const int pv = gt - NB;
                        return __all_sync(0xffffffffu, wait_bounded(o_done0 + 8u * (pv % O_DONE_RING),
                                                                    (pv / O_DONE_RING) & 1, cx, SITE_O_DONE));
                    };
                    if constexpr (!PL::S_SLOT_FIRST) {
                        if (!(ok = pv_done()))
                            break;
                    }
#pragma unroll
                    for (int ch = 0; ch < CPT; ++ch) {
                        const int pos = p0 + ch;
                        if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * (pos % NS), (pos / NS) & 1, cx,
                                                                        SITE_SLOT_FULL))))
                            break;
                    }
                    if (!ok)
                        break;
                    if constexpr (PL::S_SLOT_FIRST) {
                        if (!(ok = pv_done()))
                            break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem + L::TM_S + (gt % NB) * L::BN;
#pragma unroll
                    for (int ch = 0; ch < CPT; ++ch) {
                        const int slot = (p0 + ch) % NS;
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
                    ptx::mma_commit_w(s_full0 + 8u * (gt % NB));
                }
                if (!ok)
                    break;
                ptx::mma_commit_w(q_free0 + 8u * b);  // query tile b may take unit k + QB's Q
                g0 += n;
                pos0 += 2 * CPT * n;
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
            int g0 = 0, pos0 = 0;
            for (int k = 0; ok; ++k) {
                int u;
                if (!(ok = announced(k, u)) || u < 0)
                    break;
                const int n = unit_of(u).n;
                for (int j = 0; ok && j < n; ++j) {
                    const int gj = g0 + j;
                    const int buf = gj % NB;
                    const int p0 = pos0 + pos_v<CPT>(j, n);
                    if constexpr (CPT == 1) {  // V_j's slot first, off the P_j -> PV_j path
                        if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * (p0 % NS), (p0 / NS) & 1, cx,
                                                                        SITE_SLOT_FULL))))
                            break;
                    }
                    if (!(ok = __all_sync(0xffffffffu, wait_bounded(p_full0 + 8u * buf, (gj / NB) & 1, cx, SITE_P_FULL))))
                        break;
                    // a unit's first PV overwrites O: the previous unit's epilogue must have read it
                    if (j == 0 && k > 0 &&
                        !(ok = __all_sync(0xffffffffu, wait_bounded(o_free, (k - 1) & 1, cx, SITE_O_DONE))))
                        break;
                    ptx::tc_fence_after();
                    const uint32_t a_tmem = tmem + L::TM_S + buf * L::BN;
#pragma unroll
                    for (int ch = 0; ch < CPT; ++ch) {
                        const int pos = p0 + ch;
                        const int slot = pos % NS;
                        if constexpr (CPT != 1) {
                            if (!(ok = __all_sync(0xffffffffu, wait_bounded(slot_full0 + 8u * slot, (pos / NS) & 1, cx,
                                                                            SITE_SLOT_FULL))))
                                break;
                            ptx::tc_fence_after();
                        }
                        const uint64_t vslot = dv + static_cast<uint64_t>((slot * L::CHUNK_BYTES) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_ts_w(tmem + L::TM_O + ch * 128, a_tmem + kk * 8, vslot + ((kk * 2048) >> 4),
                                          IDESC_PV, (j > 0) || (kk > 0));
                        issued = true;
                        ptx::mma_commit_w(slot_empty0 + 8u * slot);
                    }
                    if (!ok)
                        break;
                    ptx::mma_commit_w(o_done0 + 8u * (gj % O_DONE_RING));
                }
                g0 += n;
                pos0 += 2 * CPT * n;
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
        bool ok = true;
        int g0 = 0;
        for (int k = 0; ok; ++k) {
            int u;
            if (!(ok = announced(k, u)) || u < 0)
                break;
            const Unit un = unit_of(u);
            const int n = un.n;
            float m_used = -INFINITY, l = 0.f;
            bool s_seen = false;  // S_j's barrier was seen complete while tile j-1 ended
            for (int j = 0; j < n; ++j) {
                const int gj = g0 + j;
                const int buf = gj % NB;
                if (!__all_sync(0xffffffffu, s_seen)) {
                    ok = wait_bounded(s_full0 + 8u * buf, (gj / NB) & 1, cx, SITE_S_FULL);
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

                // keys of this tile the row sees (>= 1): all < Skv, and (causal) <= the row itself;
                // only the ragged last tile or a causal diagonal takes the masked path
                const int valid = (p.causal ? min(p.Skv, un.q0 + row + 1) : p.Skv) - j * L::BN;
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
                // Poll S_{j+1}'s barrier now (same unit), so the answer returns while P_j is
                // stored and handed off; parity as in the per-unit kernel, with global tile indices.
                s_seen = j + 1 < n && ptx::mbar_test_wait(s_full0 + 8u * ((gj + 1) % NB), ((gj + 1) / NB) & 1);
                float sum0, sum1, sum2, sum3;
                ptx::f2_unpack(sum01, sum0, sum1);
                ptx::f2_unpack(sum23, sum2, sum3);
                ptx::tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
                ptx::tmem_st32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
                ptx::tmem_wait_st();
                const float tile_sum = (sum0 + sum1) + (sum2 + sum3);
                l = (j == 0) ? tile_sum : fmaf(l, alpha, tile_sum);

                // Rescale O only in warps where some row's maximum moved (they wait for PV_{gj-1}).
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
                ptx::tc_fence_before();
                ptx::mbar_arrive(p_full0 + 8u * buf);
                m_used = m_new;
            }
            if (!ok)
                break;

            // ---------------------------------------------------------- epilogue
            // O rows straight from registers to global memory (rows past Sq are not written),
            // then O's tensor memory is released to the next unit's first PV.
            {
                const int pv = g0 + n - 1;
                ok = wait_bounded(o_done0 + 8u * (pv % O_DONE_RING), (pv / O_DONE_RING) & 1, cx, SITE_O_DONE);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok)
                    break;
            }
            ptx::tc_fence_after();
            const bool row_ok = un.q0 + row < p.Sq;
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.o) +
                                                   (static_cast<size_t>(un.z_q) * p.Sq + un.q0 + row) * D);
            drain_o_row<D, BF16, 1>(t_o, 1.f / l, [&](int cc, const uint32_t (&pk)[16]) {
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[4 * cc + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            });
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(o_free);
            if (p.lse != nullptr && row_ok)
                p.lse[static_cast<size_t>(un.z_q) * p.Sq + un.q0 + row] = (m_used + ptx::lg2(l)) * LN2;
            g0 += n;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    // After an abort, loads the producer issued may still be landing: give them time.
    if (*abort_flag) {
        for (int i = 0; i < 100; ++i)
            ptx::nanosleep_ns(1000);
    }
    if (warp == 5) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// Dense launches without the causal mask (no variable-length batch, no split-KV, an O
// pointer for the row-wise stores, a claim counter) with more units than SMs. Under the
// mask the per-unit grid measured faster: causal MHA at D=128 and 16384 keys, both in the
// blocked causal unit order, -2.6 to -3.7 % for this kernel (+0.2 to +0.5 % at 8192 keys).
inline bool use_persist(const KernelParams &p, int grid)
{
    if (p.debug_flags & DEBUG_NO_PERSIST)
        return false;
    return !p.causal && p.kv_splits == 1 && p.cu_q == nullptr && p.o != nullptr && p.claim != nullptr &&
           p.num_sms > 0 && grid > p.num_sms;
}

// Host-side launcher: one CTA per SM (the units are claimed inside).
template <int D, bool BF16>
cudaError_t launch_sdp_fwd_persist(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                                   const KernelParams &p, int grid, cudaStream_t stream)
{
    static unsigned long long set = 0;
    auto kern = sdp_fwd_persist_kernel<D, BF16>;
    cudaError_t e = set_smem_once(kern, PersistLayout<D>::SMEM_BYTES, set);
    if (e != cudaSuccess)
        return e;
    e = cudaMemsetAsync(p.claim, 0, sizeof(unsigned int), stream);  // this launch's claim counter
    if (e != cudaSuccess)
        return e;
    KernelParams pp = p;
    pp.units = grid;
    const int ctas = grid < p.num_sms ? grid : p.num_sms;
    kern<<<ctas, NUM_THREADS, PersistLayout<D>::SMEM_BYTES, stream>>>(q, k, v, pp);
    return cudaGetLastError();
}

}  // namespace sdp
