// Forward masked attention on sm_103a (tcgen05 + TMEM + TMA).
//
// Passages: FlashAttention article §二.1 (tiling), §二.2 (max-subtracted
// softmax; completed here by the standard running rescale so the result is
// the exact softmax), §二.3 (QK^T and PV on tensor cores, fused in one
// kernel); blog "FlashMask技术" §2.2 (skip / full / masked block paths) and
// §4.1 items 1-3 (bounds staged in shared memory, skip decided before the KV
// block is loaded, mask fused into the softmax).
//
// Persistent: one CTA per SM walks work units (b, h, 128-row Q tile) in the
// plan's longest-first order, round robin over the CTAs; for each it walks the
// plan's list of non-skip KV tiles; skip tiles are never loaded.  Rings, score
// buffers and barrier phases follow one CTA-wide sequence of KV tiles, so the
// next unit's loads and scores overlap the current unit's last tiles and
// epilogue, and TMEM is allocated once per CTA.  Roles:
//   warp 0      TMA producer of Q (per unit) and K (three-stage ring)
//   warp 1      allocates TMEM; one thread issues the Q K^T MMAs
//   warps 2-5   softmax, KV columns [0, 64) of every row (thread = row =
//               TMEM lane)
//   warps 6-9   softmax, KV columns [64, 128)
//   warp 10     TMA producer of V (two-stage ring); stages the column bounds
//               of partial tiles with it
//   warp 11     one thread issues the P V MMAs
// Two issuing threads: the scores of later tiles are issued as soon as
// their K and score buffer are free, independently of the P V products
// waiting for the softmax (one thread doing both spent ~3,000 cycles per tile
// in waits and issue; the two streams now overlap).
// TMEM (512 columns): three score buffers S_0, S_1, S_2 at [0, 128),
// [128, 256), [256, 384) (tile t uses S_{t mod 3}) and O at [384, 384 + d).
// The scores of tile t + 1 are computed while the softmax works on tile t;
// P is written as packed bf16 over the first 64 columns of its S buffer (the
// A operand of O += P V), and the buffer is reused by the scores of tile
// t + 3 once that PV has read it.  The two softmax warpgroups exchange their
// row maxima through shared memory at a named barrier of their 256 threads
// (every thread of both reaches it on every tile, also after an abort, so it
// always completes), take the same lazy-rescale decision, and each rescales
// and finally stores its half of O's columns.
// Precise mode: P = P_hi + P_lo (P_lo = bf16(P - bf16(P))) in columns
// [0, 64) and [64, 128) of the S buffer, both multiplied by V.
// Online softmax in the base-2 domain with a lazy rescale: O and l are
// rescaled only when the row max grows by more than 2^8, which keeps every
// P <= 256 and leaves the final O / l unchanged.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

enum {
    FB_Q = 0,
    FB_KF0, FB_KF1, FB_KF2, FB_KE0, FB_KE1, FB_KE2,   // K stage loaded / released
    FB_VF0, FB_VF1, FB_VE0, FB_VE1,                   // V stage loaded / released
    FB_BF0, FB_BF1,                                   // bounds of the V stage's tile staged
    FB_S0, FB_S1, FB_S2,                              // scores of buffer b computed
    FB_P0, FB_P1, FB_P2,                              // P of buffer b written (both warpgroups)
    FB_O0, FB_O1, FB_O2,                              // O += P V of a tile using buffer b completed
    FB_QE,                                            // the last scores of a unit have read Q
    FB_OE,                                            // the epilogue of a unit has read O
    FB_UF0, FB_UF1, FB_UF2, FB_UF3,                   // unit ring: claimed unit written
    FB_UE0, FB_UE1, FB_UE2, FB_UE3,                   // unit ring: every consumer has read it
    FB_DRAIN,                                         // every MMA of the CTA completed
    FB_COUNT
};

template <int D, bool FP8 = false>
struct FwdSmem {
    static constexpr int kBox = 128 * 128;        // one 128-byte wide, 128-row box (64 bf16 or 128 e4m3 columns)
    static constexpr int kTile = 128 * D * (FP8 ? 1 : 2);   // one Q, K or V tile
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr int kQ = 0;
    static constexpr int kK = kTile;                           // [kKStages]
    static constexpr int kV = kK + kKStages * kTile;           // [kVStages]
    static constexpr int kBnd = kV + kVStages * kTile;         // int4 [kVStages][128]
    static constexpr int kMax = kBnd + kVStages * 128 * 16;    // float [2 slots][2 warpgroups][128]
    static constexpr int kSum = kMax + 2 * 2 * 128 * 4;        // float [2 slots][2 warpgroups][128]: l
    static constexpr int kUnit = kSum + 2 * 2 * 128 * 4;       // int4 [4]: unit ring (qt, bh, sidx, n)
    static constexpr int kFlag = kUnit + 4 * 16;               // int [2][8]: softmax warps' unit decisions
    static constexpr int kBar = kFlag + 16 * 4;
    static constexpr int kNumBar = FB_COUNT;
    static constexpr int kMisc = kBar + kNumBar * 8;
    // At least 120 KB so that one CTA (512 TMEM columns) is resident per SM.
    static constexpr int kBytes = (kMisc + 64 > 120 * 1024) ? kMisc + 64 : 120 * 1024;
};


constexpr int kSB = 3;              // score buffers in TMEM
constexpr int kUnitRing = 4;        // claimed units buffered between the K producer and the other roles
constexpr int kUnitReaders = 11;    // V producer, two MMA issuers, eight softmax warps

// Work counters of the persistent forward launches, one slot per launch in
// flight: {next unit to claim, CTAs finished}.  The host gives each launch
// its own slot (round robin); the launch's last CTA resets it to zero.
constexpr int kFwdSchedSlots = 64;
static __device__ unsigned int g_fwd_sched[kFwdSchedSlots][2];
constexpr int kSoftmaxBar = 1;      // named barrier of the two softmax warpgroups (256 threads)

template <int D, bool PRECISE, bool FP8>
__global__ void __launch_bounds__(384, 1)
    fm_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a)
{
    static_assert(!(PRECISE && FP8), "the FP8 path has no precise mode");
    static_assert(!FP8 || D == 128, "the FP8 path is built for d = 128");
    using S = FwdSmem<D, FP8>;
    constexpr int BOXW = FP8 ? 128 : 64;          // elements per 128-byte box row
    constexpr int NBOX = D / BOXW;
    constexpr int KS = S::kKStages, VS = S::kVStages;
    // The kernel has no static shared memory, so the dynamic window starts on
    // a 1024-byte boundary (checked below).  Pointers stay derived from the
    // __shared__ array itself, so every access compiles to a shared-memory
    // instruction rather than a generic one.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    int4 *sBnd = reinterpret_cast<int4 *>(smem + S::kBnd);
    float *sMax = reinterpret_cast<float *>(smem + S::kMax);
    float *sSum = reinterpret_cast<float *>(smem + S::kSum);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 12);
    volatile int *sUnit = reinterpret_cast<volatile int *>(smem + S::kUnit);   // [kUnitRing][4]
    volatile int *sFlag = reinterpret_cast<volatile int *>(smem + S::kFlag);

    const int warp = warp_id(), lane = lane_id();
    const PlanLayout &L = a.L;
    const int N = a.N;

    if (warp == 0) {
        const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(a.plan);
        const bool ok = ph->magic == kPlanMagic && ph->B == L.B && ph->Hm == L.Hm && ph->N == L.N &&
                        ph->bq == 128 && ph->bk == 128 && ph->q_row0 == L.q_row0 && ph->Nq == L.Nq;
        if (lane == 0) {
            if (!ok) set_status(a.status, FM_ERR_PLAN_MISMATCH);
            const bool aligned = (smem_u32(smem) & 1023u) == 0;   // 128-byte swizzle atoms need it
            if (!aligned) set_status(a.status, FM_ERR_UNSUPPORTED);
            *ok_sh = ok && aligned;
            *abort = 0;
            mbar_init(&bars[FB_Q], 1);
            for (int s = 0; s < KS; ++s) {
                mbar_init(&bars[FB_KF0 + s], 1);
                mbar_init(&bars[FB_KE0 + s], 1);
            }
            for (int s = 0; s < VS; ++s) {
                mbar_init(&bars[FB_VF0 + s], 1);
                mbar_init(&bars[FB_VE0 + s], 1);
                mbar_init(&bars[FB_BF0 + s], 32);
            }
            // One O barrier per score buffer: the PV of tile g commits to O_{g mod 3},
            // so every wait below targets a barrier at most one phase behind.
            for (int s = 0; s < kSB; ++s) {
                mbar_init(&bars[FB_S0 + s], 1);
                mbar_init(&bars[FB_P0 + s], 256);
                mbar_init(&bars[FB_O0 + s], 1);
            }
            for (int s = 0; s < kUnitRing; ++s) {
                mbar_init(&bars[FB_UF0 + s], 1);
                mbar_init(&bars[FB_UE0 + s], kUnitReaders);
            }
            mbar_init(&bars[FB_QE], 1);         // scores issuer, after a unit's last scores
            mbar_init(&bars[FB_OE], 256);       // both softmax warpgroups, after reading O
            mbar_init(&bars[FB_DRAIN], 2);      // both MMA issuers commit
            fence_barrier_init();
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Persistent CTAs with dynamic scheduling: the K producer of each CTA claims
    // the next work unit (b, h, 128-row Q tile) of the plan's longest-first order
    // from the launch's counter whenever it is ready for one, like a block
    // scheduler would, so the CTAs that run at the same time work on
    // neighbouring units of the order (which share K / V in L2) and the longest
    // lists start first.  Claimed units pass to the other roles through a ring of
    // kUnitRing entries in shared memory (-1 ends the sequence).  Every role walks
    // the same units and, across units, one CTA-wide sequence of KV tiles g:
    // rings, score buffers and barrier phases follow g, so the next unit's Q and
    // K / V loads and scores proceed while the current unit's epilogue runs.  A
    // unit with an empty list has no tiles and only writes O = 0, lse = -inf.
    const int64_t n_units = (int64_t)a.B * a.H * L.n_q;
    unsigned int *sched = g_fwd_sched[a.sched_slot];
    struct Unit {
        int qt, bh, sidx, n;
        const int32_t *list;
    };
    // Called by all 32 lanes of a warp; false on a plan that was not written by
    // the classifier (reported once, by warp 0).
    auto unit_from = [&](int c, Unit &u) -> bool {
        int ut = 0, uh = 0, ub = 0;
        if (!plan_unit(reinterpret_cast<const int32_t *>(a.plan + L.off_row_order),
                       reinterpret_cast<const int32_t *>(a.plan + L.off_row_bstart), L.n_q, a.B, a.Hm, a.H, c,
                       &ut, &uh, &ub)) {
            if (warp == 0 && lane == 0) set_status(a.status, FM_ERR_PLAN_MISMATCH);
            return false;
        }
        u.qt = ut;
        u.bh = ub * a.H + uh;
        u.sidx = ub * a.Hm + (a.Hm == 1 ? 0 : uh);
        const int64_t row = (int64_t)u.sidx * L.n_q + ut;
        u.n = reinterpret_cast<const int32_t *>(a.plan + L.off_row_cnt)[row];
        u.list = reinterpret_cast<const int32_t *>(a.plan + L.off_row_list) + row * L.n_k;
        return true;
    };
    auto list_of = [&](const Unit &u) {
        return reinterpret_cast<const int32_t *>(a.plan + L.off_row_list) + ((int64_t)u.sidx * L.n_q + u.qt) * L.n_k;
    };
    // Unit k of the ring for a reading warp: waits until it has been claimed,
    // reads it and releases the entry (lane 0 arrives for the warp); false when
    // the sequence has ended (n = -1) or a wait gave up.
    auto read_unit = [&](int k, Unit &u) -> bool {
        const int slot = k % kUnitRing;
        if (!warp_wait(&bars[FB_UF0 + slot], (k / kUnitRing) & 1, abort, a.status, a.wait_limit)) return false;
        u.qt = sUnit[slot * 4 + 0];
        u.bh = sUnit[slot * 4 + 1];
        u.sidx = sUnit[slot * 4 + 2];
        u.n = sUnit[slot * 4 + 3];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[FB_UE0 + slot]);
        u.list = list_of(u);
        return u.n >= 0;
    };

    if (*ok_sh) {
        if (warp == 0) {
            // ------------------------------------------------ K producer
            // Per unit with tiles: Q (once the previous unit's last scores have
            // read the Q buffer), then K through its ring: K of tile g is loaded
            // once the scores of tile g - KS have read the stage.
            if (lane == 0) {
                tma_prefetch_desc(&tq);
                tma_prefetch_desc(&tk);
            }
            int g = 0;    // K loads begun (CTA-wide tile counter)
            int nq = 0;   // units with tiles begun (Q loads)
            // Test hook: the first CTA withholds the K load of its second tile,
            // so that the scores' wait for it runs out (never set by a product call).
            const int withheld = (a.withhold && blockIdx.x == 0) ? 1 : -1;
            bool run = true;
            Unit u;
            for (int k = 0; run; ++k) {
                // Claim the next unit into ring entry k once every reader is done
                // with the entry's previous unit.
                const int slot = k % kUnitRing;
                if (k >= kUnitRing &&
                    !warp_wait(&bars[FB_UE0 + slot], ((k / kUnitRing) - 1) & 1, abort, a.status, a.wait_limit))
                    break;
                int c = 0;
                if (lane == 0) c = (int)atomicAdd(&sched[0], 1u);
                c = __shfl_sync(0xffffffffu, c, 0);
                bool valid = c < n_units;
                if (valid && !unit_from(c, u)) valid = false;
                if (lane == 0) {
                    sUnit[slot * 4 + 0] = valid ? u.qt : 0;
                    sUnit[slot * 4 + 1] = valid ? u.bh : 0;
                    sUnit[slot * 4 + 2] = valid ? u.sidx : 0;
                    sUnit[slot * 4 + 3] = valid ? u.n : -1;
                    mbar_arrive(&bars[FB_UF0 + slot]);
                }
                if (!valid) break;
                if (u.n == 0) continue;
                if (nq > 0 && !warp_wait(&bars[FB_QE], (nq - 1) & 1, abort, a.status, a.wait_limit)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[FB_Q], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(smem + S::kQ + x * S::kBox, &tq, &bars[FB_Q], x * BOXW, u.qt * 128, u.bh);
                }
                ++nq;
                int e_next = u.list[0];
                for (int t = 0; t < u.n; ++t, ++g) {
                    const int kb = (e_next & kTileMask) * 128;
                    if (t + 1 < u.n) e_next = u.list[t + 1];
                    const int ks = g % KS;
                    if (g >= KS && !warp_wait(&bars[FB_KE0 + ks], ((g / KS) - 1) & 1, abort, a.status, a.wait_limit)) {
                        run = false;
                        break;
                    }
                    if (lane == 0 && g != withheld) {
                        mbar_arrive_expect_tx(&bars[FB_KF0 + ks], S::kTile);
#pragma unroll
                        for (int x = 0; x < NBOX; ++x)
                            tma_load_3d(smem + S::kK + ks * S::kTile + x * S::kBox, &tk, &bars[FB_KF0 + ks], x * BOXW, kb, u.bh);
                    }
                }
            }
            // Drain copies still in flight (only possible after an abort).
            if (lane == 0 && *abort) {
                if (nq > 0) mbar_wait_drain(&bars[FB_Q], (nq - 1) & 1, a.status, a.wait_limit);
                for (int k2 = (g > KS ? g - KS : 0); k2 < g; ++k2)
                    if (k2 != withheld) mbar_wait_drain(&bars[FB_KF0 + (k2 % KS)], (k2 / KS) & 1, a.status, a.wait_limit);
            }
        } else if (warp == 10) {
            // ------------------------------------------------ V producer
            // V through its ring, and the column bounds of partial tiles staged with
            // it: the V stage (and its bounds) is free once the PV of tile g - VS
            // has completed, which follows the softmax's use of those bounds.
            if (lane == 0) tma_prefetch_desc(&tv);
            int g = 0;    // V loads begun (CTA-wide tile counter)
            bool run = true;
            Unit u;
            for (int k = 0; run; ++k) {
                if (!read_unit(k, u)) break;
                if (u.n == 0) continue;
                int e_next = u.list[0];
                for (int t = 0; t < u.n; ++t, ++g) {
                    const int e = e_next;
                    if (t + 1 < u.n) e_next = u.list[t + 1];
                    const int kb = (e & kTileMask) * 128;
                    const bool pred = ((e >> kLabelShift) == FM_TILE_PARTIAL) || kb + 128 > N;
                    const int vs = g % VS;
                    // Column bounds of a partial tile, loaded before the wait below so
                    // their latency overlaps it; stored as (start, length) pairs,
                    // columns beyond N masked for every row.
                    int4 bv[4];
                    if (pred) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int j = kb + lane * 4 + w;
                            bv[w] = make_int4(0, 0, 0, 0x7fffffff);
                            if (j < N) {
                                const int64_t o = (int64_t)u.sidx * N + j;
                                bv[w] = make_int4(a.lts[o], a.lte[o], a.uts[o], a.ute[o]);
                            }
                        }
                    }
                    if (g >= VS && !warp_wait(&bars[FB_VE0 + vs], ((g / VS) - 1) & 1, abort, a.status, a.wait_limit)) {
                        run = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[FB_VF0 + vs], S::kTile);
                        // V^T on the FP8 path, else the NBOX boxes of V
                        if (FP8)   // V^T tile: d rows x 128 key columns, [B*H][d][N] e4m3
                            tma_load_3d(smem + S::kV + vs * S::kTile, &tv, &bars[FB_VF0 + vs], kb, 0, u.bh);
                        else
                            for (int x = 0; x < NBOX; ++x)
                                tma_load_3d(smem + S::kV + vs * S::kTile + x * S::kBox, &tv, &bars[FB_VF0 + vs], x * 64, kb, u.bh);
                    }
                    if (pred) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const int4 v = bv[w];
                            sBnd[vs * 128 + lane * 4 + w] = (kb + lane * 4 + w < N)
                                                                ? make_int4(v.x, max(v.y - v.x, 0), v.z, max(v.w - v.z, 0))
                                                                : v;
                        }
                    }
                    mbar_arrive(&bars[FB_BF0 + vs]);
                }
            }
            if (lane == 0 && *abort)
                for (int k2 = (g > VS ? g - VS : 0); k2 < g; ++k2)
                    mbar_wait_drain(&bars[FB_VF0 + (k2 % VS)], (k2 / VS) & 1, a.status, a.wait_limit);
        } else if (warp == 1) {
            // ------------------------------------------------ S issuer
            // The scores of tile g as soon as its unit's Q and its K have landed and
            // its score buffer has been read by the PV of tile g - 3; runs ahead of
            // the softmax by up to the three score buffers, also into the next unit.
            // All lanes walk the units (plan_unit is warp-wide); lane 0 issues.
            constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
            const uint64_t dQ = sdesc_sw128(smem_u32(smem + S::kQ), 16, 1024);
            int g = 0, nq = 0;
            bool run = true;
            Unit u;
            for (int k = 0; run; ++k) {
                if (!read_unit(k, u)) break;
                if (u.n == 0) continue;
                if (lane == 0) {
                    run = mbar_wait(&bars[FB_Q], nq & 1, abort, a.status, a.wait_limit);
                    for (int t = 0; run && t < u.n; ++t, ++g) {
                        const int ks = g % KS;
                        // The buffer's previous tile, g - 3, must have finished its PV.
                        if (!mbar_wait(&bars[FB_KF0 + ks], (g / KS) & 1, abort, a.status, a.wait_limit) ||
                            (g >= kSB && !mbar_wait(&bars[FB_O0 + g % kSB], ((g - kSB) / kSB) & 1, abort, a.status,
                                                    a.wait_limit))) {
                            run = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t dK = sdesc_sw128(smem_u32(smem + S::kK + ks * S::kTile), 16, 1024);
                        const uint32_t tS = tmem + (g % kSB) * 128;
                        if (FP8) {
#pragma unroll
                            for (int kk = 0; kk < D / 32; ++kk)   // K = 32 e4m3 = 32 bytes per instruction
                                mma_ss_e4m3(tS, sdesc_add(dQ, kk * 32), sdesc_add(dK, kk * 32), idesc_e4m3(128, 128), kk > 0);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = (kk >> 2) * S::kBox + (kk & 3) * 32;
                                mma_ss(tS, sdesc_add(dQ, off), sdesc_add(dK, off), idS, kk > 0);
                            }
                        }
                        tc_commit(&bars[FB_S0 + g % kSB]);
                        tc_commit(&bars[FB_KE0 + ks]);
                    }
                    // Q is free for the next unit once this unit's scores complete.
                    if (run) tc_commit(&bars[FB_QE]);
                }
                ++nq;
                run = __shfl_sync(0xffffffffu, run, 0);
            }
            if (lane == 0) {
                // Every MMA of this CTA (both issuers) completes before TMEM is released.
                tc_commit(&bars[FB_DRAIN]);
                mbar_wait_drain(&bars[FB_DRAIN], 0, a.status, a.wait_limit);
            }
        } else if (warp == 11) {
            // ------------------------------------------------ PV issuer
            // O += P V of tile g once the softmax has written P and V has landed; the
            // first PV of a unit overwrites O, so it waits until the previous unit's
            // epilogue has read O.
            constexpr uint32_t idO = idesc_bf16(128, D, false, true);
            constexpr int NPART = PRECISE ? 2 : 1;
            const uint32_t tO = tmem + 384;
            int g = 0, nu = 0;
            bool run = true;
            Unit u;
            for (int k = 0; run; ++k) {
                if (!read_unit(k, u)) break;
                if (u.n == 0) continue;
                if (lane == 0) {
                    if (nu > 0) run = mbar_wait(&bars[FB_OE], (nu - 1) & 1, abort, a.status, a.wait_limit);
                    for (int t = 0; run && t < u.n; ++t, ++g) {
                        const int vs = g % VS;
                        if (!mbar_wait(&bars[FB_VF0 + vs], (g / VS) & 1, abort, a.status, a.wait_limit) ||
                            !mbar_wait(&bars[FB_P0 + g % kSB], (g / kSB) & 1, abort, a.status, a.wait_limit)) {
                            run = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t tP = tmem + (g % kSB) * 128;
                        if (FP8) {
                            // B = V^T, K-major (d rows of 128 key bytes); A = P, 4 e4m3 per column
                            const uint64_t dVt = sdesc_sw128(smem_u32(smem + S::kV + vs * S::kTile), 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ts_e4m3(tO, tP + kk * 8, sdesc_add(dVt, kk * 32), idesc_e4m3(128, D), (t > 0 || kk > 0));
                        } else {
                            const uint64_t dV = sdesc_sw128(smem_u32(smem + S::kV + vs * S::kTile), S::kBox, 1024);
#pragma unroll
                            for (int part = 0; part < NPART; ++part)   // P_hi V (+ P_lo V)
#pragma unroll
                                for (int kk = 0; kk < 8; ++kk)
                                    mma_ts(tO, tP + part * 64 + kk * 8, sdesc_add(dV, kk * 2048), idO,
                                           (t > 0 || part > 0 || kk > 0));
                        }
                        tc_commit(&bars[FB_O0 + g % kSB]);
                        tc_commit(&bars[FB_VE0 + vs]);
                    }
                }
                ++nu;
                run = __shfl_sync(0xffffffffu, run, 0);
            }
            if (lane == 0) {
                tc_commit(&bars[FB_DRAIN]);
                mbar_wait_drain(&bars[FB_DRAIN], 0, a.status, a.wait_limit);
            }
        } else {
            // ------------------------------------------------ softmax (warps 2-9)
            const int w = (warp < 6) ? 0 : 1;          // column half: KV columns [64 w, 64 w + 64)
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t tO = tmem + 384;
            constexpr int OC = D / 2;                  // O columns rescaled / stored by this warpgroup
            // softmax scale * log2(e), with the Q and K descales on the FP8 path
            const float sl2 = FP8 ? a.scale_log2 * a.descale[0] * a.descale[1] : a.scale_log2;
            // `live` turns false (for the whole warp) when a wait gives up after an
            // abort; the warp then skips its work but still reaches every named
            // barrier of the loop, so the other warpgroup is never left waiting.
            bool live = true;
            // The PV of tile k has completed (and with it every earlier MMA).
            auto wait_pv = [&](int k) {
                live = live && warp_wait(&bars[FB_O0 + k % kSB], (k / kSB) & 1, abort, a.status, a.wait_limit);
            };
            int g = 0;     // tiles begun (CTA-wide)
            int nu = 0;    // units with tiles finished
            Unit un;
            for (int k = 0;; ++k) {
                // Both warpgroups take the same decision on every unit: a wait that
                // gave up after an abort in any warp stops all eight (their named
                // barriers must stay matched).  Flags alternate between units.
                const bool got = read_unit(k, un);
                if (lane == 0) sFlag[(k & 1) * 8 + (warp - 2)] = got ? 1 : 0;
                named_bar_sync(kSoftmaxBar, 256);
                int all = sFlag[(k & 1) * 8];
#pragma unroll
                for (int q = 1; q < 8; ++q) all &= sFlag[(k & 1) * 8 + q];
                if (!all) break;
                const int li = un.qt * 128 + r;            // row of Q / O / lse
                const int i = a.q_row0 + li;               // row of the mask
                float m = -INFINITY, l = 0.f;
                int e_next = un.n > 0 ? un.list[0] : 0;
                for (int t = 0; t < un.n; ++t, ++g) {
                    const int e = e_next;
                    if (t + 1 < un.n) e_next = un.list[t + 1];
                    const int kb = (e & kTileMask) * 128;
                    const bool pred = ((e >> kLabelShift) == FM_TILE_PARTIAL) || kb + 128 > N;
                    const int bb = g % kSB, vs = g % VS;
                    const uint32_t tS = tmem + bb * 128;
                    live = live && warp_wait(&bars[FB_S0 + bb], (g / kSB) & 1, abort, a.status, a.wait_limit);
                    live = live && (!pred || warp_wait(&bars[FB_BF0 + vs], (g / VS) & 1, abort, a.status, a.wait_limit));
                    float sv[64];
                    float mxl = -INFINITY;
                    if (live) {
                        tc_fence_after();
                        uint32_t raw[2][32];
                        tmem_ld32(tS + lane_off + w * 64, raw[0]);
                        tmem_ld32(tS + lane_off + w * 64 + 32, raw[1]);
                        tmem_ld_wait();
                        tmem_reg_fence(raw[0]);
                        tmem_reg_fence(raw[1]);
#pragma unroll
                        for (int cc = 0; cc < 64; ++cc) sv[cc] = __uint_as_float(raw[cc >> 5][cc & 31]);
                        if (pred) {
                            const int4 *bnd = sBnd + vs * 128 + w * 64;
#pragma unroll
                            for (int cc = 0; cc < 64; ++cc) {
                                const int4 x = bnd[cc];
                                const bool msk = ((unsigned)(i - x.x) < (unsigned)x.y) || ((unsigned)(i - x.z) < (unsigned)x.w);
                                sv[cc] = msk ? -INFINITY : sv[cc];
                            }
                        }
                        float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                        for (int k2 = 0; k2 < 30; ++k2) mx4[k2 & 3] = fmax3(mx4[k2 & 3], sv[4 + 2 * k2], sv[5 + 2 * k2]);
                        mxl = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                    }
                    // Row max over both column halves.  Both warpgroups hold their S
                    // columns in registers once the barrier completes, so P may then
                    // overwrite the S buffer.
                    const int slot = g & 1;
                    sMax[(slot * 2 + w) * 128 + r] = mxl;
                    tc_fence_before();
                    named_bar_sync(kSoftmaxBar, 256);
                    tc_fence_after();
                    if (!live) continue;
                    const float mx = fmaxf(mxl, sMax[(slot * 2 + (1 - w)) * 128 + r]) * sl2;   // -inf stays -inf
                    float m_new = m, alpha = 1.f;
                    if (mx > m + 8.f) {
                        m_new = mx;
                        alpha = ex2(m - m_new);                  // m = -inf gives 0
                    }
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    // Rescale this warpgroup's half of O when the max moved (rare with
                    // the 2^8 threshold); the PV of the previous tile must be complete.
                    if (__any_sync(0xffffffffu, t > 0 && alpha != 1.f)) {
                        wait_pv(g - 1);
                        if (!live) continue;
                        tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < OC / 32; ++cc) {
                            uint32_t ov[32];
                            tmem_ld32(tO + lane_off + w * OC + cc * 32, ov);
                            tmem_ld_wait();
                            tmem_reg_fence(ov);
#pragma unroll
                            for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
                            tmem_st32(tO + lane_off + w * OC + cc * 32, ov);
                        }
                    }
                    // P = exp2(s * scale*log2e - m) as packed bf16 over the S buffer:
                    // this warpgroup's 64 columns go to TMEM columns [32 w, 32 w + 32)
                    // (precise mode: P_lo to [64 + 32 w, ...)).  O is normalised by the
                    // fp32 sum of P, which also gives lse (standard mode: the bf16
                    // rounding of the weights P V applied moves that sum by ~2^-9
                    // relative at most, far inside the tolerance, and summing the
                    // rounded values instead costs 1.5 instructions per element on
                    // the critical chain).  Column pairs in packed fp32.
                    const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                    uint32_t f8[16];          // FP8: the warpgroup's 64 P values, 4 e4m3 per column
                    uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(sv[hh * 32 + 2 * cc], sv[hh * 32 + 2 * cc + 1]), sc2, nm2), x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            sum2 = f2_add(sum2, f2_pack(p0, p1));
                            hi[cc] = pack_bf16x2(p0, p1);
                            if (FP8) {
                                const uint32_t e2 = pack_e4m3x2(p0, p1);     // columns 2 cc, 2 cc + 1
                                if (cc & 1) f8[hh * 8 + (cc >> 1)] |= e2 << 16;
                                else f8[hh * 8 + (cc >> 1)] = e2;
                            }
                            if (PRECISE) {
                                lo[cc] = pack_bf16x2(p0 - __uint_as_float(hi[cc] << 16),
                                                     p1 - __uint_as_float(hi[cc] & 0xffff0000u));
                            }
                        }
                        if (!FP8) tmem_st16(tS + lane_off + w * 32 + hh * 16, hi);
                        if (PRECISE) tmem_st16(tS + lane_off + 64 + w * 32 + hh * 16, lo);
                    }
                    if (FP8) tmem_st16(tS + lane_off + w * 16, f8);   // columns [16 w, 16 w + 16)
                    float s0, s1;
                    f2_unpack(sum2, s0, s1);
                    l = l * alpha + (s0 + s1);
                    m = m_new;
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars[FB_P0 + bb]);
                }
                // ------------------------------------------------ epilogue
                // Combine the two warpgroups' partial sums (one more named barrier,
                // reached by every thread of both; the slot alternates between
                // units), then each stores its half of O after the last PV.  O is
                // released to the next unit's first PV as soon as it is in
                // registers.  A unit without tiles writes O = 0, lse = -inf.
                const int su = nu & 1;
                if (un.n > 0) {
                    sSum[(su * 2 + w) * 128 + r] = l;
                    named_bar_sync(kSoftmaxBar, 256);
                    wait_pv(g - 1);
                }
                if (live) {
                    uint32_t ov[OC];
                    float lt = 0.f;
                    if (un.n > 0) {
                        tc_fence_after();
                        lt = sSum[(su * 2) * 128 + r] + sSum[(su * 2 + 1) * 128 + r];
#pragma unroll
                        for (int cc = 0; cc < OC / 32; ++cc)
                            tmem_ld32(tO + lane_off + w * OC + cc * 32, reinterpret_cast<uint32_t (&)[32]>(ov[cc * 32]));
                        tmem_ld_wait();
                        tmem_reg_fence(ov);
                        tc_fence_before();
                        mbar_arrive(&bars[FB_OE]);
                    } else {
#pragma unroll
                        for (int c = 0; c < OC; ++c) ov[c] = 0u;
                    }
                    const float inv = (lt > 0.f) ? (FP8 ? a.descale[2] : 1.f) / lt : 0.f;
                    const bool row_in = li < a.Nq;
                    const int64_t row = (int64_t)un.bh * a.Nq + li;
                    if (row_in) {
#pragma unroll
                        for (int cc = 0; cc < OC / 32; ++cc) {
                            const int col = w * OC + cc * 32;
                            const uint32_t *oc = ov + cc * 32;
                            if (a.o_f32) {
                                float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + row * D + col);
#pragma unroll
                                for (int q4 = 0; q4 < 8; ++q4)
                                    dst[q4] = make_float4(__uint_as_float(oc[4 * q4]) * inv, __uint_as_float(oc[4 * q4 + 1]) * inv,
                                                          __uint_as_float(oc[4 * q4 + 2]) * inv, __uint_as_float(oc[4 * q4 + 3]) * inv);
                            } else {
                                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + row * D + col);
#pragma unroll
                                for (int q8 = 0; q8 < 4; ++q8)
                                    dst[q8] = make_uint4(pack_bf16x2(__uint_as_float(oc[8 * q8 + 0]) * inv, __uint_as_float(oc[8 * q8 + 1]) * inv),
                                                         pack_bf16x2(__uint_as_float(oc[8 * q8 + 2]) * inv, __uint_as_float(oc[8 * q8 + 3]) * inv),
                                                         pack_bf16x2(__uint_as_float(oc[8 * q8 + 4]) * inv, __uint_as_float(oc[8 * q8 + 5]) * inv),
                                                         pack_bf16x2(__uint_as_float(oc[8 * q8 + 6]) * inv, __uint_as_float(oc[8 * q8 + 7]) * inv));
                            }
                        }
                        if (w == 0) a.lse[row] = (lt > 0.f) ? (m + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
                    }
                } else if (un.n > 0) {
                    mbar_arrive(&bars[FB_OE]);   // after an abort: nothing reads O any more
                }
                if (un.n > 0) ++nu;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // The launch's last CTA returns the work counters to zero for the next
    // launch that gets this slot (every claim precedes its CTA's count here).
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
            sched[0] = 0;
            sched[1] = 0;
            __threadfence();
        }
    }
}

}  // namespace fm

using namespace fm;

// The kernel's shared-memory limit, set once per device: later launches (also
// those captured into a graph) make no attribute call.
template <int D, bool PRECISE, bool FP8 = false>
static bool fwd_smem_ready()
{
    constexpr int smem = FwdSmem<D, FP8>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    static std::atomic<uint8_t> done[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(fm_fwd_kernel<D, PRECISE, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return false;
    done[dev].store(1, std::memory_order_release);
    return true;
}

template <int D, bool PRECISE, bool FP8 = false>
static fm_status launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const FwdArgs &a, cudaStream_t stream)
{
    constexpr int smem = FwdSmem<D, FP8>::kBytes;
    if (!fwd_smem_ready<D, PRECISE, FP8>()) return FM_ERR_CUDA;
    // Persistent: one CTA per SM (the kernel's shared memory and 512 TMEM
    // columns allow no second one), each walking units in the plan's order.
    const int64_t units = (int64_t)a.B * a.H * a.L.n_q;
    const int sms = device_sm_count();
    if (sms <= 0) return FM_ERR_CUDA;
    const unsigned grid = (unsigned)(units < sms ? units : sms);
    static std::atomic<unsigned> next_slot{0};
    FwdArgs args = a;
    args.sched_slot = (int)(next_slot.fetch_add(1, std::memory_order_relaxed) % kFwdSchedSlots);
    ProfScope ps(kKFwd, stream);
    fm_fwd_kernel<D, PRECISE, FP8><<<grid, 384, smem, stream>>>(tq, tk, tv, args);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_fwd_prepare(int d, bool precise)
{
    if (device_sm_count() <= 0) return FM_ERR_CUDA;   // cached before any stream capture
    const bool ok = d == 128 ? (precise ? fwd_smem_ready<128, true>() : fwd_smem_ready<128, false>())
                             : (precise ? fwd_smem_ready<64, true>() : fwd_smem_ready<64, false>());
    return ok ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_fwd_prepare_fp8()
{
    return (device_sm_count() > 0 && fwd_smem_ready<128, false, true>()) ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_fwd_launch_fp8(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tvt,
                            const FwdArgs &a, cudaStream_t stream)
{
    return launch_fwd<128, false, true>(tq, tk, tvt, a, stream);
}

fm_status fm_fwd_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const FwdArgs &a, int d, bool precise, cudaStream_t stream)
{
    if (d == 128)
        return precise ? launch_fwd<128, true>(tq, tk, tv, a, stream) : launch_fwd<128, false>(tq, tk, tv, a, stream);
    return precise ? launch_fwd<64, true>(tq, tk, tv, a, stream) : launch_fwd<64, false>(tq, tk, tv, a, stream);
}
