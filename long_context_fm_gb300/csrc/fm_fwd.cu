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
//   warps 2-5   softmax of the even tiles of the CTA-wide sequence, all 128
//               key columns of every row (thread = row = TMEM lane); each
//               warp turns the column bounds of its next partial tile into
//               bit masks over its 32 rows while it waits for the scores
//   warps 6-9   softmax of the odd tiles
//   warp 10     TMA producer of V (two-stage ring)
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
// t + 3 once that PV has read it.  The two softmax warpgroups take
// alternate tiles, so one's TMEM loads, waits and row max overlap the other's
// exponentials; the running row max passes from each tile's owner to the
// next through shared memory (a producer / consumer named barrier per
// direction, reached on every tile, also after an abort).  The owner of a
// tile that raises the max rescales O; each warpgroup keeps its own sum of P,
// and the epilogue combines the two and each stores half of O's columns.
// Precise mode: P = P_hi + P_lo (P_lo = bf16(P - bf16(P))) in columns
// [0, 64) and [64, 128) of the S buffer, both multiplied by V.
// Online softmax in the base-2 domain with a lazy rescale: O and l are
// rescaled only when the row max grows by more than 2^kLazy (kLazy = 32 for
// bf16 P, 8 for e4m3 P, whose largest value is 448), which keeps every P <=
// 2^kLazy and leaves the final O / l unchanged: a rescale makes the tile's
// softmax wait for the previous tile's P V, so the wider the band, the rarer
// that wait (with 2^8 the x2-scaled prefix workloads were 20-27 % slower).
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
    FB_S0, FB_S1, FB_S2,                              // scores of buffer b computed
    FB_P0, FB_P1, FB_P2,                              // P of buffer b written, first 64 keys
    FB_PB0, FB_PB1, FB_PB2,                           // P of buffer b written, last 64 keys
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
    static constexpr int kOst = kV + kVStages * kTile;         // O staging: [8 softmax warps][32 rows][64 bytes]
    static constexpr int kMask = kOst + 8 * 2048;              // uint32 [8 softmax warps][2 buffers][128 columns]
    static constexpr int kMax = kMask + 8 * 2 * 128 * 4;       // float [2 slots][2 warpgroups][128]: final m
    static constexpr int kSum = kMax + 2 * 2 * 128 * 4;        // float [2 slots][2 warpgroups][128]: l
    static constexpr int kUnit = kSum + 2 * 2 * 128 * 4;       // int4 [4]: unit ring (qt, bh, sidx, n)
    static constexpr int kFlag = kUnit + 4 * 16;               // int [2][8]: softmax warps' unit decisions
    static constexpr int kChain = kFlag + 16 * 4;              // float [128]: running row max handed between warpgroups
    static constexpr int kBar = kChain + 128 * 4;
    static constexpr int kNumBar = FB_COUNT;
    static constexpr int kMisc = kBar + kNumBar * 8;
    // At least 120 KB so that one CTA (512 TMEM columns) is resident per SM.
    static constexpr int kBytes = (kMisc + 64 > 120 * 1024) ? kMisc + 64 : 120 * 1024;
};


// Bits x of a 32-row group with lo <= x < hi (bounds clamped to [0, 32]): the
// bits at or above lo and below hi, as two clamping funnel shifts (a shift by
// 32 gives 0); empty when hi <= lo.
__device__ __forceinline__ uint32_t row_bits32(int lo, int hi)
{
    lo = min(max(lo, 0), 32);
    hi = min(max(hi, 0), 32);
    return __funnelshift_lc(0u, 0xffffffffu, (uint32_t)lo) & __funnelshift_rc(0xffffffffu, 0u, (uint32_t)(32 - hi));
}

constexpr int kSB = 3;              // score buffers in TMEM
constexpr int kUnitRing = 4;        // claimed units buffered between the K producer and the other roles
constexpr int kUnitReaders = 11;    // V producer, two MMA issuers, eight softmax warps

// Work counters of the persistent forward launches, one slot per launch in
// flight: {next unit to claim, CTAs finished}.  The host gives each launch
// its own slot (round robin); the launch's last CTA resets it to zero.
constexpr int kFwdSchedSlots = 64;
static __device__ unsigned int g_fwd_sched[kFwdSchedSlots][2];
constexpr int kSoftmaxBar = 1;      // named barrier of the two softmax warpgroups (256 threads)
// Register budgets (setmaxnreg): the four warps that issue copies or MMAs
// give registers to the eight softmax warps (128 scores each in registers);
// together they use the 384 x 168 registers the block launches with, which
// the host checks against the compiled kernel.
constexpr int kFwdLaunchRegs = 168;
constexpr int kRegsIssue = 56, kRegsSoftmax = 224;
static_assert(4 * 32 * kRegsIssue + 8 * 32 * kRegsSoftmax <= 384 * kFwdLaunchRegs, "register split of the forward");
constexpr int kChainBar = 2;        // 2 + w: row max handed on by warpgroup w (arrive) to the other (sync)

template <int D, bool PRECISE, bool FP8>
__global__ void __launch_bounds__(384, 1)
    fm_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to, const FwdArgs a)
{
    static_assert(!(PRECISE && FP8), "the FP8 path has no precise mode");
    static_assert(!FP8 || D == 128, "the FP8 path is built for d = 128");
    using S = FwdSmem<D, FP8>;
    // Lazy rescale band (base 2): P stays <= 2^kLazy.  bf16 P: terms below
    // 2^-94 of a row's maximum underflow to zero and the fp32 sums stay far
    // from overflow; e4m3 P: its largest finite value is 448.
    constexpr float kLazy = FP8 ? 8.f : 32.f;
    constexpr int BOXW = FP8 ? 128 : 64;          // elements per 128-byte box row
    constexpr int NBOX = D / BOXW;
    constexpr int KS = S::kKStages, VS = S::kVStages;
    // The kernel has no static shared memory, so the dynamic window starts on
    // a 1024-byte boundary (checked below).  Pointers stay derived from the
    // __shared__ array itself, so every access compiles to a shared-memory
    // instruction rather than a generic one.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint32_t *sMask = reinterpret_cast<uint32_t *>(smem + S::kMask);
    float *sMax = reinterpret_cast<float *>(smem + S::kMax);
    float *sSum = reinterpret_cast<float *>(smem + S::kSum);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 12);
    volatile int *dbg = reinterpret_cast<volatile int *>(smem + S::kMisc + 16);   // debug counters [3]
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
            }
            // One O barrier per score buffer: the PV of tile g commits to O_{g mod 3},
            // so every wait below targets a barrier at most one phase behind.
            for (int s = 0; s < kSB; ++s) {
                mbar_init(&bars[FB_S0 + s], 1);
                mbar_init(&bars[FB_P0 + s], 128);   // the tile's softmax warpgroup
                mbar_init(&bars[FB_PB0 + s], 128);
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
    if (kDebugChecks && threadIdx.x == 0 && (tmem & 0xffffu) != 0u) set_status(a.status, FM_ERR_DEBUG_CHECK);

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
            warp_regs_dec<kRegsIssue>();
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
            int k = 0;    // ring entries published (claims, the terminating one included)
            for (; run; ++k) {
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
                if (kDebugChecks && (u.n < 0 || u.n > L.n_k)) {
                    if (lane == 0) set_status(a.status, FM_ERR_DEBUG_CHECK);
                    *abort = 1;
                    break;
                }
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
                    if (kDebugChecks) {   // a KV tile of the row and a FULL or PARTIAL label
                        const int lab = (int)((unsigned)e_next >> kLabelShift);
                        if ((e_next & kTileMask) >= L.n_k || (lab != FM_TILE_FULL && lab != FM_TILE_PARTIAL)) {
                            if (lane == 0) set_status(a.status, FM_ERR_DEBUG_CHECK);
                            *abort = 1;
                            run = false;
                            break;
                        }
                    }
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
            if (kDebugChecks && lane == 0) dbg[2] = k + 1;
            // Drain copies still in flight (only possible after an abort).
            if (lane == 0 && *abort) {
                if (nq > 0) mbar_wait_drain(&bars[FB_Q], (nq - 1) & 1, a.status, a.wait_limit);
                for (int k2 = (g > KS ? g - KS : 0); k2 < g; ++k2)
                    if (k2 != withheld) mbar_wait_drain(&bars[FB_KF0 + (k2 % KS)], (k2 / KS) & 1, a.status, a.wait_limit);
            }
        } else if (warp == 10) {
            warp_regs_dec<kRegsIssue>();
            // ------------------------------------------------ V producer
            // V through its ring: the stage of tile g is free once the PV of tile
            // g - VS has completed.
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
                    const int vs = g % VS;
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
                }
            }
            if (lane == 0 && *abort)
                for (int k2 = (g > VS ? g - VS : 0); k2 < g; ++k2)
                    mbar_wait_drain(&bars[FB_VF0 + (k2 % VS)], (k2 / VS) & 1, a.status, a.wait_limit);
        } else if (warp == 1) {
            warp_regs_dec<kRegsIssue>();
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
                if (kDebugChecks) {
                    dbg[0] = g;
                    dbg[1] = nq;
                }
            }
        } else if (warp == 11) {
            warp_regs_dec<kRegsIssue>();
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
                        // The product in two halves over the keys: the first 64 as soon
                        // as their P is written, the rest once all of P is (the softmax
                        // releases the halves separately), so half of P V overlaps the
                        // second half's exponentials.
                        auto pv_half = [&](int h) {
                            if (FP8) {
                                // B = V^T, K-major (d rows of 128 key bytes); A = P, 4 e4m3 per column
                                const uint64_t dVt = sdesc_sw128(smem_u32(smem + S::kV + vs * S::kTile), 16, 1024);
#pragma unroll
                                for (int kk = 2 * h; kk < 2 * h + 2; ++kk)
                                    mma_ts_e4m3(tO, tP + kk * 8, sdesc_add(dVt, kk * 32), idesc_e4m3(128, D), (t > 0 || kk > 0));
                            } else {
                                const uint64_t dV = sdesc_sw128(smem_u32(smem + S::kV + vs * S::kTile), S::kBox, 1024);
#pragma unroll
                                for (int part = 0; part < NPART; ++part)   // P_hi V (+ P_lo V)
#pragma unroll
                                    for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
                                        mma_ts(tO, tP + part * 64 + kk * 8, sdesc_add(dV, kk * 2048), idO,
                                               (t > 0 || part > 0 || kk > 0));
                            }
                        };
                        pv_half(0);
                        if (!mbar_wait(&bars[FB_PB0 + g % kSB], (g / kSB) & 1, abort, a.status, a.wait_limit)) {
                            run = false;
                            break;
                        }
                        tc_fence_after();
                        pv_half(1);
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
            warp_regs_inc<kRegsSoftmax>();
            // ------------------------------------------------ softmax (warps 2-9)
            // Tile g of the CTA-wide sequence belongs to warpgroup g & 1 (warps 2-5
            // or 6-9; each covers all 128 TMEM lanes), which handles every key
            // column of its rows: thread = row = TMEM lane, 128 scores in registers.
            // The two warpgroups work on consecutive tiles at the same time, so the
            // TMEM loads, waits and row max of one overlap the exponentials of the
            // other.  Only the running row max passes from one tile to the next:
            // the owner of tile t > 0 of a unit takes the max in force after tile
            // t - 1 from the other warpgroup, decides its own and hands it on
            // before it computes its exponentials.  When the max rises the owner
            // rescales all of O once the P V of tile t - 1 has completed, before it
            // releases its own P; the P V products then accumulate in tile order.
            // Each warpgroup sums its own P relative to the max it last used; the
            // epilogue combines the two sums.
            const int w = (warp < 6) ? 0 : 1;          // warpgroup: owns the tiles g with g & 1 == w
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t tO = tmem + 384;
            constexpr int OC = D / 2;                  // O columns stored by this warpgroup
            // softmax scale * log2(e), with the Q and K descales on the FP8 path
            const float sl2 = FP8 ? a.scale_log2 * a.descale[0] * a.descale[1] : a.scale_log2;
            volatile float *sChain = reinterpret_cast<volatile float *>(smem + S::kChain);
            // `live` turns false (for the whole warp) when a wait gives up after an
            // abort; the warp then skips its work but still reaches every named
            // barrier of the loop, so the other warpgroup is never left waiting.
            bool live = true;
            // The PV of tile k has completed (and with it every earlier MMA).
            auto wait_pv = [&](int k) {
                live = live && warp_wait(&bars[FB_O0 + k % kSB], (k / kSB) & 1, abort, a.status, a.wait_limit);
            };
            int g = 0;     // tiles begun (CTA-wide, both warpgroups)
            int nu = 0;    // units with tiles finished
            int nbf = 0;   // this warpgroup's partial tiles (their masks alternate between two buffers)
            int mflag = 0; // build_mask's summary of the mask built last (read by the tile it is for)
            uint32_t *sMaskW = sMask + (warp - 2) * 256;   // this warp's two mask buffers
            // The mask of a partial tile as bits over this warp's 32 rows of the Q
            // tile (mask rows r0 + 32 quarter + x): word c has bit x set when that
            // row lies in [lts, lte) or [uts, ute) of the tile's column c; columns
            // beyond N are masked in every row.  Lane j covers columns 4 j .. 4 j + 3.
            // Built by the warp itself between its tiles, read back by all its lanes:
            // the bounds are loaded one tile ahead (load_bounds at the start of the
            // warpgroup's previous tile) and turned into bits after that tile's P
            // is released (build_mask).
            int4 bnd[4];
            // Four 16-byte loads (one per bound array) when every row of the
            // arrays starts on a 16-byte boundary: the host accepts only 16-byte
            // aligned arrays, so that holds when N is a multiple of 4.
            const bool vec_ok = (N & 3) == 0;
            auto load_bounds = [&](int e, const Unit &uu) {
                const int kb = (e & kTileMask) * 128;
                const int j0 = kb + lane * 4;
                const int64_t o0 = (int64_t)uu.sidx * N + j0;
                if (vec_ok && j0 + 4 <= N) {
                    const int4 x = *reinterpret_cast<const int4 *>(a.lts + o0), y = *reinterpret_cast<const int4 *>(a.lte + o0);
                    const int4 z = *reinterpret_cast<const int4 *>(a.uts + o0), u = *reinterpret_cast<const int4 *>(a.ute + o0);
                    bnd[0] = make_int4(x.x, y.x, z.x, u.x);
                    bnd[1] = make_int4(x.y, y.y, z.y, u.y);
                    bnd[2] = make_int4(x.z, y.z, z.z, u.z);
                    bnd[3] = make_int4(x.w, y.w, z.w, u.w);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        bnd[c] = make_int4(0, 0, 0, 0);
                        if (j0 + c < N) bnd[c] = make_int4(a.lts[o0 + c], a.lte[o0 + c], a.uts[o0 + c], a.ute[o0 + c]);
                    }
                }
            };
            // Returns, for the whole warp, 0 when none of its rows is masked in the
            // tile, 1 when all of them are masked in every column, else 2.
            auto build_mask = [&](int e, const Unit &uu, uint32_t *dst) -> int {
                const int kb = (e & kTileMask) * 128;
                const int base = a.q_row0 + uu.qt * 128 + quarter * 32;
                uint32_t wq[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int4 v = bnd[c];
                    wq[c] = (kb + lane * 4 + c < N)
                                ? (row_bits32(v.x - base, v.y - base) | row_bits32(v.z - base, v.w - base))
                                : 0xffffffffu;
                }
                *reinterpret_cast<uint4 *>(dst + lane * 4) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                const uint32_t any = __reduce_or_sync(0xffffffffu, wq[0] | wq[1] | wq[2] | wq[3]);
                const uint32_t all = __reduce_and_sync(0xffffffffu, wq[0] & wq[1] & wq[2] & wq[3]);
                __syncwarp();
                return any == 0u ? 0 : (all == 0xffffffffu ? 1 : 2);
            };
            auto is_partial = [&](int e) {
                return ((e >> kLabelShift) == FM_TILE_PARTIAL) || (e & kTileMask) * 128 + 128 > N;
            };
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
                float m = -INFINITY;   // the max this warpgroup last used (scaled, base 2)
                float l = 0.f;         // this warpgroup's sum of P, relative to m
                const int g0 = g;
                const int t0 = (w - g0) & 1;               // this warpgroup's first tile of the unit
                int e_next = t0 < un.n ? un.list[t0] : 0;
                if (live && t0 < un.n && is_partial(e_next)) {
                    load_bounds(e_next, un);
                    mflag = build_mask(e_next, un, sMaskW + (nbf & 1) * 128);
                }
                for (int t = t0; t < un.n; t += 2) {
                    const int gt = g0 + t;
                    const int e = e_next;
                    if (t + 2 < un.n) e_next = un.list[t + 2];
                    const bool next_pred = t + 2 < un.n && is_partial(e_next);
                    if (live && next_pred) load_bounds(e_next, un);   // consumed after this tile's P
                    const int kb = (e & kTileMask) * 128;
                    const bool pred = ((e >> kLabelShift) == FM_TILE_PARTIAL) || kb + 128 > N;
                    const int bb = gt % kSB;
                    const uint32_t tS = tmem + bb * 128;
                    live = live && warp_wait(&bars[FB_S0 + bb], (gt / kSB) & 1, abort, a.status, a.wait_limit);
                    uint32_t sv[128];                      // the row's scores (fp32 bits)
                    float mx = -INFINITY;
                    const uint4 *mk = reinterpret_cast<const uint4 *>(sMaskW + (nbf & 1) * 128);
                    if (pred) ++nbf;
                    if (live) {
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            tmem_ld32(tS + lane_off + c * 32, reinterpret_cast<uint32_t (&)[32]>(sv[c * 32]));
                        tmem_ld_wait();
                        tmem_reg_fence(sv);
                        if (pred && mflag != 0) {
                            // The lane is the bit of its row; masked scores become -inf
                            // (every score when the whole warp is masked, mflag == 1).
                            const uint32_t lb = 1u << lane;
                            const uint32_t all = (mflag == 1) ? 0xffffffffu : 0u;
#pragma unroll
                            for (int c4 = 0; c4 < 32; ++c4) {
                                const uint4 mw = mk[c4];
                                sv[4 * c4 + 0] = ((mw.x | all) & lb) ? 0xff800000u : sv[4 * c4 + 0];
                                sv[4 * c4 + 1] = ((mw.y | all) & lb) ? 0xff800000u : sv[4 * c4 + 1];
                                sv[4 * c4 + 2] = ((mw.z | all) & lb) ? 0xff800000u : sv[4 * c4 + 2];
                                sv[4 * c4 + 3] = ((mw.w | all) & lb) ? 0xff800000u : sv[4 * c4 + 3];
                            }
                        }
                        float mx4[4] = {__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2]),
                                        __uint_as_float(sv[3])};
#pragma unroll
                        for (int k2 = 0; k2 < 62; ++k2)
                            mx4[k2 & 3] = fmax3(mx4[k2 & 3], __uint_as_float(sv[4 + 2 * k2]), __uint_as_float(sv[5 + 2 * k2]));
                        mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;   // -inf stays -inf
                    }
                    // The max in force after tile t - 1, this tile's decision, and the
                    // hand-over to the owner of tile t + 1 (named barrier kChainBar + the
                    // producer's warpgroup: bar.arrive by the producer, bar.sync by the
                    // consumer).  Both sides depend only on t and n, so they stay
                    // matched on every tile, also after an abort.
                    float m_prev = -INFINITY;
                    if (t > 0) {
                        named_bar_sync(kChainBar + (1 - w), 256);
                        m_prev = sChain[r];
                    }
                    const float m_new = (mx > m_prev + kLazy) ? mx : m_prev;
                    if (t + 1 < un.n) {
                        sChain[r] = m_new;
                        named_bar_arrive(kChainBar + w, 256);
                    }
                    if (!live) continue;
                    // O holds tiles 0 .. t - 1 relative to m_prev: rescale it when the
                    // max rose (rare with the 2^kLazy band), after their P V completed.
                    if (__any_sync(0xffffffffu, t > 0 && m_new != m_prev)) {
                        const float alpha = (m_new != m_prev) ? ex2(m_prev - m_new) : 1.f;   // m_prev = -inf gives 0
                        wait_pv(gt - 1);
                        if (!live) continue;
                        tc_fence_after();
#pragma unroll
                        for (int cc = 0; cc < D / 16; ++cc) {
                            uint32_t ov[16];
                            tmem_ld16(tO + lane_off + cc * 16, ov);
                            tmem_ld_wait();
                            tmem_reg_fence(ov);
#pragma unroll
                            for (int u = 0; u < 16; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
                            tmem_st16(tO + lane_off + cc * 16, ov);
                        }
                    }
                    // P = exp2(s * scale*log2e - m) as packed bf16 over the first 64
                    // columns of the S buffer (precise mode: P_lo over the next 64; FP8:
                    // four e4m3 per column over the first 32).  O is normalised by the
                    // fp32 sum of P, which also gives lse (standard mode: the bf16
                    // rounding of the weights P V applied moves that sum by ~2^-9
                    // relative at most, far inside the tolerance).  Column pairs in
                    // packed fp32.
                    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                    const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_use, -m_use);
                    uint32_t f8[32];          // FP8: the row's 128 P values, 4 e4m3 per column
                    uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {          // 32 keys per step
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[hh * 32 + 2 * cc]), __uint_as_float(sv[hh * 32 + 2 * cc + 1])),
                                             sc2, nm2),
                                      x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            sum2 = f2_add(sum2, f2_pack(p0, p1));
                            if (FP8) {
                                const uint32_t e2 = pack_e4m3x2(p0, p1);     // keys hh*32 + 2 cc, + 1
                                if (cc & 1) f8[hh * 8 + (cc >> 1)] |= e2 << 16;
                                else f8[hh * 8 + (cc >> 1)] = e2;
                            } else {
                                hi[cc] = pack_bf16x2(p0, p1);
                                if (PRECISE)
                                    lo[cc] = pack_bf16x2(p0 - __uint_as_float(hi[cc] << 16),
                                                         p1 - __uint_as_float(hi[cc] & 0xffff0000u));
                            }
                        }
                        if (!FP8) tmem_st16(tS + lane_off + hh * 16, hi);
                        if (PRECISE) tmem_st16(tS + lane_off + 64 + hh * 16, lo);
                        if (hh == 1) {
                            // The first 64 keys' P is complete: release it to P V.
                            if (FP8) tmem_st16(tS + lane_off, reinterpret_cast<const uint32_t (&)[16]>(f8[0]));
                            tmem_st_wait();
                            tc_fence_before();
                            mbar_arrive(&bars[FB_P0 + bb]);
                        }
                    }
                    if (FP8) tmem_st16(tS + lane_off + 16, reinterpret_cast<const uint32_t (&)[16]>(f8[16]));
                    float s0, s1;
                    f2_unpack(sum2, s0, s1);
                    l = (m == m_new ? l : l * ex2(m - m_new)) + (s0 + s1);
                    m = m_new;
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(&bars[FB_PB0 + bb]);
                    // The mask of this warpgroup's next tile, while it waits for its scores.
                    if (next_pred) mflag = build_mask(e_next, un, sMaskW + (nbf & 1) * 128);
                }
                g = g0 + un.n;
                // ------------------------------------------------ epilogue
                // Combine the two warpgroups' sums at the final max, the larger of
                // the two they last used (one more named barrier, reached by every
                // thread of both; the slot alternates between units), then each
                // stores its half of O's columns after the last PV.  O is released to
                // the next unit's first PV as soon as it is in registers.  A unit
                // without tiles writes O = 0, lse = -inf.
                const int su = nu & 1;
                if (un.n > 0) {
                    sSum[(su * 2 + w) * 128 + r] = l;
                    sMax[(su * 2 + w) * 128 + r] = m;
                    named_bar_sync(kSoftmaxBar, 256);
                    wait_pv(g - 1);
                }
                if (live) {
                    uint32_t ov[OC];
                    float lt = 0.f, mf = -INFINITY;
                    if (un.n > 0) {
                        tc_fence_after();
                        const float m0 = sMax[(su * 2) * 128 + r], m1 = sMax[(su * 2 + 1) * 128 + r];
                        const float l0 = sSum[(su * 2) * 128 + r], l1 = sSum[(su * 2 + 1) * 128 + r];
                        mf = fmaxf(m0, m1);   // l_w > 0 implies a finite m_w <= mf
                        lt = (l0 > 0.f ? l0 * ex2(m0 - mf) : 0.f) + (l1 > 0.f ? l1 * ex2(m1 - mf) : 0.f);
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
                    // O leaves through shared memory and TMA stores: the warp stages
                    // its 32 rows x 64 bytes (16 fp32 or 32 bf16 columns) at a time in
                    // a buffer of its own with the 64-byte swizzle (16-byte chunk q of
                    // row x at chunk q ^ ((x >> 1) & 3): conflict-free), and the copy
                    // engine writes whole row segments and drops rows at or beyond
                    // Nq.  A buffer is rewritten once the previous store has read it.
                    uint8_t *stg = smem + S::kOst + (warp - 2) * 2048;
                    const int y0 = un.qt * 128 + quarter * 32;
                    auto stage_store = [&](const uint4 (&pk)[4], int x) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 4; ++q) st_shared_v4(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), pk[q]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&to, stg, x, y0, un.bh);
                            bulk_commit();
                        }
                    };
                    if (a.o_f32) {
#pragma unroll
                        for (int c = 0; c < OC / 16; ++c) {
                            uint4 pk[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                pk[q] = make_uint4(__float_as_uint(__uint_as_float(ov[c * 16 + 4 * q]) * inv),
                                                   __float_as_uint(__uint_as_float(ov[c * 16 + 4 * q + 1]) * inv),
                                                   __float_as_uint(__uint_as_float(ov[c * 16 + 4 * q + 2]) * inv),
                                                   __float_as_uint(__uint_as_float(ov[c * 16 + 4 * q + 3]) * inv));
                            stage_store(pk, w * OC + c * 16);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < OC / 32; ++c) {
                            uint4 pk[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const uint32_t *oc = ov + c * 32 + 8 * q;
                                pk[q] = make_uint4(pack_bf16x2(__uint_as_float(oc[0]) * inv, __uint_as_float(oc[1]) * inv),
                                                   pack_bf16x2(__uint_as_float(oc[2]) * inv, __uint_as_float(oc[3]) * inv),
                                                   pack_bf16x2(__uint_as_float(oc[4]) * inv, __uint_as_float(oc[5]) * inv),
                                                   pack_bf16x2(__uint_as_float(oc[6]) * inv, __uint_as_float(oc[7]) * inv));
                            }
                            stage_store(pk, w * OC + c * 32);
                        }
                    }
                    if (w == 0 && li < a.Nq)
                        a.lse[(int64_t)un.bh * a.Nq + li] = (lt > 0.f) ? (mf + __log2f(lt)) * 0.69314718055994531f : -INFINITY;
                } else if (un.n > 0) {
                    mbar_arrive(&bars[FB_OE]);   // after an abort: nothing reads O any more
                }
                if (un.n > 0) ++nu;
            }
            // Every TMA store of O has completed before the CTA leaves.
            if (lane == 0) bulk_wait_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    // Debug build: every pipeline barrier has completed as many phases as the
    // CTA's tiles (g), units with tiles and ring entries imply.
    if (kDebugChecks && threadIdx.x == 0 && *ok_sh && !*abort) {
        const int G = dbg[0], NU = dbg[1], NK = dbg[2];
        auto cnt = [](int total, int period, int idx) { return total > idx ? (total - 1 - idx) / period + 1 : 0; };
        bool good = mbar_phase_count_ok(&bars[FB_Q], NU) && mbar_phase_count_ok(&bars[FB_QE], NU) &&
                    mbar_phase_count_ok(&bars[FB_OE], NU) && mbar_phase_count_ok(&bars[FB_DRAIN], 1);
        for (int b = 0; b < kSB; ++b) {
            const int c = cnt(G, kSB, b);
            good = good && mbar_phase_count_ok(&bars[FB_S0 + b], c) && mbar_phase_count_ok(&bars[FB_P0 + b], c) &&
                   mbar_phase_count_ok(&bars[FB_PB0 + b], c) && mbar_phase_count_ok(&bars[FB_O0 + b], c);
        }
        for (int s2 = 0; s2 < KS; ++s2)
            good = good && mbar_phase_count_ok(&bars[FB_KF0 + s2], cnt(G, KS, s2)) &&
                   mbar_phase_count_ok(&bars[FB_KE0 + s2], cnt(G, KS, s2));
        for (int s2 = 0; s2 < VS; ++s2)
            good = good && mbar_phase_count_ok(&bars[FB_VF0 + s2], cnt(G, VS, s2)) &&
                   mbar_phase_count_ok(&bars[FB_VE0 + s2], cnt(G, VS, s2));
        for (int s2 = 0; s2 < kUnitRing; ++s2)
            good = good && mbar_phase_count_ok(&bars[FB_UF0 + s2], cnt(NK, kUnitRing, s2)) &&
                   mbar_phase_count_ok(&bars[FB_UE0 + s2], cnt(NK, kUnitRing, s2));
        if (!good) set_status(a.status, FM_ERR_DEBUG_CHECK);
    }
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
    // The warps' register budgets add up to the launch allocation only if the
    // kernel was compiled to exactly kFwdLaunchRegs per thread.
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, fm_fwd_kernel<D, PRECISE, FP8>) != cudaSuccess || fa.numRegs != kFwdLaunchRegs)
        return false;
    if (cudaFuncSetAttribute(fm_fwd_kernel<D, PRECISE, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return false;
    done[dev].store(1, std::memory_order_release);
    return true;
}

template <int D, bool PRECISE, bool FP8 = false>
static fm_status launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &to, const FwdArgs &a, cudaStream_t stream)
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
    fm_fwd_kernel<D, PRECISE, FP8><<<grid, 384, smem, stream>>>(tq, tk, tv, to, args);
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
                            const CUtensorMap &to, const FwdArgs &a, cudaStream_t stream)
{
    return launch_fwd<128, false, true>(tq, tk, tvt, to, a, stream);
}

fm_status fm_fwd_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &to, const FwdArgs &a, int d, bool precise, cudaStream_t stream)
{
    if (d == 128)
        return precise ? launch_fwd<128, true>(tq, tk, tv, to, a, stream)
                       : launch_fwd<128, false>(tq, tk, tv, to, a, stream);
    return precise ? launch_fwd<64, true>(tq, tk, tv, to, a, stream) : launch_fwd<64, false>(tq, tk, tv, to, a, stream);
}
