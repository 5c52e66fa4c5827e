// Backward masked attention on sm_103a: preprocess, main kernel, dQ
// postprocess.
//
// The gradients are those of plain masked softmax attention (the method is
// exact: blog "FlashMask技术" §2.2, arXiv 2410.01359 abstract), with the
// same tile skipping as the forward (blog §2.2): fully masked (Q tile, KV
// tile) pairs are never visited, fully visible pairs run without mask
// arithmetic, only partial pairs evaluate the column-interval predicate.
//
// Main kernel: one CTA = one (b, h, 128-row KV tile); it walks the plan's
// list of non-skip Q tiles of that KV tile (staged in shared memory), each as
// two 64-row halves.
//   warp 0      TMA producer (K and V once; Q, dO halves in a ring of three
//               stages; lse and D staged into shared memory by the whole warp)
//   warp 1      TMEM allocation; one thread issues the S^T MMAs
//   warps 2-17  four warpgroups, one thread per KV row j each: P^T and dS^T
//               for 16 of the half's 64 columns each
//   warps 18-21 one thread per head-dim index: drain dQ^T from TMEM into the
//               fp32 dQ accumulator with red.global.add (the caller's fp32 dQ,
//               scaled on the way, or the workspace accumulator that the
//               postprocess scales and converts to bf16)
//   warp 22     one thread issues the dQ^T MMAs
//   warp 23     one thread issues the dP^T MMAs
//   warp 24     one thread issues the dV, then dK MMAs
// The four issuing threads sit on four different sub-partitions, each
// product stream waiting only for its own inputs.
// TMEM (512 columns): dK [0, d), dV [128, 128 + d), two score buffers
// b = half & 1 with S^T [256 + 128 b, +64) and dP^T [320 + 128 b, +64).  Each
// thread overwrites the S^T columns it has read with its P^T as packed bf16
// (the A operand of dV), and the half's dQ^T lands in the dP^T columns after
// dS^T is written, so the scores of the next half run while this half is
// still being processed.
// Per half (M = 128 KV rows):
//   S^T  = K Q^T        (SS, K-major/K-major)        -> TMEM
//   dP^T = V dO^T       (SS, K-major/K-major)        -> TMEM
//   P^T  = exp2(S^T * scale*log2e - lse*log2e) as soon as S^T is written,
//   dS^T = P^T o (dP^T - D) once dP^T is written (separate barriers)
//          P^T written as bf16 into TMEM, dS^T into 128-byte-swizzled
//          shared memory (precise mode: each as two bf16 terms hi + lo, ~16
//          significant bits, both consumed by the MMAs below, so the
//          gradients do not carry a bf16 rounding of P or dS)
//   dV  += P^T dO       (TS, P^T from TMEM, dO MN-major)
//   dK  += dS^T Q       (SS, dS^T K-major, Q MN-major)
//   dQ^T = K^T dS^T     (SS, K MN-major, dS^T MN-major)
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

// ---------------------------------------------------------------- preprocess
// D[row] = sum_k dO[row, k] * O[row, k]; dQacc[row, :] = 0.  One warp per row.
template <int D>
__global__ void __launch_bounds__(256) fm_bwd_pre_kernel(const void *o, int o_f32, const uint16_t *dO,
                                                         float *Dout, float *dq_acc, int64_t rows)
{
    constexpr int PER = D / 32;   // elements per lane: 4 or 2
    const int lane = threadIdx.x & 31;
    int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (; row < rows; row += stride) {
        const int64_t base = row * D + lane * PER;
        float ov[PER], dv[PER];
        if (o_f32) {
            const float *op = reinterpret_cast<const float *>(o) + base;
            if constexpr (PER == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(op);
                ov[0] = x.x; ov[1] = x.y; ov[2] = x.z; ov[3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(op);
                ov[0] = x.x; ov[1] = x.y;
            }
        } else {
            const uint16_t *op = reinterpret_cast<const uint16_t *>(o) + base;
#pragma unroll
            for (int u = 0; u < PER; ++u) ov[u] = __uint_as_float((uint32_t)op[u] << 16);
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) dv[u] = __uint_as_float((uint32_t)dO[base + u] << 16);
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < PER; ++u) acc = fmaf(ov[u], dv[u], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) Dout[row] = acc;
        float *z = dq_acc + base;
#pragma unroll
        for (int u = 0; u < PER; ++u) z[u] = 0.f;
    }
}

// ---------------------------------------------------------------- postprocess
// bf16 gradients: dQ = scale * dQacc, rounded to bf16.  4 elements per thread.
// (fp32 gradients need no postprocess: the main kernel adds scale * dQ^T into
// the caller's buffer directly.)
__global__ void __launch_bounds__(256) fm_bwd_post_kernel(const float *dq_acc, uint16_t *dq, float scale,
                                                          int64_t n4)
{
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4;
         t += (int64_t)gridDim.x * blockDim.x) {
        const float4 x = reinterpret_cast<const float4 *>(dq_acc)[t];
        uint2 w;
        w.x = pack_bf16x2(x.x * scale, x.y * scale);
        w.y = pack_bf16x2(x.z * scale, x.w * scale);
        reinterpret_cast<uint2 *>(dq)[t] = w;
    }
}

// ---------------------------------------------------------------- main kernel
enum {
    BB_KV = 0, BB_QF0, BB_QF1, BB_QF2, BB_QE0, BB_QE1, BB_QE2, BB_SF0, BB_SF1, BB_DF0, BB_DF1, BB_PF0, BB_PF1,
    BB_PE0, BB_PE1, BB_DSE0, BB_DSE1, BB_DQF0, BB_DQF1, BB_DQE0, BB_DQE1, BB_ACC, BB_DRAIN0, BB_DRAIN1, BB_SFD0, BB_SFD1,
    BB_KVE,                                   // the unit's S^T, dP^T and dQ^T have read K and V
    BB_ACCE,                                  // the unit's epilogue has read dK and dV
    BB_STG,                                   // every P/dS warp's dK / dV stores have read their staging
    BB_UF0, BB_UF1, BB_UF2, BB_UF3,           // unit ring: claimed unit written
    BB_UE0, BB_UE1, BB_UE2, BB_UE3,           // unit ring: every reader has read it
    BB_COUNT
};

constexpr int kBwdUnitRing = 4;       // claimed units buffered between the producer and the other roles
constexpr int kBwdUnitReaders = 24;   // four MMA-issuing warps, 16 P/dS warps, 4 drain warps

// Work counters of the persistent backward launches, one slot per launch in
// flight: {next unit to claim, CTAs finished}.  The host gives each launch its
// own slot (round robin); the launch's last CTA resets it to zero.
constexpr int kBwdSchedSlots = 64;
static __device__ unsigned int g_bwd_sched[kBwdSchedSlots][2];

template <int D, bool PRECISE>
struct BwdSmem {
    // Three Q/dO stages (a stage's next load is in flight while the two
    // halves before it are processed).  Standard mode keeps two dS^T tiles
    // (dK and dQ^T of half i still read dS^T while half i+1 is written);
    // precise mode one, the low terms taking the room of the second.
    static constexpr int kStages = 3;
    static constexpr int kdSBufs = PRECISE ? 1 : 2;
    static constexpr int kKBox = 128 * 128;     // 64 columns x 128 rows
    static constexpr int kQBox = 64 * 128;      // 64 columns x 64 rows
    static constexpr int kKTile = 128 * D * 2;
    static constexpr int kQTile = 64 * D * 2;
    static constexpr int kOp = 128 * 128;       // one 128 x 64 bf16 operand tile
    static constexpr int kK = 0, kV = kKTile;
    static constexpr int kQ = 2 * kKTile;                   // [kStages]
    static constexpr int kdO = kQ + kStages * kQTile;       // [kStages]
    static constexpr int kdS = kdO + kStages * kQTile;      // dS^T (high part)  [kdSBufs]
    static constexpr int kdSlo = kdS + kdSBufs * kOp;       // precise: dS^T low part
    // dK / dV staging: the dS^T tiles and these 32 KB after them (64 KB,
    // contiguous in both modes): [16 warps][32 rows][128 bytes].
    static constexpr int kOst = PRECISE ? kdSlo + kOp : kdSlo;
    static_assert(kOst == kdS + 32768, "the staging of the dK / dV stores follows the dS^T tiles");
    static constexpr int kUnit = kOst + 16 * 2048;          // int [kBwdUnitRing][4]: unit ring
    static constexpr int kStat = kUnit + kBwdUnitRing * 16;  // -lse*log2e [kStages][64], D [kStages][64]
    static constexpr int kBar = kStat + 2 * kStages * 64 * 4;
    static constexpr int kNumBar = BB_COUNT;
    static constexpr int kMisc = kBar + kNumBar * 8;
    // At least 120 KB so that one CTA (512 TMEM columns) is resident per SM.
    static constexpr int kBytes = (kMisc + 64 + 1024 > 120 * 1024) ? kMisc + 64 + 1024 : 120 * 1024;
};


// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): the pair carries about
// 16 significant bits, so products summed by the tensor core from both
// halves lose far less than one bf16 rounding of x.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}


template <int D, bool PRECISE>
__global__ void __launch_bounds__(800, 1)
    fm_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                  const BwdArgs a)
{
    using S = BwdSmem<D, PRECISE>;
    constexpr int NBOX = D / 64;
    // The kernel has no static shared memory, so the dynamic window starts on
    // a 1024-byte boundary (checked below).  Pointers stay derived from the
    // __shared__ array itself, so every access compiles to a shared-memory
    // instruction rather than a generic one.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint8_t *sK = smem + S::kK, *sV = smem + S::kV;
    uint8_t *sQ = smem + S::kQ, *sdO = smem + S::kdO;
    uint8_t *sdS = smem + S::kdS, *sdSlo = smem + S::kdSlo;
    constexpr int NST = S::kStages;
    float *sLse = reinterpret_cast<float *>(smem + S::kStat);     // [NST][64]
    float *sD = sLse + NST * 64;                                     // [NST][64]
    volatile int *sUnit = reinterpret_cast<volatile int *>(smem + S::kUnit);   // [kBwdUnitRing][4]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 12);
    volatile int *dbg = reinterpret_cast<volatile int *>(smem + S::kMisc + 16);   // debug counters [3]

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
            mbar_init(&bars[BB_KV], 1);
            for (int s2 = 0; s2 < NST; ++s2) {
                mbar_init(&bars[BB_QF0 + s2], 33);
                mbar_init(&bars[BB_QE0 + s2], 3);     // S^T, dP^T and dV/dK issuers
            }
            mbar_init(&bars[BB_SF0], 1);      // S^T written
            mbar_init(&bars[BB_SF1], 1);
            mbar_init(&bars[BB_SFD0], 1);     // dP^T written
            mbar_init(&bars[BB_SFD1], 1);
            mbar_init(&bars[BB_DF0], 512);    // four P/dS warpgroups: dS^T written
            mbar_init(&bars[BB_DF1], 512);
            mbar_init(&bars[BB_PF0], 512);    // P^T written
            mbar_init(&bars[BB_PF1], 512);
            mbar_init(&bars[BB_PE0], 1);      // dV has read P^T
            mbar_init(&bars[BB_PE1], 1);
            mbar_init(&bars[BB_DSE0], 2);     // dQ^T and dK read dS^T
            mbar_init(&bars[BB_DSE1], 2);
            mbar_init(&bars[BB_DQF0], 1);
            mbar_init(&bars[BB_DQF1], 1);
            mbar_init(&bars[BB_DQE0], 128);
            mbar_init(&bars[BB_DQE1], 128);
            mbar_init(&bars[BB_ACC], 1);
            mbar_init(&bars[BB_KVE], 3);      // S^T, dP^T and dQ^T issuers, after a unit's last product
            mbar_init(&bars[BB_ACCE], 512);   // P/dS threads, after the unit's dK, dV epilogue
            mbar_init(&bars[BB_STG], 16);     // lane 0 of each P/dS warp, after its stores read the staging
            for (int s2 = 0; s2 < kBwdUnitRing; ++s2) {
                mbar_init(&bars[BB_UF0 + s2], 1);
                mbar_init(&bars[BB_UE0 + s2], kBwdUnitReaders);
            }
            mbar_init(&bars[BB_DRAIN0], 4);   // all four issuers
            mbar_init(&bars[BB_DRAIN1], 1);
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
    // TMEM: dK, dV, then two score buffers b = half & 1: S^T at 256 + 128 b
    // (then P^T), dP^T at 320 + 128 b (then dQ^T, once dS^T has been written).
    const uint32_t tdK = tmem, tdV = tmem + 128, tS0 = tmem + 256, tdP0 = tmem + 320;
    const int Nq = a.Nq;

    // Persistent CTAs with dynamic scheduling: the producer of each CTA claims
    // the next work unit (b, h, 128-row KV tile) of the plan's longest-first
    // order from the launch's counter whenever it is ready for one, so the CTAs
    // that run at the same time work on neighbouring units of the order and the
    // longest lists start first.  Claimed units pass to the other roles through
    // a ring of kBwdUnitRing entries in shared memory (n_it = -1 ends it).
    // Every role walks the same units and, across units, one CTA-wide sequence
    // of 64-row Q halves G: stages, score and dS^T buffers and barrier phases
    // follow G, so the next unit's loads and products start while the current
    // unit's epilogue stores dK and dV.
    const int64_t n_units = (int64_t)a.B * a.H * L.n_k;
    unsigned int *sched = g_bwd_sched[a.sched_slot];
    struct Unit {
        int kt, bh, sidx, n_it;     // n_it: 64-row Q halves of the unit's list
        const int32_t *list;
    };
    auto list_of = [&](const Unit &u) {
        return reinterpret_cast<const int32_t *>(a.plan + L.off_col_list) + ((int64_t)u.sidx * L.n_k + u.kt) * L.n_q;
    };
    // First row of half it of a unit (only the last Q tile can have a second
    // half beyond the Q rows, and it is last in the list).
    auto q0_of = [&](const Unit &u, int it) { return (u.list[it >> 1] & kTileMask) * 128 + (it & 1) * 64; };
    // Called by all 32 lanes of a warp; false on a plan that was not written by
    // the classifier (reported).
    auto unit_from = [&](int c, Unit &u) -> bool {
        int ut = 0, uh = 0, ub = 0;
        if (!plan_unit(reinterpret_cast<const int32_t *>(a.plan + L.off_col_order),
                       reinterpret_cast<const int32_t *>(a.plan + L.off_col_bstart), L.n_k, a.B, a.Hm, a.H, c,
                       &ut, &uh, &ub)) {
            if (lane == 0) set_status(a.status, FM_ERR_PLAN_MISMATCH);
            return false;
        }
        u.kt = ut;
        u.bh = ub * a.H + uh;
        u.sidx = ub * a.Hm + (a.Hm == 1 ? 0 : uh);
        u.list = list_of(u);
        const int cnt = reinterpret_cast<const int32_t *>(a.plan + L.off_col_cnt)[(int64_t)u.sidx * L.n_k + ut];
        u.n_it = (cnt > 0 && (u.list[cnt - 1] & kTileMask) * 128 + 64 >= Nq) ? 2 * cnt - 1 : 2 * cnt;
        return true;
    };
    // Unit k of the ring for a reading warp: waits until it has been claimed,
    // reads it and releases the entry (lane 0 arrives for the warp); false when
    // the sequence has ended or a wait gave up.
    auto read_unit = [&](int k, Unit &u) -> bool {
        const int slot = k % kBwdUnitRing;
        if (!warp_wait(&bars[BB_UF0 + slot], (k / kBwdUnitRing) & 1, abort, a.status, a.wait_limit)) return false;
        u.kt = sUnit[slot * 4 + 0];
        u.bh = sUnit[slot * 4 + 1];
        u.sidx = sUnit[slot * 4 + 2];
        u.n_it = sUnit[slot * 4 + 3];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[BB_UE0 + slot]);
        u.list = list_of(u);
        return u.n_it >= 0;
    };

    if (*ok_sh) {
        if (warp == 0) {
            // ------------------------------------------------ producer
            // Claims units; per unit with halves: K, V (once the previous unit's
            // S^T, dP^T and dQ^T have read them), then the Q and dO halves through
            // the three-stage ring, lse and D staged with each.
            if (lane == 0) {
                tma_prefetch_desc(&tq); tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv); tma_prefetch_desc(&tdo);
            }
            int G = 0;      // halves begun (CTA-wide)
            int nkv = 0;    // K / V loads begun (units with halves)
            // Test hook: the first CTA withholds the Q/dO load of its second half,
            // so that the scores' wait for it runs out (never set by a product call).
            const int withheld = (a.withhold && blockIdx.x == 0) ? 1 : -1;
            bool run = true;
            Unit u;
            int k = 0;      // ring entries published (claims, the terminating one included)
            for (; run; ++k) {
                // Claim the next unit into ring entry k once every reader is done
                // with the entry's previous unit.
                const int slot = k % kBwdUnitRing;
                if (k >= kBwdUnitRing &&
                    !warp_wait(&bars[BB_UE0 + slot], ((k / kBwdUnitRing) - 1) & 1, abort, a.status, a.wait_limit))
                    break;
                int c = 0;
                if (lane == 0) c = (int)atomicAdd(&sched[0], 1u);
                c = __shfl_sync(0xffffffffu, c, 0);
                bool valid = c < n_units;
                if (valid && !unit_from(c, u)) valid = false;
                if (lane == 0) {
                    sUnit[slot * 4 + 0] = valid ? u.kt : 0;
                    sUnit[slot * 4 + 1] = valid ? u.bh : 0;
                    sUnit[slot * 4 + 2] = valid ? u.sidx : 0;
                    sUnit[slot * 4 + 3] = valid ? u.n_it : -1;
                    mbar_arrive(&bars[BB_UF0 + slot]);
                }
                if (!valid) break;
                if (kDebugChecks && (u.n_it < 0 || u.n_it > 2 * L.n_q)) {
                    if (lane == 0) set_status(a.status, FM_ERR_DEBUG_CHECK);
                    *abort = 1;
                    break;
                }
                if (u.n_it == 0) continue;
                if (nkv > 0 && !warp_wait(&bars[BB_KVE], (nkv - 1) & 1, abort, a.status, a.wait_limit)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[BB_KV], 2 * S::kKTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x) {
                        tma_load_3d(sK + x * S::kKBox, &tk, &bars[BB_KV], x * 64, u.kt * 128, u.bh);
                        tma_load_3d(sV + x * S::kKBox, &tv, &bars[BB_KV], x * 64, u.kt * 128, u.bh);
                    }
                }
                ++nkv;
                for (int it = 0; it < u.n_it; ++it, ++G) {
                    if (kDebugChecks && (it & 1) == 0) {   // a Q tile of the column and a FULL or PARTIAL label
                        const int e = u.list[it >> 1];
                        const int lab = (int)((unsigned)e >> kLabelShift);
                        if ((e & kTileMask) >= L.n_q || (lab != FM_TILE_FULL && lab != FM_TILE_PARTIAL)) {
                            if (lane == 0) set_status(a.status, FM_ERR_DEBUG_CHECK);
                            *abort = 1;
                            run = false;
                            break;
                        }
                    }
                    const int q0 = q0_of(u, it);
                    const int st = G % NST;
                    // lse and D of the half's rows, loaded before the stage wait so
                    // the global latency overlaps it; rows beyond the Q rows get P = 0.
                    float lv[2], dv[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int qi = q0 + lane + rr * 32;
                        lv[rr] = INFINITY;
                        dv[rr] = 0.f;
                        if (qi < Nq) {
                            lv[rr] = a.lse[(int64_t)u.bh * Nq + qi];
                            dv[rr] = a.Dvec[(int64_t)u.bh * Nq + qi];
                        }
                    }
                    if (G >= NST &&
                        !warp_wait(&bars[BB_QE0 + st], ((G / NST) - 1) & 1, abort, a.status, a.wait_limit)) {
                        run = false;
                        break;
                    }
                    if (lane == 0 && G != withheld) {
                        mbar_arrive_expect_tx(&bars[BB_QF0 + st], 2 * S::kQTile);
#pragma unroll
                        for (int x = 0; x < NBOX; ++x) {
                            tma_load_3d(sQ + st * S::kQTile + x * S::kQBox, &tq, &bars[BB_QF0 + st], x * 64, q0, u.bh);
                            tma_load_3d(sdO + st * S::kQTile + x * S::kQBox, &tdo, &bars[BB_QF0 + st], x * 64, q0, u.bh);
                        }
                    }
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const int r = lane + rr * 32;
                        sLse[st * 64 + r] = (lv[rr] == -INFINITY) ? -INFINITY : -lv[rr] * 1.4426950408889634f;
                        sD[st * 64 + r] = dv[rr];
                    }
                    mbar_arrive(&bars[BB_QF0 + st]);     // 32 arrivals after the stores (+1 expect_tx)
                }
            }
            if (kDebugChecks && lane == 0) {
                dbg[0] = G;
                dbg[1] = nkv;
                dbg[2] = k + 1;
            }
            // Drain copies still in flight (only possible after an abort).
            if (lane == 0 && *abort) {
                if (nkv > 0) mbar_wait_drain(&bars[BB_KV], (nkv - 1) & 1, a.status, a.wait_limit);
                for (int k2 = (G > NST ? G - NST : 0); k2 < G; ++k2)
                    if (k2 != withheld) mbar_wait_drain(&bars[BB_QF0 + (k2 % NST)], (k2 / NST) & 1, a.status, a.wait_limit);
            }
        } else if (warp == 1 || warp >= 22) {
            // ------------------------------------------------ MMA issuers
            // Four issuing threads, one per product stream, each in a warp of its
            // own sub-partition: warp 1 S^T and warp 23 dP^T of each half (as soon
            // as its Q/dO have landed and their columns are free again), warp 22
            // dQ^T (once dS^T is written), warp 24 dV then dK (once P^T, dS^T are
            // written).  A Q/dO stage is released by the S^T, dP^T and dV/dK
            // threads, a dS^T buffer by the dQ^T and dK products.
            // Per unit the S^T, dP^T and dQ^T threads wait for the unit's K and V
            // (and commit the K / V release after their last product); the dV/dK
            // thread, which reads neither, instead waits until the previous unit's
            // epilogue has read dK and dV before its first product overwrites them.
            // All lanes walk the units (the ring is read warp-wide); lane 0 issues.
            const int role = (warp == 1) ? 0 : (warp == 23) ? 1 : (warp == 22) ? 2 : 3;
            constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
            constexpr uint32_t idKV = idesc_bf16(128, D, false, true);
            constexpr uint32_t idQ = idesc_bf16(128, 64, true, true);
            constexpr int NPART = PRECISE ? 2 : 1;
            const uint64_t dKk = sdesc_sw128(smem_u32(sK), 16, 1024);      // K, K-major
            const uint64_t dVk = sdesc_sw128(smem_u32(sV), 16, 1024);      // V, K-major
            const uint64_t dKm = sdesc_sw128(smem_u32(sK), S::kKBox, 1024); // K, MN-major
            const uint64_t dSk[2] = {sdesc_sw128(smem_u32(sdS), 16, 1024), sdesc_sw128(smem_u32(sdSlo), 16, 1024)};
            const uint64_t dSm[2] = {sdesc_sw128(smem_u32(sdS), S::kKBox, 1024),
                                     sdesc_sw128(smem_u32(sdSlo), S::kKBox, 1024)};
            int G = 0;      // halves begun (CTA-wide)
            int nu = 0;     // units with halves begun
            bool run = true;
            Unit u;
            for (int k = 0; run; ++k) {
                if (!read_unit(k, u)) break;
                if (u.n_it == 0) continue;
                if (lane == 0) {
                    if (role != 3) run = mbar_wait(&bars[BB_KV], nu & 1, abort, a.status, a.wait_limit);
                    else if (nu > 0) run = mbar_wait(&bars[BB_ACCE], (nu - 1) & 1, abort, a.status, a.wait_limit);
                    for (int it = 0; run && it < u.n_it; ++it, ++G) {
                        const int st = G % NST;
                        if (role <= 1) {
                            const int b = G & 1;
                            // The S^T columns of buffer b are free once dV has read the P^T
                            // of the half that used them before, the dP^T columns once the
                            // drain holds that half's dQ^T (both imply the scores were read).
                            uint64_t *free_bar = &bars[(role == 0 ? BB_PE0 : BB_DQE0) + b];
                            if (!mbar_wait(&bars[BB_QF0 + st], (G / NST) & 1, abort, a.status, a.wait_limit) ||
                                (G >= 2 && !mbar_wait(free_bar, ((G >> 1) - 1) & 1, abort, a.status, a.wait_limit))) {
                                run = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t dA = role == 0 ? dKk : dVk;                    // K for S^T, V for dP^T
                            const uint64_t dB = sdesc_sw128(smem_u32((role == 0 ? sQ : sdO) + st * S::kQTile), 16, 1024);
                            const uint32_t tD = (role == 0 ? tS0 : tdP0) + b * 128;
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t ok_ = (kk >> 2) * S::kKBox + (kk & 3) * 32;
                                const uint32_t oq = (kk >> 2) * S::kQBox + (kk & 3) * 32;
                                mma_ss(tD, sdesc_add(dA, ok_), sdesc_add(dB, oq), idS, kk > 0);
                            }
                            tc_commit(&bars[(role == 0 ? BB_SF0 : BB_SFD0) + b]);
                            tc_commit(&bars[BB_QE0 + st]);
                        } else {
                            const int qb = G & 1;          // score buffer: P^T in its S^T columns, dQ^T in its dP^T columns
                            const int pb = (S::kdSBufs == 2) ? (G & 1) : 0;   // dS^T buffer of this half
                            const uint32_t pbo = pb * S::kOp;
                            if (role == 2) {
                                if (!mbar_wait(&bars[BB_DF0 + qb], (G >> 1) & 1, abort, a.status, a.wait_limit)) {
                                    run = false;
                                    break;
                                }
                                tc_fence_after();
#pragma unroll
                                for (int part = 0; part < NPART; ++part)
#pragma unroll
                                    for (int kk = 0; kk < 8; ++kk)
                                        mma_ss(tdP0 + qb * 128, sdesc_add(dKm, kk * 2048), sdesc_add(dSm[part], pbo + kk * 2048),
                                               idQ, (part > 0 || kk > 0));
                                tc_commit(&bars[BB_DQF0 + qb]);
                                tc_commit(&bars[BB_DSE0 + pb]);
                            } else {
                                const uint64_t dQm = sdesc_sw128(smem_u32(sQ + st * S::kQTile), S::kQBox, 1024);
                                const uint64_t dOm = sdesc_sw128(smem_u32(sdO + st * S::kQTile), S::kQBox, 1024);
                                if (!mbar_wait(&bars[BB_PF0 + qb], (G >> 1) & 1, abort, a.status, a.wait_limit)) {
                                    run = false;
                                    break;
                                }
                                tc_fence_after();
                                // P^T of the 16 columns kk: TMEM columns [16 kk, 16 kk + 8) of
                                // the S^T block (the low terms in the next 8 columns).
#pragma unroll
                                for (int part = 0; part < NPART; ++part)
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        mma_ts(tdV, tS0 + qb * 128 + kk * 16 + part * 8, sdesc_add(dOm, kk * 2048), idKV,
                                               (it > 0 || part > 0 || kk > 0));
                                tc_commit(&bars[BB_PE0 + qb]);
                                if (!mbar_wait(&bars[BB_DF0 + qb], (G >> 1) & 1, abort, a.status, a.wait_limit)) {
                                    run = false;
                                    break;
                                }
                                tc_fence_after();
#pragma unroll
                                for (int part = 0; part < NPART; ++part)
#pragma unroll
                                    for (int kk = 0; kk < 4; ++kk)
                                        mma_ss(tdK, sdesc_add(dSk[part], pbo + kk * 32), sdesc_add(dQm, kk * 2048), idKV,
                                               (it > 0 || part > 0 || kk > 0));
                                tc_commit(&bars[BB_DSE0 + pb]);
                                tc_commit(&bars[BB_QE0 + st]);
                            }
                        }
                    }
                    if (run) tc_commit(&bars[role == 3 ? BB_ACC : BB_KVE]);
                }
                ++nu;
                run = __shfl_sync(0xffffffffu, run, 0);
            }
            if (lane == 0) {
                tc_commit(&bars[BB_DRAIN0]);
                mbar_wait_drain(&bars[BB_DRAIN0], 0, a.status, a.wait_limit);
            }
        } else if (warp < 18) {
            // ------------------------------------------------ P^T / dS^T
            // Four warpgroups (warps 2-5, 6-9, 10-13, 14-17) take 16 columns of
            // each half each; thread = KV row (TMEM lane).
            constexpr int CW = 16;                   // columns per thread
            const int wg = (warp - 2) >> 2;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;       // KV row within the tile
            const int c0 = wg * CW;                  // first column of this warpgroup
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            int G = 0;      // halves begun (CTA-wide)
            int nu = 0;     // units with halves finished
            int nstg = 0;   // epilogues finished (phases of BB_STG)
            bool ok = true;
            Unit u;
            for (int k = 0; ok; ++k) {
            if (!read_unit(k, u)) break;
            const int kb = u.kt * 128;
            const int j = kb + r;
            int lo0 = 0, lolen = 0, up0 = 0, uplen = 0x7fffffff;   // beyond N: masked everywhere
            if (j < N) {
                const int64_t o = (int64_t)u.sidx * N + j;
                const int l0 = a.lts[o], l1 = a.lte[o], u0 = a.uts[o], u1 = a.ute[o];
                lo0 = l0; lolen = max(l1 - l0, 0); up0 = u0; uplen = max(u1 - u0, 0);
            }
            const bool kv_tail = kb + 128 > N;
            for (int it = 0; it < u.n_it; ++it, ++G) {
                const int e = u.list[it >> 1];
                const int q0 = (e & kTileMask) * 128 + (it & 1) * 64;
                const bool pred = ((e >> kLabelShift) == FM_TILE_PARTIAL) || kv_tail;
                const int st = G % NST;
                const int b = G & 1;                      // score buffer
                // P needs only S^T: dP^T is waited for after P^T has been handed to dV.
                if (!warp_wait(&bars[BB_SF0 + b], (G >> 1) & 1, abort, a.status, a.wait_limit) ||
                    !warp_wait(&bars[BB_QF0 + st], (G / NST) & 1, abort, a.status, a.wait_limit)) { ok = false; break; }
                tc_fence_after();
                uint32_t sraw[CW], draw[CW];
                tmem_ld16(tS0 + b * 128 + lane_off + c0, sraw);
                // -lse*log2e and D of this warpgroup's columns, as packed pairs.
                uint64_t nl2[CW / 2], dd2[CW / 2];
#pragma unroll
                for (int v4 = 0; v4 < CW / 4; ++v4) {
                    const float4 x = reinterpret_cast<const float4 *>(sLse + st * 64 + c0)[v4];
                    const float4 y = reinterpret_cast<const float4 *>(sD + st * 64 + c0)[v4];
                    nl2[2 * v4] = f2_pack(x.x, x.y); nl2[2 * v4 + 1] = f2_pack(x.z, x.w);
                    dd2[2 * v4] = f2_pack(y.x, y.y); dd2[2 * v4 + 1] = f2_pack(y.z, y.w);
                }
                tmem_ld_wait();
                tmem_reg_fence(sraw);
                // Column pairs in packed fp32: x = S*scale*log2e - lse*log2e,
                // P = exp2(x), dS = P (dP - D).
                float p[CW], ds[CW];
                const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
                for (int c = 0; c < CW; c += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[c]), __uint_as_float(sraw[c + 1])), sc2, nl2[c / 2]), x0, x1);
                    float p0 = ex2(x0), p1 = ex2(x1);
                    if (pred) {
                        const int qi = a.q_row0 + q0 + c0 + c;   // row of the mask
                        const bool m0 = ((unsigned)(qi - lo0) < (unsigned)lolen) ||
                                        ((unsigned)(qi - up0) < (unsigned)uplen);
                        const bool m1 = ((unsigned)(qi + 1 - lo0) < (unsigned)lolen) ||
                                        ((unsigned)(qi + 1 - up0) < (unsigned)uplen);
                        p0 = m0 ? 0.f : p0;
                        p1 = m1 ? 0.f : p1;
                    }
                    p[c] = p0;
                    p[c + 1] = p1;
                }
                // P^T into the S^T columns this thread has read: bf16 pairs in
                // columns [c0, c0 + 8) (precise: low terms in [c0 + 8, c0 + 16)).
                if (PRECISE) {
                    uint32_t pw[16];
#pragma unroll
                    for (int w2 = 0; w2 < 8; ++w2) split_bf16x2(p[2 * w2], p[2 * w2 + 1], pw[w2], pw[8 + w2]);
                    tmem_st16(tS0 + b * 128 + lane_off + c0, pw);
                } else {
                    uint32_t pw[8];
#pragma unroll
                    for (int w2 = 0; w2 < 8; ++w2) pw[w2] = pack_bf16x2(p[2 * w2], p[2 * w2 + 1]);
                    tmem_st8(tS0 + b * 128 + lane_off + c0, pw);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[BB_PF0 + b]);
                if (!warp_wait(&bars[BB_SFD0 + b], (G >> 1) & 1, abort, a.status, a.wait_limit)) { ok = false; break; }
                tc_fence_after();
                tmem_ld16(tdP0 + b * 128 + lane_off + c0, draw);
                tmem_ld_wait();
                tmem_reg_fence(draw);
#pragma unroll
                for (int c = 0; c < CW; c += 2) {
                    const uint64_t t2 = f2_sub(f2_pack(__uint_as_float(draw[c]), __uint_as_float(draw[c + 1])), dd2[c / 2]);
                    f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]), t2), ds[c], ds[c + 1]);
                }
                // dS^T (its buffer is free once dK, dQ^T of the half that last
                // used it have completed, normally long ago), announced on DF.
                const int pb = (S::kdSBufs == 2) ? (G & 1) : 0;
                const int back = S::kdSBufs;                 // halves between two uses of a dS^T buffer
                if (G >= back && !warp_wait(&bars[BB_DSE0 + pb], ((G / back) - 1) & 1, abort, a.status, a.wait_limit)) { ok = false; break; }
                uint8_t *bdS = sdS + pb * S::kOp;
                // Row r of a 128-byte-swizzled tile: 16-byte chunk c lives at c ^ (r & 7).
#pragma unroll
                for (int u = 0; u < CW / 8; ++u) {
                    const int chunk = (c0 >> 3) + u;
                    const int off = r * 128 + ((chunk ^ (r & 7)) << 4);
                    uint32_t dh[4], dl[4];
#pragma unroll
                    for (int w2 = 0; w2 < 4; ++w2) {
                        const int c = 8 * u + 2 * w2;
                        if (PRECISE) split_bf16x2(ds[c], ds[c + 1], dh[w2], dl[w2]);
                        else dh[w2] = pack_bf16x2(ds[c], ds[c + 1]);
                    }
                    *reinterpret_cast<uint4 *>(bdS + off) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
                    if (PRECISE) *reinterpret_cast<uint4 *>(sdSlo + off) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
                }
                fence_proxy_async_smem();
                tc_fence_before();                  // dP^T reads of this half precede the dQ^T MMA
                mbar_arrive(&bars[BB_DF0 + b]);
            }
            // ------------------------------------------------ dK, dV epilogue
            // Warpgroups 0, 1 store the two column halves of dK; 2, 3 of dV.  The
            // accumulators are released to the next unit's first dV / dK product
            // once read; a unit without halves stores zeros.  The values leave
            // through shared memory and TMA stores of 32 columns x 32 rows (fp32:
            // 128-byte rows, 128-byte swizzle, 16-byte chunk q of row x at chunk
            // q ^ (x & 7); bf16: 64-byte rows, 64-byte swizzle, chunk q at
            // q ^ ((x >> 1) & 3)); the copy engine writes whole row segments and
            // drops rows at or beyond N.  Staging: 4 KB per warp in the dS^T tiles
            // and the 32 KB after them, free once the dK and dQ^T products of the
            // unit's last halves have read dS^T; the next unit's dS^T is written
            // once every warp's stores have read their staging (BB_STG).
            if (!ok) break;
            if (u.n_it > 0 && !warp_wait(&bars[BB_ACC], nu & 1, abort, a.status, a.wait_limit)) break;
            {
                const int back = S::kdSBufs;
                bool dse_ok = true;
                for (int h = (G > back ? G - back : 0); h < G && dse_ok; ++h)
                    dse_ok = warp_wait(&bars[BB_DSE0 + (h % back)], (h / back) & 1, abort, a.status, a.wait_limit);
                if (!dse_ok) break;
            }
            tc_fence_after();
            const bool is_dk = wg < 2;
            const uint32_t tsrc = is_dk ? tdK : tdV;
            const float mul = is_dk ? a.scale : 1.f;
            const CUtensorMap *tout = is_dk ? &tdk : &tdv;
            const int cbase = (wg & 1) * (D / 2);
            uint8_t *stg = sdS + (warp - 2) * 4096;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int col = cbase + cc * 32;
                uint32_t v[32];
                if (u.n_it > 0) {          // warp-uniform: every lane loads
                    tmem_ld32(tsrc + lane_off + col, v);
                    tmem_ld_wait();
                    tmem_reg_fence(v);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = 0u;
                }
                if (cc > 0) {              // the previous store has read the buffer
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                }
                if (a.g_f32) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        st_shared_v4(stg + lane * 128 + ((q ^ (lane & 7)) << 4),
                                     make_uint4(__float_as_uint(__uint_as_float(v[4 * q]) * mul),
                                                __float_as_uint(__uint_as_float(v[4 * q + 1]) * mul),
                                                __float_as_uint(__uint_as_float(v[4 * q + 2]) * mul),
                                                __float_as_uint(__uint_as_float(v[4 * q + 3]) * mul)));
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_shared_v4(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4),
                                     make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]) * mul, __uint_as_float(v[8 * q + 1]) * mul),
                                                pack_bf16x2(__uint_as_float(v[8 * q + 2]) * mul, __uint_as_float(v[8 * q + 3]) * mul),
                                                pack_bf16x2(__uint_as_float(v[8 * q + 4]) * mul, __uint_as_float(v[8 * q + 5]) * mul),
                                                pack_bf16x2(__uint_as_float(v[8 * q + 6]) * mul, __uint_as_float(v[8 * q + 7]) * mul)));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(tout, stg, col, kb + quarter * 32, u.bh);
                    bulk_commit();
                }
            }
            if (u.n_it > 0) {
                tc_fence_before();
                mbar_arrive(&bars[BB_ACCE]);
                ++nu;
            }
            // The staging (with the dS^T tiles) is free once every warp's stores
            // have read it; each warp waits for all sixteen, so the phases of
            // BB_STG stay in step with the units.
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[BB_STG]);
            if (!warp_wait(&bars[BB_STG], nstg & 1, abort, a.status, a.wait_limit)) break;
            ++nstg;
            }
            // Every TMA store of dK / dV has completed before the CTA leaves.
            if (lane == 0) bulk_wait_all();
        } else if (warp < 22) {
            // ------------------------------------------------ dQ drain
            // Thread = head-dim index (TMEM lane of dQ^T).  The half's 64 x d
            // tile goes from registers straight into the fp32 dQ accumulator
            // with red.global.add (one coalesced 128-byte request per warp and
            // row): the reductions need no staging and nothing waits for
            // them, so the drain never holds the score buffer for longer
            // than the two TMEM loads.
            const int quarter = warp & 3;
            const int dd = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const bool has_cols = quarter * 32 < D;          // warp-uniform
            // In a register: the reductions' memory clobbers would otherwise make the
            // compiler reload the parameter for every element.
            const float dq_mul = a.dq_mul;
            int G = 0;      // halves begun (CTA-wide)
            bool run = true;
            Unit u;
            for (int k = 0; run && read_unit(k, u); ++k)
            for (int it = 0; it < u.n_it; ++it, ++G) {
                const int q0 = q0_of(u, it);
                const int qb = G & 1;
                if (!warp_wait(&bars[BB_DQF0 + qb], (G >> 1) & 1, abort, a.status, a.wait_limit)) {
                    run = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[2][32];
                tmem_ld32(tdP0 + qb * 128 + lane_off, v[0]);
                tmem_ld32(tdP0 + qb * 128 + lane_off + 32, v[1]);
                tmem_ld_wait();
                tmem_reg_fence(v[0]);
                tmem_reg_fence(v[1]);
                // The factor in packed fp32 pairs, before the arrive: a scalar
                // multiply folded into each reduction below measured 40 % slower.
                {
                    const uint64_t m2 = f2_pack(dq_mul, dq_mul);
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float x0, x1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(v[c >> 5][c & 31]),
                                                 __uint_as_float(v[c >> 5][(c & 31) + 1])), m2), x0, x1);
                        v[c >> 5][c & 31] = __float_as_uint(x0);
                        v[c >> 5][(c & 31) + 1] = __float_as_uint(x1);
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars[BB_DQE0 + qb]);   // score buffer qb is free again
                if (!has_cols) continue;
                float *dst = a.dq_acc + ((int64_t)u.bh * Nq + q0) * D + dd;
                const int lim = min(64, Nq - q0);      // rows beyond the Q rows: nothing to add
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c < lim) red_add_f32(dst + (int64_t)c * D, __uint_as_float(v[c >> 5][c & 31]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // Debug build: every pipeline barrier has completed as many phases as the
    // CTA's halves (G), units with halves, units and ring entries imply.
    if (kDebugChecks && threadIdx.x == 0 && *ok_sh && !*abort) {
        const int G = dbg[0], NU = dbg[1], NK = dbg[2];
        auto cnt = [](int total, int period, int idx) { return total > idx ? (total - 1 - idx) / period + 1 : 0; };
        bool good = mbar_phase_count_ok(&bars[BB_KV], NU) && mbar_phase_count_ok(&bars[BB_KVE], NU) &&
                    mbar_phase_count_ok(&bars[BB_ACC], NU) && mbar_phase_count_ok(&bars[BB_ACCE], NU) &&
                    mbar_phase_count_ok(&bars[BB_STG], NK - 1) && mbar_phase_count_ok(&bars[BB_DRAIN0], 1) &&
                    mbar_phase_count_ok(&bars[BB_DRAIN1], 0);
        for (int s2 = 0; s2 < NST; ++s2)
            good = good && mbar_phase_count_ok(&bars[BB_QF0 + s2], cnt(G, NST, s2)) &&
                   mbar_phase_count_ok(&bars[BB_QE0 + s2], cnt(G, NST, s2));
        for (int b = 0; b < 2; ++b) {
            const int c = cnt(G, 2, b);
            good = good && mbar_phase_count_ok(&bars[BB_SF0 + b], c) && mbar_phase_count_ok(&bars[BB_SFD0 + b], c) &&
                   mbar_phase_count_ok(&bars[BB_PF0 + b], c) && mbar_phase_count_ok(&bars[BB_PE0 + b], c) &&
                   mbar_phase_count_ok(&bars[BB_DF0 + b], c) && mbar_phase_count_ok(&bars[BB_DQF0 + b], c) &&
                   mbar_phase_count_ok(&bars[BB_DQE0 + b], c);
        }
        for (int b = 0; b < S::kdSBufs; ++b)
            good = good && mbar_phase_count_ok(&bars[BB_DSE0 + b], cnt(G, S::kdSBufs, b));
        for (int s2 = 0; s2 < kBwdUnitRing; ++s2)
            good = good && mbar_phase_count_ok(&bars[BB_UF0 + s2], cnt(NK, kBwdUnitRing, s2)) &&
                   mbar_phase_count_ok(&bars[BB_UE0 + s2], cnt(NK, kBwdUnitRing, s2));
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

fm_status fm_bwd_pre_launch(const void *o, int o_f32, const void *dO, float *Dout, float *dq_acc,
                            int64_t rows, int d, cudaStream_t stream)
{
    const int64_t warps_needed = rows;
    int64_t blocks = (warps_needed + 7) / 8;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    ProfScope ps(kKBwdPre, stream);
    if (d == 128)
        fm_bwd_pre_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(o, o_f32, (const uint16_t *)dO, Dout, dq_acc, rows);
    else
        fm_bwd_pre_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(o, o_f32, (const uint16_t *)dO, Dout, dq_acc, rows);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

// The kernel's shared-memory limit, set once per device: later launches (also
// those captured into a graph) make no attribute call.
template <int D, bool PRECISE>
static bool bwd_smem_ready()
{
    constexpr int smem = BwdSmem<D, PRECISE>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    static std::atomic<uint8_t> done[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(fm_bwd_kernel<D, PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return false;
    done[dev].store(1, std::memory_order_release);
    return true;
}

template <int D, bool PRECISE>
static fm_status launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv,
                            const BwdArgs &a, cudaStream_t stream)
{
    constexpr int smem = BwdSmem<D, PRECISE>::kBytes;
    if (!bwd_smem_ready<D, PRECISE>()) return FM_ERR_CUDA;
    // Persistent: one CTA per SM (shared memory and 512 TMEM columns allow no
    // second one), each claiming units of the plan's order.
    const int64_t units = (int64_t)a.B * a.H * a.L.n_k;
    const int sms = device_sm_count();
    if (sms <= 0) return FM_ERR_CUDA;
    const unsigned grid = (unsigned)(units < sms ? units : sms);
    static std::atomic<unsigned> next_slot{0};
    BwdArgs args = a;
    args.sched_slot = (int)(next_slot.fetch_add(1, std::memory_order_relaxed) % kBwdSchedSlots);
    ProfScope ps(kKBwd, stream);
    fm_bwd_kernel<D, PRECISE><<<grid, 800, smem, stream>>>(tq, tk, tv, tdo, tdk, tdv, args);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_bwd_prepare(int d, bool precise)
{
    if (device_sm_count() <= 0) return FM_ERR_CUDA;   // cached before any stream capture
    const bool ok = d == 128 ? (precise ? bwd_smem_ready<128, true>() : bwd_smem_ready<128, false>())
                             : (precise ? bwd_smem_ready<64, true>() : bwd_smem_ready<64, false>());
    return ok ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_bwd_main_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv,
                             const BwdArgs &a, int d, bool precise, cudaStream_t stream)
{
    if (d == 128)
        return precise ? launch_bwd<128, true>(tq, tk, tv, tdo, tdk, tdv, a, stream)
                       : launch_bwd<128, false>(tq, tk, tv, tdo, tdk, tdv, a, stream);
    return precise ? launch_bwd<64, true>(tq, tk, tv, tdo, tdk, tdv, a, stream)
                   : launch_bwd<64, false>(tq, tk, tv, tdo, tdk, tdv, a, stream);
}

fm_status fm_bwd_post_launch(const float *dq_acc, void *dq, float scale, int64_t n, cudaStream_t stream)
{
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    ProfScope ps(kKBwdPost, stream);
    fm_bwd_post_kernel<<<(unsigned)blocks, 256, 0, stream>>>(dq_acc, reinterpret_cast<uint16_t *>(dq), scale, n4);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
