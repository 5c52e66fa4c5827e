// Backward main kernel, standard precision, on whole 128-row Q tiles.
//
// The gradients are those of plain masked softmax attention (the method is
// exact: blog "FlashMask技术" §2.2, arXiv 2410.01359 abstract), with the
// forward's tile skipping (blog §2.2): fully masked (Q tile, KV tile) pairs
// are never visited, fully visible pairs run without mask arithmetic, only
// partial pairs evaluate the column-interval predicate.
//
// One CTA = one (b, h, 128-row KV tile); it walks the plan's list of non-skip
// Q tiles of that KV tile, one whole 128-row Q tile per step, so every one of
// the five products is an M = 128 MMA with N = 128 (or d) and K = 128:
//   S^T  = K Q^T        (SS, K-major / K-major)          -> TMEM S
//   dP^T = V dO^T       (SS, K-major / K-major)          -> TMEM dP
//   P^T  = exp2(S^T * scale*log2e - lse*log2e), written as packed bf16 over
//          the S^T columns it was computed from (the A operand of dV)
//   dS^T = P^T o (dP^T - D), written as bf16 into 128-byte-swizzled shared
//          memory (A of dK, B of dQ^T)
//   dV  += P^T dO       (TS, P^T from TMEM, dO MN-major)
//   dK  += dS^T Q       (SS, dS^T K-major, Q MN-major)
//   dQ^T = K^T dS^T     (SS, K MN-major, dS^T MN-major)  -> TMEM dP columns
// TMEM (512 columns): dK [0, 128), dV [128, 256), S^T / P^T [256, 384),
// dP^T / dQ^T [384, 512).  With one score buffer the scores of step t + 1
// wait for dV of step t (S columns) and for the drain of dQ^T of step t (dP
// columns); the other products of neighbouring steps fill the tensor pipe
// meanwhile.  Shared memory (d = 128): K, V, two Q stages, two dO stages
// (each released by its own two readers), one dS^T tile, lse and D per
// stage: 226 KB.
// Roles:
//   warp 0      TMA producer (K, V once; Q and dO per step into their rings;
//               lse and D staged into shared memory by the whole warp)
//   warp 1      TMEM allocation; one thread issues S^T
//   warps 2-17  four warpgroups, thread = KV row j: P^T and dS^T for 32 of
//               the step's 128 Q columns each
//   warps 18-21 thread = head-dim index: drain dQ^T from TMEM into the fp32
//               dQ accumulator with red.global.add
//   warp 22     one thread issues dQ^T
//   warp 23     one thread issues dP^T
//   warp 24     one thread issues dV, then dK
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

enum {
    B2_KV = 0, B2_QF0, B2_QF1, B2_OF0, B2_OF1, B2_QE0, B2_QE1, B2_OE0, B2_OE1,
    B2_SF, B2_PF, B2_PE, B2_DPF, B2_DF, B2_DSE, B2_DQF, B2_DQE, B2_ACC, B2_DRAIN, B2_COUNT
};

template <int D>
struct Bwd128Smem {
    static constexpr int kStages = 2;
    static constexpr int kBox = 128 * 128;          // 64 bf16 columns x 128 rows, 128-byte swizzle
    static constexpr int kTile = 128 * D * 2;       // one 128-row tile of K, V, Q or dO
    static constexpr int kK = 0, kV = kTile;
    static constexpr int kQ = 2 * kTile;                    // [kStages]
    static constexpr int kdO = kQ + kStages * kTile;        // [kStages]
    static constexpr int kdS = kdO + kStages * kTile;       // dS^T: 128 KV rows x 128 Q columns
    static constexpr int kStat = kdS + 2 * kBox;            // -lse*log2e [kStages][128], D [kStages][128]
    static constexpr int kList = kStat + 2 * kStages * 128 * 4;
    static constexpr int kListCap = 128;                    // Q tiles staged from the plan
    static constexpr int kBar = kList + kListCap * 4;
    static constexpr int kMisc = kBar + B2_COUNT * 8;
    static constexpr int kBytes0 = kMisc + 64;
    // At least 120 KB so that one CTA (512 TMEM columns) is resident per SM.
    static constexpr int kBytes = kBytes0 > 120 * 1024 ? kBytes0 : 120 * 1024;
};

template <int D>
__global__ void __launch_bounds__(800, 1)
    fm_bwd128_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                     const BwdArgs a)
{
    using S = Bwd128Smem<D>;
    constexpr int NBOX = D / 64;
    constexpr int NST = S::kStages;
    constexpr int KSTEPS = D / 16;              // K = 16 slices of the head dim
    // No static shared memory: the dynamic window starts on a 1024-byte
    // boundary (checked below); pointers stay derived from the __shared__
    // array so that every access is a shared-memory instruction.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    uint8_t *sK = smem + S::kK, *sV = smem + S::kV;
    uint8_t *sQ = smem + S::kQ, *sdO = smem + S::kdO, *sdS = smem + S::kdS;
    float *sLse = reinterpret_cast<float *>(smem + S::kStat);    // [NST][128]
    float *sD = sLse + NST * 128;                                   // [NST][128]
    int32_t *sList = reinterpret_cast<int32_t *>(smem + S::kList);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *cnt_sh = reinterpret_cast<int *>(smem + S::kMisc + 8);
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 12);
    int *unit_sh = reinterpret_cast<int *>(smem + S::kMisc + 16);   // KV tile, head, batch

    const int warp = warp_id(), lane = lane_id();
    const PlanLayout &L = a.L;
    const int N = a.N;

    if (warp == 0) {
        const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(a.plan);
        bool ok = ph->magic == kPlanMagic && ph->B == L.B && ph->Hm == L.Hm && ph->N == L.N &&
                  ph->bq == 128 && ph->bk == 128 && ph->q_row0 == L.q_row0 && ph->Nq == L.Nq;
        int ut = 0, uh = 0, ub = 0;
        const int64_t cta = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
        if (ok)
            ok = plan_unit(reinterpret_cast<const int32_t *>(a.plan + L.off_col_order),
                           reinterpret_cast<const int32_t *>(a.plan + L.off_col_bstart), L.n_k, a.B, a.Hm, a.H, cta,
                           &ut, &uh, &ub);
        if (lane == 0) {
            if (!ok) set_status(a.status, FM_ERR_PLAN_MISMATCH);
            const bool aligned = (smem_u32(smem) & 1023u) == 0;   // 128-byte swizzle atoms need it
            if (!aligned) set_status(a.status, FM_ERR_UNSUPPORTED);
            *ok_sh = ok && aligned;
            unit_sh[0] = ut; unit_sh[1] = uh; unit_sh[2] = ub;
            const int us = ub * a.Hm + (a.Hm == 1 ? 0 : uh);
            *cnt_sh = ok ? reinterpret_cast<const int32_t *>(a.plan + L.off_col_cnt)[(int64_t)us * L.n_k + ut] : 0;
            *abort = 0;
            mbar_init(&bars[B2_KV], 1);
            for (int s = 0; s < NST; ++s) {
                mbar_init(&bars[B2_QF0 + s], 33);    // expect_tx + the 32 lanes' lse / D stores
                mbar_init(&bars[B2_OF0 + s], 1);
                mbar_init(&bars[B2_QE0 + s], 2);     // S^T and dK have read Q
                mbar_init(&bars[B2_OE0 + s], 2);     // dP^T and dV have read dO
            }
            mbar_init(&bars[B2_SF], 1);      // S^T written
            mbar_init(&bars[B2_PF], 512);    // P^T written (all P/dS threads)
            mbar_init(&bars[B2_PE], 1);      // dV has read P^T: S columns free
            mbar_init(&bars[B2_DPF], 1);     // dP^T written
            mbar_init(&bars[B2_DF], 512);    // dS^T written
            mbar_init(&bars[B2_DSE], 2);     // dK and dQ^T have read dS^T
            mbar_init(&bars[B2_DQF], 1);     // dQ^T written
            mbar_init(&bars[B2_DQE], 128);   // drain has read dQ^T: dP columns free
            mbar_init(&bars[B2_ACC], 1);     // last dK (and every dV) complete
            mbar_init(&bars[B2_DRAIN], 4);   // all four issuers
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
    const int kt = unit_sh[0], h = unit_sh[1], b = unit_sh[2];
    const int sidx = b * a.Hm + (a.Hm == 1 ? 0 : h);
    const int bh = b * a.H + h;
    const int kb = kt * 128;
    const uint32_t tdK = tmem, tdV = tmem + 128, tS = tmem + 256, tdP = tmem + 384;
    const int cnt = *cnt_sh;
    const int32_t *glist =
        reinterpret_cast<const int32_t *>(a.plan + L.off_col_list) + ((int64_t)sidx * L.n_k + kt) * L.n_q;
    for (int i = threadIdx.x; i < cnt && i < S::kListCap; i += blockDim.x) sList[i] = glist[i];
    __syncthreads();
    auto entry = [&](int t) { return t < S::kListCap ? sList[t] : glist[t]; };
    const int Nq = a.Nq;

    if (*ok_sh) {
        if (warp == 0) {
            // ------------------------------------------------ producer
            if (lane == 0 && cnt > 0) {
                tma_prefetch_desc(&tq); tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv); tma_prefetch_desc(&tdo);
                mbar_arrive_expect_tx(&bars[B2_KV], 2 * S::kTile);
#pragma unroll
                for (int x = 0; x < NBOX; ++x) {
                    tma_load_3d(sK + x * S::kBox, &tk, &bars[B2_KV], x * 64, kb, bh);
                    tma_load_3d(sV + x * S::kBox, &tv, &bars[B2_KV], x * 64, kb, bh);
                }
            }
            int t = 0, nq = 0, no = 0;   // steps begun, Q loads issued, dO loads issued
            for (; t < cnt; ++t) {
                const int q0 = (entry(t) & kTileMask) * 128;
                const int st = t % NST;
                // lse and D of the step's rows, loaded before the stage waits so
                // the global latency overlaps them; rows beyond the Q rows get P = 0.
                float lv[4], dv[4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int qi = q0 + lane + rr * 32;
                    lv[rr] = INFINITY;
                    dv[rr] = 0.f;
                    if (qi < Nq) {
                        lv[rr] = a.lse[(int64_t)bh * Nq + qi];
                        dv[rr] = a.Dvec[(int64_t)bh * Nq + qi];
                    }
                }
                // dO first: its stage is released by dV, which completes before dK
                // releases the Q stage.
                if (t >= NST && !warp_wait(&bars[B2_OE0 + st], ((t / NST) - 1) & 1, abort, a.status)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[B2_OF0 + st], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(sdO + st * S::kTile + x * S::kBox, &tdo, &bars[B2_OF0 + st], x * 64, q0, bh);
                }
                ++no;
                if (t >= NST && !warp_wait(&bars[B2_QE0 + st], ((t / NST) - 1) & 1, abort, a.status)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[B2_QF0 + st], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(sQ + st * S::kTile + x * S::kBox, &tq, &bars[B2_QF0 + st], x * 64, q0, bh);
                }
                ++nq;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int r = lane + rr * 32;
                    sLse[st * 128 + r] = (lv[rr] == -INFINITY) ? -INFINITY : -lv[rr] * 1.4426950408889634f;
                    sD[st * 128 + r] = dv[rr];
                }
                mbar_arrive(&bars[B2_QF0 + st]);     // 32 arrivals after the stores (+1 expect_tx)
            }
            // Drain copies still in flight (only possible after an abort).
            if (lane == 0 && *abort) {
                if (cnt > 0) mbar_wait_drain(&bars[B2_KV], 0, a.status);
                for (int k2 = (nq > NST ? nq - NST : 0); k2 < nq; ++k2)
                    mbar_wait_drain(&bars[B2_QF0 + (k2 % NST)], (k2 / NST) & 1, a.status);
                for (int k2 = (no > NST ? no - NST : 0); k2 < no; ++k2)
                    mbar_wait_drain(&bars[B2_OF0 + (k2 % NST)], (k2 / NST) & 1, a.status);
            }
        } else if (warp == 1 || warp >= 22) {
            // ------------------------------------------------ MMA issuers
            const int role = (warp == 1) ? 0 : (warp == 23) ? 1 : (warp == 22) ? 2 : 3;
            if (lane == 0 && cnt > 0) {
                constexpr uint32_t idS = idesc_bf16(128, 128, false, false);   // S^T, dP^T
                constexpr uint32_t idKV = idesc_bf16(128, D, false, true);     // dV, dK
                constexpr uint32_t idQ = idesc_bf16(128, 128, true, true);     // dQ^T
                const uint64_t dKk = sdesc_sw128(smem_u32(sK), 16, 1024);          // K, K-major
                const uint64_t dVk = sdesc_sw128(smem_u32(sV), 16, 1024);          // V, K-major
                const uint64_t dKm = sdesc_sw128(smem_u32(sK), S::kBox, 1024);     // K, MN-major
                const uint64_t dSk = sdesc_sw128(smem_u32(sdS), 16, 1024);         // dS^T, K-major
                const uint64_t dSm = sdesc_sw128(smem_u32(sdS), S::kBox, 1024);    // dS^T, MN-major
                bool ok = mbar_wait(&bars[B2_KV], 0, abort, a.status);
                for (int t = 0; ok && t < cnt; ++t) {
                    const int st = t % NST;
                    const uint32_t sp = (t / NST) & 1, up = t & 1;
                    if (role <= 1) {
                        // S^T once Q has landed and dV of the previous step has read
                        // P^T; dP^T once dO has landed and the drain holds the
                        // previous step's dQ^T.
                        uint64_t *full = &bars[(role == 0 ? B2_QF0 : B2_OF0) + st];
                        uint64_t *free_bar = &bars[role == 0 ? B2_PE : B2_DQE];
                        if (!mbar_wait(full, sp, abort, a.status) ||
                            (t > 0 && !mbar_wait(free_bar, up ^ 1, abort, a.status))) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dA = role == 0 ? dKk : dVk;
                        const uint64_t dB = sdesc_sw128(smem_u32((role == 0 ? sQ : sdO) + st * S::kTile), 16, 1024);
                        const uint32_t tD = role == 0 ? tS : tdP;
#pragma unroll
                        for (int kk = 0; kk < KSTEPS; ++kk) {
                            const uint32_t off = (kk >> 2) * S::kBox + (kk & 3) * 32;
                            mma_ss(tD, sdesc_add(dA, off), sdesc_add(dB, off), idS, kk > 0);
                        }
                        tc_commit(&bars[role == 0 ? B2_SF : B2_DPF]);
                        tc_commit(&bars[(role == 0 ? B2_QE0 : B2_OE0) + st]);
                    } else if (role == 2) {
                        // dQ^T = K^T dS^T into the dP columns once dS^T is written
                        // (which also means dP^T has been read).
                        if (!mbar_wait(&bars[B2_DF], up, abort, a.status)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tdP, sdesc_add(dKm, kk * 2048), sdesc_add(dSm, kk * 2048), idQ, kk > 0);
                        tc_commit(&bars[B2_DQF]);
                        tc_commit(&bars[B2_DSE]);
                    } else {
                        const uint64_t dQm = sdesc_sw128(smem_u32(sQ + st * S::kTile), S::kBox, 1024);
                        const uint64_t dOm = sdesc_sw128(smem_u32(sdO + st * S::kTile), S::kBox, 1024);
                        if (!mbar_wait(&bars[B2_PF], up, abort, a.status)) { ok = false; break; }
                        tc_fence_after();
                        // P^T of Q columns [16 kk, 16 kk + 16): warpgroup kk / 2 wrote
                        // its 32 columns packed into TMEM columns [32 (kk / 2), +16).
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tdV, tS + (kk >> 1) * 32 + (kk & 1) * 8, sdesc_add(dOm, kk * 2048), idKV,
                                   (t > 0 || kk > 0));
                        tc_commit(&bars[B2_PE]);
                        tc_commit(&bars[B2_OE0 + st]);
                        if (!mbar_wait(&bars[B2_DF], up, abort, a.status)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tdK, sdesc_add(dSk, (kk >> 2) * S::kBox + (kk & 3) * 32),
                                   sdesc_add(dQm, kk * 2048), idKV, (t > 0 || kk > 0));
                        tc_commit(&bars[B2_DSE]);
                        tc_commit(&bars[B2_QE0 + st]);
                    }
                }
                if (ok && role == 3) tc_commit(&bars[B2_ACC]);
            }
            if (lane == 0) {
                tc_commit(&bars[B2_DRAIN]);
                mbar_wait_drain(&bars[B2_DRAIN], 0, a.status);
            }
        } else if (warp < 18) {
            // ------------------------------------------------ P^T / dS^T
            // Four warpgroups (warps 2-5, 6-9, 10-13, 14-17) take 32 Q columns of
            // each step each; thread = KV row (TMEM lane).
            constexpr int CW = 32;
            const int wg = (warp - 2) >> 2;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;       // KV row within the tile
            const int c0 = wg * CW;                  // first Q column of this warpgroup
            const int j = kb + r;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            int lo0 = 0, lolen = 0, up0 = 0, uplen = 0x7fffffff;   // beyond N: masked everywhere
            if (j < N) {
                const int64_t o = (int64_t)sidx * N + j;
                const int l0 = a.lts[o], l1 = a.lte[o], u0 = a.uts[o], u1 = a.ute[o];
                lo0 = l0; lolen = max(l1 - l0, 0); up0 = u0; uplen = max(u1 - u0, 0);
            }
            const bool kv_tail = kb + 128 > N;
            // dS^T of row r, Q columns [c0, c0 + 32): box c0 / 64, 16-byte chunks
            // (c0 % 64) / 8 + u at chunk ^ (r & 7) (128-byte swizzle).
            uint8_t *dS_row = sdS + (c0 >> 6) * S::kBox + r * 128;
            const int chunk0 = (c0 & 63) >> 3;
            const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2);
            bool ok = true;
            for (int t = 0; t < cnt; ++t) {
                const int e = entry(t);
                const int q0 = (e & kTileMask) * 128;
                const bool pred = ((e >> kLabelShift) == FM_TILE_PARTIAL) || kv_tail;
                const int st = t % NST;
                const uint32_t up = t & 1;
                if (!warp_wait(&bars[B2_SF], up, abort, a.status) ||
                    !warp_wait(&bars[B2_QF0 + st], (t / NST) & 1, abort, a.status)) { ok = false; break; }
                tc_fence_after();
                uint32_t sraw[CW];
                tmem_ld32(tS + lane_off + c0, sraw);
                tmem_ld_wait();
                tmem_reg_fence(sraw);
                // x = S*scale*log2e - lse*log2e in packed fp32 pairs, P = exp2(x).
                float p[CW];
                const float4 *lse4 = reinterpret_cast<const float4 *>(sLse + st * 128 + c0);
#pragma unroll
                for (int v4 = 0; v4 < CW / 4; ++v4) {
                    const float4 nl = lse4[v4];
                    float x0, x1, x2, x3;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[4 * v4]), __uint_as_float(sraw[4 * v4 + 1])), sc2,
                                     f2_pack(nl.x, nl.y)), x0, x1);
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[4 * v4 + 2]), __uint_as_float(sraw[4 * v4 + 3])), sc2,
                                     f2_pack(nl.z, nl.w)), x2, x3);
                    p[4 * v4] = ex2(x0);
                    p[4 * v4 + 1] = ex2(x1);
                    p[4 * v4 + 2] = ex2(x2);
                    p[4 * v4 + 3] = ex2(x3);
                }
                if (pred) {
#pragma unroll
                    for (int c = 0; c < CW; ++c) {
                        const int qi = a.q_row0 + q0 + c0 + c;   // row of the mask
                        const bool m = ((unsigned)(qi - lo0) < (unsigned)lolen) || ((unsigned)(qi - up0) < (unsigned)uplen);
                        p[c] = m ? 0.f : p[c];
                    }
                }
                // P^T over the first 16 of this warpgroup's 32 S^T columns, packed.
                {
                    uint32_t pw[16];
#pragma unroll
                    for (int w2 = 0; w2 < 16; ++w2) pw[w2] = pack_bf16x2(p[2 * w2], p[2 * w2 + 1]);
                    tmem_st16(tS + lane_off + c0, pw);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[B2_PF]);
                if (!warp_wait(&bars[B2_DPF], up, abort, a.status)) { ok = false; break; }
                tc_fence_after();
                // dS = P (dP - D), packed as bf16 pairs; dP^T read in two halves
                // of 16 columns to keep the live registers down.
                uint32_t dsw[CW / 2];
                const float4 *d4 = reinterpret_cast<const float4 *>(sD + st * 128 + c0);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t draw[16];
                    tmem_ld16(tdP + lane_off + c0 + 16 * hh, draw);
                    tmem_ld_wait();
                    tmem_reg_fence(draw);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        const float4 dd = d4[4 * hh + v4];
                        const int c = 16 * hh + 4 * v4;
                        float s0, s1, s2, s3;
                        f2_unpack(f2_mul(f2_pack(p[c], p[c + 1]),
                                         f2_sub(f2_pack(__uint_as_float(draw[4 * v4]), __uint_as_float(draw[4 * v4 + 1])),
                                                f2_pack(dd.x, dd.y))), s0, s1);
                        f2_unpack(f2_mul(f2_pack(p[c + 2], p[c + 3]),
                                         f2_sub(f2_pack(__uint_as_float(draw[4 * v4 + 2]), __uint_as_float(draw[4 * v4 + 3])),
                                                f2_pack(dd.z, dd.w))), s2, s3);
                        dsw[c / 2] = pack_bf16x2(s0, s1);
                        dsw[c / 2 + 1] = pack_bf16x2(s2, s3);
                    }
                }
                // The dS^T tile is free once dK and dQ^T of the previous step have read it.
                if (t > 0 && !warp_wait(&bars[B2_DSE], up ^ 1, abort, a.status)) { ok = false; break; }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    *reinterpret_cast<uint4 *>(dS_row + (((chunk0 + u) ^ (r & 7)) << 4)) =
                        make_uint4(dsw[4 * u], dsw[4 * u + 1], dsw[4 * u + 2], dsw[4 * u + 3]);
                fence_proxy_async_smem();
                tc_fence_before();                  // dP^T reads precede the dQ^T MMA
                mbar_arrive(&bars[B2_DF]);
            }
            // ------------------------------------------------ dK, dV epilogue
            // Warpgroups 0, 1 store the two column halves of dK; 2, 3 of dV.
            if (ok && (cnt == 0 || warp_wait(&bars[B2_ACC], 0, abort, a.status))) {
                tc_fence_after();
                const bool row_in = j < N;
                const int64_t row = (int64_t)bh * N + j;
                const bool is_dk = wg < 2;
                const uint32_t tsrc = is_dk ? tdK : tdV;
                const float mul = is_dk ? a.scale : 1.f;
                void *dst = is_dk ? a.dk : a.dv;
                const int cbase = (wg & 1) * (D / 2);
#pragma unroll
                for (int cc = 0; cc < D / 64; ++cc) {
                    const int col = cbase + cc * 32;
                    uint32_t v[32];
                    if (cnt > 0) {            // warp-uniform: every lane loads
                        tmem_ld32(tsrc + lane_off + col, v);
                        tmem_ld_wait();
                        tmem_reg_fence(v);
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u) v[u] = 0u;
                    }
                    if (!row_in) continue;
                    if (a.g_f32) {
                        float4 *pp = reinterpret_cast<float4 *>(reinterpret_cast<float *>(dst) + row * D + col);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            pp[u] = make_float4(__uint_as_float(v[4 * u]) * mul, __uint_as_float(v[4 * u + 1]) * mul,
                                                __uint_as_float(v[4 * u + 2]) * mul, __uint_as_float(v[4 * u + 3]) * mul);
                    } else {
                        uint4 *pp = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(dst) + row * D + col);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            pp[u] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * u]) * mul, __uint_as_float(v[8 * u + 1]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul),
                                               pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul));
                    }
                }
            }
        } else if (warp < 22) {
            // ------------------------------------------------ dQ drain
            // Thread = head-dim index (TMEM lane of dQ^T).  The step's 128 x d
            // tile goes from registers straight into the fp32 dQ accumulator with
            // red.global.add (one coalesced 128-byte request per warp and row), in
            // two halves of 64 Q rows; the dP columns are released once both
            // halves are in registers.
            const int quarter = warp & 3;
            const int dd = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const bool has_cols = quarter * 32 < D;          // warp-uniform
            for (int t = 0; t < cnt; ++t) {
                const int q0 = (entry(t) & kTileMask) * 128;
                if (!warp_wait(&bars[B2_DQF], t & 1, abort, a.status)) break;
                tc_fence_after();
                float *dst = a.dq_acc + ((int64_t)bh * Nq + q0) * D + dd;
                const int lim = min(128, Nq - q0);      // rows beyond the Q rows: nothing to add
                uint32_t v[2][32];
                tmem_ld32(tdP + lane_off, v[0]);
                tmem_ld32(tdP + lane_off + 32, v[1]);
                tmem_ld_wait();
                tmem_reg_fence(v[0]);
                tmem_reg_fence(v[1]);
                if (has_cols) {
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c < lim) red_add_f32(dst + (int64_t)c * D, __uint_as_float(v[c >> 5][c & 31]));
                }
                tmem_ld32(tdP + lane_off + 64, v[0]);
                tmem_ld32(tdP + lane_off + 96, v[1]);
                tmem_ld_wait();
                tmem_reg_fence(v[0]);
                tmem_reg_fence(v[1]);
                tc_fence_before();
                mbar_arrive(&bars[B2_DQE]);   // the dP columns are free again
                if (!has_cols) continue;
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c + 64 < lim) red_add_f32(dst + (int64_t)(c + 64) * D, __uint_as_float(v[c >> 5][c & 31]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fm

using namespace fm;

// The kernel's shared-memory limit, set once per device: later launches (also
// those captured into a graph) make no attribute call.
template <int D>
static bool bwd128_smem_ready()
{
    constexpr int smem = Bwd128Smem<D>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    static std::atomic<uint8_t> done[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(fm_bwd128_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return false;
    done[dev].store(1, std::memory_order_release);
    return true;
}

fm_status fm_bwd128_prepare(int d)
{
    return (d == 128 ? bwd128_smem_ready<128>() : bwd128_smem_ready<64>()) ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_bwd128_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &tdo, const BwdArgs &a, int d, cudaStream_t stream)
{
    if (fm_bwd128_prepare(d) != FM_OK) return FM_ERR_CUDA;
    ProfScope ps(kKBwd, stream);
    if (d == 128)
        fm_bwd128_kernel<128><<<dim3(a.L.n_k, a.H, a.B), 800, Bwd128Smem<128>::kBytes, stream>>>(tq, tk, tv, tdo, a);
    else
        fm_bwd128_kernel<64><<<dim3(a.L.n_k, a.H, a.B), 800, Bwd128Smem<64>::kBytes, stream>>>(tq, tk, tv, tdo, a);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
