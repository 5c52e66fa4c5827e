// Forward masked attention on sm_103a (tcgen05 + TMEM + TMA).
//
// Passages: FlashAttention article §二.1 (tiling), §二.2 (max-subtracted
// softmax; completed here by the standard running rescale so the result is
// the exact softmax), §二.3 (QK^T and PV on tensor cores, fused in one
// kernel); blog "FlashMask技术" §2.2 (skip / full / masked block paths) and
// §4.1 items 1-3 (bounds staged in shared memory, skip decided before the KV
// block is loaded, mask fused into the softmax).
//
// One CTA = one (b, h) and two consecutive 128-row Q tiles (Q0, Q1) that
// share every K/V load.  The CTA walks the union of the two tiles' lists of
// non-skip KV tiles (from the plan, staged in shared memory); a KV tile that
// only one Q tile needs is multiplied only for that tile, and skip tiles are
// never loaded.  Roles:
//   warp 0      TMA producer: Q0, Q1 once; K and V through a two-stage ring;
//               the column bounds of partial tiles into shared memory
//   warp 1      allocates TMEM; one thread issues the tcgen05 MMAs of Q0
//   warps 2-5   softmax of Q0, one thread per row = TMEM lane
//   warps 6-9   softmax of Q1
//   warp 10     one thread issues the tcgen05 MMAs of Q1
// TMEM (512 columns): S0, S1 = Qi K^T at [0, 128) and [128, 256), each
// overwritten in place by P as packed bf16 (the A operand of Oi += P V; in
// precise mode a second term P_lo = bf16(P - bf16(P)) follows in the upper
// 64 columns and Oi += P_hi V + P_lo V); O0, O1 accumulate at [256, 384) and
// [384, 512).  The two (Q tile, softmax, issuer) streams run independently:
// while one softmax works on its scores the tensor core runs the other
// tile's products.
// Online softmax in the base-2 domain with a lazy rescale: O and l are
// rescaled only when the row max grows by more than 2^8, which keeps every
// P <= 256 and leaves the final O / l unchanged.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

template <int D>
struct FwdSmem {
    static constexpr int kBox = 128 * 128;        // one 64-column, 128-row bf16 box
    static constexpr int kTile = 128 * D * 2;     // one Q, K or V tile
    static constexpr int kQ0 = 0, kQ1 = kTile;
    static constexpr int kK = 2 * kTile;          // [2] stages
    static constexpr int kV = 4 * kTile;          // [2] stages
    static constexpr int kBnd = 6 * kTile;        // int4 [2][128]
    static constexpr int kListCap = 2048;         // KV tiles per Q tile staged from the plan
    static constexpr int kList0 = kBnd + 4096;
    static constexpr int kList1 = kList0 + kListCap * 4;
    static constexpr int kBar = kList1 + kListCap * 4;
    static constexpr int kNumBar = 22;
    static constexpr int kMisc = kBar + kNumBar * 8;
    // At least 120 KB so that one CTA (512 TMEM columns) is resident per SM.
    static constexpr int kBytes = (kMisc + 64 + 1024 > 120 * 1024) ? kMisc + 64 + 1024 : 120 * 1024;
};

enum {
    FB_Q = 0, FB_KF0, FB_KF1, FB_KE0, FB_KE1, FB_VF0, FB_VF1, FB_VE0, FB_VE1, FB_BF0, FB_BF1,
    FB_S0, FB_S1, FB_P0, FB_P1, FB_O0, FB_O1, FB_DRAIN0, FB_DRAIN1, FB_TK0, FB_TK1
};

// Walks the union of two ascending lists of KV tiles (entries tile | label << 28).
struct TileMerge {
    const int32_t *s0, *s1, *g0, *g1;
    int n0, n1, i0, i1, cap;
    __device__ __forceinline__ int32_t at0(int i) const { return i < cap ? s0[i] : g0[i]; }
    __device__ __forceinline__ int32_t at1(int i) const { return i < cap ? s1[i] : g1[i]; }
    // kt: next KV tile; lab0 / lab1: its label for Q0 / Q1, or -1 if that
    // Q tile skips it.
    __device__ __forceinline__ bool next(int &kt, int &lab0, int &lab1)
    {
        if (i0 >= n0 && i1 >= n1) return false;
        const int32_t e0 = i0 < n0 ? at0(i0) : INT_MAX, e1 = i1 < n1 ? at1(i1) : INT_MAX;
        const int k0 = i0 < n0 ? (e0 & kTileMask) : INT_MAX, k1 = i1 < n1 ? (e1 & kTileMask) : INT_MAX;
        kt = min(k0, k1);
        lab0 = -1;
        lab1 = -1;
        if (k0 == kt) { lab0 = e0 >> kLabelShift; ++i0; }
        if (k1 == kt) { lab1 = e1 >> kLabelShift; ++i1; }
        return true;
    }
};

template <int D, bool PRECISE>
__global__ void __launch_bounds__(352, 1)
    fm_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a)
{
    using S = FwdSmem<D>;
    constexpr int NBOX = D / 64;
    // The kernel has no static shared memory, so the dynamic window starts on
    // a 1024-byte boundary (checked below).  Pointers stay derived from the
    // __shared__ array itself, so every access compiles to a shared-memory
    // instruction rather than a generic one.
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    int4 *sBnd = reinterpret_cast<int4 *>(smem + S::kBnd);
    int32_t *sList0 = reinterpret_cast<int32_t *>(smem + S::kList0);
    int32_t *sList1 = reinterpret_cast<int32_t *>(smem + S::kList1);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *cnt_sh = reinterpret_cast<int *>(smem + S::kMisc + 8);   // [2]
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 16);

    const int warp = warp_id(), lane = lane_id();
    const PlanLayout &L = a.L;
    const int pair = (int)gridDim.x - 1 - (int)blockIdx.x;   // heavy causal tiles first
    const int qt0 = 2 * pair;
    const bool has1 = qt0 + 1 < L.n_q;
    const int h = blockIdx.y, b = blockIdx.z;
    const int sidx = b * a.Hm + (a.Hm == 1 ? 0 : h);
    const int bh = b * a.H + h;
    const int N = a.N;

    if (threadIdx.x == 0) {
        const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(a.plan);
        const bool ok = ph->magic == kPlanMagic && ph->B == L.B && ph->Hm == L.Hm && ph->N == L.N &&
                        ph->bq == 128 && ph->bk == 128;
        if (!ok) set_status(a.status, FM_ERR_PLAN_MISMATCH);
        const bool aligned = (smem_u32(smem) & 1023u) == 0;   // 128-byte swizzle atoms need it
        if (!aligned) set_status(a.status, FM_ERR_UNSUPPORTED);
        *ok_sh = ok && aligned;
        const int32_t *rc = reinterpret_cast<const int32_t *>(a.plan + L.off_row_cnt) + (int64_t)sidx * L.n_q;
        cnt_sh[0] = ok ? rc[qt0] : 0;
        cnt_sh[1] = (ok && has1) ? rc[qt0 + 1] : 0;
        *abort = 0;
        mbar_init(&bars[FB_Q], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[FB_KF0 + s], 1);
            mbar_init(&bars[FB_KE0 + s], 2);    // one arrival per stream
            mbar_init(&bars[FB_VF0 + s], 1);
            mbar_init(&bars[FB_VE0 + s], 2);
            mbar_init(&bars[FB_BF0 + s], 32);
            mbar_init(&bars[FB_S0 + s], 1);
            mbar_init(&bars[FB_P0 + s], 128);
            mbar_init(&bars[FB_O0 + s], 1);
        }
        mbar_init(&bars[FB_DRAIN0], 1);
        mbar_init(&bars[FB_DRAIN1], 1);
        mbar_init(&bars[FB_TK0], 128);   // exponential-phase token for softmax 0 / 1
        mbar_init(&bars[FB_TK1], 128);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int n0 = cnt_sh[0], n1 = cnt_sh[1];
    const int32_t *g0 =
        reinterpret_cast<const int32_t *>(a.plan + L.off_row_list) + ((int64_t)sidx * L.n_q + qt0) * L.n_k;
    const int32_t *g1 = g0 + L.n_k;
    for (int i = threadIdx.x; i < S::kListCap; i += blockDim.x) {
        if (i < n0) sList0[i] = g0[i];
        if (i < n1) sList1[i] = g1[i];
    }
    __syncthreads();
    TileMerge walk{sList0, sList1, g0, g1, n0, n1, 0, 0, S::kListCap};
    const bool any = n0 + n1 > 0;

    if (*ok_sh) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0 && any) {
                tma_prefetch_desc(&tq);
                tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv);
                mbar_arrive_expect_tx(&bars[FB_Q], (has1 ? 2 : 1) * S::kTile);
#pragma unroll
                for (int x = 0; x < NBOX; ++x) {
                    tma_load_3d(smem + S::kQ0 + x * S::kBox, &tq, &bars[FB_Q], x * 64, qt0 * 128, bh);
                    if (has1) tma_load_3d(smem + S::kQ1 + x * S::kBox, &tq, &bars[FB_Q], x * 64, qt0 * 128 + 128, bh);
                }
            }
            int t = 0, kt, l0, l1;
            for (; walk.next(kt, l0, l1); ++t) {
                const int st = t & 1;
                const uint32_t ph = ((t >> 1) - 1) & 1;
                const int kb = kt * 128;
                const bool pred = l0 == FM_TILE_PARTIAL || l1 == FM_TILE_PARTIAL || kb + 128 > N;
                // Column bounds of a partial tile, loaded before the waits below so
                // their latency overlaps them; stored as (start, length) pairs,
                // columns beyond N masked for every row.
                int4 bv[4];
                if (pred) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = kb + lane * 4 + u;
                        bv[u] = make_int4(0, 0, 0, 0x7fffffff);
                        if (j < N) {
                            const int64_t o = (int64_t)sidx * N + j;
                            bv[u] = make_int4(a.lts[o], a.lte[o], a.uts[o], a.ute[o]);
                        }
                    }
                }
                if (t >= 2 && !warp_wait(&bars[FB_KE0 + st], ph, abort, a.status)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[FB_KF0 + st], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(smem + S::kK + st * S::kTile + x * S::kBox, &tk, &bars[FB_KF0 + st], x * 64,
                                    kb, bh);
                }
                if (t >= 2 && !warp_wait(&bars[FB_VE0 + st], ph, abort, a.status)) {
                    ++t;   // K of this tile is in flight
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars[FB_VF0 + st], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(smem + S::kV + st * S::kTile + x * S::kBox, &tv, &bars[FB_VF0 + st], x * 64,
                                    kb, bh);
                }
                if (pred) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int4 v = bv[u];
                        sBnd[st * 128 + lane * 4 + u] = (kb + lane * 4 + u < N)
                                                            ? make_int4(v.x, max(v.y - v.x, 0), v.z, max(v.w - v.z, 0))
                                                            : v;
                    }
                }
                mbar_arrive(&bars[FB_BF0 + st]);
            }
            // Drain copies still in flight (only possible after an abort).
            if (lane == 0 && *abort) {
                if (any) mbar_wait_drain(&bars[FB_Q], 0, a.status);
                for (int k2 = (t > 2 ? t - 2 : 0); k2 < t; ++k2) {
                    mbar_wait_drain(&bars[FB_KF0 + (k2 & 1)], (k2 >> 1) & 1, a.status);
                    mbar_wait_drain(&bars[FB_VF0 + (k2 & 1)], (k2 >> 1) & 1, a.status);
                }
            }
        } else if (warp == 1 || warp == 10) {
            // ------------------------------------------------ MMA issuers
            // One issuing thread per Q tile (warp 1 for Q0, warp 10 for Q1):
            // each alternates S_q = Q_q K^T and O_q += P_q V over its own
            // tiles, so one stream blocking on the tensor-core queue or on its
            // softmax never holds back the other.  Both threads walk every
            // tile of the union: a tile's K (V) stage is released by one
            // arrival per stream, a commit after its S (PV) if the stream needs
            // the tile, a plain arrive after seeing the tile land if not.
            if (lane == 0 && any) {
                const int q = (warp == 1) ? 0 : 1;
                constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
                constexpr uint32_t idO = idesc_bf16(128, D, false, true);
                constexpr int NPART = PRECISE ? 2 : 1;
                const uint64_t dQ = sdesc_sw128(smem_u32(smem + (q ? S::kQ1 : S::kQ0)), 16, 1024);
                const uint32_t tSq = tmem + q * 128, tOq = tmem + 256 + q * 128;
                bool ok = mbar_wait(&bars[FB_Q], 0, abort, a.status);
                int c = 0, t = 0, kt, lab[2];
                for (; ok && walk.next(kt, lab[0], lab[1]); ++t) {
                    const int st = t & 1;
                    const uint32_t ph = (t >> 1) & 1;
                    const bool mine = lab[q] >= 0;
                    if (!mbar_wait(&bars[FB_KF0 + st], ph, abort, a.status)) { ok = false; break; }
                    if (mine) {
                        // S_q aliases P_q of this stream's previous tile: wait for that PV.
                        if (c > 0 && !mbar_wait(&bars[FB_O0 + q], (c - 1) & 1, abort, a.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dK = sdesc_sw128(smem_u32(smem + S::kK + st * S::kTile), 16, 1024);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * S::kBox + (kk & 3) * 32;
                            mma_ss(tSq, sdesc_add(dQ, off), sdesc_add(dK, off), idS, kk > 0);
                        }
                        tc_commit(&bars[FB_S0 + q]);
                        tc_commit(&bars[FB_KE0 + st]);
                    } else {
                        mbar_arrive(&bars[FB_KE0 + st]);
                    }
                    if (!mbar_wait(&bars[FB_VF0 + st], ph, abort, a.status)) { ok = false; break; }
                    if (mine) {
                        if (!mbar_wait(&bars[FB_P0 + q], c & 1, abort, a.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dV = sdesc_sw128(smem_u32(smem + S::kV + st * S::kTile), S::kBox, 1024);
#pragma unroll
                        for (int part = 0; part < NPART; ++part)   // P_hi V (+ P_lo V)
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                mma_ts(tOq, tSq + part * 64 + kk * 8, sdesc_add(dV, kk * 2048), idO,
                                       (c > 0 || part > 0 || kk > 0));
                        tc_commit(&bars[FB_O0 + q]);
                        tc_commit(&bars[FB_VE0 + st]);
                        ++c;
                    } else {
                        mbar_arrive(&bars[FB_VE0 + st]);
                    }
                }
            }
            if (lane == 0) {
                // Every MMA of this CTA completes before TMEM is released.
                tc_commit(&bars[FB_DRAIN0 + (warp == 1 ? 0 : 1)]);
                mbar_wait_drain(&bars[FB_DRAIN0 + (warp == 1 ? 0 : 1)], 0, a.status);
            }
        } else if (warp < 10) {
            // ------------------------------------------------ softmax (Q0: warps 2-5, Q1: warps 6-9)
            const int q = (warp < 6) ? 0 : 1;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int i = (qt0 + q) * 128 + r;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t tS = tmem + q * 128, tO = tmem + 256 + q * 128;
            float m = -INFINITY, l = 0.f, lr = 0.f;
            int cnt = 0;
            bool done = true;
            int t = 0, kt, lab[2];
            // The two softmax warpgroups take turns on the exponential phase
            // (MUFU), tile by tile of the union walk: 0 runs tile t after 1
            // has finished (or skipped) tile t - 1, and 1 runs tile t after 0
            // has finished (or skipped) tile t.  While one exponentiates, the
            // tensor core runs the other stream's products.  A warpgroup
            // always waits for its turn before handing it on, so neither
            // token barrier runs more than one phase ahead of its waiter.
            auto take_turn = [&](int tt) {
                if (q == 0) return tt == 0 || warp_wait(&bars[FB_TK0], (tt - 1) & 1, abort, a.status);
                return warp_wait(&bars[FB_TK1], tt & 1, abort, a.status);
            };
            auto pass_turn = [&]() { mbar_arrive(&bars[q == 0 ? FB_TK1 : FB_TK0]); };
            for (; walk.next(kt, lab[0], lab[1]); ++t) {
                if (lab[q] < 0) {
                    if (!take_turn(t)) { done = false; break; }
                    pass_turn();
                    continue;
                }
                const int st = t & 1;
                const bool pred = (lab[q] == FM_TILE_PARTIAL) || (kt * 128 + 128 > N);
                if (!warp_wait(&bars[FB_S0 + q], cnt & 1, abort, a.status)) { done = false; break; }
                if (pred && !warp_wait(&bars[FB_BF0 + st], (t >> 1) & 1, abort, a.status)) { done = false; break; }
                tc_fence_after();
                uint32_t raw[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + lane_off + cc * 32, raw[cc]);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tmem_reg_fence(raw[cc]);
                float sv[128];
#pragma unroll
                for (int cc = 0; cc < 128; ++cc) sv[cc] = __uint_as_float(raw[cc >> 5][cc & 31]);
                if (pred) {
                    const int4 *bnd = sBnd + st * 128;
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc) {
                        const int4 x = bnd[cc];
                        const bool msk = ((unsigned)(i - x.x) < (unsigned)x.y) || ((unsigned)(i - x.z) < (unsigned)x.w);
                        sv[cc] = msk ? -INFINITY : sv[cc];
                    }
                }
                float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                for (int k2 = 0; k2 < 62; ++k2) mx4[k2 & 3] = fmax3(mx4[k2 & 3], sv[4 + 2 * k2], sv[5 + 2 * k2]);
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * a.scale_log2;   // -inf stays -inf
                float m_new = m, alpha = 1.f;
                if (mx > m + 8.f) {
                    m_new = mx;
                    alpha = ex2(m - m_new);                  // m = -inf gives 0
                }
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                if (!take_turn(t)) { done = false; break; }
                // P = exp2(s * scale*log2e - m), written over S as packed bf16.
                // Precise mode: two terms, P_hi = bf16(P) in columns [0, 64) and
                // P_lo = bf16(P - P_hi) in columns [64, 128).  Standard mode:
                // P_hi only, and O is normalised by the sum of the rounded P,
                // i.e. of the weights the PV product really applied, so the
                // normalised weights sum to one.  lse uses the fp32 sum.
                // Column pairs in packed fp32: x = s * scale*log2e - m, and the
                // running sums of P and of the rounded P.
                const uint64_t sc2 = f2_pack(a.scale_log2, a.scale_log2), nm2 = f2_pack(-m_use, -m_use);
                uint64_t sum2 = f2_pack(0.f, 0.f), rs2 = f2_pack(0.f, 0.f);
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(sv[hh * 32 + 2 * cc], sv[hh * 32 + 2 * cc + 1]), sc2, nm2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        sum2 = f2_add(sum2, f2_pack(p0, p1));
                        hi[cc] = pack_bf16x2(p0, p1);
                        if (PRECISE) {
                            lo[cc] = pack_bf16x2(p0 - __uint_as_float(hi[cc] << 16),
                                                 p1 - __uint_as_float(hi[cc] & 0xffff0000u));
                        } else {
                            rs2 = f2_add(rs2, f2_pack(__uint_as_float(hi[cc] << 16), __uint_as_float(hi[cc] & 0xffff0000u)));
                        }
                    }
                    tmem_st16(tS + lane_off + hh * 16, hi);
                    if (PRECISE) tmem_st16(tS + lane_off + 64 + hh * 16, lo);
                }
                pass_turn();
                float s0, s1;
                f2_unpack(sum2, s0, s1);
                l = l * alpha + (s0 + s1);
                if (!PRECISE) {
                    f2_unpack(rs2, s0, s1);
                    lr = lr * alpha + (s0 + s1);
                }
                m = m_new;
                // Rescale O when the max moved (O holds this tile's earlier KV
                // tiles; their PV finished before this S was computed).
                if (__any_sync(0xffffffffu, cnt > 0 && alpha != 1.f)) {
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        tmem_ld32(tO + lane_off + cc * 32, ov);
                        tmem_ld_wait();
                        tmem_reg_fence(ov);
#pragma unroll
                        for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
                        tmem_st32(tO + lane_off + cc * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[FB_P0 + q]);
                ++cnt;
            }
            // ------------------------------------------------ epilogue
            const bool tile_exists = q == 0 || has1;
            if (tile_exists && done && (cnt == 0 || warp_wait(&bars[FB_O0 + q], (cnt - 1) & 1, abort, a.status))) {
                tc_fence_after();
                const float nrm = PRECISE ? l : lr;
                const float inv = (nrm > 0.f) ? 1.f / nrm : 0.f;
                const bool row_in = i < N;
                const int64_t row = (int64_t)bh * N + i;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    if (cnt > 0) {
                        tmem_ld32(tO + lane_off + cc * 32, ov);
                        tmem_ld_wait();
                        tmem_reg_fence(ov);
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u) ov[u] = 0u;
                    }
                    if (!row_in) continue;
                    if (a.o_f32) {
                        float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + row * D + cc * 32);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            dst[u] = make_float4(__uint_as_float(ov[4 * u]) * inv, __uint_as_float(ov[4 * u + 1]) * inv,
                                                 __uint_as_float(ov[4 * u + 2]) * inv, __uint_as_float(ov[4 * u + 3]) * inv);
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + row * D + cc * 32);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            dst[u] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * u + 0]) * inv, __uint_as_float(ov[8 * u + 1]) * inv),
                                                pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv),
                                                pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv),
                                                pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv));
                    }
                }
                if (row_in)
                    a.lse[row] = (l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
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

template <int D, bool PRECISE>
static fm_status launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const FwdArgs &a, cudaStream_t stream)
{
    constexpr int smem = FwdSmem<D>::kBytes;
    static_assert(smem <= 227 * 1024, "shared memory budget");
    if (cudaFuncSetAttribute(fm_fwd_kernel<D, PRECISE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
        return FM_ERR_CUDA;
    ProfScope ps(kKFwd, stream);
    fm_fwd_kernel<D, PRECISE><<<dim3((a.L.n_q + 1) / 2, a.H, a.B), 352, smem, stream>>>(tq, tk, tv, a);
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}

fm_status fm_fwd_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const FwdArgs &a, int d, bool precise, cudaStream_t stream)
{
    if (d == 128)
        return precise ? launch_fwd<128, true>(tq, tk, tv, a, stream) : launch_fwd<128, false>(tq, tk, tv, a, stream);
    return precise ? launch_fwd<64, true>(tq, tk, tv, a, stream) : launch_fwd<64, false>(tq, tk, tv, a, stream);
}
