// Forward masked attention on sm_103a (tcgen05 + TMEM + TMA).
//
// Passages: FlashAttention article §二.1 (tiling), §二.2 (max-subtracted
// softmax; completed here by the standard running rescale so the result is
// the exact softmax), §二.3 (QK^T and PV on tensor cores, fused in one
// kernel); blog "FlashMask技术" §2.2 (skip / full / masked block paths) and
// §4.1 items 1-3 (bounds staged in shared memory, skip decided before the KV
// block is loaded, mask fused into the softmax).
//
// One CTA = one (b, h, 128-row Q tile).  Roles:
//   warp 0      TMA producer: Q once, then K and V of each non-skip KV tile
//               from the plan's ordered list (skip tiles are never loaded);
//   warp 1      allocates TMEM, one thread issues the tcgen05 MMAs;
//   warps 2-5   softmax, one thread per Q row = TMEM lane.
// TMEM (256 columns): S = Q K^T at columns [0, 128) (fp32), then overwritten
// in place by P as two packed-bf16 terms (P_hi, P_lo: 64 columns each), the A
// operands of O += P_hi V + P_lo V; O accumulates at columns [128, 128 + d).
// Online softmax in the base-2 domain with a lazy rescale: O and l are
// rescaled only when the row max grows by more than 2^8, which keeps every
// P <= 256 and leaves the final O / l unchanged.
// Two CTAs share an SM (about 100 KB shared memory and 256 TMEM columns each)
// so one CTA's softmax overlaps the other's MMAs.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

template <int D>
struct FwdSmem {
    static constexpr int kBox = 128 * 128;        // one 64-column, 128-row bf16 box
    static constexpr int kTile = 128 * D * 2;     // Q, K or V tile
    static constexpr int kQ = 0, kK = kTile, kV = 2 * kTile;
    static constexpr int kBnd = 3 * kTile;        // int4 [2][128]
    static constexpr int kBar = kBnd + 4096;
    static constexpr int kNumBar = 10;
    static constexpr int kMisc = kBar + kNumBar * 8;
    static constexpr int kUsed = kMisc + 64;
    // Request at least 100 KB so that no more than two CTAs (2 x 256 TMEM
    // columns) are resident on one SM.
    static constexpr int kBytes = (kUsed + 1024 > 100 * 1024) ? kUsed + 1024 : 100 * 1024;
};

enum { FB_Q = 0, FB_K, FB_V, FB_KE, FB_VE, FB_S, FB_P, FB_O, FB_DRAIN, FB_BND };

template <int D>
__global__ void __launch_bounds__(192, 2)
    fm_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdArgs a)
{
    using S = FwdSmem<D>;
    constexpr int NBOX = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem + S::kQ, *sK = smem + S::kK, *sV = smem + S::kV;
    int4 *sBnd = reinterpret_cast<int4 *>(smem + S::kBnd);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::kBar);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + S::kMisc);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + S::kMisc + 4);
    int *cnt_sh = reinterpret_cast<int *>(smem + S::kMisc + 8);
    int *ok_sh = reinterpret_cast<int *>(smem + S::kMisc + 12);

    const int warp = warp_id(), lane = lane_id();
    const PlanLayout &L = a.L;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;   // heavy causal tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int sidx = b * a.Hm + (a.Hm == 1 ? 0 : h);
    const int bh = b * a.H + h;
    const int N = a.N;

    if (threadIdx.x == 0) {
        const PlanHeader *ph = reinterpret_cast<const PlanHeader *>(a.plan);
        const bool ok = ph->magic == kPlanMagic && ph->B == L.B && ph->Hm == L.Hm && ph->N == L.N &&
                        ph->bq == 128 && ph->bk == 128;
        if (!ok) set_status(a.status, FM_ERR_PLAN_MISMATCH);
        *ok_sh = ok;
        *cnt_sh = ok ? reinterpret_cast<const int32_t *>(a.plan + L.off_row_cnt)[(int64_t)sidx * L.n_q + qt] : 0;
        *abort = 0;
        mbar_init(&bars[FB_Q], 1);
        mbar_init(&bars[FB_K], 1);
        mbar_init(&bars[FB_V], 1);
        mbar_init(&bars[FB_KE], 1);
        mbar_init(&bars[FB_VE], 1);
        mbar_init(&bars[FB_S], 1);
        mbar_init(&bars[FB_P], 128);
        mbar_init(&bars[FB_O], 1);
        mbar_init(&bars[FB_DRAIN], 1);
        mbar_init(&bars[FB_BND], 128);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS = tmem, tO = tmem + 128;
    const int cnt = *cnt_sh;
    const int32_t *list =
        reinterpret_cast<const int32_t *>(a.plan + L.off_row_list) + ((int64_t)sidx * L.n_q + qt) * L.n_k;

    if (*ok_sh) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&tq);
                tma_prefetch_desc(&tk);
                tma_prefetch_desc(&tv);
                int issued = 0;
                if (cnt > 0) {
                    mbar_arrive_expect_tx(&bars[FB_Q], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(sQ + x * S::kBox, &tq, &bars[FB_Q], x * 64, qt * 128, bh);
                }
                for (int t = 0; t < cnt; ++t) {
                    const int kt = list[t] & kTileMask;
                    if (t > 0 && !mbar_wait(&bars[FB_KE], (t - 1) & 1, abort, a.status)) break;
                    mbar_arrive_expect_tx(&bars[FB_K], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(sK + x * S::kBox, &tk, &bars[FB_K], x * 64, kt * 128, bh);
                    if (t > 0 && !mbar_wait(&bars[FB_VE], (t - 1) & 1, abort, a.status)) {
                        issued = -(t + 1);   // K of tile t in flight, V not
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[FB_V], S::kTile);
#pragma unroll
                    for (int x = 0; x < NBOX; ++x)
                        tma_load_3d(sV + x * S::kBox, &tv, &bars[FB_V], x * 64, kt * 128, bh);
                    issued = t + 1;
                }
                // Drain: every issued copy must land before the CTA exits.
                if (*abort) {
                    const int nk = issued < 0 ? -issued : issued, nv = issued < 0 ? -issued - 1 : issued;
                    if (cnt > 0) mbar_wait_drain(&bars[FB_Q], 0, a.status);
                    if (nk > 0) mbar_wait_drain(&bars[FB_K], (nk - 1) & 1, a.status);
                    if (nv > 0) mbar_wait_drain(&bars[FB_V], (nv - 1) & 1, a.status);
                }
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
                constexpr uint32_t idO = idesc_bf16(128, D, false, true);
                const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
                if (cnt > 0 && mbar_wait(&bars[FB_Q], 0, abort, a.status)) {
                    for (int t = 0; t < cnt; ++t) {
                        if (!mbar_wait(&bars[FB_K], t & 1, abort, a.status)) break;
                        if (t > 0 && !mbar_wait(&bars[FB_O], (t - 1) & 1, abort, a.status)) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * S::kBox + (kk & 3) * 32;
                            mma_ss(tS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024),
                                   idS, kk > 0);
                        }
                        tc_commit(&bars[FB_S]);
                        tc_commit(&bars[FB_KE]);
                        if (!mbar_wait(&bars[FB_P], t & 1, abort, a.status)) break;
                        if (!mbar_wait(&bars[FB_V], t & 1, abort, a.status)) break;
                        tc_fence_after();
#pragma unroll
                        for (int part = 0; part < 2; ++part)     // P_hi V, then P_lo V
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                mma_ts(tO, tS + part * 64 + kk * 8, sdesc_sw128(aV + kk * 2048, S::kBox, 1024),
                                       idO, (t > 0 || part > 0 || kk > 0));
                        tc_commit(&bars[FB_O]);
                        tc_commit(&bars[FB_VE]);
                    }
                }
                // Every MMA of this CTA completes before TMEM is released.
                tc_commit(&bars[FB_DRAIN]);
                mbar_wait_drain(&bars[FB_DRAIN], 0, a.status);
            }
        } else {
            // ------------------------------------------------ softmax
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int i = qt * 128 + r;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            float m = -INFINITY, l = 0.f;
            int npart = 0;
            bool done = true;
            for (int t = 0; t < cnt; ++t) {
                const int32_t e = list[t];
                const int kt = e & kTileMask, lab = e >> kLabelShift;
                const int kb = kt * 128;
                const bool pred = (lab == FM_TILE_PARTIAL) || (kb + 128 > N);
                int4 *bnd = sBnd + (npart & 1) * 128;
                if (pred) {
                    const int j = kb + r;
                    int4 v;
                    if (j < N) {
                        const int64_t o = (int64_t)sidx * N + j;
                        const int l0 = a.lts[o], l1 = a.lte[o], u0 = a.uts[o], u1 = a.ute[o];
                        v = make_int4(l0, max(l1 - l0, 0), u0, max(u1 - u0, 0));
                    } else {
                        v = make_int4(0, 0, 0, 0x7fffffff);   // beyond N: masked for every row
                    }
                    bnd[r] = v;
                    mbar_arrive(&bars[FB_BND]);
                    if (!warp_wait(&bars[FB_BND], npart & 1, abort, a.status)) { done = false; break; }
                    ++npart;
                }
                if (!warp_wait(&bars[FB_S], t & 1, abort, a.status)) { done = false; break; }
                tc_fence_after();
                uint32_t raw[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, raw[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_reg_fence(raw[c]);
                float sv[128];
#pragma unroll
                for (int c = 0; c < 128; ++c) sv[c] = __uint_as_float(raw[c >> 5][c & 31]);
                if (pred) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const int4 x = bnd[c];
                        const bool msk = ((unsigned)(i - x.x) < (unsigned)x.y) ||
                                         ((unsigned)(i - x.z) < (unsigned)x.w);
                        sv[c] = msk ? -INFINITY : sv[c];
                    }
                }
                float mx0 = sv[0], mx1 = sv[1], mx2 = sv[2], mx3 = sv[3];
#pragma unroll
                for (int c = 4; c < 128; c += 4) {
                    mx0 = fmaxf(mx0, sv[c]);
                    mx1 = fmaxf(mx1, sv[c + 1]);
                    mx2 = fmaxf(mx2, sv[c + 2]);
                    mx3 = fmaxf(mx3, sv[c + 3]);
                }
                const float rowmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
                const float mx = rowmax * a.scale_log2;     // -inf stays -inf
                float m_new = m, alpha = 1.f;
                if (mx > m + 8.f) {
                    m_new = mx;
                    alpha = ex2(m - m_new);                  // m = -inf gives 0
                }
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                // P = exp2(s * scale*log2e - m), written over S as two packed bf16
                // terms: P_hi = bf16(P) in columns [0, 64) and P_lo = bf16(P - P_hi)
                // in columns [64, 128).  O accumulates P_hi V + P_lo V, so O carries
                // ~16 significant bits of P instead of one bf16 rounding (the
                // backward's D = rowsum(dO * O) depends on that accuracy).
                float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float p0 = ex2(fmaf(sv[hh * 32 + 2 * c], a.scale_log2, -m_use));
                        const float p1 = ex2(fmaf(sv[hh * 32 + 2 * c + 1], a.scale_log2, -m_use));
                        sum0 += p0;
                        sum1 += p1;
                        hi[c] = pack_bf16x2(p0, p1);
                        lo[c] = pack_bf16x2(p0 - __uint_as_float(hi[c] << 16), p1 - __uint_as_float(hi[c] & 0xffff0000u));
                    }
                    tmem_st16(tS + lane_off + hh * 16, hi);
                    tmem_st16(tS + lane_off + 64 + hh * 16, lo);
                }
                l = l * alpha + (sum0 + sum1);
                m = m_new;
                // Rescale O when the max moved (O holds tiles 0..t-1; the PV MMA
                // of tile t is issued only after this thread's arrive below).
                if (__any_sync(0xffffffffu, t > 0 && alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tO + lane_off + c * 32, ov);
                        tmem_ld_wait();
                        tmem_reg_fence(ov);
#pragma unroll
                        for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
                        tmem_st32(tO + lane_off + c * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[FB_P]);
            }
            // ------------------------------------------------ epilogue
            if (done && (cnt == 0 || warp_wait(&bars[FB_O], (cnt - 1) & 1, abort, a.status))) {
                tc_fence_after();
                const float inv = (l > 0.f) ? 1.f / l : 0.f;
                const bool row_in = i < N;
                const int64_t row = (int64_t)bh * N + i;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    if (cnt > 0) {
                        tmem_ld32(tO + lane_off + c * 32, ov);
                        tmem_ld_wait();
                        tmem_reg_fence(ov);
                    } else {
#pragma unroll
                        for (int u = 0; u < 32; ++u) ov[u] = 0u;
                    }
                    if (row_in) {
                        if (a.o_f32) {
                            float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.o) + row * D + c * 32);
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                dst[u] = make_float4(__uint_as_float(ov[4 * u]) * inv, __uint_as_float(ov[4 * u + 1]) * inv,
                                                     __uint_as_float(ov[4 * u + 2]) * inv, __uint_as_float(ov[4 * u + 3]) * inv);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.o) + row * D + c * 32);
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                uint4 w;
                                w.x = pack_bf16x2(__uint_as_float(ov[8 * u + 0]) * inv, __uint_as_float(ov[8 * u + 1]) * inv);
                                w.y = pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv);
                                w.z = pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv);
                                w.w = pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv);
                                dst[u] = w;
                            }
                        }
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
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace fm

using namespace fm;

fm_status fm_fwd_launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const FwdArgs &a, int d, cudaStream_t stream)
{
    const dim3 grid(a.L.n_q, a.H, a.B);
    if (d == 128) {
        constexpr int smem = FwdSmem<128>::kBytes;
        if (cudaFuncSetAttribute(fm_fwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return FM_ERR_CUDA;
        ProfScope ps(kKFwd, stream);
        fm_fwd_kernel<128><<<grid, 192, smem, stream>>>(tq, tk, tv, a);
    } else {
        constexpr int smem = FwdSmem<64>::kBytes;
        if (cudaFuncSetAttribute(fm_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return FM_ERR_CUDA;
        ProfScope ps(kKFwd, stream);
        fm_fwd_kernel<64><<<grid, 192, smem, stream>>>(tq, tk, tv, a);
    }
    return cudaPeekAtLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
