// Tile classification (blog "FlashMask技术" §2.2: per (Q block, KV block)
// skip / full GEMM / masked GEMM; §4.1 item 2: decide before a KV block is
// loaded).  Three launches:
//   1. minmax: one CTA per (b*Hm, KV tile) reduces the tile's canonicalised
//      column bounds to 8 int32 (min and max of each bound), validates the
//      bounds and writes the plan header;
//   2. lists:  one CTA per (b*Hm, Q tile) writes that Q tile's label row and
//      the ordered list of its non-skip KV tiles; one CTA per (b*Hm, KV tile)
//      writes the list of non-skip Q tiles of that KV tile (for the
//      KV-major backward).  Labels are recomputed from the 8 numbers, so the
//      two halves need no other dependency;
//   3. order:  a stable counting sort by list length, longest first, one CTA
//      per direction (for the backward a KV tile's length is that of the
//      longest list in its group, see below); the attention kernels claim
//      their units in this order, so the longest lists (a sink column, a long
//      document) start first, and a document's KV tiles run together in the
//      backward (sharing their Q / dO tiles and dQ rows in L2).
// HBM traffic: 16 bytes per column read, n_q*n_k label bytes and <= 8 bytes
// per non-skip pair written.
#include <cuda_runtime.h>

#include "fm_internal.h"
#include "fm_ptx.cuh"

namespace fm {

struct TileMinMax {  // canonical empty lower = (N, N), empty upper = (0, 0)
    int32_t L0max, L0min, L1min, L1max, U0max, U0min, U1min, U1max;
};

__device__ __forceinline__ int tile_label(const TileMinMax &t, int qb, int qe)
{
    const bool skip = (t.L0max <= qb && t.L1min >= qe) || (t.U0max <= qb && t.U1min >= qe);
    if (skip) return FM_TILE_SKIP;
    const bool lower_clear = t.L0min >= qe || t.L1max <= qb;
    const bool upper_clear = t.U0min >= qe || t.U1max <= qb;
    return (lower_clear && upper_clear) ? FM_TILE_FULL : FM_TILE_PARTIAL;
}

__global__ void __launch_bounds__(128) classify_minmax_kernel(fm_bounds m, PlanLayout L,
                                                              uint8_t *plan, int32_t *status)
{
    const int kt = blockIdx.x, s = blockIdx.y;
    const int N = L.N, bk = L.bk;
    const int j = kt * bk + threadIdx.x;
    const bool in = threadIdx.x < bk && j < N;
    int l0 = N, l1 = N, u0 = 0, u1 = 0;
    if (in) {
        const int64_t o = (int64_t)s * N + j;
        l0 = m.lts[o]; l1 = m.lte[o]; u0 = m.uts[o]; u1 = m.ute[o];
        if ((unsigned)l0 > (unsigned)N || (unsigned)l1 > (unsigned)N || (unsigned)u0 > (unsigned)N ||
            (unsigned)u1 > (unsigned)N)
            set_status(status, FM_ERR_BAD_BOUNDS);
        if (l0 >= l1) { l0 = N; l1 = N; }
        if (u0 >= u1) { u0 = 0; u1 = 0; }
    }
    // max-reductions: the max of x and the max of -x (= -min)
    int v[8] = {in ? l0 : INT_MIN, in ? -l0 : INT_MIN, in ? -l1 : INT_MIN, in ? l1 : INT_MIN,
                in ? u0 : INT_MIN, in ? -u0 : INT_MIN, in ? -u1 : INT_MIN, in ? u1 : INT_MIN};
#pragma unroll
    for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v[q] = max(v[q], __shfl_xor_sync(0xffffffffu, v[q], off));
    __shared__ int red[4][8];
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int q = 0; q < 8; ++q) red[w][q] = v[q];
    __syncthreads();
    if (threadIdx.x < 8) {
        int r = red[0][threadIdx.x];
        for (int ww = 1; ww < (int)(blockDim.x >> 5); ++ww) r = max(r, red[ww][threadIdx.x]);
        const bool neg = (threadIdx.x == 1 || threadIdx.x == 2 || threadIdx.x == 5 || threadIdx.x == 6);
        int32_t *mm = reinterpret_cast<int32_t *>(plan + L.off_minmax) + ((int64_t)s * L.n_k + kt) * 8;
        mm[threadIdx.x] = neg ? -r : r;
    }
    if (kt == 0 && s == 0 && threadIdx.x == 0) {
        PlanHeader *h = reinterpret_cast<PlanHeader *>(plan);
        h->B = L.B; h->Hm = L.Hm; h->N = L.N; h->bq = L.bq; h->bk = L.bk;
        h->n_q = L.n_q; h->n_k = L.n_k; h->total = L.total;
        h->off_row_order = L.off_row_order; h->off_col_order = L.off_col_order;
        h->off_row_bstart = L.off_row_bstart; h->off_col_bstart = L.off_col_bstart;
        h->q_row0 = L.q_row0; h->Nq = L.Nq;
        __threadfence();
        h->magic = kPlanMagic;
    }
}

__device__ __forceinline__ TileMinMax load_minmax(const int32_t *p)
{
    TileMinMax t;
    t.L0max = p[0]; t.L0min = p[1]; t.L1min = p[2]; t.L1max = p[3];
    t.U0max = p[4]; t.U0min = p[5]; t.U1min = p[6]; t.U1max = p[7];
    return t;
}

// blockIdx.x < n_q: row job for Q tile blockIdx.x; otherwise column job for
// KV tile blockIdx.x - n_q.  128 threads; ordered compaction by warp ballots.
__global__ void __launch_bounds__(128) classify_lists_kernel(PlanLayout L, uint8_t *plan,
                                                             uint8_t *labels_out)
{
    const int s = blockIdx.y;
    const int32_t *mm = reinterpret_cast<const int32_t *>(plan + L.off_minmax) + (int64_t)s * L.n_k * 8;
    __shared__ int warp_cnt[4];
    __shared__ int base_sh;
    const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
    if (threadIdx.x == 0) base_sh = 0;
    __syncthreads();

    const bool row_job = (int)blockIdx.x < L.n_q;
    const int idx = row_job ? blockIdx.x : blockIdx.x - L.n_q;
    const int n_other = row_job ? L.n_k : L.n_q;
    int32_t *list;
    int32_t *cnt;
    uint8_t *lbl_row = nullptr, *lbl_out = nullptr;
    TileMinMax own{};
    int qb = 0, qe = 0;
    if (row_job) {
        list = reinterpret_cast<int32_t *>(plan + L.off_row_list) + ((int64_t)s * L.n_q + idx) * L.n_k;
        cnt = reinterpret_cast<int32_t *>(plan + L.off_row_cnt) + (int64_t)s * L.n_q + idx;
        lbl_row = plan + L.off_labels + ((int64_t)s * L.n_q + idx) * L.n_k;
        if (labels_out) lbl_out = labels_out + ((int64_t)s * L.n_q + idx) * L.n_k;
        qb = L.q_row0 + idx * L.bq;
        qe = min(qb + L.bq, L.q_row0 + L.Nq);
    } else {
        list = reinterpret_cast<int32_t *>(plan + L.off_col_list) + ((int64_t)s * L.n_k + idx) * L.n_q;
        cnt = reinterpret_cast<int32_t *>(plan + L.off_col_cnt) + (int64_t)s * L.n_k + idx;
        own = load_minmax(mm + (int64_t)idx * 8);
    }
    for (int c0 = 0; c0 < n_other; c0 += 128) {
        const int c = c0 + threadIdx.x;
        int lab = FM_TILE_SKIP;
        if (c < n_other) {
            if (row_job) {
                lab = tile_label(load_minmax(mm + (int64_t)c * 8), qb, qe);
                lbl_row[c] = (uint8_t)lab;
                if (lbl_out) lbl_out[c] = (uint8_t)lab;
            } else {
                const int b0 = L.q_row0 + c * L.bq;
                lab = tile_label(own, b0, min(b0 + L.bq, L.q_row0 + L.Nq));
            }
        }
        const bool keep = c < n_other && lab != FM_TILE_SKIP;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (ln == 0) warp_cnt[w] = __popc(bal);
        __syncthreads();
        int before = base_sh;
        for (int ww = 0; ww < w; ++ww) before += warp_cnt[ww];
        if (keep) list[before + __popc(bal & ((1u << ln) - 1u))] = c | (lab << kLabelShift);
        __syncthreads();
        if (threadIdx.x == 0) base_sh += warp_cnt[0] + warp_cnt[1] + warp_cnt[2] + warp_cnt[3];
        __syncthreads();
    }
    if (threadIdx.x == 0) *cnt = base_sh;
}

constexpr int kOrderThreads = 1024;

// blockIdx.x == 0: order of the B*Hm*n_q Q-tile entries by row-list length;
// blockIdx.x == 1: order of the B*Hm*n_k KV-tile entries by column-list length.
// A counting sort over the length buckets of order_bucket (longest first),
// stable: inside a bucket entries keep their index order, so the plan is
// deterministic.  Also writes the first entry of every bucket.
// Backward order: the KV tiles whose Q-tile lists end at the same Q tile form
// a group (under causal masks within documents: the KV tiles of one
// document); their lists read the same Q / dO tiles and add into the same dQ
// rows, so the order keeps a group together: an entry's bucket is that of the
// longest list in its group (largest groups first), and the stable sort keeps
// index order inside a bucket, hence the group's tiles contiguous (measured at
// 128K packing: 1-3 % faster backward; the same grouping of the forward's Q
// tiles by their lists' first KV tile made document packing 3 % slower, so
// the forward order keys each tile by its own list length).  Segments with
// more than kGroupCap tiles use the entry's own list length.
constexpr int kGroupCap = 8192;

__global__ void __launch_bounds__(kOrderThreads) classify_order_kernel(PlanLayout L, uint8_t *plan)
{
    const bool rows = blockIdx.x == 0;
    const int n_t = rows ? L.n_q : L.n_k;              // tiles per (b, hm) segment
    const int n_other = rows ? L.n_k : L.n_q;          // list capacity per tile
    const int64_t n_seg = (int64_t)L.B * L.Hm;
    const int32_t *len = reinterpret_cast<const int32_t *>(plan + (rows ? L.off_row_cnt : L.off_col_cnt));
    const int32_t *lists = reinterpret_cast<const int32_t *>(plan + (rows ? L.off_row_list : L.off_col_list));
    int32_t *order = reinterpret_cast<int32_t *>(plan + (rows ? L.off_row_order : L.off_col_order));
    int32_t *bstart = reinterpret_cast<int32_t *>(plan + (rows ? L.off_row_bstart : L.off_col_bstart));

    __shared__ int hist[kOrderBuckets];
    __shared__ int next[kOrderBuckets];
    __shared__ int gmax[kGroupCap];
    const int t = threadIdx.x, w = t >> 5, ln = t & 31;
    const bool grouped = !rows && n_t <= kGroupCap;
    // Group key of entry e (a tile index), or -1 for an empty list.
    auto key_of = [&](int64_t e) -> int {
        const int n = len[e];
        if (n <= 0) return -1;
        return lists[e * n_other + (rows ? 0 : n - 1)] & kTileMask;
    };
    // gmax[key] = longest list of the group, for segment sg (whole block).
    auto group_max = [&](int64_t sg) {
        for (int i = t; i < n_t; i += kOrderThreads) gmax[i] = 0;
        __syncthreads();
        for (int i = t; i < n_t; i += kOrderThreads) {
            const int64_t e = sg * n_t + i;
            const int k = key_of(e);
            if (k >= 0) atomicMax(&gmax[k], len[e]);
        }
        __syncthreads();
    };
    auto weight_of = [&](int64_t e) -> int {
        if (!grouped) return len[e];
        const int k = key_of(e);
        return k < 0 ? 0 : gmax[k];
    };
    if (t < kOrderBuckets) hist[t] = 0;
    __syncthreads();
    for (int64_t sg = 0; sg < n_seg; ++sg) {
        if (grouped) group_max(sg);
        for (int i = t; i < n_t; i += kOrderThreads) atomicAdd(&hist[order_bucket(weight_of(sg * n_t + i))], 1);
        __syncthreads();
    }
    if (t == 0) {
        int run = 0;
        for (int k = 0; k < kOrderBuckets; ++k) {
            next[k] = run;
            bstart[k] = run;
            run += hist[k];
        }
        bstart[kOrderBuckets] = run;
    }
    __syncthreads();
    // stable scatter, one chunk of 1024 entries at a time: rank inside the warp
    // (peers with the same bucket), then a scan of the warps' counts per bucket.
    __shared__ uint8_t wcnt[kOrderThreads / 32][kOrderBuckets];
    __shared__ int wbase[kOrderThreads / 32][kOrderBuckets];
    for (int64_t sg = 0; sg < n_seg; ++sg)
    for (int c0 = 0; c0 < n_t; c0 += kOrderThreads) {
        if (c0 == 0 && grouped) group_max(sg);
        for (int i = t; i < (kOrderThreads / 32) * kOrderBuckets; i += kOrderThreads) (&wcnt[0][0])[i] = 0;
        __syncthreads();
        const int64_t e = sg * n_t + c0 + t;
        const int bk = (c0 + t < n_t) ? order_bucket(weight_of(e)) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, bk);
        const int rank = __popc(peers & ((1u << ln) - 1u));
        if (bk >= 0 && rank == 0) wcnt[w][bk] = (uint8_t)__popc(peers);
        __syncthreads();
        if (t < kOrderBuckets) {
            int run = next[t];
            for (int ww = 0; ww < kOrderThreads / 32; ++ww) {
                wbase[ww][t] = run;
                run += wcnt[ww][t];
            }
            next[t] = run;
        }
        __syncthreads();
        if (bk >= 0) order[wbase[w][bk] + rank] = (int32_t)e;
        __syncthreads();
    }
}

}  // namespace fm

using namespace fm;

fm_status fm_classify_launch(fm_bounds m, int q_row0, int Nq, int bq, int bk, void *plan, uint8_t *labels,
                             int32_t *status, cudaStream_t stream)
{
    PlanLayout L;
    if (!plan_layout(m.B, m.Hm, m.N, bq, bk, &L, q_row0, Nq)) return FM_ERR_INVALID_ARG;
    const int S = m.B * m.Hm;
    if (L.n_k > 65535 * 64 || S > 65535) return FM_ERR_UNSUPPORTED;
    {
        ProfScope ps(kKClassifyMinmax, stream);
        classify_minmax_kernel<<<dim3(L.n_k, S), 128, 0, stream>>>(m, L, (uint8_t *)plan, status);
    }
    if (cudaPeekAtLastError() != cudaSuccess) return FM_ERR_CUDA;
    {
        ProfScope ps(kKClassifyLists, stream);
        classify_lists_kernel<<<dim3(L.n_q + L.n_k, S), 128, 0, stream>>>(L, (uint8_t *)plan, labels);
    }
    if (cudaPeekAtLastError() != cudaSuccess) return FM_ERR_CUDA;
    {
        ProfScope ps(kKClassifyOrder, stream);
        classify_order_kernel<<<2, kOrderThreads, 0, stream>>>(L, (uint8_t *)plan);
    }
    if (cudaPeekAtLastError() != cudaSuccess) return FM_ERR_CUDA;
    return FM_OK;
}
