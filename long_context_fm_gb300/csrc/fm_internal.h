// Internal definitions shared by the library's host and device code.
#pragma once

#include <cstddef>
#include <cstdint>

#include "fm.h"

#if defined(__CUDACC__)
#define FM_HD __host__ __device__ __forceinline__
#else
#define FM_HD inline
#endif

namespace fm {

constexpr uint32_t kPlanMagic = 0x464D5031u;  // "FMP1"
constexpr int kLabelShift = 28;               // list entry = tile | (label << 28)
constexpr int32_t kTileMask = (1 << kLabelShift) - 1;

// Plan layout: header, per-KV-tile min/max, labels, per-Q-tile lists (CSR),
// per-KV-tile lists (CSC), and the two work orders.  Every section starts on a
// 256-byte boundary.
struct PlanLayout {
    int32_t B, Hm, N, bq, bk, n_q, n_k;
    int32_t q_row0, Nq;    // Q rows [q_row0, q_row0 + Nq) of the N x N mask (whole mask: 0, N)
    int64_t off_minmax;    // int32 [B*Hm][n_k][8]
    int64_t off_labels;    // uint8 [B*Hm][n_q][n_k]
    int64_t off_row_cnt;   // int32 [B*Hm][n_q]
    int64_t off_row_list;  // int32 [B*Hm][n_q][n_k]  kv tile | label << 28
    int64_t off_col_cnt;   // int32 [B*Hm][n_k]
    int64_t off_col_list;  // int32 [B*Hm][n_k][n_q]  q tile | label << 28
    int64_t off_row_order; // int32 [B*Hm*n_q]  entries s*n_q + q tile, longest list first
    int64_t off_col_order; // int32 [B*Hm*n_k]  entries s*n_k + kv tile, longest list first
    int64_t off_row_bstart;// int32 [kOrderBuckets + 1]  first row-order entry of each bucket
    int64_t off_col_bstart;// int32 [kOrderBuckets + 1]  first col-order entry of each bucket
    int64_t total;
};

// Work-order buckets: list length len > 0 falls in half-octave 2*floor(log2 len)
// + (second bit of len), len = 0 in the last bucket; bucket 0 holds the
// longest lists.  Within a bucket entries keep their index order.
constexpr int kOrderBuckets = 64;
FM_HD int order_bucket(int len)
{
    if (len <= 0) return kOrderBuckets - 1;
    int lg = 0;
    while ((len >> lg) > 1) ++lg;
    const int half = lg > 0 ? (len >> (lg - 1)) & 1 : 0;
    return kOrderBuckets - 2 - (2 * lg + half);          // lg <= 30: result in [0, 62]
}

struct PlanHeader {        // first 128 bytes of a plan, written by the classifier
    uint32_t magic;
    int32_t B, Hm, N, bq, bk, n_q, n_k;
    int64_t total;
    int64_t off_row_order, off_col_order, off_row_bstart, off_col_bstart;
    int32_t q_row0, Nq;
    int32_t pad[12];
};
static_assert(sizeof(PlanHeader) == 128, "plan header size");

FM_HD int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

// Plan of the Q rows [q_row0, q_row0 + Nq) against all N key columns;
// q_row0 is a multiple of bq, so local Q tile t covers global rows
// [q_row0 + t bq, ...).  Nq < 0 means the whole mask (q_row0 = 0, Nq = N).
FM_HD bool plan_layout(int B, int Hm, int N, int bq, int bk, PlanLayout *L, int q_row0 = 0, int Nq = -1)
{
    if (Nq < 0) { q_row0 = 0; Nq = N; }
    if (B <= 0 || Hm <= 0 || N <= 0 || Nq <= 0 || q_row0 < 0) return false;
    if (!((bq == 64 || bq == 128) && (bk == 64 || bk == 128))) return false;
    if (q_row0 % bq != 0 || (int64_t)q_row0 + Nq > N) return false;
    const int64_t n_q = (Nq + bq - 1) / bq, n_k = (N + bk - 1) / bk;
    if (n_q >= kTileMask || n_k >= kTileMask) return false;
    const int64_t S = (int64_t)B * Hm;
    if (S * (n_q > n_k ? n_q : n_k) >= ((int64_t)1 << 31)) return false;   // order entries are int32
    L->B = B; L->Hm = Hm; L->N = N; L->bq = bq; L->bk = bk;
    L->q_row0 = q_row0; L->Nq = Nq;
    L->n_q = (int32_t)n_q; L->n_k = (int32_t)n_k;
    int64_t off = 256;
    L->off_minmax = off;   off = align256(off + S * n_k * 8 * 4);
    L->off_labels = off;   off = align256(off + S * n_q * n_k);
    L->off_row_cnt = off;  off = align256(off + S * n_q * 4);
    L->off_row_list = off; off = align256(off + S * n_q * n_k * 4);
    L->off_col_cnt = off;  off = align256(off + S * n_k * 4);
    L->off_col_list = off; off = align256(off + S * n_k * n_q * 4);
    L->off_row_order = off; off = align256(off + S * n_q * 4);
    L->off_col_order = off; off = align256(off + S * n_k * 4);
    L->off_row_bstart = off; off = align256(off + (kOrderBuckets + 1) * 4);
    L->off_col_bstart = off; off = align256(off + (kOrderBuckets + 1) * 4);
    L->total = off;
    return true;
}

#if defined(__CUDACC__)
// Work unit of the attention CTA with linear block index c, for a grid of
// n_tiles x H x B CTAs; called by all 32 lanes of one warp, result valid in
// every lane.  Order entries (s * n_tiles + tile, s = b * Hm + hm) are grouped
// into length buckets, longest first; one entry stands for the rep heads that
// read mask head hm (rep = H for a shared mask, else 1).  Inside a bucket the
// heads are outermost, so CTAs that run together mostly share a head and read
// neighbouring tiles.  Returns false on a plan not written by the classifier.
__device__ __forceinline__ bool plan_unit(const int32_t *order, const int32_t *bstart, int n_tiles, int B,
                                          int Hm, int H, int64_t c, int *tile, int *h, int *b)
{
    const int lane = threadIdx.x & 31;
    const int64_t rep = (Hm == 1) ? H : 1;
    const int64_t n_e = (int64_t)B * Hm * n_tiles;
    // bucket starts: lane l holds buckets l and l + 32, lane 0 also the end
    const int64_t s0 = bstart[lane], s1 = bstart[lane + 32], s_end = bstart[kOrderBuckets];
    if (__any_sync(0xffffffffu, s0 < 0 || s0 > n_e || s1 < 0 || s1 > n_e) || s_end != n_e) return false;
    // last bucket whose first unit is <= c (buckets may be empty: take the last such start)
    const unsigned m0 = __ballot_sync(0xffffffffu, s0 * rep <= c);
    const unsigned m1 = __ballot_sync(0xffffffffu, s1 * rep <= c);
    const int k = m1 ? 32 + 31 - __clz(m1) : 31 - __clz(m0);
    if (k < 0 || c >= n_e * rep) return false;
    const int64_t kb = __shfl_sync(0xffffffffu, k < 32 ? s0 : s1, k & 31);
    const int64_t knext = (k + 1 < kOrderBuckets)
                              ? __shfl_sync(0xffffffffu, (k + 1) < 32 ? s0 : s1, (k + 1) & 31)
                              : s_end;
    const int64_t cnt = knext - kb;
    if (cnt <= 0 || knext > n_e) return false;
    const int64_t local = c - kb * rep;
    const int64_t hr = local / cnt;
    const int32_t v = order[kb + (local - hr * cnt)];
    if (v < 0 || (int64_t)v >= n_e) return false;
    const int s = v / n_tiles;
    *tile = v - s * n_tiles;
    *b = s / Hm;
    *h = (Hm == 1) ? (int)hr : s - *b * Hm;
    return true;
}
#endif

// Arguments of the forward kernel (everything but the TMA descriptors).
struct FwdArgs {
    const int32_t *lts, *lte, *uts, *ute;
    const uint8_t *plan;
    PlanLayout L;
    void *o;
    float *lse;
    int32_t *status;
    int B, H, Hm, N;
    int q_row0, Nq;       // Q, O, lse hold rows [q_row0, q_row0 + Nq) of the mask
    float scale_log2;     // softmax scale * log2(e)
    int o_f32;
    const float *descale; // FP8 path: device [3], the Q, K, V descales (else unused)
    long long wait_limit; // bound of every device-side wait, SM cycles (kWaitLimitCycles)
    int withhold;         // test hook (0 in every product launch): CTA 0 skips its second K load
    int sched_slot;       // work-counter slot of this launch (persistent scheduling)
};

// Arguments of the backward main kernel.
struct BwdArgs {
    const int32_t *lts, *lte, *uts, *ute;
    const uint8_t *plan;
    PlanLayout L;
    const float *lse;     // forward logsumexp, natural log
    const float *Dvec;    // rowsum(dO * O)
    float *dq_acc;        // fp32 dQ accumulator: the caller's dq (fp32 gradients) or the workspace
    float dq_mul;         // factor of the accumulated dQ^T: scale (caller's dq) or 1 (workspace, scaled later)
    void *dk, *dv;
    int32_t *status;
    int B, H, Hm, N;
    int q_row0, Nq;       // Q, dO, lse, D, dQ hold rows [q_row0, q_row0 + Nq); K, V, dK, dV all N
    float scale, scale_log2;
    int g_f32;
    long long wait_limit; // bound of every device-side wait, SM cycles (kWaitLimitCycles)
    int withhold;         // test hook (0 in every product launch): CTA 0 skips its second Q/dO load
    int sched_slot;       // work-counter slot of this launch (persistent scheduling)
};

// Kernel ids for the profiler.
enum KernelId {
    kKClassifyMinmax = FM_K_CLASSIFY_MINMAX,
    kKClassifyLists = FM_K_CLASSIFY_LISTS,
    kKFwd = FM_K_FWD,
    kKBwdPre = FM_K_BWD_PRE,
    kKBwd = FM_K_BWD,
    kKBwdPost = FM_K_BWD_POST,
    kKClassifyOrder = FM_K_CLASSIFY_ORDER,
    kKFp8Amax = FM_K_FP8_AMAX,
    kKFp8Convert = FM_K_FP8_CONVERT,
};

// Devices a process may use (per-device caches of kernel attributes).
constexpr int kMaxDevices = 64;

// Device-side checks of the FM_DEBUG build (a compile definition; the release
// build compiles them out): plan entries within range, the TMEM allocation
// at column 0, and at the end of each CTA every pipeline mbarrier's phase
// parity against the number of tiles, halves and units the CTA processed.  A
// failed check records FM_ERR_DEBUG_CHECK in the caller's status word.
#ifdef FM_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Default limit of every bounded device-side wait, in SM clock cycles
// (about 1.5 s at 1.4-2.1 GHz): far above any legitimate wait inside a CTA.
constexpr long long kWaitLimitCycles = 3000000000LL;

}  // namespace fm

// Host-side helpers implemented in fm_api.cu.
namespace fm {
// Number of SMs of the current device (cached per device; 0 on error): the
// grid of the persistent attention kernels.
int device_sm_count();

// Shape checks shared by every attention entry point: FM_ERR_INVALID_ARG for
// non-positive or overflowing sizes, FM_ERR_UNSUPPORTED for a head dim other
// than 64 / 128 or B, H beyond the launch grid.
fm_status check_shapes(int B, int H, int N, int d);

struct ProfScope {
    // Records a start event on construction and a stop event on destruction
    // when profiling is on.
    ProfScope(int kernel, void *stream);
    ~ProfScope();
    int slot;
    void *stream;
};
}  // namespace fm
