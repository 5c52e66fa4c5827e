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
// per-KV-tile lists (CSC).  Every section starts on a 256-byte boundary.
struct PlanLayout {
    int32_t B, Hm, N, bq, bk, n_q, n_k;
    int64_t off_minmax;    // int32 [B*Hm][n_k][8]
    int64_t off_labels;    // uint8 [B*Hm][n_q][n_k]
    int64_t off_row_cnt;   // int32 [B*Hm][n_q]
    int64_t off_row_list;  // int32 [B*Hm][n_q][n_k]  kv tile | label << 28
    int64_t off_col_cnt;   // int32 [B*Hm][n_k]
    int64_t off_col_list;  // int32 [B*Hm][n_k][n_q]  q tile | label << 28
    int64_t total;
};

struct PlanHeader {        // first 64 bytes of a plan, written by the classifier
    uint32_t magic;
    int32_t B, Hm, N, bq, bk, n_q, n_k;
    int64_t total;
    int32_t pad[6];
};
static_assert(sizeof(PlanHeader) == 64, "plan header size");

FM_HD int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

FM_HD bool plan_layout(int B, int Hm, int N, int bq, int bk, PlanLayout *L)
{
    if (B <= 0 || Hm <= 0 || N <= 0) return false;
    if (!((bq == 64 || bq == 128) && (bk == 64 || bk == 128))) return false;
    const int64_t n_q = (N + bq - 1) / bq, n_k = (N + bk - 1) / bk;
    if (n_q >= kTileMask || n_k >= kTileMask) return false;
    const int64_t S = (int64_t)B * Hm;
    L->B = B; L->Hm = Hm; L->N = N; L->bq = bq; L->bk = bk;
    L->n_q = (int32_t)n_q; L->n_k = (int32_t)n_k;
    int64_t off = 256;
    L->off_minmax = off;   off = align256(off + S * n_k * 8 * 4);
    L->off_labels = off;   off = align256(off + S * n_q * n_k);
    L->off_row_cnt = off;  off = align256(off + S * n_q * 4);
    L->off_row_list = off; off = align256(off + S * n_q * n_k * 4);
    L->off_col_cnt = off;  off = align256(off + S * n_k * 4);
    L->off_col_list = off; off = align256(off + S * n_k * n_q * 4);
    L->total = off;
    return true;
}

// Arguments of the forward kernel (everything but the TMA descriptors).
struct FwdArgs {
    const int32_t *lts, *lte, *uts, *ute;
    const uint8_t *plan;
    PlanLayout L;
    void *o;
    float *lse;
    int32_t *status;
    int B, H, Hm, N;
    float scale_log2;     // softmax scale * log2(e)
    int o_f32;
};

// Arguments of the backward main kernel.
struct BwdArgs {
    const int32_t *lts, *lte, *uts, *ute;
    const uint8_t *plan;
    PlanLayout L;
    const float *lse;     // forward logsumexp, natural log
    const float *Dvec;    // rowsum(dO * O)
    float *dq_acc;        // fp32 dQ accumulator (unscaled)
    void *dk, *dv;
    int32_t *status;
    int B, H, Hm, N;
    float scale, scale_log2;
    int g_f32;
};

// Kernel ids for the profiler.
enum KernelId {
    kKClassifyMinmax = FM_K_CLASSIFY_MINMAX,
    kKClassifyLists = FM_K_CLASSIFY_LISTS,
    kKFwd = FM_K_FWD,
    kKBwdPre = FM_K_BWD_PRE,
    kKBwd = FM_K_BWD,
    kKBwdPost = FM_K_BWD_POST,
};

// Default limit of every bounded device-side wait, in SM clock cycles
// (about 1.5 s at 1.4-2.1 GHz): far above any legitimate wait inside a CTA.
constexpr long long kWaitLimitCycles = 3000000000LL;

}  // namespace fm

// Host-side helpers implemented in fm_api.cu.
namespace fm {
struct ProfScope {
    // Records a start event on construction and a stop event on destruction
    // when profiling is on.
    ProfScope(int kernel, void *stream);
    ~ProfScope();
    int slot;
    void *stream;
};
}  // namespace fm
