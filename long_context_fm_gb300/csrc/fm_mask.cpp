// Host converter: per-row inclusive attend intervals -> column-wise masked
// row ranges.
//
// Row form: blog "FlashMask技术" §2.1 (causal: col_start = 0, col_end = i)
// and §3.3 (document packing: (offset, offset + i) inside each document).
// Column form: FlashMask's column-wise sparse encoding (arXiv 2410.01359),
// two masked row ranges per key column.
//
// Method.  For a fixed column j the attend indicator a(i) = [cs_i <= j <= ce_i]
// changes value between rows i-1 and i exactly on the columns of the
// symmetric difference of the two rows' intervals (at most two column
// ranges).  A difference array over columns therefore counts, for every
// column, how often its indicator flips (O(N)).  A column with R attended
// runs has R-1 masked gaps between them plus a masked head and tail when row
// 0 / row N-1 is masked; more than two masked runs cannot be encoded and is
// rejected before anything else is done.  Otherwise every column flips at
// most six times, so listing the flip rows column by column costs O(N) in
// total, and the runs follow directly.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "fm.h"

namespace {

struct Span {  // half-open column range [a, b)
    int64_t a, b;
    bool empty() const { return a >= b; }
};

// Columns whose attend flag differs between two rows with half-open column
// ranges x and y: up to two ranges.
int sym_diff(Span x, Span y, Span out[2])
{
    int n = 0;
    if (x.empty() && y.empty()) return 0;
    if (x.empty()) { out[n++] = y; return n; }
    if (y.empty()) { out[n++] = x; return n; }
    if (x.b <= y.a || y.b <= x.a) {        // disjoint
        out[n++] = x;
        out[n++] = y;
        return n;
    }
    Span lo{std::min(x.a, y.a), std::max(x.a, y.a)};
    Span hi{std::min(x.b, y.b), std::max(x.b, y.b)};
    if (!lo.empty()) out[n++] = lo;
    if (!hi.empty()) out[n++] = hi;
    return n;
}

fm_status convert_one(const int32_t *cs, const int32_t *ce, int64_t N, int32_t *lts, int32_t *lte,
                      int32_t *uts, int32_t *ute)
{
    auto row_span = [&](int64_t i) -> Span {
        if (i < 0 || i >= N) return Span{0, 0};
        if (cs[i] > ce[i]) return Span{0, 0};
        return Span{cs[i], (int64_t)ce[i] + 1};
    };
    for (int64_t i = 0; i < N; ++i)
        if (cs[i] <= ce[i] && (cs[i] < 0 || ce[i] >= N)) return FM_ERR_BAD_BOUNDS;

    // 1. flips per column by a difference array (rows -1 and N are empty).
    std::vector<int32_t> diff(N + 1, 0);
    for (int64_t i = 0; i <= N; ++i) {
        Span d[2];
        const int nd = sym_diff(row_span(i - 1), row_span(i), d);
        for (int t = 0; t < nd; ++t) {
            diff[d[t].a] += 1;
            diff[d[t].b] -= 1;
        }
    }
    std::vector<uint8_t> nflip(N);
    {
        int64_t run = 0;
        for (int64_t j = 0; j < N; ++j) {
            run += diff[j];
            const int64_t flips = run;           // even: 2 * attended runs
            const int64_t R = flips / 2;
            if (R > 3) return FM_ERR_UNREPRESENTABLE;
            nflip[j] = (uint8_t)flips;
        }
    }
    // 2. flip rows per column (each column has at most 6, so O(N) total);
    //    masked-run counting needs a(0) and a(N-1), read off the flip list.
    std::vector<int32_t> flip(6 * N);
    std::vector<uint8_t> fill(N, 0);
    for (int64_t i = 0; i <= N; ++i) {
        Span d[2];
        const int nd = sym_diff(row_span(i - 1), row_span(i), d);
        for (int t = 0; t < nd; ++t)
            for (int64_t j = d[t].a; j < d[t].b; ++j) flip[6 * j + fill[j]++] = (int32_t)i;
    }
    // 3. masked runs = complement of the attended runs [f0,f1), [f2,f3), ...
    for (int64_t j = 0; j < N; ++j) {
        const int nf = nflip[j];
        const int32_t *f = &flip[6 * j];
        Span runs[4];
        int nr = 0;
        int64_t prev = 0;
        for (int t = 0; t + 1 < nf; t += 2) {
            if (f[t] > prev) runs[nr++] = Span{prev, f[t]};
            prev = f[t + 1];
            if (nr > 2) return FM_ERR_UNREPRESENTABLE;
        }
        if (prev < N) runs[nr++] = Span{prev, N};
        if (nr > 2) return FM_ERR_UNREPRESENTABLE;
        int32_t L0 = (int32_t)N, L1 = (int32_t)N, U0 = 0, U1 = 0;
        if (nr == 1) {
            if (runs[0].a == 0) { U0 = 0; U1 = (int32_t)runs[0].b; }
            else { L0 = (int32_t)runs[0].a; L1 = (int32_t)runs[0].b; }
        } else if (nr == 2) {
            U0 = (int32_t)runs[0].a; U1 = (int32_t)runs[0].b;
            L0 = (int32_t)runs[1].a; L1 = (int32_t)runs[1].b;
        }
        lts[j] = L0; lte[j] = L1; uts[j] = U0; ute[j] = U1;
    }
    return FM_OK;
}

}  // namespace

extern "C" fm_status fm_mask_from_rows(const int32_t *cs, const int32_t *ce, int B, int Hm, int N,
                                       int32_t *lts, int32_t *lte, int32_t *uts, int32_t *ute)
{
    if (!cs || !ce || !lts || !lte || !uts || !ute) return FM_ERR_INVALID_ARG;
    if (B <= 0 || Hm <= 0 || N <= 0) return FM_ERR_INVALID_ARG;
    if ((int64_t)B * Hm * N > ((int64_t)1 << 40)) return FM_ERR_INVALID_ARG;
    for (int64_t s = 0; s < (int64_t)B * Hm; ++s) {
        const int64_t o = s * N;
        const fm_status st = convert_one(cs + o, ce + o, N, lts + o, lte + o, uts + o, ute + o);
        if (st != FM_OK) return st;
    }
    return FM_OK;
}
