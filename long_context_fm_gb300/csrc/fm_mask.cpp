// Host converter: per-row attend intervals -> column-wise masked row ranges.
//
// Row form: blog "FlashMask技术" §2.1 (causal: col_start = 0, col_end = i),
// §3.3 (document packing: (offset, offset + i) inside each document), and the
// multi-interval extension of §6.1 item 1 (several disjoint intervals per row,
// e.g. row 0 -> (0, 100), (200, 300)); the window-with-sink-tokens mask of the
// §5 streaming-inference example is one such two-interval row form.  Column
// form: FlashMask's column-wise sparse encoding (arXiv 2410.01359), two masked
// row ranges per key column.
//
// Method.  Each row's intervals are first normalised into sorted, disjoint,
// non-touching half-open column spans.  For a fixed column j the attend
// indicator a(i) changes value between rows i-1 and i exactly on the columns
// of the symmetric difference of the two rows' attended sets; with sorted
// span lists that difference is read off the merged boundary sequences (a
// boundary present in both lists cancels).  A difference array over columns
// then counts, for every column, how often its indicator flips (O(total
// spans + N)).  A column with R attended runs has R-1 masked gaps between them
// plus a masked head and tail when row 0 / row N-1 is masked; more than two
// masked runs cannot be encoded and is rejected before anything else is done.
// Otherwise every column flips at most six times, so listing the flip rows
// column by column costs O(N) in total, and the runs follow directly.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "fm.h"

namespace {

struct Span {  // half-open column range [a, b)
    int64_t a, b;
};

// Attended spans of every row of one (b, hm): row i owns sp[off[i], off[i+1]),
// sorted by start, pairwise disjoint and not touching (b < next a).
struct RowSpans {
    std::vector<int64_t> off;
    std::vector<Span> sp;
};

// starts / ends: [N, K] inclusive intervals; start > end is an unused slot.
fm_status normalise_rows(const int32_t *starts, const int32_t *ends, int64_t N, int64_t K, RowSpans &rs)
{
    rs.off.assign(N + 1, 0);
    rs.sp.clear();
    rs.sp.reserve(N * std::min<int64_t>(K, 4));
    std::vector<Span> tmp;
    for (int64_t i = 0; i < N; ++i) {
        rs.off[i] = (int64_t)rs.sp.size();
        tmp.clear();
        for (int64_t k = 0; k < K; ++k) {
            const int64_t s = starts[i * K + k], e = ends[i * K + k];
            if (s > e) continue;
            if (s < 0 || e >= N) return FM_ERR_BAD_BOUNDS;
            tmp.push_back(Span{s, e + 1});
        }
        if (tmp.size() > 1)
            std::sort(tmp.begin(), tmp.end(), [](const Span &x, const Span &y) { return x.a < y.a; });
        for (const Span &s : tmp) {
            if ((int64_t)rs.sp.size() > rs.off[i] && s.a <= rs.sp.back().b)
                rs.sp.back().b = std::max(rs.sp.back().b, s.b);     // overlapping or touching
            else
                rs.sp.push_back(s);
        }
    }
    rs.off[N] = (int64_t)rs.sp.size();
    return FM_OK;
}

// Columns whose attend flag differs between rows p and q (either may be -1 or
// N: an empty row), appended to out.  Each normalised list contributes the
// strictly increasing boundaries a0 < b0 < a1 < b1 < ...; a point is inside a
// list's set when an odd number of its boundaries are <= it, so the symmetric
// difference is the odd-count set of the merged sequence, where a boundary
// present in both lists cancels.
void sym_diff(const RowSpans &rs, int64_t N, int64_t p, int64_t q, std::vector<Span> &out)
{
    out.clear();
    auto range = [&](int64_t i, int64_t &lo, int64_t &hi) {
        if (i < 0 || i >= N) { lo = hi = 0; return; }
        lo = 2 * rs.off[i];
        hi = 2 * rs.off[i + 1];
    };
    auto bound = [&](int64_t t) { return (t & 1) ? rs.sp[t >> 1].b : rs.sp[t >> 1].a; };
    int64_t x, xe, y, ye;
    range(p, x, xe);
    range(q, y, ye);
    bool open = false;
    int64_t start = 0;
    auto toggle = [&](int64_t v) {
        if (!open) { start = v; open = true; }
        else { out.push_back(Span{start, v}); open = false; }
    };
    while (x < xe || y < ye) {
        if (y >= ye || (x < xe && bound(x) < bound(y))) toggle(bound(x++));
        else if (x >= xe || bound(y) < bound(x)) toggle(bound(y++));
        else { ++x; ++y; }                                         // equal: cancels
    }
}

fm_status convert_one(const RowSpans &rs, int64_t N, int32_t *lts, int32_t *lte, int32_t *uts, int32_t *ute)
{
    std::vector<Span> d;
    // 1. flips per column by a difference array (rows -1 and N are empty).
    std::vector<int32_t> diff(N + 1, 0);
    for (int64_t i = 0; i <= N; ++i) {
        sym_diff(rs, N, i - 1, i, d);
        for (const Span &s : d) {
            diff[s.a] += 1;
            diff[s.b] -= 1;
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
        sym_diff(rs, N, i - 1, i, d);
        for (const Span &s : d)
            for (int64_t j = s.a; j < s.b; ++j) flip[6 * j + fill[j]++] = (int32_t)i;
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

extern "C" fm_status fm_mask_from_row_intervals(const int32_t *starts, const int32_t *ends, int K, int B, int Hm,
                                                int N, int32_t *lts, int32_t *lte, int32_t *uts, int32_t *ute)
{
    if (!starts || !ends || !lts || !lte || !uts || !ute) return FM_ERR_INVALID_ARG;
    if (K <= 0 || B <= 0 || Hm <= 0 || N <= 0) return FM_ERR_INVALID_ARG;
    if ((int64_t)B * Hm * N * K > ((int64_t)1 << 40)) return FM_ERR_INVALID_ARG;
    RowSpans rs;
    for (int64_t s = 0; s < (int64_t)B * Hm; ++s) {
        const int64_t o = s * N;
        fm_status st = normalise_rows(starts + o * K, ends + o * K, N, K, rs);
        if (st == FM_OK) st = convert_one(rs, N, lts + o, lte + o, uts + o, ute + o);
        if (st != FM_OK) return st;
    }
    return FM_OK;
}

extern "C" fm_status fm_mask_from_rows(const int32_t *cs, const int32_t *ce, int B, int Hm, int N,
                                       int32_t *lts, int32_t *lte, int32_t *uts, int32_t *ute)
{
    return fm_mask_from_row_intervals(cs, ce, 1, B, Hm, N, lts, lte, uts, ute);
}
