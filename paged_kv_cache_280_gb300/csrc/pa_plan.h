// The decode's work plan, shared by the kernels and the host (pa_decode_build_plan): the
// per-sequence block prefix sums, the CTA ranges over the list of tiles, and the piece walk
// of a range.  The host builds exactly what a launch would compute on the device.
#pragma once

#include <stdint.h>

#include "pa_internal.h"

#if defined(__CUDACC__)
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

// a / b with a 32-bit divide when both fit (the common case): the 64-bit one
// is a long instruction sequence, and the plan runs before any tile is issued
PA_HD int64_t div_nonneg(int64_t a, int64_t b) {
    if (((uint64_t)a >> 32) == 0 && ((uint64_t)b >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// Where the tiles of one CTA start and end, and who holds which partial.
struct Plan {
    const int32_t* pref;   // pref[b] = blocks of sequences < b (per KV head)
    const int32_t* upref;  // same in partitions (fixed mode)
    int32_t B, Hkv, C, PT;
    int32_t A;     // no partitions: a tile weighs kTileUnits units, a segment A more
    static constexpr int K = kTileUnits;
    int64_t T, U;  // total tiles; total partitions, or total weighted units
    // Shares of the CTAs (no partitions): CTA c belongs to dispatch wave c / WV (WV = the SM count,
    // NWV waves) and takes a share kWaveWeight + KS (NWV - 1 - 2 wave) of the units, so with KS > 0
    // the CTAs dispatched first to an SM, which its warp scheduler favours, take more.  KS = 0:
    // equal shares.  WC = the weight of CTAs 0 .. C - 1.
    int32_t WV, NWV, KS;
    int64_t WC;

    // weight of CTAs 0 .. c - 1 (c <= C)
    PA_HD int64_t weight_before(int c) const {
        if (KS == 0) return c;
        const int s = c / WV;
        int64_t w = 0;
        for (int v = 0; v < s; ++v) w += (int64_t)WV * (kWaveWeight + KS * (NWV - 1 - 2 * v));
        return w + (int64_t)(c - s * WV) * (kWaveWeight + KS * (NWV - 1 - 2 * s));
    }
    // largest c in [0, C - 1] with weight_before(c) <= y (y >= 0)
    PA_HD int cta_at_weight(int64_t y) const {
        if (KS == 0) return (int)(y < C - 1 ? y : C - 1);
        int64_t w0 = 0;
        for (int s = 0;; ++s) {
            const int64_t ws = kWaveWeight + KS * (NWV - 1 - 2 * s);
            const int64_t c = (int64_t)s * WV + (y - w0) / ws;
            if (c < (int64_t)(s + 1) * WV || s + 1 >= NWV) return (int)(c < C - 1 ? c : C - 1);
            w0 += (int64_t)WV * ws;
        }
    }
    // the first unit of CTA c's range (no partitions): ceil(W(c) U / W(C))
    PA_HD int64_t start_unit(int c) const { return div_nonneg(weight_before(c) * U + WC - 1, WC); }
    // the CTA whose range holds unit x < U (no partitions): the largest c with start_unit(c) <= x
    PA_HD int cta_of_unit(int64_t x) const { return cta_at_weight(div_nonneg(x * WC, U)); }

    PA_HD int nblocks(int b) const { return pref[b + 1] - pref[b]; }
    PA_HD int64_t seg_start(int b, int h) const {
        return (int64_t)Hkv * pref[b] + (int64_t)h * nblocks(b);
    }
    // largest b in [0, B) with Hkv * pre[b] <= x
    // (Hkv * pre[b] <= Hkv * pre[B] < 2^31: tiles and partitions are counted in 32 bits; x < 2^31)
    PA_HD int find_seq(const int32_t* pre, int64_t x) const {
        const int32_t x32 = (int32_t)x;
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (Hkv * pre[mid] <= x32)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    }
    // *split = the first tile of the segment the returned tile falls strictly inside, else -1;
    // *seq = a sequence at or before the one that holds the returned tile
    PA_HD int64_t tile_of_unit(int64_t u, int64_t* split, int* seq) const {
        *split = -1;
        *seq = 0;
        if (u >= U) return T;
        int b = find_seq(upref, u);
        *seq = b;
        int64_t local = u - (int64_t)Hkv * upref[b];
        int ub = upref[b + 1] - upref[b];
        int h = (int)(local / ub), part = (int)(local % ub);
        if (part > 0) *split = seg_start(b, h);
        return seg_start(b, h) + (int64_t)part * PT;
    }
    // Weighted units (no partitions): tile t of segment (b, h) sits at unit
    //   K t + A (Hkv b + h + 1),
    // i.e. every segment's tiles are preceded by A units of fixed work.
    PA_HD int64_t unit_of_tile(int64_t t) const {
        const int b = find_seq(pref, t);
        const int h = (int)((t - (int64_t)Hkv * pref[b]) / nblocks(b));
        return (int64_t)K * t + (int64_t)A * ((int64_t)Hkv * b + h + 1);
    }
    // the first tile at or after weighted unit x; *split and *seq as in tile_of_unit
    PA_HD int64_t first_tile_at_unit(int64_t x, int64_t* split, int* seq) const {
        *split = -1;
        int lo = 0, hi = B - 1;  // largest b whose units start at or before x
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((int64_t)Hkv * ((int64_t)K * pref[mid] + (int64_t)A * mid) <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo, nb = nblocks(b);
        *seq = b;
        const int64_t local = x - (int64_t)Hkv * ((int64_t)K * pref[b] + (int64_t)A * b);
        const int64_t span = (int64_t)K * nb + A;  // units of one segment of sequence b
        if (span == 0) return (int64_t)Hkv * pref[b];  // A = 0 and b empty: not reached (b is the last with its start)
        const int64_t h = div_nonneg(local, span), r = local - h * span;
        const int64_t j = r <= A ? 0 : (r - A + K - 1) / K;  // at most nb: then the next segment's first tile
        if (j > 0 && j < nb) *split = (int64_t)Hkv * pref[b] + h * nb;
        return (int64_t)Hkv * pref[b] + h * nb + j;
    }
    // the first tile of CTA c's range; *split: the first tile of the segment that tile splits
    // (it then continues the range of CTA c - 1), else -1; *seq: a sequence at or before the one
    // that holds the tile (a start for the piece walk's forward search)
    PA_HD int64_t cta_start(int c, int64_t* split, int* seq) const {
        *split = -1;
        *seq = 0;
        if (PT == 0) return c >= C ? T : first_tile_at_unit(start_unit(c), split, seq);
        return tile_of_unit((int64_t)c * U / C, split, seq);
    }
    // the CTA whose range holds tile t of segment (b, h)
    PA_HD int cta_of_seg(int64_t t, int b, int h) const {
        if (PT == 0) return cta_of_unit((int64_t)K * t + (int64_t)A * ((int64_t)Hkv * b + h + 1));
        return cta_of(t);
    }
    // the CTA whose range holds tile t
    PA_HD int cta_of(int64_t t) const {
        if (PT == 0) return cta_of_unit(unit_of_tile(t));
        int b = find_seq(pref, t);
        int64_t local = t - (int64_t)Hkv * pref[b];
        int nb = nblocks(b), ub = upref[b + 1] - upref[b];
        int h = (int)(local / nb), j = (int)(local % nb);
        int64_t u = (int64_t)Hkv * upref[b] + (int64_t)h * ub + j / PT;
        return (int)(((u + 1) * C - 1) / U);
    }
};

// The pieces of a CTA range [t0, t1).  When the range ends inside a segment that starts inside
// it at tile ta (the first piece of a segment split with the next CTA), the walk takes [ta, t1)
// first and then [t0, ta): a CTA's split pieces then both come early in its range, and so does
// the merge of a segment split between two CTAs, while the grid still streams.  (The partial
// slots follow j0: a piece with j0 > 0 continues its segment, slot 0; a split segment's first
// piece, slot 1.)  ROT = false: no rotation (the walk is [t0, t1) in order).
template <bool ROT>
struct PieceIter {
    // Tile indices fit in 32 bits (the host refuses num_seqs * Hkv * max_blocks_per_seq >= 2^31),
    // so the walk uses 32-bit arithmetic: it runs before any tile is requested.
    int32_t t, t1, t0, ta;  // walking [t, t1); then [t0, ta) while ta > t0
    int b, b0;              // the walk's sequence; a sequence at or before the one holding t0
    // seq0 / seq1: sequences at or before the ones holding t0 / the tile t1 splits
    PA_HD void init(const Plan& P, int64_t t0_, int64_t t1_, int64_t ta_, int seq0, int seq1) {
        t0 = (int32_t)t0_;
        t1 = (int32_t)t1_;
        ta = ROT && ta_ > t0_ && ta_ < t1_ ? (int32_t)ta_ : t0;
        t = ta;
        b0 = seq0;
        b = ta > t0 ? seq1 : seq0;
    }
    PA_HD bool next(const Plan& P, int& b_out, int& h, int& j0, int& j1) {
        if (t >= t1) {
            if (!ROT || ta <= t0) return false;
            t1 = ta;  // the part before the rotated piece
            ta = t = t0;
            b = b0;
        }
        while (P.Hkv * P.pref[b + 1] <= t) ++b;
        const int nb = P.nblocks(b);
        const uint32_t local = (uint32_t)(t - P.Hkv * P.pref[b]);
        h = (int)(local / (uint32_t)nb);
        j0 = (int)(local - (uint32_t)h * (uint32_t)nb);
        const int32_t room = t1 - t;
        j1 = nb - j0 < room ? nb : j0 + room;
        t += j1 - j0;
        b_out = b;
        return true;
    }
    // no piece left after the one next() returned last
    PA_HD bool done() const { return t >= t1 && (!ROT || ta <= t0); }
};

PA_HD int clamp_len(int len, int max_len) { return len < 0 ? 0 : (len > max_len ? max_len : len); }

// The plan of a decode launch of C CTAs over the scanned batch.  Only the first
// min(C, T) CTAs (min(C, U) with partitions) take work.  A split segment's
// pieces then come from consecutive CTAs, which the slot rule and the merge
// rely on: with partitions every working CTA owns at least one; without, a
// range is at least K units wide, so no range falls between two tiles of one
// segment (only in the gap at a segment's start can one be empty).
//
// wave_ctas (the SM count) and wave_skew weigh the CTAs by dispatch wave as Plan describes, over
// num_ctas / wave_ctas waves.  The weights apply only without partitions, and only when the
// lightest range still spans K units (U w_min >= K C w_max); otherwise the shares are equal.
PA_HD Plan plan_from_prefix(const int32_t* pref, const int32_t* upref, int B, int Hkv, int partition_tiles,
                           int seg_units, int num_ctas, int wave_ctas, int wave_skew) {
    Plan P;
    const bool fixed = partition_tiles > 0;
    P.pref = pref;
    P.upref = upref;
    P.B = B;
    P.Hkv = Hkv;
    P.PT = partition_tiles;
    P.A = seg_units;
    P.T = (int64_t)Hkv * pref[B];
    P.U = fixed ? (int64_t)Hkv * upref[B] : (int64_t)P.K * P.T + (int64_t)P.A * Hkv * B;
    const int64_t units = fixed ? P.U : P.T;
    int64_t ce = units < (int64_t)num_ctas ? units : num_ctas;
    if (fixed && ce > 0) {
        // Partitions are coarse: give every working CTA the same number of them
        // (the fewest CTAs with the same largest share), so none is left with
        // one partition more than the rest at the end of the kernel.
        const int64_t per = (units + ce - 1) / ce;
        ce = (units + per - 1) / per;
    }
    P.C = (int32_t)ce;
    P.WV = wave_ctas > 0 ? wave_ctas : 1;
    P.NWV = (num_ctas + P.WV - 1) / P.WV;
    P.KS = 0;
    P.WC = P.C;
    if (!fixed && wave_skew > 0 && P.NWV > 1 && kWaveWeight - wave_skew * (P.NWV - 1) > 0) {
        const int64_t wmin = kWaveWeight - (int64_t)wave_skew * (P.NWV - 1);
        const int64_t wmax = kWaveWeight + (int64_t)wave_skew * (P.NWV - 1);
        if (P.U * wmin >= (int64_t)P.K * P.C * wmax) {
            P.KS = wave_skew;
            P.WC = P.weight_before(P.C);
        }
    }
    return P;
}

// ---- host-built plans (pa_decode_build_plan) ----------------------------------
// A plan buffer is int32 words: a header, then pref[B + 1], upref[B + 1] (zeros without
// partitions) and the clamped lengths[B], then one record per CTA of the launch's grid.  A
// record holds the CTA's range ends, the rotation point, the piece walk's sequence hints and
// the block-table entries of the first 32 tiles of its first piece.
constexpr int32_t kPlanMagic = 0x4c504150;  // "PAPL"
constexpr int kPlanHeaderWords = 16;
constexpr int kPlanRecWords = 40;
constexpr int kPlanChunk = 32;
enum PlanHeaderWord {
    kPlanWMagic = 0,
    kPlanWNumSeqs,
    kPlanWGrid,
    kPlanWKvHeads,
    kPlanWPartitionTiles,
    kPlanWSegUnits,
    kPlanWBlockSize,
    kPlanWMaxLen,
    kPlanWMergeInKernel,
    kPlanWMaxBlocks,
    kPlanWWaveCtas,
    kPlanWWaveSkew,
};
enum PlanRecWord { kRecT0 = 0, kRecT1, kRecTa, kRecSeq0, kRecSeq1, kRecFirst = 8 };
PA_HD int64_t plan_words(int num_seqs, int grid) {
    return kPlanHeaderWords + 3 * (int64_t)num_seqs + 2 + (int64_t)kPlanRecWords * grid;
}
PA_HD int64_t plan_rec_off(int num_seqs, int c) { return kPlanHeaderWords + 3 * (int64_t)num_seqs + 2 + (int64_t)kPlanRecWords * c; }

}  // namespace pa
