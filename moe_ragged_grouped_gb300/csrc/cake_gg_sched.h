// cake_gg_sched.h -- ragged tile walk of the persistent grouped-GEMM kernel.
//
// Shared by the kernel (device) and by cake_gg_tile_walk (host) so that the
// host replica used in tests is the same code the GPU runs.
//
// Tiles.  Every pass computes C[m, n] = sum_k A[m, k] B[n, k] on 128 x tile_n
// output tiles.
//  * forward / data gradient: m runs over an expert's rows (ragged), n over
//    the output columns (N resp. K); the reduction (K resp. N) is dense.
//  * weight gradient: m runs over N (or over K when swap_ab), n over the
//    other one; the reduction runs over the expert's rows (ragged).  A long
//    reduction may be split into chunks of `split_chunk` 64-row k-blocks; the
//    number of splits of expert e, S_e, depends only on its row count.
//
// Pairs.  With pair = 2, two CTAs of a cluster take one unit together: rank r
// computes m-tile 2 * m_unit + r (its own 128-row output tile) and both share
// the unit's B operand (n-tile, k-range), each loading half of it for both.
// A rank whose m-tile lies past the output computes masked garbage only.
//
// Order.  Experts are walked in a processing order and, inside an expert, in
// m-tile-major order (n fastest, then split).  The weight gradient walks its
// experts heaviest-first (most k-blocks per split first, ties by index) when
// E <= kSortMaxE, so the longest tiles start first ("unsorted" group orders
// in flashinfer PR #8258's row classes do not change the tail).  CTAs take
// tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...  Which CTA takes a tile
// never changes what the tile computes.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define CAKE_HD __host__ __device__ __forceinline__
#else
#define CAKE_HD inline
#endif

namespace cakegg {

constexpr int kModeFwd = 0;
constexpr int kModeDgrad = 1;
constexpr int kModeWgrad = 2;
// The FP32 router GEMM (BF16x3): the forward pass's walk and epilogue, FP32
// operand tiles split into BF16 high and low parts inside the kernel.
constexpr int kModeRouter = 3;
// the weight gradient with N-split tail pieces compiled in (a kernel of its own,
// so that the other weight-gradient kernels carry none of that code)
constexpr int kModeWgradNT = 4;

constexpr int kTileM = 128;     // MMA rows (TMEM lanes)
constexpr int kTileK = 64;      // reduction elements of one k-chunk (one 128-byte swizzle row)
constexpr int kMaxE = 1024;     // experts supported by the on-chip tables
constexpr int kSortMaxE = 256;  // heaviest-first walk only up to this many experts

struct Geom {
    int32_t mode;
    int32_t E;
    int32_t N;
    int32_t K;
    int64_t M_max;
    int32_t bn;           // tile_n
    int32_t swap;         // weight gradient: m over K
    int32_t kchunk;       // weight gradient: k-blocks per split (0 = none)
    int32_t n_tiles;      // output column tiles
    int32_t m_tiles_w;    // weight gradient: output row tiles
    int32_t nkb;          // forward / data gradient: reduction k-blocks
    int32_t pair;         // CTAs per unit (1, or 2 for a 2-SM pair sharing one MMA)
    int32_t bk;           // reduction elements per pipeline stage (64 * k-chunks per stage)
    int32_t csplit;       // weight gradient: splits of a tile run by one cluster (0 = off)
    int32_t tail;         // weight gradient: the last `tail` units of the walk are split ...
    int32_t tail_s;       // ... into tail_s pieces each (0 = no tail split)
    int32_t sk;           // weight gradient, one expert: stream-K segment length in k-blocks (0 = off)
    int32_t ntail;        // weight gradient: the last `ntail` units of the walk run ...
    int32_t ntq;          // ... as ntq column pieces each, every piece over all of its k-blocks (0 = off)
};

CAKE_HD int32_t ceil_div_i(int32_t a, int32_t b) { return (a + b - 1) / b; }

CAKE_HD Geom make_geom(int32_t mode, int32_t E, int32_t N, int32_t K, int64_t M_max, int32_t bn,
                       int32_t swap, int32_t kchunk, int32_t pair = 1, int32_t bk = kTileK,
                       int32_t csplit = 0, int32_t tail = 0, int32_t tail_s = 0, int32_t sk = 0,
                       int32_t ntail = 0, int32_t ntq = 0)
{
    Geom g;
    g.ntail = mode == kModeWgrad && ntq > 1 ? ntail : 0;
    g.ntq = mode == kModeWgrad && ntq > 1 ? ntq : 0;
    g.sk = mode == kModeWgrad ? sk : 0;
    g.tail = tail_s > 1 ? tail : 0;
    g.tail_s = tail_s > 1 ? tail_s : 0;
    g.pair = pair;
    g.bk = bk;
    g.csplit = csplit;
    g.mode = mode;
    g.E = E;
    g.N = N;
    g.K = K;
    g.M_max = M_max;
    g.bn = bn;
    g.swap = swap;
    g.kchunk = kchunk;
    if (mode == kModeFwd) {
        g.n_tiles = ceil_div_i(N, bn);
        g.nkb = ceil_div_i(K, bk);
        g.m_tiles_w = 0;
    } else if (mode == kModeDgrad) {
        g.n_tiles = ceil_div_i(K, bn);
        g.nkb = ceil_div_i(N, bk);
        g.m_tiles_w = 0;
    } else {
        const int32_t mdim = swap ? K : N;
        const int32_t ndim = swap ? N : K;
        g.m_tiles_w = ceil_div_i(mdim, kTileM);
        g.n_tiles = ceil_div_i(ndim, bn);
        g.nkb = 0;
    }
    return g;
}

// Splits of an expert with `rows` rows (weight gradient); 1 when unsplit or empty.
// With cluster splits every tile has csplit splits, one per CTA of a cluster,
// walked as a single unit.
CAKE_HD int32_t expert_splits(const Geom &g, int32_t rows)
{
    if (g.mode == kModeWgrad && g.csplit > 0) return g.csplit;
    if (g.mode != kModeWgrad || g.kchunk <= 0) return 1;
    const int32_t nkb = ceil_div_i(rows, g.bk);
    return nkb <= 0 ? 1 : ceil_div_i(nkb, g.kchunk);
}

// Output row tiles of the weight gradient taken per unit (pairs share a unit).
CAKE_HD int32_t m_units_w(const Geom &g) { return ceil_div_i(g.m_tiles_w, g.pair); }

// Units of one expert (a unit is one tile, or one tile per CTA of a pair).
CAKE_HD int32_t expert_tiles(const Geom &g, int32_t rows)
{
    if (g.mode == kModeWgrad) return m_units_w(g) * g.n_tiles * (g.csplit > 0 ? 1 : expert_splits(g, rows));
    return ceil_div_i(rows, kTileM * g.pair) * g.n_tiles;
}

// Sort key of the heaviest-first walk: k-blocks in one split of the expert.
CAKE_HD int32_t expert_cost(const Geom &g, int32_t rows)
{
    const int32_t nkb = ceil_div_i(rows, g.bk);
    const int32_t s = expert_splits(g, rows);
    return ceil_div_i(nkb, s);
}

CAKE_HD bool walk_is_sorted(const Geom &g) { return g.mode == kModeWgrad && g.E <= kSortMaxE; }

// ---- stream-K walk (weight gradient of one expert) ----
//
// The work is n_tiles x KB k-blocks per m-unit (KB = the expert's k-blocks).
// It is cut into segments of sk consecutive k-blocks in (n-tile, k-block)
// order; segment j is processed by m_units virtual pairs at once, one per
// m-unit (v = j * m_units + mu), so the m-units of an n-tile read the same
// rows of the wide operand at the same time.  A segment covers the end of
// one n-tile and the start of the next (or more): each such piece is its own
// unit, and a tile's pieces are summed in k order through partial slots.  A
// unit id is v * pmax + piece.  The walk depends on the plan and the offsets
// only, never on which pair runs a virtual pair.

// k-blocks of the expert (at least 1, so an empty expert still writes its zero tiles)
CAKE_HD int32_t sk_kb(const Geom &g, int32_t rows)
{
    const int32_t kb = ceil_div_i(rows, g.bk);
    return kb > 0 ? kb : 1;
}

// Largest number of pieces of one segment.
CAKE_HD int32_t sk_pmax(const Geom &g, int32_t KB) { return ceil_div_i(g.sk, KB) + 1; }

// Segments (each run by m_units virtual pairs).
CAKE_HD int32_t sk_segments(const Geom &g, int32_t KB) { return ceil_div_i(g.n_tiles * KB, g.sk); }

// Virtual pairs of the walk.
CAKE_HD int32_t sk_virtual(const Geom &g, int32_t KB)
{
    return ceil_div_i(g.m_tiles_w, g.pair) * sk_segments(g, KB);
}

// Pieces of virtual pair v's segment.
CAKE_HD int32_t sk_pieces(const Geom &g, int32_t KB, int32_t v)
{
    const int32_t j = v / ceil_div_i(g.m_tiles_w, g.pair);
    const int32_t a = j * g.sk;
    const int32_t w = g.n_tiles * KB;
    const int32_t b = a + g.sk < w ? a + g.sk : w;
    return (b - 1) / KB - a / KB + 1;
}

// Partial slots reserved per output tile: the most pieces a tile of at most
// KB_max k-blocks can have.
CAKE_HD int32_t sk_slots_per_tile(int32_t KB_max, int32_t sk) { return (KB_max > 0 ? KB_max - 1 : 0) / sk + 2; }

// One unit of work.
struct Tile {
    int32_t e;        // expert
    int32_t mt;       // output row tile
    int32_t nt;       // output column tile
    int32_t s;        // split index
    int32_t S;        // splits of this output tile
    int32_t kb0;      // first k-block (g.bk reduction elements each)
    int32_t kb1;      // one past the last k-block
    int32_t row0;     // fwd/dgrad: first row of the tile; wgrad: first row of the expert
    int32_t row_end;  // one past the expert's last row
    int32_t ticket;   // wgrad: output tile index e * (m_tiles_w * n_tiles) + mt * n_tiles + nt
    int64_t slot;     // wgrad split: partial slot of this split
    int32_t c0;       // wgrad N-split tail piece: first column of the piece within the tile (else 0)
    int32_t cw;       // columns of the tile this unit computes (tile_n, or the piece's width)
    bool valid;       // false for a pair rank whose tile lies past the output
    bool tail;        // a piece of a split tail unit (partials in slots, also when non-deterministic)
};

// Slack placement of the split tail (flashinfer PR #8258, opening summary,
// 2nd paragraph: while the full-wave tiles run, the clusters are ranked by
// load; if the less-loaded ones have room -- each stays within the largest
// load plus one tail share -- every tail tile goes whole to one of them, with
// no tail sums; otherwise the split tail runs).  Here the loads are projected
// from the offsets, not measured: the walk's units are taken in walk order by
// the first of P pairs to become free (what the unit counter does on equal-
// speed pairs), a unit lasting its k-blocks, up to the last g.tail units.
// Then each tail unit in turn goes to a least-loaded pair, which must stay
// within the largest load plus one tail share (the unit's k-blocks /
// g.tail_s) plus what splitting itself costs (split_overhead_kblocks: the
// pages' test alone split the tail on ragged "random" workloads where the
// decision protocol measured the split slower).  True: the tail units run
// whole.  A function of the offsets and
// the fixed wave P alone, so every CTA (and the host walk) decides alike and
// deterministic results do not depend on max_sms.  Loads are kept as at most
// kSlackClasses (load, pairs) classes; more distinct loads -> the split tail.
constexpr int kSlackClasses = 48;
constexpr int kWaveCtas = 152;      // GB300 SMs: the fixed wave plans and projections assume
constexpr int kSlackMaxE = 64;      // projection only up to this many experts (else the 80 % rule below)

// The cheaper rule used above kSlackMaxE experts: the tail stays split when the
// walk's last units are about as long as its first (the lightest expert costs
// at least 80 % of the heaviest).
CAKE_HD bool tail_active(const Geom &g, const int32_t *off, const int32_t *order)
{
    if (g.mode != kModeWgrad || g.tail <= 0) return false;
    const int32_t e_hi = order[0], e_lo = order[g.E - 1];
    const int64_t c_hi = expert_cost(g, off[e_hi + 1] - off[e_hi]);
    const int64_t c_lo = expert_cost(g, off[e_lo + 1] - off[e_lo]);
    return 5 * c_lo >= 4 * c_hi;
}

CAKE_HD void slack_add(int64_t *val, int32_t *cnt, int &nc, int64_t v, int32_t k)
{
    int i = 0;
    while (i < nc && val[i] < v) ++i;
    if (i < nc && val[i] == v) {
        cnt[i] += k;
        return;
    }
    for (int j = nc; j > i; --j) {
        val[j] = val[j - 1];
        cnt[j] = cnt[j - 1];
    }
    val[i] = v;
    cnt[i] = k;
    ++nc;
}

// What splitting a unit costs on top of its pieces, in k-blocks: the FP32
// partial tile's write and read (x2 margin) and the finish -- the cost the
// planner's split model charges (rounded up).
CAKE_HD int64_t split_overhead_kblocks(int32_t bn, int32_t bk)
{
    const int64_t num = int64_t(4096) * bn * 64;
    const int64_t den = (int64_t(16384) + int64_t(128) * bn) * bk;
    return (num + den - 1) / den + (4 * 64 + bk - 1) / bk;
}

CAKE_HD bool tail_fits_whole(const Geom &g, const int32_t *off, const int32_t *order, int32_t P)
{
    if (g.mode != kModeWgrad || g.tail <= 0 || g.tail_s <= 1) return true;
    if (g.E > kSlackMaxE) return !tail_active(g, off, order);
    int64_t val[kSlackClasses + 1];
    int32_t cnt[kSlackClasses + 1];
    int nc = 1;
    val[0] = 0;
    cnt[0] = P;
    int64_t units = 0;
    for (int i = 0; i < g.E; ++i) units += expert_tiles(g, off[order[i] + 1] - off[order[i]]);
    int64_t before = units - g.tail;   // units of the walk ahead of the tail
    for (int i = 0; i < g.E; ++i) {
        const int32_t rows = off[order[i] + 1] - off[order[i]];
        const int64_t c = ceil_div_i(rows, g.bk);   // k-blocks of a whole unit of this expert
        int64_t n = expert_tiles(g, rows);
        while (n > 0) {
            if (before > 0) {
                // the next units of the walk go to the least-loaded pairs
                int64_t k = n < cnt[0] ? n : cnt[0];
                if (k > before) k = before;
                const int64_t v = val[0] + c;
                cnt[0] -= int32_t(k);
                if (cnt[0] == 0) {
                    for (int j = 0; j + 1 < nc; ++j) {
                        val[j] = val[j + 1];
                        cnt[j] = cnt[j + 1];
                    }
                    --nc;
                }
                slack_add(val, cnt, nc, v, int32_t(k));
                if (nc > kSlackClasses) return false;
                n -= k;
                before -= k;
            } else {
                // a tail unit, whole, on a least-loaded pair: within the largest
                // load plus one tail share -- the share a piece would take, with
                // what splitting costs on top of the pieces?
                const int64_t vmax = val[nc - 1];
                const int64_t ovh = split_overhead_kblocks(g.bn, g.bk);
                if ((val[0] + c - vmax - ovh) * g.tail_s > c) return false;
                const int64_t v = val[0] + c;
                if (--cnt[0] == 0) {
                    for (int j = 0; j + 1 < nc; ++j) {
                        val[j] = val[j + 1];
                        cnt[j] = cnt[j + 1];
                    }
                    --nc;
                }
                slack_add(val, cnt, nc, v, 1);
                if (nc > kSlackClasses) return false;
                --n;
            }
        }
    }
    return true;
}

// Positions in the walk: the weight gradient's last g.tail units each take
// g.tail_s positions (one per piece).
CAKE_HD int64_t walk_length(const Geom &g, int64_t units)
{
    return units + int64_t(g.tail) * (g.tail_s > 1 ? g.tail_s - 1 : 0) +
           int64_t(g.ntail) * (g.ntq > 1 ? g.ntq - 1 : 0);
}

// Tables: off[E+1] offsets; order[E] processing position -> expert;
// pref[E+1] tile prefix in processing order; spref[E+1] split prefix by
// expert id (weight gradient).
CAKE_HD Tile decode_tile(const Geom &g, int64_t t, const int32_t *off, const int32_t *order,
                         const int32_t *pref, const int32_t *spref, int32_t rank = 0)
{
    // a piece of a split tail unit: position -> (unit, piece)
    int32_t tail_piece = -1;
    int64_t tail_unit = 0;
    if (g.mode == kModeWgrad && g.tail > 0) {
        const int64_t main_units = int64_t(pref[g.E]) - g.tail;
        if (t >= main_units) {
            const int64_t j = t - main_units;
            tail_unit = j / g.tail_s;
            tail_piece = int32_t(j - tail_unit * g.tail_s);
            t = main_units + tail_unit;
        }
    }
    // a column piece of an N-split tail unit: position -> (unit, piece)
    int32_t npiece = -1;
    if (g.mode == kModeWgrad && g.ntail > 0) {
        const int64_t main_units = int64_t(pref[g.E]) - g.ntail;
        if (t >= main_units) {
            const int64_t j = t - main_units;
            const int64_t u = j / g.ntq;
            npiece = int32_t(j - u * g.ntq);
            t = main_units + u;
        }
    }
    // last position p with pref[p] <= t (positions of empty experts have
    // pref[p] == pref[p+1] and are never selected since t < pref[E])
    int32_t lo = 0, hi = g.E - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (static_cast<int64_t>(pref[mid]) <= t) lo = mid; else hi = mid - 1;
    }
    Tile ti;
    ti.tail = false;
    ti.c0 = 0;
    ti.cw = g.bn;
    const int32_t e = order[lo];
    const int32_t local = static_cast<int32_t>(t - pref[lo]);
    const int32_t r0 = off[e];
    const int32_t r1 = off[e + 1];
    ti.e = e;
    ti.row_end = r1;
    if (g.mode == kModeWgrad && g.csplit > 0) {
        // one unit per output tile (per pair tile); cluster rank r is split
        // s = r / pair, which takes the s-th of csplit contiguous k-block chunks
        // (possibly empty for a short expert), and half r % pair of a pair
        const int32_t S = g.csplit;
        const int32_t s = rank / g.pair;
        const int32_t nkb_e = ceil_div_i(r1 - r0, g.bk);
        const int32_t chunk = ceil_div_i(nkb_e, S);
        ti.nt = local % g.n_tiles;
        ti.mt = (local / g.n_tiles) * g.pair + (rank - s * g.pair);
        ti.s = s;
        ti.S = S;
        ti.kb0 = s * chunk < nkb_e ? s * chunk : nkb_e;
        ti.kb1 = (s + 1) * chunk < nkb_e ? (s + 1) * chunk : nkb_e;
        ti.row0 = r0;
        ti.ticket = (e * g.m_tiles_w + ti.mt) * g.n_tiles + ti.nt;
        ti.slot = 0;
        ti.valid = ti.mt < g.m_tiles_w;
    } else if (g.mode == kModeWgrad && g.sk > 0) {
        // stream-K piece: unit id = v * pmax + piece (see sk_kb)
        const int32_t KB = sk_kb(g, r1 - r0);
        const int32_t pmax = sk_pmax(g, KB);
        const int32_t mu_n = ceil_div_i(g.m_tiles_w, g.pair);
        const int32_t v = int32_t(t / pmax);
        const int32_t pc = int32_t(t - int64_t(v) * pmax);
        const int32_t mu = v % mu_n;
        const int32_t j = v / mu_n;
        const int32_t a = j * g.sk;
        const int32_t w = g.n_tiles * KB;
        const int32_t b = a + g.sk < w ? a + g.sk : w;
        const int32_t nt = a / KB + pc;
        const int32_t base = nt * KB;
        ti.nt = nt;
        ti.mt = mu * g.pair + rank;
        ti.kb0 = (a > base ? a : base) - base;
        ti.kb1 = (b < base + KB ? b : base + KB) - base;
        // cuts (multiples of sk) inside the tile before this piece, and in all of it
        ti.s = (base + ti.kb0) / g.sk - base / g.sk;
        ti.S = ceil_div_i(base + KB, g.sk) - base / g.sk;
        ti.row0 = r0;
        ti.ticket = (e * g.m_tiles_w + ti.mt) * g.n_tiles + ti.nt;
        const int32_t spt = sk_slots_per_tile(int32_t((g.M_max + g.bk - 1) / g.bk), g.sk);
        ti.slot = int64_t(ti.ticket) * spt + ti.s;
        ti.valid = ti.mt < g.m_tiles_w;
        ti.tail = true;   // partials in slots, summed in piece order in both modes
    } else if (g.mode == kModeWgrad) {
        const int32_t S = expert_splits(g, r1 - r0);
        const int32_t nkb_e = ceil_div_i(r1 - r0, g.bk);
        const int32_t s = local % S;
        const int32_t rest = local / S;
        // m-units fastest: the units of a wave share the wide operand's columns
        // (fewer L2 misses than walking the n-tiles first)
        ti.nt = rest / m_units_w(g);
        ti.mt = (rest % m_units_w(g)) * g.pair + rank;
        ti.s = s;
        ti.S = S;
        const int32_t chunk = S > 1 ? g.kchunk : nkb_e;
        ti.kb0 = s * chunk;
        ti.kb1 = (s + 1) * chunk < nkb_e ? (s + 1) * chunk : nkb_e;
        ti.row0 = r0;
        ti.ticket = (e * g.m_tiles_w + ti.mt) * g.n_tiles + ti.nt;
        ti.slot = (static_cast<int64_t>(spref[e]) * g.m_tiles_w * g.n_tiles) +
                  static_cast<int64_t>(ti.mt * g.n_tiles + ti.nt) * S + s;
        ti.valid = ti.mt < g.m_tiles_w;
        if (tail_piece >= 0) {
            // piece `tail_piece` of the expert's k-blocks, split into g.tail_s
            // contiguous chunks; slots per (tail unit, pair rank, piece)
            const int32_t ch = ceil_div_i(nkb_e, g.tail_s);
            ti.s = tail_piece;
            ti.S = g.tail_s;
            ti.kb0 = tail_piece * ch < nkb_e ? tail_piece * ch : nkb_e;
            ti.kb1 = (tail_piece + 1) * ch < nkb_e ? (tail_piece + 1) * ch : nkb_e;
            ti.slot = (tail_unit * g.pair + rank) * g.tail_s + tail_piece;
            ti.tail = true;
        }
        if (npiece >= 0) {
            // the same k-blocks over a narrower column range: each output element's
            // reduction order is unchanged (one rounding, the bits of the whole unit)
            ti.cw = g.bn / g.ntq;
            ti.c0 = npiece * ti.cw;
        }
    } else {
        ti.mt = (local / g.n_tiles) * g.pair + rank;
        ti.nt = local % g.n_tiles;
        ti.s = 0;
        ti.S = 1;
        ti.kb0 = 0;
        ti.kb1 = g.nkb;
        ti.row0 = r0 + ti.mt * kTileM;
        ti.ticket = 0;
        ti.slot = 0;
        ti.valid = ti.row0 < r1;
    }
    return ti;
}

}  // namespace cakegg
