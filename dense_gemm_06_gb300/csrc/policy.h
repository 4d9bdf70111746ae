// policy.h -- the host-side choices the library makes automatically, as plain
// C++ (no CUDA), so they can be compiled and checked on a machine without a
// GPU: the FFMA kernel's K-split of the tiles left after its last full round,
// whether a K-major fp32 operand is first transposed, the row panels
// gemm_host() pipelines its copies over, and the tensor-core kernel's tile
// shape and split of its last round.
#pragma once

#include <cstdint>
#include <numeric>

namespace libgemm {

// K-split of the FFMA kernel's tail. Tiles 0 .. dp_tiles-1 (raster order) run
// whole; every later tile is cut into `splits` K-slices of `kt_slice` k-tiles,
// one CTA each, summed in slice order by a fixup kernel.
struct TailSplit {
    int dp_tiles;
    int splits;
    int kt_slice;
};

// Model: an SM finishes the same tile work per unit of time whether it holds
// one CTA or two, so a launch takes (most tile-units on one SM) x (work of a
// unit). With P SMs and T tiles, q = T / P full rounds and r = T mod P tail
// tiles: whole, the tail adds one round; cut into s K-slices (one CTA each),
// it adds ceil(r s / P) / s. split_mode 0 (automatic): with no full round (the
// GPU under-filled) or at least two, the s in 2..8 (slices of at least 32
// k-tiles: shorter ones spend too much of their time filling the pipeline
// and writing partial sums) with the shortest time, if that saves at least
// 10% against no split. With exactly one full round the model fails
// (measured at 2048^3: 4 slices ran 12% slower than whole tiles), so that
// case is not split. split_mode 1: never. split_mode 2 (tests): always cut
// the last wave of `slots` resident CTAs (all tiles if T < slots) into 2-4
// slices. slots <= 0 (occupancy unknown) or sm_count <= 0: never.
inline TailSplit plan_tail_split(int64_t T, int slots, int sm_count, int nkt, int split_mode) {
    TailSplit t{(int)T, 1, nkt};
    if (split_mode == 1 || slots <= 0 || sm_count <= 0 || T <= 0) return t;
    if (split_mode == 2) {
        int64_t r = T % slots;
        if (r == 0) r = T < slots ? T : slots;
        int s = (int)(slots / r);
        s = s < 2 ? 2 : (s > 4 ? 4 : s);
        t.dp_tiles = (int)(T - r);
        t.splits = s;
        t.kt_slice = (nkt + s - 1) / s;
        return t;
    }
    const int64_t P = sm_count, q = T / P, r = T % P;
    if (r == 0 || q == 1) return t;
    const double whole = (double)(q + 1);
    double best = whole;
    int best_s = 1;
    for (int s = 2; s <= 8 && nkt >= 32 * s; ++s) {
        const double time = (double)q + (double)((r * s + P - 1) / P) / s;
        if (time < best - 1e-9) {
            best = time;
            best_s = s;
        }
    }
    if (best_s == 1 || best > 0.9 * whole) return t;
    t.dp_tiles = (int)(T - r);
    t.splits = best_s;
    t.kt_slice = (nkt + best_s - 1) / best_s;
    return t;
}

// Stream-K plan of the TMA-fed FFMA kernel: tiles 0 .. dp_tiles-1 (raster
// order) run whole, one CTA each; the k-iterations of the later tiles (tile
// t, k-tile k is iteration (t - dp_tiles) * nkt + k) are shared evenly by
// sk_ctas CTAs, each taking one contiguous range (at most one tile's worth,
// so at most two tile segments). sk_ctas == 0: no stream-K.
struct StreamK {
    int dp_tiles;
    int sk_ctas;
};

// Model: with P SMs, `slots` = 2 P resident CTAs (two per SM) and
// P <= T < 2 P tiles, whole tiles give some SMs two tiles, so the launch
// takes two tiles' time. Sharing every tile's k-iterations evenly over all
// `slots` CTAs gives every CTA, wherever the block scheduler places it, the
// same T / (2 P) tiles' worth, so every SM does T / P: split_mode 0
// (automatic) uses that when it saves at least 10% (T <= 1.8 P) and a tile
// has at least 32 k-tiles. (Mixing whole-tile CTAs with stream-K CTAs
// measured slower: co-resident CTAs come from neighbouring block indices,
// so two whole tiles could share an SM.) split_mode 3 (tests): stream-K
// whatever it saves, a third of the tiles whole and the rest shared by 3/2
// as many CTAs as tiles. Otherwise no stream-K.
inline StreamK plan_stream_k(int64_t T, int slots, int sm_count, int nkt, int split_mode) {
    StreamK s{(int)T, 0};
    if (T <= 0 || nkt <= 0) return s;
    if (split_mode == 3) {
        const int64_t dp = T / 3, rest = T - dp;
        const int64_t g = rest + (rest + 1) / 2;
        s.dp_tiles = (int)dp;
        s.sk_ctas = (int)(g < rest * nkt ? g : rest * nkt);  // no CTA without iterations
        return s;
    }
    if (split_mode != 0 || sm_count <= 0 || slots < 2 * sm_count || nkt < 32) return s;
    const int64_t P = sm_count;
    if (T < P || T >= 2 * P || 10 * T > 18 * P) return s;
    s.dp_tiles = 0;
    s.sk_ctas = (int)(2 * P);
    return s;
}

// Whether to give the FFMA kernel an MN-major copy of a K-major operand.
// The kernel reads MN-major tiles with 16-byte copies (or TMA) and K-major
// ones with transposing 4-byte copies (about 10% slower at 8192^3); a
// transpose costs two HBM passes over the operand, 48/n of the GEMM time for
// the other dimension n, so it pays when n >= 512 and the product is large
// enough for the extra launch not to matter. mode: 0 automatic, 1 never,
// 2 always.
inline bool want_transpose(int64_t other_dim, int64_t M, int64_t N, int64_t K, int mode) {
    if (mode == 1) return false;
    if (mode == 2) return true;
    return other_dim >= 512 && (double)M * (double)N * (double)K >= 2147483648.0;
}

// gemm_host(): with more than one row panel and an fp32 C, the first panel
// runs as host_k_pieces() GEMMs over consecutive ranges of K, each adding its
// product to C (fused epilogue, beta = 1), so the first one starts once a
// quarter of B (and of that panel's A) is in instead of all of it. A 16-bit C
// would be rounded between the pieces, and K below 4 x 256 would leave pieces
// too short to pay for their launches: those run whole (1 piece).
constexpr int kHostKPieces = 4;
inline int host_k_pieces(int64_t panels, int out_bytes, int64_t K) {
    return panels > 1 && out_bytes == 4 && K >= kHostKPieces * 256 ? kHostKPieces : 1;
}

// First k of piece j of `pieces` (j == pieces: K): K j / pieces rounded up to
// a multiple of 64, so every piece but the last covers whole 64-deep k-tiles.
inline int64_t host_k_bound(int64_t K, int pieces, int j) {
    if (j >= pieces) return K;
    const int64_t b = (K * j / pieces + 63) / 64 * 64;
    return b < K ? b : K;
}

// Rows of the normalised C per gemm_host() panel: a whole number of waves of
// the kernel that computes it (so no panel adds a partial wave), at most
// about 8 panels; M itself when the product is too small (M N K < 1e10) for
// overlapping the copies with compute to pay. f32: the FFMA kernel (128 x
// 128 tiles, `ctas_per_sm` resident CTAs per SM); otherwise the tensor-core
// kernel with CTA group `cta_group` (1: 128 x 256 tiles, one CTA each; 2:
// 256 x 256 tiles per CTA pair) and operand multicast (2: clusters of two
// pairs, 512 x 256).
inline int64_t host_panel_rows(int64_t M, int64_t N, int64_t K, bool f32, int ctas_per_sm,
                               int cta_group, int multicast, int sm_count) {
    if (K == 0 || (double)M * (double)N * (double)K < 1.0e10) return M;
    const bool one_cta = f32 || cta_group == 1;
    const int64_t tm = f32 ? 128 : (cta_group == 1 ? 128 : (multicast == 2 ? 512 : 256));
    const int64_t tn = f32 ? 128 : 256;
    int64_t slots = f32 ? (int64_t)sm_count * ctas_per_sm
                        : (int64_t)sm_count / (one_cta ? 1 : (multicast == 2 ? 4 : 2));
    if (slots < 1) slots = 1;
    const int64_t tiles_m = (M + tm - 1) / tm, tiles_n = (N + tn - 1) / tn;
    int64_t r = slots / std::gcd(slots, tiles_n);
    while (r * 8 < tiles_m) r *= 2;
    return r >= tiles_m ? M : r * tm;
}

// Tensor-core tile shape: the CTA group (1: a CTA per 128-row tile, 2: a
// CTA pair per 256-row tile) and the tile width in columns (64, 128 or 256;
// at least 64 per CTA of the group). cta_group / tile_n: the value asked for,
// or 0 for automatic. Automatic: a problem with fewer 256 x 256 pair tiles
// than a quarter of the SMs (fewer than half the CTA pairs would get one)
// runs one CTA per tile, in the narrowest width that still fits every tile
// into one round over the SMs, so its epilogue (the part of a short problem
// that takes longest) is spread over as many SMs as possible; everything
// else runs 256 x 256 pair tiles. Operand multicast always runs 256 x 256
// pair tiles.
struct TcShape {
    int cta_group;
    int tile_n;
};

inline TcShape plan_tc_shape(int64_t M, int64_t N, int cta_group, int tile_n, bool multicast,
                             int sm_count) {
    TcShape s{cta_group, tile_n};
    if (multicast) return TcShape{2, 256};
    if (s.cta_group != 1 && s.cta_group != 2) {
        const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
        s.cta_group = pair_tiles * 4 < (int64_t)sm_count ? 1 : 2;
    }
    if (s.tile_n != 64 && s.tile_n != 128 && s.tile_n != 256) {
        s.tile_n = 256;
        if (s.cta_group == 1)
            for (int tn = 64; tn < 256; tn *= 2)
                if (((M + 127) / 128) * ((N + tn - 1) / tn) <= (int64_t)sm_count) {
                    s.tile_n = tn;
                    break;
                }
    }
    if (s.tile_n < 64 * s.cta_group) s.tile_n = 64 * s.cta_group;
    return s;
}

// The first tile (raster order) of a tensor-core launch that runs as two
// work units of half the width. With `slots` clusters resident at once and T
// tiles, the last round holds r = T mod slots tiles; when at least two rounds
// are needed and r is at most half the slots, splitting those r tiles makes
// the last round take half as long (2 r half units still fit in one round):
// at 8192^3 (1024 pair tiles on 76 pairs, r = 36) 14 rounds become 13.5.
// split_mode 0: automatic; 1: never; 2 (tests): split the last round's
// tiles (every tile when there is less than one round) whatever it saves.
// Half units need half the width to hold 64 columns per CTA; operand
// multicast never splits. Returns T for no split.
inline int64_t plan_tc_split(int64_t T, int64_t slots, int tile_n, int cta_group,
                             bool multicast, int split_mode) {
    if (split_mode == 1 || multicast || tile_n / 2 < 64 * cta_group || slots <= 0 || T <= 0)
        return T;
    int64_t r = T % slots;
    if (split_mode == 2) {
        if (r == 0) r = T < slots ? T : slots;
        return T - r;
    }
    if (T <= slots || r == 0 || 2 * r > slots) return T;
    return T - r;
}

}  // namespace libgemm
