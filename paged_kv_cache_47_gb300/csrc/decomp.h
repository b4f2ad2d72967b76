// Work decomposition of one split-K decode launch.
//
// A *unit* is one (sequence s, kv head g, query-head chunk c): the q heads of
// kv head g are cut into chunks of at most `gc_max` heads, so a unit carries a
// fixed number of q heads whatever the grouping. Units of one sequence all
// have the sequence's context length L_s and are cut into tiles of
// PKV_TILE_TOKENS tokens (the last one ragged): n_s = ceil(L_s / TILE).
//
// Tiles are laid out flat, sequence-major, then unit within the sequence,
// then tile within the unit:
//     seq_prefix[s] = U * sum_{s' < s} n_{s'},   NT = seq_prefix[S]
// where U = units per sequence. Unit (s, u) starts at tile
//     T = seq_prefix[s] + u * n_s.
//
// CTA c of C processes the contiguous tile range [split(c), split(c+1)) with
// split(c) = floor(c * NT / C) ("stream-K"): every CTA gets the same number of
// tiles to within one, whatever the spread of context lengths, so no CTA waits
// on a long sequence. A unit cut by a CTA boundary yields one partial result
// per CTA that touches it; the CTA that writes the last of them (found with
// an arrival counter per unit) merges them by log-sum-exp. A unit entirely
// inside one CTA range is finished by that CTA directly.
//
// Partial slots: each CTA owns two partial slots. Its first segment (which
// may continue a unit from the previous CTA) uses slot 0; its last segment,
// when it is a different unit than the first and runs past the range end,
// uses slot 1. For unit starting at tile T handled by CTA c:
//     slot(c, T) = (T > split(c)) ? 1 : 0.
//
// This header is plain C++ usable on the host and the device (the host-side
// checker compiles it with a C++ compiler and no CUDA).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__ __forceinline__
#else
#define PKV_HD inline
#endif

#define PKV_TILE_TOKENS 64

PKV_HD int64_t pkv_split(int c, int C, int64_t NT) { return ((int64_t)c * NT) / C; }

// The CTA owning tile tau: the largest c with split(c) <= tau.
PKV_HD int pkv_owner(int64_t tau, int C, int64_t NT) {
    return (int)(((tau + 1) * (int64_t)C - 1) / NT);
}

// True when CTA c has no tiles (more CTAs than tiles): it writes no partial.
PKV_HD bool pkv_cta_empty(int c, int C, int64_t NT) {
    return pkv_split(c, C, NT) == pkv_split(c + 1, C, NT);
}

// Tiles of a unit of L tokens; tt is the tile size (PKV_TILE_TOKENS unless a
// kernel variant uses larger tiles).
PKV_HD int pkv_tiles_of_len(int L, int tt = PKV_TILE_TOKENS) { return (L + tt - 1) / tt; }

PKV_HD int pkv_partial_slot(int c, int C, int64_t NT, int64_t unit_start) {
    return unit_start > pkv_split(c, C, NT) ? 1 : 0;
}

// Number of partials of the unit of n tiles starting at tile T (the CTAs
// whose range meets [T, T + n)). With NT >= C every CTA has at least one tile,
// so they are all CTAs from owner(T) to owner(T + n - 1); with NT < C every
// CTA has at most one tile, so there is one CTA per tile.
PKV_HD int pkv_unit_parts(int64_t T, int n, int C, int64_t NT) {
    if (NT < C) return n;
    return pkv_owner(T + n - 1, C, NT) - pkv_owner(T, C, NT) + 1;
}

// Clamp a device-provided context length to [0, max_len]; sets *bad on clamp.
PKV_HD int pkv_clamp_len(int L, int max_len, int *bad) {
    if (L < 0) { *bad = 1; return 0; }
    if (L > max_len) { *bad = 1; return max_len; }
    return L;
}

// Sequence holding tile tau: the largest s with seq_prefix[s] <= tau
// (sequences with no tiles are skipped because their prefix equals the next).
PKV_HD int pkv_find_seq(const int *seq_prefix, int S, int64_t tau) {
    int lo = 0, hi = S;  // invariant: seq_prefix[lo] <= tau < seq_prefix[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((int64_t)seq_prefix[mid] <= tau) lo = mid; else hi = mid;
    }
    return lo;
}

// Position of tile tau in the flattened tile space: sequence s (context L,
// n tiles per unit), unit u of the sequence, tile ti of the unit.
struct PkvCursor {
    int s, u, ti, n, L;
};

PKV_HD void pkv_cursor_at(PkvCursor &c, int64_t tau, const int *seq_prefix, const int *seq_len,
                          int S, int tt = PKV_TILE_TOKENS) {
    c.s = pkv_find_seq(seq_prefix, S, tau);
    c.L = seq_len[c.s];
    c.n = pkv_tiles_of_len(c.L, tt);
    const int off = (int)(tau - seq_prefix[c.s]);
    c.u = off / c.n;
    c.ti = off - c.u * c.n;
}

// The next tile in flat order, skipping sequences with no tiles. Past the
// last tile c.s becomes S and the other fields are left as they were.
PKV_HD void pkv_cursor_next(PkvCursor &c, const int *seq_len, int S, int U,
                            int tt = PKV_TILE_TOKENS) {
    if (++c.ti < c.n) return;
    c.ti = 0;
    if (++c.u < U) return;
    c.u = 0;
    do {
        ++c.s;
    } while (c.s < S && seq_len[c.s] == 0);
    if (c.s < S) {
        c.L = seq_len[c.s];
        c.n = pkv_tiles_of_len(c.L, tt);
    }
}
