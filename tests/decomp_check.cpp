// Host-side check of the split-K work decomposition (csrc/decomp.h).
//
// For random batches it replays what the split-K kernel's producer decides
// for every CTA (segments, whole-unit writes, partial slots) and how the
// partials of a cut unit are merged: each CTA holding one counts itself in
// the counter of the unit's first owner, CTAs finishing in a random order,
// and the one that brings the count to pkv_unit_parts merges. It checks that
//   * every tile belongs to exactly one CTA and pkv_owner inverts pkv_split,
//   * each CTA writes at most one partial per slot,
//   * the producer's cursor (pkv_cursor_at / pkv_cursor_next) names the
//     right sequence, unit and tile at every step of a CTA's walk, for
//     64-token and 128-token tiles,
//   * no two cut units share a counter, pkv_unit_parts equals the number of
//     CTAs that touch the unit, and every counter ends back at zero,
//   * every unit is finished exactly once: either whole by one CTA, or merged
//     once from exactly the partials written for it, which together cover
//     all its tiles.
// Prints "OK" and exits 0 on success.
#include <cstdio>
#include <algorithm>
#include <cstdlib>
#include <random>
#include <vector>

#include "decomp.h"

static int fails = 0;
#define CHECK(c, ...)                                 \
    do {                                              \
        if (!(c)) {                                   \
            if (fails++ < 10) {                       \
                std::printf("FAIL %s:%d ", __FILE__, __LINE__); \
                std::printf(__VA_ARGS__);             \
                std::printf("\n");                    \
            }                                         \
        }                                             \
    } while (0)

int main() {
    std::mt19937_64 rng(12345);
    for (int trial = 0; trial < 3000 && fails == 0; ++trial) {
        const int S = 1 + rng() % 40;
        const int U = 1 + rng() % 6;
        int C = 1 + rng() % 200;
        const int tt = (trial & 1) ? 128 : 64;
        std::vector<int> len(S), n(S), prefix(S + 1, 0);
        for (int s = 0; s < S; ++s) {
            const int kind = rng() % 6;
            len[s] = kind == 0 ? 0 : (kind == 1 ? 1 + rng() % 64 : 1 + rng() % 3000);
            n[s] = pkv_tiles_of_len(len[s], tt);
            CHECK(len[s] <= (int64_t)n[s] * tt && (n[s] == 0 || len[s] > (int64_t)(n[s] - 1) * tt),
                  "tiles of length %d", len[s]);
            prefix[s + 1] = prefix[s] + n[s] * U;
        }
        const int64_t NT = prefix[S];
        if (NT == 0) continue;
        if (trial % 4 == 3) {
            // C near NT: uneven shares, empty CTAs, the switch to the weighted split
            C = (int)std::max<int64_t>(1, std::min<int64_t>(4096, NT / 2 + (int64_t)(rng() % (NT + 1))));
        }
        const int units = S * U;
        std::vector<int> whole(units, 0), merged(units, 0), covered(units, 0);
        std::vector<int> slot_unit(2 * C, -1), slot_tiles(2 * C, 0);
        // cut segments each CTA reports at its end: (unit, unit start tile)
        std::vector<std::vector<std::pair<int, int64_t>>> arrivals(C);
        std::vector<int> counter(C, 0), counter_unit(C, -1), touching(units, 0);

        // with NT >= C every CTA holds a tile (pkv_unit_parts counts on it)
        if (NT >= C)
            for (int c = 0; c < C; ++c)
                CHECK(!pkv_cta_empty(c, C, NT), "CTA %d of %d empty with %lld tiles", c, C,
                      (long long)NT);
        for (int64_t t = 0; t < NT; ++t) {
            const int c = pkv_owner(t, C, NT);
            CHECK(c >= 0 && c < C && pkv_split(c, C, NT) <= t && t < pkv_split(c + 1, C, NT),
                  "owner of tile %lld", (long long)t);
        }
        // producer replay
        for (int c = 0; c < C; ++c) {
            const int64_t t0 = pkv_split(c, C, NT), t1 = pkv_split(c + 1, C, NT);
            int64_t t = t0;
            while (t < t1) {
                const int s = pkv_find_seq(prefix.data(), S, t);
                CHECK(prefix[s] <= t && t < prefix[s + 1], "find_seq");
                const int u = (int)((t - prefix[s]) / n[s]);
                const int64_t Tu = prefix[s] + (int64_t)u * n[s];
                const int64_t seg_end = (Tu + n[s] < t1) ? Tu + n[s] : t1;
                const int unit = s * U + u;
                touching[unit]++;
                const bool is_whole = Tu >= t0 && Tu + n[s] <= t1;
                if (is_whole) {
                    whole[unit]++;
                } else {
                    const int slot = Tu > t0 ? 1 : 0;
                    CHECK(slot == pkv_partial_slot(c, C, NT, Tu), "slot rule");
                    CHECK(slot_unit[2 * c + slot] == -1, "CTA %d writes slot %d twice", c, slot);
                    slot_unit[2 * c + slot] = unit;
                    slot_tiles[2 * c + slot] = (int)(seg_end - t);
                    arrivals[c].push_back({unit, Tu});
                }
                t = seg_end;
            }
            if (t1 > t0) {
                // the producer's cursor walks [t0, t1) in flat order (and one step
                // past it, which the lookahead cursor takes)
                PkvCursor cur;
                pkv_cursor_at(cur, t0, prefix.data(), len.data(), S, tt);
                for (int64_t tau = t0; tau <= t1 && tau < NT; ++tau) {
                    const int s = pkv_find_seq(prefix.data(), S, tau);
                    const int off = (int)(tau - prefix[s]);
                    CHECK(cur.s == s && cur.u == off / n[s] && cur.ti == off % n[s] &&
                              cur.n == n[s] && cur.L == len[s],
                          "CTA %d: cursor (%d,%d,%d) at tile %lld", c, cur.s, cur.u, cur.ti,
                          (long long)tau);
                    pkv_cursor_next(cur, len.data(), S, U, tt);
                }
            }
        }
        // arrival replay, CTAs finishing in a random order
        std::vector<int> order(C);
        for (int c = 0; c < C; ++c) order[c] = c;
        std::shuffle(order.begin(), order.end(), rng);
        for (int c : order) {
            for (const auto &a : arrivals[c]) {
                const int unit = a.first, s = unit / U;
                const int64_t Tu = a.second;
                const int cf = pkv_owner(Tu, C, NT);
                CHECK(counter_unit[cf] == -1 || counter_unit[cf] == unit,
                      "units %d and %d share counter %d", counter_unit[cf], unit, cf);
                counter_unit[cf] = unit;
                const int parts = pkv_unit_parts(Tu, n[s], C, NT);
                CHECK(parts == touching[unit], "unit %d: %d parts, %d CTAs touch it", unit, parts,
                      touching[unit]);
                if (++counter[cf] != parts) continue;
                counter[cf] = 0;   // the merging warp puts the counter back
                merged[unit]++;
                const int cl = pkv_owner(Tu + n[s] - 1, C, NT);
                const int slot_first = pkv_partial_slot(cf, C, NT, Tu);
                for (int c2 = cf; c2 <= cl; ++c2) {
                    if (pkv_cta_empty(c2, C, NT)) continue;
                    const int slot = c2 == cf ? slot_first : 0;
                    CHECK(slot_unit[2 * c2 + slot] == unit, "merge of unit %d reads CTA %d slot %d",
                          unit, c2, slot);
                    covered[unit] += slot_tiles[2 * c2 + slot];
                }
            }
        }
        for (int c = 0; c < C; ++c) CHECK(counter[c] == 0, "counter %d left at %d", c, counter[c]);
        for (int s = 0; s < S; ++s)
            for (int u = 0; u < U; ++u) {
                const int unit = s * U + u;
                if (n[s] == 0) {
                    CHECK(whole[unit] == 0 && merged[unit] == 0, "empty unit touched");
                    continue;
                }
                CHECK(whole[unit] + merged[unit] == 1, "unit %d finished %d+%d times (trial %d)",
                      unit, whole[unit], merged[unit], trial);
                if (merged[unit]) CHECK(covered[unit] == n[s], "unit %d covers %d of %d tiles", unit,
                                        covered[unit], n[s]);
            }
    }
    if (fails) return 1;
    std::printf("OK\n");
    return 0;
}
