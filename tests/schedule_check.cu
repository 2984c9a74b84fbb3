// Host-side check of the balanced Wgrad's work split (test helper, compiled
// and run by tests/test_schedule.py; no GPU needed).  It calls the same
// __host__ __device__ functions of gemm.cuh that the kernel's producers, MMA
// thread and promotion warps call, over many grid and problem sizes, and
// checks that
//  - every reduction chunk of every output tile belongs to exactly one
//    cluster's segment, whole-tile rounds first in tile order;
//  - each cluster's segments add up to the chunk count its MMA thread issues;
//  - a cluster has at most two remainder segments, in distinct split slots,
//    and every slot and arrival counter index lies inside the scratch the
//    host allocates;
//  - the parts the last-arriving warp sums for a remaining tile are exactly
//    the clusters that wrote a partial of it.
// Prints "schedule ok: <cases> cases, max <parts> parts" and exits 0, or
// prints the first failure and exits 1.
#include <cstdio>
#include <cstdint>
#include <set>
#include <vector>

#include "gemm.cuh"

using fp8bq::GemmParams;

static bool fail(const char* what, int tiles, int KC, int n, int a, int b) {
    std::printf("FAIL %s: tiles %d KC %d clusters %d (%d, %d)\n", what, tiles, KC, n, a, b);
    return false;
}

// The sizes the library runs in the balanced order (the host's rule).
static bool balanced(int tiles, int KC, int n) {
    const int64_t rem = tiles % n;
    return n >= 2 && tiles >= n && rem > 0 && 10 * rem <= 9 * static_cast<int64_t>(n) &&
           rem * KC * static_cast<int64_t>(n) < (int64_t(1) << 31);
}

static bool check(int tiles, int KC, int n, int& max_parts) {
    GemmParams p = {};
    p.KC = KC;
    p.num_tiles = tiles;
    const int R = tiles / n, rem = tiles - R * n;
    std::vector<int> owner(static_cast<size_t>(tiles) * KC, -1);
    std::vector<std::set<int>> writers(rem);
    for (int cid = 0; cid < n; ++cid) {
        int tile, c_lo, c_hi, rt, k = 0;
        int64_t chunks = 0;
        bool slot_used[2] = {false, false};
        while (fp8bq::hyb_segment(p, cid, n, k, tile, c_lo, c_hi, rt)) {
            if (k > R + 1) return fail("more than two remainder segments", tiles, KC, n, cid, k);
            if (tile < 0 || tile >= tiles || c_lo < 0 || c_lo >= c_hi || c_hi > KC)
                return fail("segment out of range", tiles, KC, n, cid, k);
            if (k < R && (rt != -1 || tile != cid + k * n || c_lo != 0 || c_hi != KC))
                return fail("whole-tile round not in tile order", tiles, KC, n, cid, k);
            if (k >= R) {
                if (rt < 0 || rt >= rem || tile != R * n + rt) return fail("remaining tile index", tiles, KC, n, cid, k);
                const int j = fp8bq::hyb_slot_segment(p, n, cid, rt);
                if (j < 0 || j > 1 || slot_used[j]) return fail("split slot", tiles, KC, n, cid, j);
                slot_used[j] = true;
                // slot (cid, j, CTA rank 1) inside n clusters' slots; counter
                // (rt, rank 1, warp 7) inside (n - 1) tiles' counters
                if ((static_cast<int64_t>(cid) * 2 + j) * 2 + 1 >= static_cast<int64_t>(n) * 2 * 2)
                    return fail("slot index", tiles, KC, n, cid, j);
                if ((static_cast<int64_t>(rt) * 2 + 1) * fp8bq::kPromoWarps + fp8bq::kPromoWarps - 1 >=
                    static_cast<int64_t>(n - 1) * fp8bq::kSplitTileCounters)
                    return fail("counter index", tiles, KC, n, cid, rt);
                writers[rt].insert(cid);
            }
            for (int c = c_lo; c < c_hi; ++c) {
                int& o = owner[static_cast<size_t>(tile) * KC + c];
                if (o != -1) return fail("chunk covered twice", tiles, KC, n, tile, c);
                o = cid;
            }
            chunks += c_hi - c_lo;
            ++k;
        }
        if (chunks != fp8bq::hyb_chunk_count(p, cid, n)) return fail("chunk count", tiles, KC, n, cid, int(chunks));
    }
    for (size_t i = 0; i < owner.size(); ++i)
        if (owner[i] < 0) return fail("chunk not covered", tiles, KC, n, int(i / KC), int(i % KC));
    for (int rt = 0; rt < rem; ++rt) {
        int first, last;
        fp8bq::hyb_part_range(p, n, rt, first, last);
        if (first < 0 || last >= n || first > last) return fail("part range", tiles, KC, n, first, last);
        std::set<int> parts;
        for (int c = first; c <= last; ++c)
            if (fp8bq::hyb_meets(p, n, c, rt)) parts.insert(c);
        if (parts != writers[rt] || parts.empty()) return fail("parts summed != parts written", tiles, KC, n, rt, 0);
        if (static_cast<int>(parts.size()) > max_parts) max_parts = static_cast<int>(parts.size());
    }
    return true;
}

int main() {
    int cases = 0, max_parts = 0;
    const int ns[] = {2, 3, 5, 7, 16, 37, 73, 74};
    const int kcs[] = {1, 2, 3, 5, 8, 16, 24, 48, 64, 256};
    for (int n : ns)
        for (int KC : kcs)
            for (int m : {1, 2, 3, 5, 7, 10})
                for (int extra : {1, 2, n / 3, n / 2, (9 * n) / 10, n - 1}) {
                    const int tiles = m * n + extra;
                    if (!balanced(tiles, KC, n)) continue;
                    if (!check(tiles, KC, n, max_parts)) return 1;
                    ++cases;
                }
    // the 3.8B layer's and the test shapes' Wgrads on 74 clusters
    const int real[][2] = {{384, 256}, {768, 256}, {768, 64}, {192, 128}, {81, 16}, {75, 32}, {81, 8}};
    for (const auto& s : real) {
        if (!balanced(s[0], s[1], 74)) continue;
        if (!check(s[0], s[1], 74, max_parts)) return 1;
        ++cases;
    }
    // seeded pseudo-random sizes (64-bit LCG)
    uint64_t x = 0x9E3779B97F4A7C15ull;
    auto next = [&](int mod) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        return static_cast<int>((x >> 33) % static_cast<uint64_t>(mod));
    };
    for (int i = 0; i < 600; ++i) {
        const int n = 2 + next(73), KC = 1 + next(300), tiles = n + next(20 * n);
        if (!balanced(tiles, KC, n)) continue;
        if (!check(tiles, KC, n, max_parts)) return 1;
        ++cases;
    }
    std::printf("schedule ok: %d cases, max %d parts\n", cases, max_parts);
    return 0;
}
