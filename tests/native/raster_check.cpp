/*
 * Host-side check of the GEMM kernel's tile rasterisation (tcg::raster in
 * tcg_internal.h, shared by the host planner and the kernel): for a grid of
 * num_m_tiles x num_n_tiles tiles per batch entry, linear tile ids 0 .. tiles-1
 * must map one to one onto (batch, m-tile, n-tile), batch entries in order, and
 * every run of consecutive ids inside a group must stay within that group's
 * group_m rows of m-tiles, walking them m fastest and then n (the L2-locality
 * order the planner relies on).  Test code only.
 */
#include <cstdint>
#include <vector>

#include "tcg_internal.h"

extern "C" int64_t raster_mismatches(int num_m_tiles, int num_n_tiles, int batch, int group_m)
{
    tcg::GemmArgs p{};
    p.num_m_tiles = num_m_tiles;
    p.num_n_tiles = num_n_tiles;
    p.batch = batch;
    p.group_m = group_m;
    const int64_t per_batch = static_cast<int64_t>(num_m_tiles) * num_n_tiles;
    const int64_t tiles = per_batch * batch;
    std::vector<uint8_t> seen(static_cast<size_t>(tiles), 0);
    int64_t bad = 0;
    int prev_b = 0, prev_m = -1, prev_n = -1;
    for (int64_t t = 0; t < tiles; ++t) {
        int b = -1, mt = -1, nt = -1;
        tcg::raster(p, static_cast<int>(t), b, mt, nt);
        if (b < 0 || b >= batch || mt < 0 || mt >= num_m_tiles || nt < 0 || nt >= num_n_tiles) {
            ++bad;
            continue;
        }
        const int64_t id = (static_cast<int64_t>(b) * num_m_tiles + mt) * num_n_tiles + nt;
        if (seen[static_cast<size_t>(id)]++)
            ++bad;                                   // visited twice
        if (b != t / per_batch)
            ++bad;                                   // batch entries not in order
        // Inside a batch entry: the group of m-tiles [g*group_m, g*group_m + size) is
        // walked column by column, m fastest.
        const int r = static_cast<int>(t % per_batch);
        const int g = r / (group_m * num_n_tiles);
        const int first = g * group_m;
        const int size = num_m_tiles - first < group_m ? num_m_tiles - first : group_m;
        if (mt < first || mt >= first + size)
            ++bad;
        if (b == prev_b && prev_m >= 0 && r % (group_m * num_n_tiles) != 0) {
            const bool next_m = nt == prev_n && mt == prev_m + 1;
            const bool next_col = nt == prev_n + 1 && mt == first && prev_m == first + size - 1;
            if (!next_m && !next_col)
                ++bad;
        }
        prev_b = b;
        prev_m = mt;
        prev_n = nt;
    }
    for (int64_t i = 0; i < tiles; ++i)
        if (seen[static_cast<size_t>(i)] != 1)
            ++bad;                                   // never visited (or counted above)
    return bad;
}
