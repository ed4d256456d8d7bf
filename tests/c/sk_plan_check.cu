// Host-only check of the stream-K schedule (tg::sk_plan, tg::sk_bound,
// tg::sk_owner, tg::sk_piece: the functions the kernel and the host API use).
// For every (tiles, units, k_blocks) of a sweep it replays each unit's work
// items as the kernel does and checks that
//   - the units' ranges are non-empty and partition the stream-K k-blocks;
//   - every stream-K tile is covered exactly once by its pieces, which carry the
//     slice indices 0 .. slices-1 in k order (or slices == 0 for a tile held by
//     one range), with slices <= max_slices so that every partial slab lies in
//     the workspace the host allocates;
//   - every whole tile is taken by exactly one unit;
//   - ranges differ in length by at most SK_QUANTUM k-blocks plus the remainder
//     that the last range takes;
//   - the tile raster (tg::raster) visits every (M-tile, N-tile) of a problem
//     exactly once, for every band width.
// Prints one line per failure and "OK <plans> <stream-K plans>" at the end;
// exit status 1 on any failure.
#include <cstdio>
#include <vector>

#include "tg_kernel.cuh"

static int failures = 0;

static void fail(const char* what, long long T, long long U, long long KB, long long a, long long b) {
    if (failures < 20) std::printf("FAIL %s tiles=%lld units=%lld k_blocks=%lld (%lld, %lld)\n", what, T, U, KB, a, b);
    ++failures;
}

int main() {
    const long long units_list[] = {2, 3, 7, 76, 148, 152};
    const long long kb_list[] = {1, 4, 7, 8, 9, 16, 17, 63, 64, 65, 128, 129, 1000};
    long long plans = 0, sk_plans = 0;
    for (long long U_all : units_list)
        for (long long KB : kb_list)
            for (long long T = 1; T <= 420; ++T) {
                ++plans;
                const tg::SkPlan sp = tg::sk_plan(T, U_all, KB);
                const long long R = sp.tiles, U = sp.units;
                if (R == 0) {
                    if (sp.units != 0) fail("units without tiles", T, U_all, KB, U, 0);
                } else {
                    ++sk_plans;
                    if (U <= R || U > U_all) fail("unit count", T, U_all, KB, U, R);
                    if (sp.max_slices > tg::SK_MAX_PIECES + 1) fail("too many pieces", T, U_all, KB, sp.max_slices, 0);
                }
                const long long total = R * KB;
                // coverage count of every stream-K k-block, and the pieces of each tile in k order
                std::vector<int> cover(static_cast<size_t>(total), 0);
                std::vector<std::vector<std::pair<int, int>>> pieces(static_cast<size_t>(R));   // (kb0, slice)
                std::vector<int> slices_of(static_cast<size_t>(R), -1);
                long long min_len = total + 1, max_len = -1;
                for (long long u = 0; u < U; ++u) {
                    const long long b0 = tg::sk_bound(u, U, total), b1 = tg::sk_bound(u + 1, U, total);
                    if (b1 <= b0) { fail("empty range", T, U_all, KB, u, b1 - b0); continue; }
                    if (u + 1 < U) { min_len = b1 - b0 < min_len ? b1 - b0 : min_len; }
                    max_len = b1 - b0 > max_len ? b1 - b0 : max_len;
                    for (long long cur = b0; cur < b1;) {
                        const tg::SkPiece q = tg::sk_piece(cur, b1, static_cast<int>(KB), U, total, u);
                        if (q.t < 0 || q.t >= R || q.kb0 < 0 || q.kb1 <= q.kb0 || q.kb1 > KB ||
                            q.t * KB + q.kb0 != cur) {
                            fail("bad piece", T, U_all, KB, u, cur);
                            break;
                        }
                        for (long long k = q.t * KB + q.kb0; k < q.t * KB + q.kb1; ++k) cover[static_cast<size_t>(k)]++;
                        if (q.slices == 0) {
                            if (q.kb0 != 0 || q.kb1 != KB) fail("single piece is not the whole tile", T, U_all, KB, u, q.t);
                        } else if (q.slice < 0 || q.slice >= q.slices || q.slices > sp.max_slices) {
                            fail("slice index", T, U_all, KB, q.slice, q.slices);
                        }
                        if (slices_of[static_cast<size_t>(q.t)] < 0) slices_of[static_cast<size_t>(q.t)] = q.slices;
                        else if (slices_of[static_cast<size_t>(q.t)] != q.slices) fail("slices disagree", T, U_all, KB, q.t, q.slices);
                        pieces[static_cast<size_t>(q.t)].push_back({q.kb0, q.slice});
                        cur += q.kb1 - q.kb0;
                    }
                }
                for (long long k = 0; k < total; ++k)
                    if (cover[static_cast<size_t>(k)] != 1) { fail("k-block coverage", T, U_all, KB, k, cover[static_cast<size_t>(k)]); break; }
                for (long long t = 0; t < R; ++t) {
                    const auto& ps = pieces[static_cast<size_t>(t)];
                    const int n = static_cast<int>(ps.size());
                    const int sl = slices_of[static_cast<size_t>(t)];
                    if ((sl == 0 && n != 1) || (sl != 0 && sl != n)) fail("piece count", T, U_all, KB, t, n);
                    for (int i = 0; i < n; ++i) {
                        // pieces were appended in unit order, which is k order
                        if (i > 0 && ps[i].first <= ps[i - 1].first) fail("piece order", T, U_all, KB, t, i);
                        if (sl != 0 && ps[i].second != i) fail("slice numbering", T, U_all, KB, t, i);
                    }
                }
                if (U > 1 && max_len - min_len > tg::SK_QUANTUM + (total % tg::SK_QUANTUM))
                    fail("range balance", T, U_all, KB, min_len, max_len);
                // whole tiles: unit u takes R + u, R + u + U_all, ...
                std::vector<int> taken(static_cast<size_t>(T), 0);
                for (long long u = 0; u < U_all; ++u)
                    for (long long t = R + u; t < T; t += U_all) taken[static_cast<size_t>(t)]++;
                for (long long t = R; t < T; ++t)
                    if (taken[static_cast<size_t>(t)] != 1) { fail("whole tile coverage", T, U_all, KB, t, taken[static_cast<size_t>(t)]); break; }
            }
    // the raster visits every (M-tile, N-tile) of a problem exactly once
    long long rasters = 0;
    for (int tm = 1; tm <= 40; ++tm)
        for (int tn = 1; tn <= 40; ++tn)
            for (int band : {1, 2, 3, 4, 8, 16}) {
                ++rasters;
                std::vector<int> seen(static_cast<size_t>(tm * tn), 0);
                for (long long l = 0; l < static_cast<long long>(tm) * tn; ++l) {
                    int mb = -1, nb = -1;
                    tg::raster(l, tm, tn, band, mb, nb);
                    if (mb < 0 || mb >= tm || nb < 0 || nb >= tn) { fail("raster out of range", tm, tn, band, mb, nb); break; }
                    seen[static_cast<size_t>(mb * tn + nb)]++;
                }
                for (int i = 0; i < tm * tn; ++i)
                    if (seen[static_cast<size_t>(i)] != 1) { fail("raster coverage", tm, tn, band, i, seen[static_cast<size_t>(i)]); break; }
            }
    std::printf("%s %lld %lld %lld\n", failures ? "FAILED" : "OK", plans, sk_plans, rasters);
    return failures ? 1 : 0;
}
