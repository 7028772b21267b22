// Work order of dense launches (prefill and backward) whose streamed tiles do
// not fit in L2.
//
// A prefill item is one (b, h) and one block qb of two 128-row Q tiles; a causal
// item reads the KV tiles up to its diagonal, so its length grows with qb. The
// kernel deals positions of a schedule to its persistent CTAs in rounds of G
// (one position per CTA), alternating direction from round to round, and each
// CTA runs its positions in order.
//
// The nominal order (no table) runs round r over block NQB-1-r of every (b, h):
// longest first, well balanced, but a head's blocks are one round apart, so
// once B*H heads of K and V exceed L2 each block reads its head's K and V from
// DRAM again. The blocked order here keeps the balance and the reuse:
//   * the heads are taken in order and their items cut into blocks of two
//     rounds (2 G positions); within a block, items run longest first. Two
//     rounds cover 2G/NQB heads, whose K and V then stay in L2 while all of
//     their blocks run.
//   * in the alternating deal a CTA gets rank c of the first round and rank
//     2G-1-c of the block (the c-th shortest) in the second, so a block of
//     whole heads, whose lengths 2, 4, ..., 2 NQB pair up symmetrically, gives
//     every CTA the same load;
//   * the positions that do not fill a last pair of rounds go to the shortest
//     items of the launch (qb = 0 of every head first), placed last: either the
//     partial last round only, or ("even body") also one full round so that the
//     body is a whole number of blocks.
// A load model (the item's KV tiles plus a fixed cost per item) picks the better
// of the two and falls back to the nominal order if neither is within 2% of its
// balance. The backward's one-tile items (dK/dV per KV tile, dQ per query tile)
// take the same construction, ranked by their length; without the causal mask
// every item has the same length and the blocked order is taken as it is.
//
// Plain C++ (no CUDA types): the host builds the table once per shape, and the
// tests compile this header with the host compiler.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

namespace alibi {
namespace order {

// KV tiles of causal item block qb out of NQT Q tiles (the second Q tile 2 qb + 1
// may be past the end).
inline int item_tiles(int qb, int NQT)
{
    const int t1 = 2 * qb + 1;
    return t1 < NQT ? t1 + 1 : t1;
}

// The CTA that runs schedule position idx when G CTAs take rounds of G positions
// in alternating direction.
inline long cta_of(long idx, long G)
{
    const long k = idx / G, c = idx - k * G;
    return (k & 1) ? G - 1 - c : c;
}

// Item (b h * NQB + qb) at position idx of the nominal order.
inline long nominal_item(long idx, long BH, int NQB)
{
    const long r = idx / BH;
    return (idx - r * BH) * NQB + (NQB - 1 - r);
}

// Largest per-CTA load of a schedule (empty: the nominal order): the KV tiles
// len(qb) of its items plus per_item for each item's fill and epilogue.
template <class Len>
inline double makespan_by(const std::vector<int64_t> &sched, long BH, int NQB, Len len, long G, double per_item)
{
    const long n = BH * NQB;
    std::vector<double> load(static_cast<size_t>(G), 0.0);
    for (long i = 0; i < n; ++i) {
        const long item = sched.empty() ? nominal_item(i, BH, NQB) : static_cast<long>(sched[i]);
        load[cta_of(i, G)] += len(static_cast<int>(item % NQB)) + per_item;
    }
    return *std::max_element(load.begin(), load.end());
}

// The prefill's items: len = item_tiles.
inline double makespan(const std::vector<int64_t> &sched, long BH, int NQB, int NQT, long G, double per_item)
{
    return makespan_by(sched, BH, NQB, [NQT](int qb) { return item_tiles(qb, NQT); }, G, per_item);
}

// The blocked order (see above); even_body also holds back one full round when
// the full rounds are odd in number. Only the ranking matters here: items with a
// larger qb are longer.
inline std::vector<int64_t> blocked(long BH, int NQB, long G, bool even_body)
{
    const long n = BH * NQB;
    const long rounds = n / G;
    const long held = n % G + ((even_body && (rounds & 1)) ? G : 0);
    // held back: the `held` shortest items, block index ascending, heads ascending;
    // item (bh, qb) is among them iff qb * BH + bh < held
    std::vector<int64_t> sched;
    sched.reserve(static_cast<size_t>(n));
    for (long bh = 0; bh < BH; ++bh)
        for (int qb = 0; qb < NQB; ++qb)
            if (static_cast<long>(qb) * BH + bh >= held) sched.push_back(bh * NQB + qb);
    const long body = static_cast<long>(sched.size());
    const auto longer = [NQB](int64_t a, int64_t b) { return a % NQB > b % NQB; };
    for (long s = 0; s < body; s += 2 * G)
        std::stable_sort(sched.begin() + s, sched.begin() + std::min(body, s + 2 * G), longer);
    for (int qb = NQB - 1; qb >= 0; --qb)
        for (long bh = 0; bh < BH; ++bh)
            if (static_cast<long>(qb) * BH + bh < held) sched.push_back(bh * NQB + qb);
    return sched;
}

// Fixed cost of an item in KV-tile units in the load model (fill and epilogue).
constexpr double kItemCost = 2.0;

// The schedule to launch with, or an empty vector for the nominal order, for
// items whose length len(qb) grows with qb.
template <class Len>
inline std::vector<int64_t> choose_by(long BH, int NQB, Len len, long G, double per_item)
{
    const long n = BH * NQB;
    if (NQB < 2 || G < 1 || n <= 2 * G) return {};
    std::vector<int64_t> a = blocked(BH, NQB, G, false), b = blocked(BH, NQB, G, true);
    const double ma = makespan_by(a, BH, NQB, len, G, per_item), mb = makespan_by(b, BH, NQB, len, G, per_item);
    const double m0 = makespan_by({}, BH, NQB, len, G, per_item);
    if (std::min(ma, mb) > 1.02 * m0) return {};
    return mb < ma ? b : a;
}

// The prefill's schedule.
inline std::vector<int64_t> choose(long BH, int NQB, int NQT, long G)
{
    return choose_by(BH, NQB, [NQT](int qb) { return item_tiles(qb, NQT); }, G, kItemCost);
}

// Items of equal length (the symmetric, non-causal bias: every item visits all
// tiles): any order is as balanced as the nominal one, so the blocked order.
inline std::vector<int64_t> choose_uniform(long BH, int per_head, long G)
{
    return choose_by(BH, per_head, [](int) { return 1; }, G, 0.0);
}

// The backward's schedule: NT one-tile items per head, ranked r = 0 .. NT-1 by
// length r + 1 (dK/dV: KV tile NT-1-r meets r + 1 query tiles; dQ: query tile r
// meets r + 1 KV tiles).
inline std::vector<int64_t> choose_single(long BH, int NT, long G)
{
    return choose_by(BH, NT, [](int r) { return r + 1; }, G, 1.0);
}

}  // namespace order
}  // namespace alibi
