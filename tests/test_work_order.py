"""The blocked work order of dense launches (csrc/work_order.h), on the host.

The header is plain C++; a small program compiled with g++ checks, over a grid of
shapes (ragged Q-tile counts, G = 1, G above the item count, odd NQB):

* the schedule is a permutation of every item (b h * NQB + qb), so no block of
  rows is computed twice or left out;
* cta_of inverts the kernel's alternating deal (position k G + c in even rounds,
  (k + 1) G - 1 - c in odd ones) and nominal_item is the kernel's nominal decode;
* the items held back for the last rounds are the launch's shortest (no held
  item has a larger block index than any body item);
* each two-round block of the body spans at most ceil(2G / m) + 1 heads, m the
  fewest items a head keeps in the body (the locality the order exists for);
* for whole-head blocks (nothing held back, NQB divides 2G) every CTA gets the
  same load over each complete block;
* choose() (prefill items) and choose_single() (the backward's one-tile items)
  never return a schedule the load model puts more than 2% above the nominal
  order, and return the nominal order where ordering cannot matter;
  choose_uniform() (equal lengths, no causal mask) takes the blocked order.

Plus the loads worked out by hand for one small case. No GPU involved."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "alibi_positional_bias_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <set>
#include "work_order.h"
using namespace alibi::order;
static int fails = 0;
#define EXPECT(c, ...) do { if (!(c)) { std::printf("FAIL line %d: %s |", __LINE__, #c); std::printf(__VA_ARGS__); std::printf("\n"); ++fails; } } while (0)

static void check_schedule(const std::vector<int64_t> &s, long BH, int NQB, int NQT, long G, bool even)
{
    const long n = BH * NQB;
    EXPECT((long)s.size() == n, "size %zu n %ld", s.size(), n);
    std::vector<char> seen(n, 0);
    for (auto x : s) {
        EXPECT(x >= 0 && x < n, "item %lld", (long long)x);
        if (x >= 0 && x < n) { EXPECT(!seen[x], "dup %lld", (long long)x); seen[x] = 1; }
    }
    const long rounds = n / G;
    const long held = n % G + ((even && (rounds & 1)) ? G : 0);
    const long body = n - held;
    int max_held_qb = -1, min_body_qb = NQB;
    for (long i = 0; i < n; ++i) {
        const int qb = (int)(s[i] % NQB);
        if (i < body) min_body_qb = std::min(min_body_qb, qb); else max_held_qb = std::max(max_held_qb, qb);
    }
    EXPECT(held == 0 || max_held_qb <= min_body_qb, "held qb %d body qb %d", max_held_qb, min_body_qb);
    // within the body: each block of 2G positions runs longest first and spans few
    // heads (a head keeps at least NQB - ceil(held / BH) items in the body)
    const long per_head = NQB - (held + BH - 1) / BH;
    const long span_max = per_head > 0 ? (2 * G + per_head - 1) / per_head + 1 : BH;
    for (long b0 = 0; b0 < body; b0 += 2 * G) {
        std::set<long> heads;
        const long e = std::min(body, b0 + 2 * G);
        for (long i = b0; i < e; ++i) {
            heads.insert(s[i] / NQB);
            if (i > b0) EXPECT(s[i - 1] % NQB >= s[i] % NQB, "not longest first at %ld", i);
        }
        EXPECT((long)heads.size() <= span_max, "block at %ld spans %zu heads (max %ld)", b0, heads.size(), span_max);
    }
    // the held-back part runs longest first too
    for (long i = body + 1; i < n; ++i) EXPECT(s[i - 1] % NQB >= s[i] % NQB, "held not sorted at %ld", i);
    // whole-head blocks (nothing held back, NQB divides 2G): equal load per CTA over
    // each block of two rounds
    if (held == 0 && (2 * G) % NQB == 0 && NQT == 2 * NQB) {
        for (long b0 = 0; b0 + 2 * G <= body; b0 += 2 * G) {
            std::vector<long> load(G, 0);
            for (long i = b0; i < b0 + 2 * G; ++i) load[cta_of(i, G)] += item_tiles((int)(s[i] % NQB), NQT);
            for (long c = 1; c < G; ++c) EXPECT(load[c] == load[0], "block %ld cta %ld load %ld vs %ld", b0, c, load[c], load[0]);
        }
    }
}

int main()
{
    // the kernel's deal and nominal decode
    for (long G : {1L, 2L, 7L, 152L})
        for (long k = 0; k < 5; ++k)
            for (long c = 0; c < G; ++c) {
                const long idx = (k & 1) ? (k + 1) * G - 1 - c : k * G + c;
                EXPECT(cta_of(idx, G) == c, "G %ld k %ld c %ld", G, k, c);
            }
    for (long idx = 0; idx < 6 * 5; ++idx) {
        const long BH = 6; const int NQB = 5;
        const long r = idx / BH;
        EXPECT(nominal_item(idx, BH, NQB) == (idx % BH) * NQB + (NQB - 1 - r), "nominal %ld", idx);
    }
    // KV tiles of an item: both Q tiles present, or only the first at an odd end
    EXPECT(item_tiles(0, 2) == 2 && item_tiles(3, 8) == 8 && item_tiles(3, 7) == 7 && item_tiles(0, 1) == 1, "tiles");

    // hand-worked case: 4 heads x 3 blocks on G = 4 CTAs, NQT = 6: 12 items, 3 rounds,
    // nothing held back without the even body: blocks of 8 positions
    {
        auto s = blocked(4, 3, 4, false);
        // body block 0: heads 0, 1 (6 items) and head 2 qb 0, 1 -> sorted by qb desc, stable
        const int64_t want0[8] = {0 * 3 + 2, 1 * 3 + 2, 0 * 3 + 1, 1 * 3 + 1, 2 * 3 + 1, 0 * 3 + 0, 1 * 3 + 0, 2 * 3 + 0};
        for (int i = 0; i < 8; ++i) EXPECT(s[i] == want0[i], "hand block pos %d: %lld", i, (long long)s[i]);
        // block 1 (partial, 4 positions): head 2 qb 2, head 3 qb 0..2 -> qb 2, 2, 1, 0
        const int64_t want1[4] = {2 * 3 + 2, 3 * 3 + 2, 3 * 3 + 1, 3 * 3 + 0};
        for (int i = 0; i < 4; ++i) EXPECT(s[8 + i] == want1[i], "hand block1 pos %d: %lld", i, (long long)s[8 + i]);
        // loads (tiles 2, 4, 6 for qb 0, 1, 2, plus 2 per item): round 0 gives CTAs 0..3 qb 2, 2, 1, 1;
        // round 1 (reversed) gives CTA 3..0 qb 1, 0, 0, 0; round 2 gives CTAs 0..3 qb 2, 2, 1, 0
        // CTA0: 6+2 + 2+2 + 6+2 = 20; CTA1: 8 + 4 + 8 = 20; CTA2: 6 + 4 + 6 = 16; CTA3: 6 + 6 + 4 = 16
        EXPECT(makespan(s, 4, 3, 6, 4, 2.0) == 20.0, "hand makespan %f", makespan(s, 4, 3, 6, 4, 2.0));
        // the nominal order: rounds of qb 2 (4 items), 1, 0 -> every CTA 8 + 6 + 4 = 18
        EXPECT(makespan({}, 4, 3, 6, 4, 2.0) == 18.0, "hand nominal %f", makespan({}, 4, 3, 6, 4, 2.0));
        // with the even body the odd third round is held back: qb 0 of the 4 heads last;
        // the body (qb 2 x 4, then qb 1 x 4) gives every CTA 8 + 6, the last round 4: 18
        auto e = blocked(4, 3, 4, true);
        const int64_t wante[12] = {2, 5, 8, 11, 1, 4, 7, 10, 0, 3, 6, 9};
        for (int i = 0; i < 12; ++i) EXPECT(e[i] == wante[i], "hand even pos %d: %lld", i, (long long)e[i]);
        EXPECT(makespan(e, 4, 3, 6, 4, 2.0) == 18.0, "hand even makespan %f", makespan(e, 4, 3, 6, 4, 2.0));
        // so choose() takes the even body (18 < 20, and within 2% of the nominal 18)
        EXPECT(choose(4, 3, 6, 4) == e, "hand choose");
    }

    // the grid of shapes
    const long BHs[] = {1, 3, 12, 16, 32, 64, 128, 160, 320, 512, 1000};
    const int NQBs[] = {1, 2, 3, 4, 7, 8, 16, 32, 64};
    const long Gs[] = {1, 5, 152};
    for (long BH : BHs)
        for (int NQB : NQBs)
            for (int odd = 0; odd < 2; ++odd)
                for (long G0 : Gs) {
                    const int NQT = 2 * NQB - odd;
                    if (NQT < 1) continue;
                    const long n = BH * NQB;
                    const long G = std::min(n, G0);
                    for (int even = 0; even < 2; ++even) check_schedule(blocked(BH, NQB, G, even), BH, NQB, NQT, G, even);
                    auto c = choose(BH, NQB, NQT, G);
                    if (NQB < 2 || n <= 2 * G) EXPECT(c.empty(), "choose BH %ld NQB %d G %ld", BH, NQB, G);
                    if (!c.empty()) {
                        EXPECT((long)c.size() == n, "choose size");
                        const double m0 = makespan({}, BH, NQB, NQT, G, kItemCost), m = makespan(c, BH, NQB, NQT, G, kItemCost);
                        EXPECT(m <= 1.02 * m0, "choose BH %ld NQB %d G %ld: %f vs %f", BH, NQB, G, m, m0);
                        EXPECT(c == blocked(BH, NQB, G, false) || c == blocked(BH, NQB, G, true), "choose is one of the two");
                    }
                }
    // the backward's one-tile items (lengths r + 1) and equal-length items
    for (long BH : {1L, 12L, 128L, 320L, 512L})
        for (int NT : {1, 2, 5, 16, 31, 32})
            for (long G0 : {5L, 152L}) {
                const long n = BH * NT, G = std::min(n, G0);
                const auto len1 = [](int r) { return r + 1; };
                auto c = choose_single(BH, NT, G);
                if (NT < 2 || n <= 2 * G) EXPECT(c.empty(), "single BH %ld NT %d G %ld", BH, NT, G);
                if (!c.empty()) {
                    check_schedule(c, BH, NT, 2 * NT, G, c == blocked(BH, NT, G, true) && c != blocked(BH, NT, G, false));
                    EXPECT(makespan_by(c, BH, NT, len1, G, 1.0) <= 1.02 * makespan_by({}, BH, NT, len1, G, 1.0),
                           "single balance BH %ld NT %d G %ld", BH, NT, G);
                }
                auto u = choose_uniform(BH, NT, G);
                if (NT >= 2 && n > 2 * G) {
                    EXPECT(u == blocked(BH, NT, G, false), "uniform BH %ld NT %d G %ld", BH, NT, G);
                    // as balanced as the nominal order: item counts per CTA differ by at most one
                    const auto one = [](int) { return 1; };
                    EXPECT(makespan_by(u, BH, NT, one, G, 0.0) == makespan_by({}, BH, NT, one, G, 0.0), "uniform count");
                } else {
                    EXPECT(u.empty(), "uniform small BH %ld NT %d G %ld", BH, NT, G);
                }
            }
    // a decoder-layer launch (B = 4, H = 32, N = 2048: 128 heads x 8 blocks on 152 CTAs)
    // gets the blocked order with the nominal order's balance
    {
        auto c = choose(128, 8, 16, 152);
        EXPECT(!c.empty(), "layer shape keeps the nominal order");
        if (!c.empty()) EXPECT(makespan(c, 128, 8, 16, 152, kItemCost) <= makespan({}, 128, 8, 16, 152, kItemCost), "layer balance");
    }
    std::printf(fails ? "%d failures\n" : "ok\n", fails);
    return fails != 0;
}
"""


def test_work_order_on_host(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "order.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "order"
    subprocess.run([cxx, "-std=c++17", "-O2", f"-I{CSRC}", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr
    assert r.stdout.strip().endswith("ok")


def test_flag_values_match_header():
    """The Python constants are the header's #define values."""
    import re
    import alibi_positional_bias_gb300 as ab
    hdr = open(os.path.join(os.path.dirname(HERE), "include", "alibi.h")).read()
    defs = dict(re.findall(r"#define (ALIBI_FWD_\w+) (\d+)u", hdr))
    assert set(defs) == {"ALIBI_FWD_SKIP_UNDERFLOW", "ALIBI_FWD_CLAMP", "ALIBI_FWD_LOGDIST", "ALIBI_FWD_SOFTCAP",
                         "ALIBI_FWD_NOMINAL_ORDER"}
    for name, val in defs.items():
        assert getattr(ab, name) == int(val), name
