// plan_host_check.cpp -- runs the library's host/device planning rules
// (csrc/sp_rules.h, csrc/sp_plan.h) on the CPU so that tests can compare
// what the kernels would attend over with the oracle's visibility sets,
// without a GPU.  Test infrastructure only: built by tests/test_plan_host.py.
//
// Input (stdin): a case count, then one case per line:
//   mode kind sink window P n i_lo i_hi n_idx idx...
// mode 0  prefill plan of query rows i_lo..i_hi over a unit holding n tokens
//         of history (n = n_b); for each row: "R i count sum sumsq", and the
//         sorted visible positions ("L i p...") for the first, middle and
//         last row.  Checks, reported as "ERR ..." lines: cursor walk equals
//         indexed tiles; tile widths are whole 16-key steps of at most 128
//         keys; paged tiles start on a page and stay inside the unit's pages;
//         a tile marked full (no mask in the kernels) passes the masked rule
//         for every row and valid key;
//         no row sees a position twice.
// mode 1  decode ranges of a query at t = i_lo in a unit holding n tokens:
//         "D count sum sumsq" and "L t p..." (positions read through the
//         slot rule); "ERR" on an empty or duplicated slot.
// mode 2  slot table of a unit holding n tokens: "S pages" then one line
//         "P pos..." per page (-1 = empty slot).
// mode 3  the writes of i_lo chunks (sizes follow the index list) applied
//         one after another as the scatter kernel applies them (kept tokens
//         from retained_items, slots from unit_slot): after each chunk the
//         table in mode 2's format; "ERR" on a slot outside the unit's pages.
#include <algorithm>
#include <cstdio>
#include <vector>

#include "sp_plan.h"

using namespace sp;

static UnitPol make_pol(int kind, int sink, int window, int P, int n_idx) {
    UnitPol u{};
    u.kind = kind;
    if (kind == kLocal) {
        u.sink = sink;
        u.window = window;
        u.ring = (window + P - 1) / P + 1;
        u.sink_pages = (sink + P - 1) / P;
    }
    u.n_idx = n_idx;
    return u;
}

static bool same_tile(const KvTile& a, const KvTile& b) {
    return a.paged == b.paged && a.nvalid == b.nvalid && a.nkeys == b.nkeys && a.full == b.full &&
           a.table == b.table && a.start == b.start;
}

static void prefill_case(const UnitPol& u, const int32_t* idx, int P, int64_t n_b, int64_t i_lo,
                         int64_t i_hi) {
    const Plan pl = make_plan(u, idx, n_b, i_lo, i_hi, P);
    const int64_t rows = i_hi - i_lo + 1;
    std::vector<std::vector<int64_t>> vis(rows);
    const int64_t owned = unit_pages(u, idx, n_b, P);
    TileCursor cur = cursor_begin(pl);
    for (int64_t t = 0; t < pl.ntiles; ++t) {
        const KvTile kt = plan_tile(pl, u, t, i_lo, i_hi);
        const KvTile kc = cursor_tile(cur, u, (int32_t)i_lo, (int32_t)i_hi);
        cursor_next(pl, cur);
        if (!same_tile(kt, kc)) printf("ERR tile %lld: cursor and index disagree\n", (long long)t);
        // a cursor placed straight on tile t (where a piece of a split item starts)
        const KvTile ka = cursor_tile(cursor_at(pl, t), u, (int32_t)i_lo, (int32_t)i_hi);
        if (!same_tile(kt, ka)) printf("ERR tile %lld: cursor placed on it disagrees\n", (long long)t);
        if (kt.nkeys % 16 != 0 || kt.nkeys > kTileKeys || kt.nvalid < 1 || kt.nvalid > kt.nkeys)
            printf("ERR tile %lld: width %d valid %d\n", (long long)t, kt.nkeys, kt.nvalid);
        if (kt.paged) {
            if (kt.start % P != 0) printf("ERR tile %lld: paged tile off a page\n", (long long)t);
            const int64_t last_page = (kt.start + kt.nkeys - 1) / P;
            if (last_page >= owned)
                printf("ERR tile %lld: page %lld of %lld owned\n", (long long)t, (long long)last_page,
                       (long long)owned);
        }
        if (kt.paged) {
            // the arithmetic row mask of history tiles against the per-key rule
            for (int64_t r = 0; r < rows; ++r) {
                uint32_t vm[4];
                paged_row_mask(kt, u, (int32_t)n_b, (int32_t)(i_lo + r), P, vm);
                for (int c = 0; c < kTileKeys; ++c) {
                    const int64_t pos = tile_key_position(kt, u, idx, n_b, c, P);
                    const bool want = c < kt.nkeys && key_visible<int64_t>(kt, u, i_lo + r, c, pos);
                    const bool got = (vm[c >> 5] >> (c & 31)) & 1u;
                    if (want != got)
                        printf("ERR tile %lld: row mask of key %d (position %lld) for row %lld is %d\n",
                               (long long)t, c, (long long)pos, (long long)(i_lo + r), (int)got);
                }
            }
        }
        for (int c = 0; c < kt.nkeys; ++c) {
            const int64_t pos = tile_key_position(kt, u, idx, n_b, c, P);
            for (int64_t r = 0; r < rows; ++r) {
                const int64_t i = i_lo + r;
                const bool v = key_visible<int64_t>(kt, u, i, c, pos);
                if (kt.full && c < kt.nvalid) {
                    // the unmasked shortcut must agree with the masked rule
                    KvTile km = kt;
                    km.full = 0;
                    km.table = kt.paged ? 1 : kt.table;
                    if (!key_visible<int64_t>(km, u, i, c, pos))
                        printf("ERR tile %lld: marked full, key %d (position %lld) hidden from row %lld\n",
                               (long long)t, c, (long long)pos, (long long)i);
                }
                if (v) vis[r].push_back(pos);
            }
        }
    }
    if (cur.s != kMaxSegs) printf("ERR cursor not at the end after %lld tiles\n", (long long)pl.ntiles);
    for (int64_t r = 0; r < rows; ++r) {
        std::vector<int64_t>& s = vis[r];
        std::sort(s.begin(), s.end());
        if (std::adjacent_find(s.begin(), s.end()) != s.end())
            printf("ERR row %lld sees a position twice\n", (long long)(i_lo + r));
        long long sum = 0, sq = 0;
        for (int64_t p : s) { sum += p; sq += p * p; }
        printf("R %lld %zu %lld %lld\n", (long long)(i_lo + r), s.size(), sum, sq);
        if (r == 0 || r == rows - 1 || r == rows / 2) {
            printf("L %lld", (long long)(i_lo + r));
            for (int64_t p : s) printf(" %lld", (long long)p);
            printf("\n");
        }
    }
}

static void decode_case(const UnitPol& u, const int32_t* idx, int P, int64_t n, int64_t t) {
    const SlotRanges rg = decode_ranges(u, idx, t, P);
    std::vector<int64_t> s;
    for (int k = 0; k < rg.count; ++k)
        for (int64_t us = rg.lo[k]; us < rg.hi[k]; ++us) {
            const int64_t p = slot_position(u, idx, us, n, P);
            if (p < 0) printf("ERR decode range slot %lld is empty\n", (long long)us);
            else s.push_back(p);
        }
    std::sort(s.begin(), s.end());
    if (std::adjacent_find(s.begin(), s.end()) != s.end()) printf("ERR decode sees a position twice\n");
    long long sum = 0, sq = 0;
    for (int64_t p : s) { sum += p; sq += p * p; }
    printf("D %zu %lld %lld\n", s.size(), sum, sq);
    printf("L %lld", (long long)t);
    for (int64_t p : s) printf(" %lld", (long long)p);
    printf("\n");
}

static void slot_case(const UnitPol& u, const int32_t* idx, int P, int64_t n) {
    const int64_t pages = unit_pages(u, idx, n, P);
    printf("S %lld\n", (long long)pages);
    for (int64_t pg = 0; pg < pages; ++pg) {
        printf("P");
        for (int sl = 0; sl < P; ++sl)
            printf(" %lld", (long long)slot_position(u, idx, pg * P + sl, n, P));
        printf("\n");
    }
}

static void write_case(const UnitPol& u, const int32_t* idx, int P, const std::vector<int64_t>& chunks) {
    std::vector<int64_t> table;
    int64_t n = 0;
    for (int64_t c : chunks) {
        const int64_t n_new = n + c;
        const int64_t pages = unit_pages(u, idx, n_new, P);
        table.resize(pages * P, -1);
        const ItemRanges r = retained_items(u, idx, n, n_new, P);
        for (int k = 0; k < 2; ++k)
            for (int64_t it = r.lo[k]; it < r.hi[k]; ++it) {
                const int64_t pos = u.kind == kRetrieval ? idx[it] : it;
                const int64_t us = unit_slot(u, idx, pos, P);
                if (us < 0 || us >= pages * P) {
                    printf("ERR token %lld to slot %lld of %lld\n", (long long)pos, (long long)us,
                           (long long)(pages * P));
                    continue;
                }
                table[us] = pos;
            }
        n = n_new;
        printf("S %lld\n", (long long)pages);
        for (int64_t pg = 0; pg < pages; ++pg) {
            printf("P");
            for (int sl = 0; sl < P; ++sl) printf(" %lld", (long long)table[pg * P + sl]);
            printf("\n");
        }
    }
}

int main() {
    int cases = 0;
    if (scanf("%d", &cases) != 1) return 2;
    for (int k = 0; k < cases; ++k) {
        int mode, kind, sink, window, P, n_idx;
        long long n, i_lo, i_hi;
        if (scanf("%d %d %d %d %d %lld %lld %lld %d", &mode, &kind, &sink, &window, &P, &n, &i_lo,
                  &i_hi, &n_idx) != 9)
            return 2;
        std::vector<int32_t> idx(n_idx > 0 ? n_idx : 1, 0);
        for (int j = 0; j < n_idx; ++j)
            if (scanf("%d", &idx[j]) != 1) return 2;
        std::vector<int64_t> chunks;
        if (mode == 3)
            for (long long j = 0; j < i_lo; ++j) {
                long long c;
                if (scanf("%lld", &c) != 1) return 2;
                chunks.push_back(c);
            }
        const UnitPol u = make_pol(kind, sink, window, P, n_idx);
        printf("C %d\n", k);
        if (mode == 3) write_case(u, idx.data(), P, chunks);
        else if (mode == 0) prefill_case(u, idx.data(), P, n, i_lo, i_hi);
        else if (mode == 1) decode_case(u, idx.data(), P, n, i_lo);
        else slot_case(u, idx.data(), P, n);
    }
    return 0;
}
