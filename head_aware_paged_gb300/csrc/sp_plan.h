// sp_plan.h -- the key tiles one prefill work item attends over.
//
// A work item is 128 consecutive query rows (positions i_lo .. i_hi) of one
// or two query heads of one KV head.  Its visible keys (the union of V(i)
// over its rows) are covered by "segments" -- runs of keys from one source:
//   * chunk: the call's own K/V rows, positions p >= n_b (rows of the chunk);
//   * paged: unit slots of the cache pages (history, positions < n_b).
// Each segment is cut into tiles of at most 128 keys; a tile's MMA width is
// its valid key count rounded up to 16 (so a 4-token sink costs a 16-wide
// tile, not 128).  Segments never overlap, so every visible key is counted
// exactly once, and keys a tile holds that a row must not see are masked:
//   * chunk tiles (GLOBAL / LOCAL): position p0 + c, mask by arithmetic;
//   * paged tiles and RETRIEVAL chunk tiles: per-key position table.
// A tile is "full" when every row of the item sees every key of it; only
// tiles that are not full are masked.  The same functions run on the host
// (work estimates, ordering) and in the kernels.
#pragma once
#include "sp_rules.h"

namespace sp {

constexpr int kTileKeys = 128;
constexpr int kMaxSegs = 5;

struct Seg {
    int64_t start;     // first position (chunk) or first unit slot (paged, page aligned)
    int64_t len;       // keys (chunk) or slots (paged); 0 = unused slot
};

// Segment slots are fixed per class (static indexing keeps a plan in
// registers):  GLOBAL  0 history pages, 1 chunk;
//              LOCAL   0 sink pages, 1 sink rows of the chunk, 2 and 3 ring
//                      pages (the ring may wrap once), 4 window rows of the chunk;
//              RETRIEVAL 0 history pages, 1 chunk rows from the first index.
struct Plan {
    Seg seg[kMaxSegs];
    int64_t ntiles;
};

struct KvTile {
    int32_t paged;
    int32_t nvalid;    // keys in the tile that belong to the segment
    int32_t nkeys;     // MMA width: nvalid rounded up to 16
    int32_t full;      // every row sees every valid key; no mask needed
    int32_t table;     // mask needs a per-key position table
    int64_t start;     // position of key 0 (chunk) or unit slot of key 0 (paged)
};

SP_HD bool seg_paged(int kind, int s) {
    return kind == kLocal ? (s == 0 || s == 2 || s == 3) : s == 0;
}

SP_HD int64_t seg_tiles(int64_t len) { return len > 0 ? (len + kTileKeys - 1) / kTileKeys : 0; }

// Segments of one work item.  n_b: tokens the unit already holds (history);
// rows i_lo .. i_hi (positions, i_lo >= n_b).
SP_HD Plan make_plan(const UnitPol& u, const int32_t* idx, int64_t n_b, int64_t i_lo,
                     int64_t i_hi, int P) {
    Plan pl;
    #pragma unroll
    for (int s = 0; s < kMaxSegs; ++s) { pl.seg[s].start = 0; pl.seg[s].len = 0; }
    if (u.kind == kGlobal) {
        pl.seg[0].start = 0;   pl.seg[0].len = n_b;
        pl.seg[1].start = n_b; pl.seg[1].len = i_hi + 1 - n_b;
    } else if (u.kind == kLocal) {
        const int64_t se = min64(u.sink, i_hi + 1);            // sink positions [0, se)
        pl.seg[0].start = 0;   pl.seg[0].len = min64(se, n_b);
        pl.seg[1].start = n_b; pl.seg[1].len = se - n_b;
        const int64_t wa = max64(u.sink, i_lo - u.window + 1);  // window positions [wa, i_hi]
        if (wa < n_b && wa <= i_hi) {
            const int64_t e = min64(i_hi + 1, n_b);
            const int64_t ring = u.ring, base = (int64_t)u.sink_pages * P;
            const int64_t qa = (wa - u.sink) % (ring * P);
            const int64_t fa = qa / P;
            const int64_t np = (qa + (e - wa) - 1) / P - fa + 1;  // ring pages touched (<= ring)
            const int64_t n1 = min64(np, ring - fa);
            pl.seg[2].start = base + fa * P; pl.seg[2].len = n1 * P;
            pl.seg[3].start = base;          pl.seg[3].len = (np - n1) * P;
        }
        const int64_t ca = max64(wa, n_b);
        pl.seg[4].start = ca; pl.seg[4].len = i_hi + 1 - ca;
    } else {
        const int64_t cnt_h = count_below(idx, u.n_idx, n_b);
        pl.seg[0].start = 0; pl.seg[0].len = cnt_h;
        if (cnt_h < u.n_idx && idx[cnt_h] <= i_hi) {
            const int64_t f = idx[cnt_h];
            pl.seg[1].start = f; pl.seg[1].len = i_hi + 1 - f;
        }
    }
    pl.ntiles = 0;
    #pragma unroll
    for (int s = 0; s < kMaxSegs; ++s) pl.ntiles += seg_tiles(pl.seg[s].len);
    return pl;
}

// Tile t (0 <= t < pl.ntiles) of a plan.
SP_HD KvTile plan_tile(const Plan& pl, const UnitPol& u, int64_t t, int64_t i_lo,
                       int64_t i_hi) {
    KvTile k;
    k.paged = 0; k.nvalid = 0; k.nkeys = 0; k.full = 0; k.table = 0; k.start = 0;
    bool found = false;
    #pragma unroll
    for (int s = 0; s < kMaxSegs; ++s) {
        const int64_t nt = seg_tiles(pl.seg[s].len);
        if (!found && t < nt) {
            found = true;
            const bool paged = seg_paged(u.kind, s);
            k.paged = paged;
            k.start = pl.seg[s].start + t * kTileKeys;
            k.nvalid = (int32_t)min64(kTileKeys, pl.seg[s].len - t * kTileKeys);
            k.nkeys = (k.nvalid + 15) & ~15;
            const bool exact = k.nkeys == k.nvalid;
            if (paged) {
                // history: every stored position is < n_b <= i_lo; GLOBAL and
                // RETRIEVAL slots and LOCAL sink slots are visible to all rows
                k.full = exact && (u.kind != kLocal || s == 0);
                k.table = !k.full;
            } else {
                const int64_t p0 = k.start, p1 = k.start + k.nvalid - 1;
                bool full = exact && p1 <= i_lo && u.kind != kRetrieval;
                if (u.kind == kLocal) full = full && (p1 < u.sink || p0 >= i_hi - u.window + 1);
                k.full = full;
                k.table = u.kind == kRetrieval;
            }
        } else if (!found) {
            t -= nt;
        }
    }
    return k;
}

// Incremental walk over a plan's tiles (tile t+1 from tile t without
// re-scanning the segments).  Positions and slots fit in 32 bits.
struct TileCursor {
    int32_t s;        // current segment (kMaxSegs = done)
    int32_t t_in;     // tile within the segment
    int32_t nt_s;     // tiles in the segment
    int32_t start;    // segment start
    int32_t len;      // segment length
};

SP_HD void cursor_load(const Plan& pl, TileCursor& c) {
    // first non-empty segment at or after c.s (static indexing only)
    int32_t s = kMaxSegs, start = 0, len = 0;
    #pragma unroll
    for (int q = kMaxSegs - 1; q >= 0; --q)
        if (q >= c.s && pl.seg[q].len > 0) { s = q; start = (int32_t)pl.seg[q].start; len = (int32_t)pl.seg[q].len; }
    c.s = s;
    c.start = start;
    c.len = len;
    c.t_in = 0;
    c.nt_s = (len + kTileKeys - 1) / kTileKeys;
}

SP_HD TileCursor cursor_begin(const Plan& pl) {
    TileCursor c;
    c.s = 0;
    cursor_load(pl, c);
    return c;
}

SP_HD void cursor_next(const Plan& pl, TileCursor& c) {
    if (++c.t_in < c.nt_s) return;
    c.s += 1;
    cursor_load(pl, c);
}

// A cursor on tile t of the plan (0 <= t < pl.ntiles): where a piece of a
// work item split along its keys starts.
SP_HD TileCursor cursor_at(const Plan& pl, int64_t t) {
    TileCursor c;
    c.s = 0;
    cursor_load(pl, c);
    while (c.s < kMaxSegs && t >= c.nt_s) {
        t -= c.nt_s;
        c.s += 1;
        cursor_load(pl, c);
    }
    c.t_in = (int32_t)t;
    return c;
}

// The tile under the cursor (same result as plan_tile for that index).
SP_HD KvTile cursor_tile(const TileCursor& c, const UnitPol& u, int32_t i_lo, int32_t i_hi) {
    KvTile k;
    const bool paged = seg_paged(u.kind, c.s);
    k.paged = paged;
    k.start = (int64_t)c.start + (int64_t)c.t_in * kTileKeys;
    const int32_t rest = c.len - c.t_in * kTileKeys;
    k.nvalid = rest < kTileKeys ? rest : kTileKeys;
    k.nkeys = (k.nvalid + 15) & ~15;
    const bool exact = k.nkeys == k.nvalid;
    if (paged) {
        k.full = exact && (u.kind != kLocal || c.s == 0);
        k.table = !k.full;
    } else {
        const int32_t p0 = (int32_t)k.start, p1 = p0 + k.nvalid - 1;
        bool full = exact && p1 <= i_lo && u.kind != kRetrieval;
        if (u.kind == kLocal) full = full && (p1 < u.sink || p0 >= i_hi - u.window + 1);
        k.full = full;
        k.table = u.kind == kRetrieval;
    }
    return k;
}

// Position of key c of a tile, as the mask sees it (-1 = never visible).
SP_HD int64_t tile_key_position(const KvTile& k, const UnitPol& u, const int32_t* idx,
                                int64_t n_b, int c, int P) {
    if (c >= k.nvalid) return -1;
    if (k.paged) return slot_position(u, idx, k.start + c, n_b, P);
    const int64_t p = k.start + c;
    if (u.kind == kRetrieval) {
        const int64_t r = count_below(idx, u.n_idx, p);
        return (r < u.n_idx && idx[r] == p) ? p : -1;
    }
    return p;
}

// Does query position i see key position p (p >= 0) under the unit's class.
SP_HD bool sees(const UnitPol& u, int64_t p, int64_t i) {
    if (p < 0 || p > i) return false;
    if (u.kind == kLocal) return p < u.sink || p > i - u.window;
    return true;
}

// Is key c of tile k visible to the query at position i?  table_pos is the
// key's entry of the position table (used only when k.table is set).
template <typename I>
SP_HD bool key_visible(const KvTile& k, const UnitPol& u, I i, int c, I table_pos) {
    if (c >= k.nvalid) return false;
    if (k.full) return true;
    const I p = k.table ? table_pos : (I)k.start + (I)c;
    if (p < 0 || p > i) return false;
    if (u.kind == kLocal) return p < (I)u.sink || p > i - (I)u.window;
    return true;
}


// Bits [0, n) set, n clamped to [0, 32].
SP_HD uint32_t low_bits32(int64_t n) {
    return n <= 0 ? 0u : n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
}

// Visibility bits of a paged (history) tile for the query at position i
// (key c -> bit c % 32 of vm[c / 32]); the unit holds n_b <= i tokens, so
// every stored position is below i.  GLOBAL and RETRIEVAL slots and LOCAL
// sink slots are seen by every row: the tile's first nvalid keys.  LOCAL
// ring slots hold consecutive positions with one break at the ring's newest
// slot h (newest = n_b - 1 - sink = K * ring_slots + h, see slot_position):
// A + c up to the break, A - ring_slots + c after it (slots not yet written
// when K = 0); a row sees those at or after i - window + 1.  Same bits as
// key_visible on the slots' positions.  Positions and slots fit in 32 bits.
SP_HD void paged_row_mask(const KvTile& k, const UnitPol& u, int32_t n_b, int32_t i, int P,
                          uint32_t (&vm)[4]) {
    const int32_t base = u.sink_pages * P, start = (int32_t)k.start;
    if (u.kind != kLocal || start < base) {
        for (int w = 0; w < 4; ++w) vm[w] = low_bits32((int64_t)k.nvalid - 32 * w);
        return;
    }
    const int32_t rs = u.ring * P, q0 = start - base, newest = n_b - 1 - u.sink;
    const int32_t K = newest / rs, h = newest - K * rs;     // a ring tile exists: newest >= 0
    const int64_t A = (int64_t)u.sink + (int64_t)K * rs + q0;   // position of key 0, before the break
    const int64_t lo = (int64_t)i - u.window + 1;                // oldest position the row sees
    const int64_t brk = min64(max64((int64_t)h - q0 + 1, 0), 128);
    const int64_t v1 = min64(max64(lo - A, 0), 128);
    const int64_t v2 = K > 0 ? min64(max64(lo - (A - rs), 0), 128) : 128;
    for (int w = 0; w < 4; ++w) {
        const uint32_t before = low_bits32(brk - 32 * w);
        vm[w] = low_bits32((int64_t)k.nvalid - 32 * w) &
                ((before & ~low_bits32(v1 - 32 * w)) | (~before & ~low_bits32(v2 - 32 * w)));
    }
}

}  // namespace sp
