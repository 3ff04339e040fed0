// sp_rules.h -- the storage and visibility rules of the head-aware paged KV
// cache, as __host__ __device__ functions shared by the host planner and the
// kernels (one definition for both sides).
//
// Head classes and their visible sets follow the RedKnot SegPagedAttention
// runtime article, section 2 (GLOBAL: the whole history; LOCAL: sink tokens
// plus a recent window; RETRIEVAL: selected tokens); the storage follows its
// section 3 (per-head page lists in one pool; a local head keeps only sink and
// recent-window pages, so its page count stops growing with the context).
//
// Slot layout of one unit (= one (sequence, layer, KV head)); a "unit slot"
// is page_index * P + slot_in_page:
//   GLOBAL      token t at unit slot t.
//   LOCAL       t < sink at unit slot t (sink pages = ceil(sink / P));
//               t >= sink at sink_pages*P + (t - sink) mod (ring*P), with
//               ring = ceil(window / P) + 1 pages; newer tokens overwrite.
//   RETRIEVAL   only t in idx, at unit slot rank(t) (its index in idx).
// A unit holding n tokens owns exactly unit_pages(n) pages.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define SP_HD __host__ __device__ __forceinline__
#else
#define SP_HD inline
#endif

namespace sp {

enum : int32_t { kGlobal = 0, kLocal = 1, kRetrieval = 2 };

// Device/host record of one unit's policy (32 bytes).
struct UnitPol {
    int32_t kind;
    int32_t sink;
    int32_t window;
    int32_t ring;        // LOCAL: ring pages = ceil(window / P) + 1
    int32_t sink_pages;  // LOCAL: ceil(sink / P)
    int32_t idx_off;     // RETRIEVAL: offset of the list in the sequence's index area
    int32_t n_idx;       // RETRIEVAL: list length
    int32_t pad;
};

SP_HD int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
SP_HD int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
SP_HD int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// Number of list entries below n (lower bound in an ascending list).
SP_HD int64_t count_below(const int32_t* idx, int64_t n_idx, int64_t n) {
    int64_t lo = 0, hi = n_idx;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)idx[mid] < n) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Pages a unit owns once it holds n tokens.
SP_HD int64_t unit_pages(const UnitPol& u, const int32_t* idx, int64_t n, int P) {
    if (n <= 0) return 0;
    if (u.kind == kGlobal) return cdiv64(n, P);
    if (u.kind == kLocal) {
        const int64_t sink_part = cdiv64(min64(n, u.sink), P);
        const int64_t ring_part = min64((int64_t)u.ring, cdiv64(max64(0, n - u.sink), P));
        return sink_part + ring_part;
    }
    return cdiv64(count_below(idx, u.n_idx, n), P);
}

// Unit slot token t is written to, or -1 if the unit does not store it.
SP_HD int64_t unit_slot(const UnitPol& u, const int32_t* idx, int64_t t, int P) {
    if (u.kind == kGlobal) return t;
    if (u.kind == kLocal) {
        if (t < u.sink) return t;
        const int64_t ring_slots = (int64_t)u.ring * P;
        return (int64_t)u.sink_pages * P + (t - u.sink) % ring_slots;
    }
    const int64_t k = count_below(idx, u.n_idx, t);
    return (k < u.n_idx && idx[k] == t) ? k : -1;
}

// Token held by unit slot us once the unit holds n tokens (-1 = empty).
SP_HD int64_t slot_position(const UnitPol& u, const int32_t* idx, int64_t us,
                            int64_t n, int P) {
    if (u.kind == kGlobal) return us < n ? us : -1;
    if (u.kind == kLocal) {
        const int64_t base = (int64_t)u.sink_pages * P;
        if (us < base) return us < min64(n, u.sink) ? us : -1;
        const int64_t q = us - base;
        const int64_t ring_slots = (int64_t)u.ring * P;
        if (q >= ring_slots) return -1;
        const int64_t newest = n - 1 - u.sink;      // largest offset t - sink written
        if (newest < q) return -1;
        return u.sink + q + ((newest - q) / ring_slots) * ring_slots;
    }
    const int64_t cnt = count_below(idx, u.n_idx, n);
    return us < cnt ? (int64_t)idx[us] : -1;
}

// Tokens of [n_old, n_new) the unit keeps after the write, as up to two
// ranges of "items".  For GLOBAL and LOCAL an item is a position; for
// RETRIEVAL an item is a rank into idx (position idx[rank]).
struct ItemRanges { int64_t lo[2], hi[2]; };

SP_HD ItemRanges retained_items(const UnitPol& u, const int32_t* idx,
                                int64_t n_old, int64_t n_new, int P) {
    ItemRanges r;
    r.lo[0] = r.hi[0] = r.lo[1] = r.hi[1] = 0;
    if (u.kind == kGlobal) {
        r.lo[0] = n_old; r.hi[0] = n_new;
    } else if (u.kind == kLocal) {
        // sink tokens, then only the newest ring*P non-sink tokens survive
        r.lo[0] = n_old; r.hi[0] = max64(n_old, min64(n_new, u.sink));
        const int64_t ring_slots = (int64_t)u.ring * P;
        r.lo[1] = max64(max64((int64_t)u.sink, n_new - ring_slots), n_old);
        r.hi[1] = max64(r.lo[1], n_new);
    } else {
        r.lo[0] = count_below(idx, u.n_idx, n_old);
        r.hi[0] = count_below(idx, u.n_idx, n_new);
    }
    return r;
}

// Visible unit-slot ranges of a query at position t when the unit holds
// n >= t + 1 tokens and the visible tokens all live in the unit (decode).
// At most three ranges (sink, and a ring window that may wrap once).
struct SlotRanges { int64_t lo[3], hi[3]; int count; };

SP_HD SlotRanges decode_ranges(const UnitPol& u, const int32_t* idx, int64_t t, int P) {
    SlotRanges r;
    r.count = 0;
    for (int k = 0; k < 3; ++k) r.lo[k] = r.hi[k] = 0;
    if (t < 0) return r;
    if (u.kind == kGlobal) {
        r.lo[0] = 0; r.hi[0] = t + 1; r.count = 1;
    } else if (u.kind == kLocal) {
        const int64_t sink_end = min64(u.sink, t + 1);
        if (sink_end > 0) { r.lo[r.count] = 0; r.hi[r.count] = sink_end; ++r.count; }
        const int64_t w0 = max64(max64(t - u.window + 1, 0), sink_end);
        if (w0 <= t) {
            const int64_t base = (int64_t)u.sink_pages * P;
            const int64_t ring_slots = (int64_t)u.ring * P;
            const int64_t q0 = (w0 - u.sink) % ring_slots;
            const int64_t len = t - w0 + 1;
            if (q0 + len <= ring_slots) {
                r.lo[r.count] = base + q0; r.hi[r.count] = base + q0 + len; ++r.count;
            } else {
                r.lo[r.count] = base + q0; r.hi[r.count] = base + ring_slots; ++r.count;
                r.lo[r.count] = base; r.hi[r.count] = base + q0 + len - ring_slots; ++r.count;
            }
        }
    } else {
        const int64_t cnt = count_below(idx, u.n_idx, t + 1);
        if (cnt > 0) { r.lo[0] = 0; r.hi[0] = cnt; r.count = 1; }
    }
    return r;
}

// |V(i)| of a query at position i (any i >= 0), from the class definition.
SP_HD int64_t visible_count(const UnitPol& u, const int32_t* idx, int64_t i) {
    if (i < 0) return 0;
    if (u.kind == kGlobal) return i + 1;
    if (u.kind == kLocal) return min64(i + 1, (int64_t)u.sink + u.window);
    return count_below(idx, u.n_idx, i + 1);
}

// Pages a set of slot ranges touches (one decode work item per page piece).
SP_HD int64_t range_pages(int64_t lo, int64_t hi, int P) {
    return hi > lo ? (hi - 1) / P - lo / P + 1 : 0;
}

SP_HD int64_t decode_items(const SlotRanges& r, int P) {
    int64_t n = 0;
    for (int k = 0; k < r.count; ++k) n += range_pages(r.lo[k], r.hi[k], P);
    return n;
}

}  // namespace sp
