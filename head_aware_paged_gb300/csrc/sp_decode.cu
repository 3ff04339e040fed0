// sp_decode.cu -- split-KV decode over each head's own visible pages.
//
// One query per sequence reads, for every (sequence, KV head) unit, only the
// pages holding that head's visible tokens (RedKnot SegPagedAttention runtime
// article section 4: each head attends over its own page table, no mask;
// section 5: decode is where the saving grows with the context).  Decode is
// HBM-bound (KV-cache tutorial section 3.3), so the design goal is a
// continuous, balanced page stream:
//
//   * The visible pages of all units of the call form one list of work items
//     (one item = one page with a valid slot range).  The persistent grid
//     splits that list evenly: CTA c streams items [T c / G, T (c+1) / G), so
//     every SM reads the same number of pages whatever the head classes.
//   * One producer lane streams the pages with 2D TMA loads (128-byte
//     swizzle) into a ring of shared-memory stages; each stage belongs to one
//     of the consumer warps, which takes the whole page (blocks of 32 keys)
//     and computes QK^T and PV for all query heads of the KV head at once
//     with mma.sync m16n8k16 (rows = query heads, so each K/V byte is read
//     once for the whole GQA group), with an online softmax in registers
//     (tutorial section 10.2) and deferred normalisation (section 10.4).
//     The warps' partial states are merged at the end of each unit.
//   * Where a unit's items span several CTAs (split-KV), each CTA writes an
//     unnormalised partial (o, m, l); the last CTA to finish the unit (atomic
//     ticket, no waiting) merges them: m* = max m_s, l* = sum 2^(m_s-m*) l_s,
//     O = sum 2^(m_s-m*) o_s / l*.
#include "sp_internal.h"
#include "sp_device.cuh"

namespace sp {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 12;

template <int D, int P, bool F8 = false>
struct DecodeShape {
    static constexpr int kElem = F8 ? 1 : 2;            // bytes per stored element
    static constexpr int kHalves = D * kElem / 128;     // 128-byte column blocks per row
    // FP8 pages of 64 or more keys stream as two stages of half a page: twice
    // the stages in the same memory, so every consumer warp owns three and
    // has two in flight while it computes one (whole 8 KB-per-K pages gave
    // six stages, three owner warps, one page in flight each)
    static constexpr int kSub = (F8 && P >= 64) ? 2 : 1;   // stages per page
    static constexpr int kStageKeys = P / kSub;
    static constexpr int kHalfBytes = kStageKeys * 128;
    static constexpr int kTileBytes = kHalves * kHalfBytes;   // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    // FP8 runs two CTAs per SM (twice the warps to hide the per-block
    // latency chain), each with half the stage memory
    static constexpr int kCtasPerSm = F8 ? 2 : 1;
    // Shared memory a CTA may use: all of an SM's, or half of it for two CTAs.
    // The stages get what the merge buffers (sized by the call's group and
    // grid) and the barriers leave, up to kMaxStages; bf16 stages are capped
    // at 192 KB (six 32 KB stages at P = 64, owned by three warps).
    static constexpr int kSmemCap = F8 ? 113 * 1024 : 227 * 1024;
    static constexpr int kStageCap = F8 ? kSmemCap : 192 * 1024;
    static constexpr int kMiscBytes = kMaxStages * 16 /*full, empty*/ + kMaxStages * 16 /*desc*/
                                      + 16 /*flags*/ + 32 * 16 /*producer batch*/
                                      + 16 /*barrier alignment*/ + 1024 /*base alignment*/;
};

__device__ __forceinline__ int64_t cta_of_item(int64_t x, int64_t T, int G) {
    return (x * G + G - 1) / T;
}

template <int D, int P, bool F8>
__global__ void __launch_bounds__(kDecodeThreads, F8 ? 2 : 1)
k_decode(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmK,
         const __grid_constant__ CUtensorMap tmV) {
    using S = DecodeShape<D, P, F8>;
    const int NST = p.nst;
    constexpr int BK = P >= 32 ? 32 : 16;     // keys per warp block
    constexpr int NT = BK / 8;                // S n-tiles per block
    constexpr int NB = S::kStageKeys / BK;    // blocks per stage (1, 2 or 4)
    static_assert(NB == 1 || NB == 2 || NB == 4, "blocks per page must divide the warp count");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;
    // merge_o: [4][group][D] partial outputs, later [2][grid][group] merge weights
    float* merge_o = reinterpret_cast<float*>(smem + NST * S::kStageBytes);
    float* merge_ml = merge_o + p.merge_floats;                               // [4][group][2]
    uint64_t* full = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(merge_ml + kConsumerWarps * p.geo.group * 2) + 15) & ~uintptr_t(15));
    uint64_t* empty = full + NST;
    int4* desc = reinterpret_cast<int4*>(empty + NST);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(desc + NST);
    int* flag_last = const_cast<int*>(abort_flag) + 1;
    int4* batch = reinterpret_cast<int4*>(const_cast<int*>(abort_flag) + 4);   // [32] producer batch

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int64_t T = p.total_items;
    const int64_t x0 = T * c / G, x1 = T * (c + 1) / G;
    const Geo& g = p.geo;
    const int group = g.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }   // one consumer warp per page
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: stream this CTA's pages ----------------
        // The warp resolves the pages of 32 work items at a time (one per lane:
        // unit, policy, visible ranges, page-table entry -- dependent global
        // loads whose latency the lanes overlap), then lane 0 waits for free
        // stages and issues the TMA loads in item order.
        if (x0 < x1) {
            if (lane == 0) { prefetch_tmap(&tmK); prefetch_tmap(&tmV); }
            int issued = 0;
            int ps = 0;               // stage of the next load
            uint32_t pk = 0;          // times that stage has been filled before
            for (int64_t base = x0; base < x1; base += 32) {
                const int64_t x = base + lane;
                if (x < x1) {
                    int lo_u = 0, hi_u = p.n_units - 1;      // unit holding item x
                    while (lo_u < hi_u) {
                        const int mid = (lo_u + hi_u) >> 1;
                        if (p.item_off[mid + 1] <= x) lo_u = mid + 1; else hi_u = mid;
                    }
                    const int u = lo_u;
                    const int b = u / g.hkv, h = u % g.hkv;
                    const int seq = p.seq[b];
                    const int64_t row = g.unit_row(seq, p.layer, h);
                    const UnitPol pol = p.meta.pol[row];
                    const int32_t* idx = p.meta.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
                    const SlotRanges rg = decode_ranges(pol, idx, p.tq[b], P);
                    int64_t j = x - p.item_off[u];
                    int64_t pidx = 0, lo = 0, hi = 0;
                    for (int q = 0; q < rg.count; ++q) {
                        const int64_t np = range_pages(rg.lo[q], rg.hi[q], P);
                        if (j < np) {
                            pidx = rg.lo[q] / P + j;
                            lo = max64(rg.lo[q], pidx * P) - pidx * P;
                            hi = min64(rg.hi[q], (pidx + 1) * P) - pidx * P;
                            break;
                        }
                        j -= np;
                    }
                    int32_t page = p.meta.ptab[row * g.max_pages_unit + pidx];
                    if (page < 0 || page >= g.num_pages) {
                        atomicOr(p.meta.status, kStatusBadPage);
                        page = 0; lo = hi = 0;          // load something harmless, use nothing
                    }
                    batch[lane] = make_int4(u, (int)lo | ((int)hi << 16), page, 0);
                }
                __syncwarp();
                if (lane == 0) {
                    const int n = (int)min64(32, x1 - base);
                    bool stop = false;
                    for (int i = 0; i < n && !stop; ++i) {
                        const int4 bi = batch[i];
                        const int lo = bi.y & 0xFFFF, hi = bi.y >> 16;
                        #pragma unroll
                        for (int sub = 0; sub < S::kSub; ++sub) {
                            if (pk > 0 && !mbar_wait(&empty[ps], (pk - 1) & 1, abort_flag, p.meta.status)) {
                                stop = true;
                                break;
                            }
                            // this stage's slot range, relative to its first key
                            const int k0 = sub * S::kStageKeys;
                            const int slo = max(lo - k0, 0), shi = min(hi - k0, S::kStageKeys);
                            desc[ps] = make_int4(bi.x, slo < shi ? slo | (shi << 16) : 0, bi.w, 0);
                            if (slo < shi) {
                                mbar_arrive_expect_tx(&full[ps], S::kStageBytes);
                                uint8_t* kdst = stages + ps * S::kStageBytes;
                                uint8_t* vdst = kdst + S::kTileBytes;
                                #pragma unroll
                                for (int hh = 0; hh < S::kHalves; ++hh) {
                                    tma_load_2d(kdst + hh * S::kHalfBytes, &tmK, &full[ps], hh * 64, bi.z * P + k0);
                                    tma_load_2d(vdst + hh * S::kHalfBytes, &tmV, &full[ps], hh * 64, bi.z * P + k0);
                                }
                            } else {
                                mbar_arrive(&full[ps]);     // no visible slot: nothing to load
                            }
                            ++issued;
                            if (++ps == NST) { ps = 0; ++pk; }
                        }
                    }
                }
                __syncwarp();
                if (*abort_flag) break;
            }
            // Leave only after every load this CTA issued has landed (bounded,
            // also after an abort).
            if (lane == 0) {
                for (int s = 0; s < NST && s < issued; ++s) {
                    const int last_k = (issued - 1 - s) / NST;
                    mbar_wait(&full[s], (uint32_t)(last_k & 1), nullptr, nullptr);
                }
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int ctid = threadIdx.x;     // 0..127
    // Units with no visible token: O = 0, LSE = -inf (one CTA each).
    for (int u = c; u < p.n_units; u += G) {
        if (p.item_off[u + 1] != p.item_off[u]) continue;
        const int b = u / g.hkv, h = u % g.hkv;
        for (int e = ctid; e < group * D; e += kConsumerWarps * 32) {
            const int r = e / D, col = e % D;
            p.out[((int64_t)b * g.hq + h * group + r) * D + col] = __float2bfloat16(0.f);
            if (col == 0 && p.lse) p.lse[(int64_t)b * g.hq + h * group + r] = -INFINITY;
        }
    }
    if (x0 >= x1) return;

    const int qr = lane >> 2, qc = (lane & 3) * 2;   // fragment row / column base
    uint32_t qa[D / 16][4];
    float m_run[2], l_run[2];
    float o_acc[D / 8][4];
    // Consumer warp w < W takes stages w, w+W, w+2W, ... of this CTA's stream
    // (whole pages, or half pages for FP8), so a warp only handles the keys
    // it computes.  W divides
    // the stage count (the launcher makes NST a multiple of 4, or W = NST
    // below 4 stages), so stage s always belongs to warp s % W and each warp
    // waits for its stages' fills in order -- never for a fill two phases
    // ahead.  All four warps walk the same list of units and merge at the
    // end of each, whatever their own pages were; after a failed wait a warp
    // only keeps walking, so that every merge barrier still sees all four.
    const int W = p.owners;
    const bool owner = warp < W;
    int xi = warp;                    // this warp's next stage fill, relative to x0 * kSub
    int s = warp;                     // its stage (xi % NST)
    uint32_t rounds = 0;              // times that stage has been filled before
    bool dead = false;
    int u_lo = 0, u_hi = p.n_units - 1;     // first unit with an item >= x0
    while (u_lo < u_hi) {
        const int mid = (u_lo + u_hi) >> 1;
        if (p.item_off[mid + 1] <= x0) u_lo = mid + 1; else u_hi = mid;
    }
    for (int u = u_lo; u < p.n_units && p.item_off[u] < x1; ++u) {
        const int64_t ua = max64(p.item_off[u], x0), ub = min64(p.item_off[u + 1], x1);
        if (ua >= ub) continue;       // no pages (handled above) or none in this CTA
        const int b = u / g.hkv, h = u - (u / g.hkv) * g.hkv;
        {
            const __nv_bfloat16* qb = p.q + ((int64_t)b * g.hq + h * group) * D;
            auto ld = [&](int r, int cc) -> uint32_t {
                return r < group ? *reinterpret_cast<const uint32_t*>(qb + (int64_t)r * D + cc) : 0u;
            };
            if constexpr (F8) {
                // q * k_scale as f16 (q . (code * s) = (q * s) . code), with
                // the reduction index of step kk, lane quad j mapped to dims
                // j*32 + kk*4 + {0,1 | 2,3}: one 32-bit word of a key's codes
                // then feeds both halves of the B fragment
                const float* ks = p.meta.kscale + ((int64_t)p.layer * g.hkv + h) * D;
                auto ldq = [&](int r, int cc) -> uint32_t {
                    const uint32_t w = ld(r, cc);
                    const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w);
                    return pack_f16(__low2float(v2) * ks[cc], __high2float(v2) * ks[cc + 1]);
                };
                const int j = lane & 3;
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int col = j * 32 + kk * 4;
                    qa[kk][0] = ldq(qr, col);
                    qa[kk][1] = ldq(qr + 8, col);
                    qa[kk][2] = ldq(qr, col + 2);
                    qa[kk][3] = ldq(qr + 8, col + 2);
                }
            } else {
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const int col = kk * 16 + qc;
                    qa[kk][0] = ld(qr, col);
                    qa[kk][1] = ld(qr + 8, col);
                    qa[kk][2] = ld(qr, col + 8);
                    qa[kk][3] = ld(qr + 8, col + 8);
                }
            }
            m_run[0] = m_run[1] = -INFINITY;
            l_run[0] = l_run[1] = 0.f;
            #pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                #pragma unroll
                for (int e = 0; e < 4; ++e) o_acc[nt][e] = 0.f;
        }
        for (; owner && x0 * S::kSub + xi < ub * S::kSub; xi += W) {
        if (!dead && !mbar_wait(&full[s], rounds & 1, abort_flag, p.meta.status)) dead = true;
        if (dead) continue;
        const int4 dd = desc[s];
        const int lo = dd.y & 0xFFFF, hi = dd.y >> 16;
        if (dd.x != u && lane == 0) atomicOr(p.meta.status, kStatusBadState);
        const uint32_t kbase = smem_u32(stages + s * S::kStageBytes);
        const uint32_t vbase = kbase + S::kTileBytes;
        #pragma unroll 1
        for (int blk = 0; blk < NB; ++blk) {
        const int key0 = blk * BK;
        if (key0 < hi && key0 + BK > lo) {
            // S = Q K^T for BK keys: NT n-tiles of 8 keys
            float sc[NT][4];
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            if constexpr (F8) {
                // B fragments straight from the codes: lane (n, j) reads bytes
                // j*32 .. j*32+31 of key n of each n-tile; word kk of them is
                // dims j*32 + kk*4 .. +3 (e4m3 -> f16 is exact)
                const uint8_t* tk = stages + s * S::kStageBytes;
                const int j = lane & 3, n = lane >> 2;
                uint32_t w[NT][8];
                #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int key = key0 + nt * 8 + n;
                    const uint4 c0 = *reinterpret_cast<const uint4*>(tk + sw128(key, 2 * j));
                    const uint4 c1 = *reinterpret_cast<const uint4*>(tk + sw128(key, 2 * j + 1));
                    w[nt][0] = c0.x; w[nt][1] = c0.y; w[nt][2] = c0.z; w[nt][3] = c0.w;
                    w[nt][4] = c1.x; w[nt][5] = c1.y; w[nt][6] = c1.z; w[nt][7] = c1.w;
                }
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        uint32_t b0, b1;
                        f16x2x2_of_e4m3x4(w[nt][kk], b0, b1);
                        mma_f16_16816(sc[nt], qa[kk], b0, b1);
                    }
            } else {
                const int mi = lane >> 3;
                #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t chunk = kk * 2 + (mi & 1);
                    #pragma unroll
                    for (int hb = 0; hb < NT / 2; ++hb) {
                        const uint32_t key = key0 + hb * 16 + (lane & 7) + (mi >= 2 ? 8 : 0);
                        const uint32_t addr = kbase + (chunk >> 3) * S::kHalfBytes + sw128(key, chunk & 7);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(addr, r0, r1, r2, r3);
                        mma_bf16_16816(sc[2 * hb], qa[kk], r0, r1);
                        mma_bf16_16816(sc[2 * hb + 1], qa[kk], r2, r3);
                    }
                }
            }
            // scale to log2 units, mask keys outside [lo, hi) (only for a
            // block that straddles the range), online softmax
            float mx[2] = {-INFINITY, -INFINITY};
            if (key0 >= lo && key0 + BK <= hi) {
                #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        sc[nt][e] *= p.scale_log2;
                        mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
                    }
            } else {
                #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + nt * 8 + qc + (e & 1);
                        float v = sc[nt][e] * p.scale_log2;
                        if (key < lo || key >= hi) v = -INFINITY;
                        sc[nt][e] = v;
                        mx[e >> 1] = fmaxf(mx[e >> 1], v);
                    }
            }
            #pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            }
            // rescale the running state only when a row's maximum grows
            // (otherwise the factor is exactly 1)
            if (__any_sync(0xffffffffu, mx[0] > m_run[0] || mx[1] > m_run[1])) {
                #pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float m_new = fmaxf(m_run[r], mx[r]);
                    const float alpha = fast_exp2(m_run[r] - (m_new == -INFINITY ? 0.f : m_new));
                    m_run[r] = m_new;
                    l_run[r] *= alpha;
                    #pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt) {
                        o_acc[nt][2 * r] *= alpha;
                        o_acc[nt][2 * r + 1] *= alpha;
                    }
                }
            }
            const float mbase[2] = {m_run[0] == -INFINITY ? 0.f : m_run[0],
                                    m_run[1] == -INFINITY ? 0.f : m_run[1]};
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pv = fast_exp2(sc[nt][e] - mbase[e >> 1]);
                    sc[nt][e] = pv;
                    l_run[e >> 1] += pv;
                }
            // O += P V, 16 keys at a time: P from the S fragments (rows = heads)
            #pragma unroll
            for (int hb = 0; hb < NT / 2; ++hb) {
                uint32_t pa[4];
                if constexpr (F8) {
                    pa[0] = pack_f16(sc[2 * hb][0], sc[2 * hb][1]);
                    pa[1] = pack_f16(sc[2 * hb][2], sc[2 * hb][3]);
                    pa[2] = pack_f16(sc[2 * hb + 1][0], sc[2 * hb + 1][1]);
                    pa[3] = pack_f16(sc[2 * hb + 1][2], sc[2 * hb + 1][3]);
                    // The output dims of n-tile nt, column n are n*16 + nt, so
                    // lane (n, j) needs dims n*16 .. n*16+15 (chunk n) of keys
                    // 2j, 2j+1, 2j+8, 2j+9; byte interleaves pair consecutive
                    // keys per dim.  V's scales are applied to the finished sums.
                    const uint8_t* tv = stages + s * S::kStageBytes + S::kTileBytes;
                    const int j = lane & 3, n = lane >> 2, kb = key0 + hb * 16 + 2 * j;
                    const uint4 r0 = *reinterpret_cast<const uint4*>(tv + sw128(kb, n));
                    const uint4 r1 = *reinterpret_cast<const uint4*>(tv + sw128(kb + 1, n));
                    const uint4 r8 = *reinterpret_cast<const uint4*>(tv + sw128(kb + 8, n));
                    const uint4 r9 = *reinterpret_cast<const uint4*>(tv + sw128(kb + 9, n));
                    const uint32_t a0[4] = {r0.x, r0.y, r0.z, r0.w}, a1[4] = {r1.x, r1.y, r1.z, r1.w};
                    const uint32_t a8[4] = {r8.x, r8.y, r8.z, r8.w}, a9[4] = {r9.x, r9.y, r9.z, r9.w};
                    #pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {     // dims n*16 + 4wd .. +3: n-tiles 4wd .. 4wd+3
                        uint32_t lo0, lo1, lo2, lo3, hi0, hi1, hi2, hi3;
                        f16x2x2_of_e4m3x4(prmt(a0[wd], a1[wd], 0x5140u), lo0, lo1);   // bytes 0,1
                        f16x2x2_of_e4m3x4(prmt(a0[wd], a1[wd], 0x7362u), lo2, lo3);   // bytes 2,3
                        f16x2x2_of_e4m3x4(prmt(a8[wd], a9[wd], 0x5140u), hi0, hi1);
                        f16x2x2_of_e4m3x4(prmt(a8[wd], a9[wd], 0x7362u), hi2, hi3);
                        mma_f16_16816(o_acc[4 * wd + 0], pa, lo0, hi0);
                        mma_f16_16816(o_acc[4 * wd + 1], pa, lo1, hi1);
                        mma_f16_16816(o_acc[4 * wd + 2], pa, lo2, hi2);
                        mma_f16_16816(o_acc[4 * wd + 3], pa, lo3, hi3);
                    }
                } else {
                    pa[0] = pack_bf16(sc[2 * hb][0], sc[2 * hb][1]);
                    pa[1] = pack_bf16(sc[2 * hb][2], sc[2 * hb][3]);
                    pa[2] = pack_bf16(sc[2 * hb + 1][0], sc[2 * hb + 1][1]);
                    pa[3] = pack_bf16(sc[2 * hb + 1][2], sc[2 * hb + 1][3]);
                    const int mi = lane >> 3;
                    const uint32_t key = key0 + hb * 16 + (lane & 7) + ((mi & 1) ? 8 : 0);
                    #pragma unroll
                    for (int np = 0; np < D / 16; ++np) {
                        const uint32_t chunk = np * 2 + (mi >> 1);
                        const uint32_t addr = vbase + (chunk >> 3) * S::kHalfBytes + sw128(key, chunk & 7);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_t(addr, r0, r1, r2, r3);
                        mma_bf16_16816(o_acc[2 * np], pa, r0, r1);
                        mma_bf16_16816(o_acc[2 * np + 1], pa, r2, r3);
                    }
                }
            }
        }
        }   // blocks of the page
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        s += W;
        if (s >= NST) { s -= NST; ++rounds; }
        }   // this warp's pages of the unit

        // ------------- merge the four warps' partial states -------------
        #pragma unroll
        for (int r = 0; r < 2; ++r) {
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
            l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        }
        #pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = qr + 8 * r;
            if (row < group) {
                float* mo = merge_o + ((size_t)warp * group + row) * D;
                if constexpr (F8) {       // column c of n-tile nt is dim c*16 + nt; times V's scale
                    const float* vs = p.meta.vscale + ((int64_t)p.layer * g.hkv + h) * D;
                    #pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt) {
                        const int d0 = qc * 16 + nt, d1 = (qc + 1) * 16 + nt;
                        mo[d0] = o_acc[nt][2 * r] * vs[d0];
                        mo[d1] = o_acc[nt][2 * r + 1] * vs[d1];
                    }
                } else {
                    #pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt) {
                        mo[nt * 8 + qc] = o_acc[nt][2 * r];
                        mo[nt * 8 + qc + 1] = o_acc[nt][2 * r + 1];
                    }
                }
                if ((lane & 3) == 0) {
                    merge_ml[(warp * group + row) * 2] = m_run[r];
                    merge_ml[(warp * group + row) * 2 + 1] = l_run[r];
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));

        const int64_t ia = p.item_off[u], ib = p.item_off[u + 1];
        const int c_first = (int)cta_of_item(ia, T, G), c_last = (int)cta_of_item(ib - 1, T, G);
        const bool whole = c_first == c_last;
        const int64_t part = (int64_t)u + c;
        for (int e = ctid; e < group * D; e += kConsumerWarps * 32) {
            const int r = e / D, col = e % D;
            float mst = -INFINITY;
            #pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mst = fmaxf(mst, merge_ml[(w * group + r) * 2]);
            float lst = 0.f, ost = 0.f;
            #pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float sc_w = fast_exp2(merge_ml[(w * group + r) * 2] - mst);
                lst += sc_w * merge_ml[(w * group + r) * 2 + 1];
                ost += sc_w * merge_o[((size_t)w * group + r) * D + col];
            }
            const int64_t orow = (int64_t)b * g.hq + h * group + r;
            if (whole) {
                p.out[orow * D + col] = __float2bfloat16(ost / lst);
                if (col == 0 && p.lse) p.lse[orow] = (mst + __log2f(lst)) * 0.69314718055994531f;
            } else {
                p.part_o[(part * group + r) * D + col] = ost;
                if (col == 0) {
                    p.part_ml[(part * group + r) * 2] = mst;
                    p.part_ml[(part * group + r) * 2 + 1] = lst;
                }
            }
        }
        if (!whole) {
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
            if (ctid == 0) {
                int target = 0;
                for (int cc = c_first; cc <= c_last; ++cc)
                    target += (T * cc / G) < (T * (cc + 1) / G) ? 1 : 0;
                const int old = atomicAdd(&p.counters[u], 1);
                *flag_last = (old == target - 1) ? 1 : 0;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
            if (*flag_last) {
                // Merge the unit's partials.  Segment sg is CTA c_first + sg
                // (skipped if its item range is empty).  Stage the (m, l) pairs in
                // shared memory (the intra-CTA merge buffers are free now), turn
                // them into weights 2^(m - m*), then sum the weighted partial
                // outputs with several independent loads in flight per thread.
                __threadfence();
                const int nseg = c_last - c_first + 1;
                float* wts = merge_o;                          // [nseg][group] weights
                float* mls = merge_o + p.merge_floats / 2;     // [nseg][group] l
                float* mstar = merge_ml;                       // [group] m*, then 1 / l*
                for (int e = ctid; e < nseg * group; e += kConsumerWarps * 32) {
                    const int sg = e / group, r = e % group;
                    const int cc = c_first + sg;
                    const bool live = (T * cc / G) < (T * (cc + 1) / G);
                    const int64_t pi = (int64_t)u + cc;
                    wts[e] = live ? __ldcg(&p.part_ml[(pi * group + r) * 2]) : -INFINITY;
                    mls[e] = live ? __ldcg(&p.part_ml[(pi * group + r) * 2 + 1]) : 0.f;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
                if (ctid < group) {
                    const int r = ctid;
                    float mst = -INFINITY;
                    for (int sg = 0; sg < nseg; ++sg) mst = fmaxf(mst, wts[sg * group + r]);
                    float lst = 0.f;
                    for (int sg = 0; sg < nseg; ++sg) {
                        const float w = fast_exp2(wts[sg * group + r] - mst);
                        wts[sg * group + r] = w;
                        lst += w * mls[sg * group + r];
                    }
                    mstar[2 * r] = mst;
                    mstar[2 * r + 1] = lst;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
                for (int e = ctid; e < group * D; e += kConsumerWarps * 32) {
                    const int r = e / D, col = e % D;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    int sg = 0;
                    for (; sg + 4 <= nseg; sg += 4) {
                        float v4[4];
                        #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float w = wts[(sg + q) * group + r];
                            const int64_t pi = (int64_t)u + c_first + sg + q;
                            v4[q] = w != 0.f ? __ldcg(&p.part_o[(pi * group + r) * D + col]) * w : 0.f;
                        }
                        #pragma unroll
                        for (int q = 0; q < 4; ++q) acc[q] += v4[q];
                    }
                    for (; sg < nseg; ++sg) {
                        const float w = wts[sg * group + r];
                        const int64_t pi = (int64_t)u + c_first + sg;
                        if (w != 0.f) acc[0] += w * __ldcg(&p.part_o[(pi * group + r) * D + col]);
                    }
                    const float ost = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                    const float lst = mstar[2 * r + 1];
                    const int64_t orow = (int64_t)b * g.hq + h * group + r;
                    p.out[orow * D + col] = __float2bfloat16(ost / lst);
                    if (col == 0 && p.lse) p.lse[orow] = (mstar[2 * r] + __log2f(lst)) * 0.69314718055994531f;
                }
                if (ctid == 0) p.counters[u] = 0;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));
    }
}

template <int D, int P, bool F8 = false>
cudaError_t launch_decode_t(const sp_cache* c, DecodeParams& p, int grid, cudaStream_t s) {
    using Sh = DecodeShape<D, P, F8>;
    // merge buffer: the four warps' [group][D] partials, or two [grid][group]
    // arrays for the cross-CTA merge, whichever is larger (a multiple of 4)
    const int group = c->geo.group;
    const int mo = std::max(kConsumerWarps * group * D, 2 * grid * group);
    p.merge_floats = (mo + 3) & ~3;
    const int merge_bytes = (p.merge_floats + kConsumerWarps * group * 2) * 4;
    const int room = std::min(Sh::kStageCap, Sh::kSmemCap - merge_bytes - Sh::kMiscBytes);
    // the deepest ring whose stages split evenly over at least three warps
    // (or over all of them when there are fewer than three stages)
    p.nst = 0;
    for (int n = std::min(kMaxStages, room / Sh::kStageBytes); n >= 2 && p.nst == 0; --n) {
        const int w = n % 4 == 0 ? 4 : n % 3 == 0 ? 3 : n % 2 == 0 ? 2 : 1;
        if (w >= std::min(3, n)) { p.nst = n; p.owners = w; }
    }
    if (p.nst < 2) return cudaErrorInvalidConfiguration;
    const int smem = p.nst * Sh::kStageBytes + merge_bytes + Sh::kMiscBytes;
    cudaError_t e = cudaFuncSetAttribute(k_decode<D, P, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Sh::kSmemCap);
    if (e != cudaSuccess) return e;
    if (Sh::kCtasPerSm > 1) {
        e = cudaFuncSetAttribute(k_decode<D, P, F8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    // the tensor maps' box is one stage's keys: a whole page, or half a page
    const CUtensorMap& tk = Sh::kSub == 2 ? c->tm_kpool_half : c->tm_kpool;
    const CUtensorMap& tv = Sh::kSub == 2 ? c->tm_vpool_half : c->tm_vpool;
    k_decode<D, P, F8><<<grid, kDecodeThreads, smem, s>>>(p, tk, tv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const sp_cache* c, DecodeParams& p, cudaStream_t s) {
    // Persistent grid, but at least kMinItemsPerCta pages per CTA: a small batch
    // then spreads one head over a few CTAs instead of dozens (fewer partials
    // to merge).
    constexpr int64_t kMinItemsPerCta = 8;
    int grid = c->decode_ctas;
    const int64_t want = (p.total_items + kMinItemsPerCta - 1) / kMinItemsPerCta;
    if (want < grid) grid = (int)(want > 0 ? want : 1);
    const int D = c->geo.d, P = c->geo.page;
    if (c->geo.fp8) {   // FP8 pages: head_dim 128 only (checked at create)
        if (D != 128) return cudaErrorInvalidValue;
        if (P == 16) return launch_decode_t<128, 16, true>(c, p, grid, s);
        if (P == 32) return launch_decode_t<128, 32, true>(c, p, grid, s);
        if (P == 64) return launch_decode_t<128, 64, true>(c, p, grid, s);
        if (P == 128) return launch_decode_t<128, 128, true>(c, p, grid, s);
        return cudaErrorInvalidValue;
    }
#define SP_DEC(DD, PP) if (D == DD && P == PP) return launch_decode_t<DD, PP>(c, p, grid, s);
    SP_DEC(64, 16) SP_DEC(64, 32) SP_DEC(64, 64) SP_DEC(64, 128)
    SP_DEC(128, 16) SP_DEC(128, 32) SP_DEC(128, 64) SP_DEC(128, 128)
#undef SP_DEC
    return cudaErrorInvalidValue;
}

}  // namespace sp
