// sp_prefill.cu -- mask-free causal prefill over each head's own visible keys
// (RedKnot SegPagedAttention runtime article section 4: every (query head, KV
// head) pair attends over exactly its own tokens in one fused varlen call, no
// attention mask is built).  The FlashAttention forward recurrence follows the
// KV-cache tutorial section 10.2 (tiling with an online softmax) and 10.4
// (normalise once at the end); its Hopper FA-3 kernel is prior art only.
//
// sm_103a design (one persistent CTA per SM, 12 warps = 3 warpgroups):
//   warp 8       TMA producer: the work item's Q tiles (128 rows of one or two
//                query heads of one KV head), then its K/V tiles from the
//                chunk (2D tensor map) or from cache pages (tensor map over
//                the page pool), 128-byte swizzled, into a ring of stages.
//   warp 9       TMEM owner and tcgen05 MMA issuer (one thread): S_t = Q_t K^T
//                into TMEM, later O_t += P_t V with P_t read from TMEM.
//   warp 10      second MMA issuer (bf16 K/V, head_dim 128, two query tiles:
//                warp 9 issues tile 0's MMAs, warp 10 tile 1's); with FP8
//                history warps 10-11 turn page codes into bf16 stage rows;
//                otherwise idle (the producer/MMA warpgroup gives its
//                registers to the softmax warpgroups with setmaxnreg).
//   warps 0-3    softmax + epilogue of query tile 0; warps 4-7 of tile 1.
//                Each thread owns one query row: it reads its S row from
//                TMEM into registers, masks (only on tiles that need it, see
//                sp_plan.h),
//                keeps the running max / sum, writes P (bf16 pairs) back into
//                TMEM over its S tile, where the PV MMA reads it as the A
//                operand, and rescales its O row in TMEM only when the max
//                grew by more than 2^8 (lazy rescale).
//   The two query tiles share every K/V tile and ping-pong on the tensor core:
//   while one softmax group works, the MMA warp runs the other's PV and next QK.
//   With bf16 K/V and head_dim 128 each query tile has its own issuing thread
//   (warps 9 and 10) and the two take turns block by block.
// Work items are assigned to CTAs on the host, longest first, each to the
// CTA with the least work so far (greedy), so no SM idles at the tail; when
// the call's K/V exceeds about half of L2, one (sequence, KV head) unit after
// another, so the CTAs share one unit's K/V in L2 at a time.  Items much
// longer than a CTA's share are split along their keys into pieces whose
// partial results a small merge kernel combines.
// Every wait is bounded (sp_device.cuh); on a time-out the CTA drains its
// copies and MMAs, frees TMEM and returns with the status word set.
#include <algorithm>
#include <climits>
#include <cmath>
#include <memory>
#include <functional>
#include <utility>
#include <vector>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_plan.h"
#include "sp_prefill.h"
#include "sp_tcgen05.cuh"

namespace sp {

namespace {

constexpr int kPfThreads = 384;        // 3 warpgroups: 2 softmax, 1 producer/MMA
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMmaWarp2 = 10;          // second MMA issuer (bf16 pages, two query tiles)
// Register split between the warpgroups (setmaxnreg).  The block is launched
// with kLaunchRegs per thread (384 threads x 168 = 64512 of the SM's 65536);
// the producer/MMA warpgroup drops to kLowRegs and each softmax warpgroup
// rises to kHighRegs: 2 x 208 + 88 = 3 x 168, so the increase never waits for
// registers that do not exist.  The host checks kLaunchRegs before launching.
constexpr int kLaunchRegs = 168;
constexpr int kHighRegs = 208;
constexpr int kLowRegs = 88;
static_assert(2 * kHighRegs + kLowRegs == 3 * kLaunchRegs, "register split must add up");
constexpr int kSmemLimit = 232448;     // 227 KB per CTA
constexpr int kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;   // lazy-rescale threshold (log2 units)
constexpr int kPrefetchTiles = 3;      // K/V tiles brought into L2 ahead of their loads
// Two MMA issuers: the turn passes this many MMAs before the end of a block
// (1, 2 and 3 measured within 1 % of each other; at the very end, the hand-over
// left the tensor pipe idle: 0.67 instead of 0.73 of peak on 128K calls).
constexpr int kTurnEarly = 2;
constexpr int64_t kSpecTilesPerItem = 32;   // speculative exponentials above this mean item length
constexpr int64_t kTileCost = 160;     // work-assignment cost of one K/V tile
constexpr int64_t kItemCost = 480;     // and of one work item's fixed part
constexpr int kMinPieceTiles = 6;      // key tiles of a piece of a split item, at least
constexpr int64_t kL2UnitOrderBytes = int64_t(64) << 20;   // K/V of a call above which units go in turn

constexpr int kInlineWords = 1344;     // int4 words of work list carried in the parameters
struct PrefillParams {
    Meta meta;
    Geo geo;
    int32_t layer;
    int32_t nq;                  // query tiles per item: 2 (head pairs) or 1
    int32_t n_items;
    float scale_log2;            // log2(e) / sqrt(d)
    // work items {b | first tile << 10, kv head, pair | row block << 8,
    // tiles | (partial slot + 1) << 20}, grouped by CTA
    const int4* items;
    const int32_t* cta_off;      // items of CTA c: [cta_off[c], cta_off[c+1])
    __nv_bfloat16* out;
    float* lse;
    // A piece of an item split along its keys writes its unnormalised O
    // ([slot][query tile][d / 4][128 rows] float4) and its row max / sum
    // ([slot][query tile][128 rows] float2) here; k_prefill_merge combines
    // the pieces.
    float4* split_o;
    float2* split_ml;
    int32_t seq[kMaxCallSeqs];
    int32_t n_b[kMaxCallSeqs];   // tokens held before the chunk
    int32_t cnt[kMaxCallSeqs];   // chunk rows
    int32_t row0[kMaxCallSeqs];  // first chunk row in q / k / v
    // A work list that fits travels inside the parameters (items, then the
    // CTA offsets as int32 packed four to an int4); inline_words = 0 means
    // it was uploaded to items / cta_off.  Inline, the launch carries it and
    // no copy engine is involved, so the kernel never queues behind the
    // caller's own host<->device transfers.
    int32_t inline_words;
    int4 inl[kInlineWords];
};

template <int D, bool F8 = false>
struct PfShape {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = 128 * 128;            // 128 rows x 128 bytes
    static constexpr int kQBytes = kHalves * kHalfBytes;     // one Q tile
    static constexpr int kKVBytes = kHalves * kHalfBytes;    // one K or V tile
    // FP8 history pages land in one of two code slots (128 keys x 128 bytes)
    // before the converter warps write them into a bf16 stage
    static constexpr int kF8Slot = 128 * 128;
    static constexpr int kFixed = 2 * kQBytes + (F8 ? 2 * kF8Slot : 0);
    static constexpr int kMisc = 2048;                       // barriers, flags, alignment slack
    static constexpr int kStagesFit = (kSmemLimit - kFixed - kMisc) / kKVBytes;
    static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
    static constexpr int kSmem = kFixed + kStages * kKVBytes + kMisc;
    static_assert(kStages >= 2, "not enough shared memory for two K/V stages");
};

struct Item {
    int b, kvh, h0, rows;
    int t0, nt, slot;                    // first plan tile, tiles, partial slot (-1: whole item)
    int64_t n_b, i_lo, i_hi, row_base;   // row_base: chunk row of query row 0
    int64_t key_row0;                    // chunk row of position n_b
    UnitPol pol;
    const int32_t* idx;
    const int32_t* ptab;
};

__device__ __forceinline__ Item load_item(const PrefillParams& p, const int4* items, int n) {
    const int4 it = items[n];
    Item m;
    m.b = it.x & 1023;
    m.t0 = (int)((uint32_t)it.x >> 10);
    m.nt = it.w & 0xFFFFF;
    m.slot = (int)((uint32_t)it.w >> 20) - 1;
    m.kvh = it.y;
    const Geo& g = p.geo;
    m.h0 = it.y * g.group + (it.z & 255) * p.nq;
    const int seq = p.seq[m.b];
    const int r0 = (it.z >> 8) * 128;
    m.rows = min(128, p.cnt[m.b] - r0);
    m.n_b = p.n_b[m.b];
    m.i_lo = m.n_b + r0;
    m.i_hi = m.i_lo + m.rows - 1;
    m.key_row0 = p.row0[m.b];
    m.row_base = p.row0[m.b] + r0;
    const int64_t urow = g.unit_row(seq, p.layer, m.kvh);
    m.pol = p.meta.pol[urow];
    m.idx = p.meta.idx + (int64_t)seq * g.max_idx_per_seq + m.pol.idx_off;
    m.ptab = p.meta.ptab + urow * g.max_pages_unit;
    return m;
}

// Packed fp32x2 helpers (sm_100 and later): two lanes of fp32 in one 64-bit
// register, one instruction per pair.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Bits [0, n) set, n clamped to [0, 32].
__device__ __forceinline__ uint32_t lowmask32(int32_t n) {
    return n <= 0 ? 0u : n >= 32 ? 0xFFFFFFFFu : ((1u << n) - 1u);
}

template <int D, int P, bool F8, bool TWO = false, bool SPEC = false>
__global__ void __launch_bounds__(kPfThreads, 1)
k_prefill(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmQ,
          const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
          const __grid_constant__ CUtensorMap tmKp, const __grid_constant__ CUtensorMap tmVp) {
    using S = PfShape<D, F8>;
    constexpr int NS = S::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                               // [2][halves][128][128 B]
    uint8_t* sKV = sQ + 2 * S::kQBytes;               // [NS][halves][128][128 B]
    uint8_t* sF8 = sKV + NS * S::kKVBytes;            // FP8 only: [2][128][128 B] code slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(sF8 + (F8 ? 2 * S::kF8Slot : 0));
    uint64_t* q_full = bars;
    uint64_t* q_empty = bars + 1;
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = kv_full + NS;
    uint64_t* s_full = kv_empty + NS;                 // [2]
    uint64_t* p_full = s_full + 2;                    // [2]
    uint64_t* o_full = p_full + 2;                    // [2]
    uint64_t* o_empty = o_full + 2;                   // [2]
    uint64_t* mma_done = o_empty + 2;
    uint64_t* f_full = mma_done + 1;                  // [2] FP8 code slot landed
    uint64_t* f_empty = f_full + 2;                   // [2] FP8 code slot converted
    // turn tokens of the two MMA issuers: issuer t arrives on tok[t] after
    // each block it issued
    uint64_t* tok = f_empty + 2;                      // [2]
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tok + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // MMA width (keys) of the tile each K/V stage holds, written by the
    // producer before the stage's copies; read by the MMA thread after the
    // stage's full barrier (the arrive orders the write before it)
    volatile int32_t* stage_keys = abort_flag + 4;
    // FP8: the conversion job of each code slot {bf16 stage, K or V, KV head,
    // rows}, or {-1, ...} = no more jobs; written by the producer before the
    // slot's full barrier
    int4* jobs = reinterpret_cast<int4*>(
        (reinterpret_cast<uintptr_t>(stage_keys + 8) + 15) & ~uintptr_t(15));
    int* status = p.meta.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const Geo& g = p.geo;
    const int nq = p.nq;
    // the work list: in the parameters (generic loads of the parameter
    // space; no __ldg there) or in the workspace
    const int4* items = p.inline_words ? p.inl : p.items;
    const int32_t* cta_off = p.inline_words ? reinterpret_cast<const int32_t*>(p.inl + p.n_items) : p.cta_off;
    // TWO (two query tiles, bf16 K/V, head_dim 128; the host's choice): one
    // MMA-issuing thread per query tile (warps 9 and 10), taking turns block
    // by block.  A separate instance: the one-issuer kernel (FP8 history,
    // one query tile, head_dim 64) keeps its code size.
    static_assert(!(TWO && F8), "FP8 history keeps warp 10 for the code conversion");
    // SPEC (calls of long items, with TWO; the host's choice): each softmax
    // row takes its exponentials against its running max at once and this
    // tile's max alongside, redoing them only when the max grew past the lazy
    // rescale's 2^8 or on an item's first tile.  Measured +4 % on 128K-token
    // calls (about 130 tiles an item) and -2 % on 8K-token calls (about 12),
    // whose first tiles take two passes: a separate instance.
    constexpr bool two = TWO;
    constexpr uint32_t nissue = TWO ? 2u : 1u;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, nissue);          // released by every issuer's last QK
        for (int s = 0; s < NS; ++s) { mbar_init(&kv_full[s], 1); mbar_init(&kv_empty[s], nissue); }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);          // one arrival per softmax warp
            mbar_init(&o_full[t], 1);
            mbar_init(&o_empty[t], 4);
        }
        mbar_init(mma_done, nissue);
        for (int f = 0; f < 2; ++f) { mbar_init(&f_full[f], 1); mbar_init(&f_empty[f], 1); }
        mbar_init(&tok[0], 1);
        mbar_init(&tok[1], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp >= 8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLowRegs));
      if (warp == kProducerWarp && lane == 0) {
        // ------------------------------ producer ------------------------------
        prefetch_tmap(&tmQ); prefetch_tmap(&tmK); prefetch_tmap(&tmV);
        prefetch_tmap(&tmKp); prefetch_tmap(&tmVp);
        uint32_t q_loads = 0, L = 0, F = 0;     // F: FP8 code slots filled
        bool ok = true;
        for (int n = cta_off[cta]; n < cta_off[cta + 1] && ok; ++n) {
            const Item it = load_item(p, items, n);
            if (it.nt == 0) continue;
            const Plan pl = make_plan(it.pol, it.idx, it.n_b, it.i_lo, it.i_hi, P);
            if (q_loads > 0 && !mbar_wait(q_empty, (q_loads - 1) & 1, abort_flag, status)) { ok = false; break; }
            mbar_arrive_expect_tx(q_full, nq * S::kQBytes);
            for (int t = 0; t < nq; ++t)
                for (int hf = 0; hf < S::kHalves; ++hf)
                    tma_load_2d(sQ + t * S::kQBytes + hf * S::kHalfBytes, &tmQ, q_full,
                                (it.h0 + t) * D + hf * 64, (int32_t)it.row_base);
            ++q_loads;
            // L2 prefetch of K/V tiles kPrefetchTiles ahead of their loads (a
            // prefetch of the next item's Q measured 1-2 % slower)
            auto prefetch_tile = [&](const KvTile& pk) {
                if (!pk.paged) {
                    const int32_t y = (int32_t)(it.key_row0 + (pk.start - it.n_b));
                    for (int hf = 0; hf < S::kHalves; ++hf) {
                        tma_prefetch_2d(&tmK, it.kvh * D + hf * 64, y);
                        tma_prefetch_2d(&tmV, it.kvh * D + hf * 64, y);
                    }
                } else {
                    const int np = (pk.nkeys + P - 1) / P;
                    for (int pg = 0; pg < np; ++pg) {
                        const int32_t phys = it.ptab[pk.start / P + pg];
                        if (phys < 0 || phys >= g.num_pages) continue;
                        for (int hf = 0; hf < (F8 ? 1 : S::kHalves); ++hf) {   // FP8 rows: one 128-byte box
                            tma_prefetch_2d(&tmKp, hf * 64, phys * P);
                            tma_prefetch_2d(&tmVp, hf * 64, phys * P);
                        }
                    }
                }
            };
            const int32_t ilo32 = (int32_t)it.i_lo, ihi32 = (int32_t)it.i_hi;
            TileCursor cur = cursor_at(pl, it.t0), pre = cur;
            int64_t pj = 0;
            for (; pj < it.nt && pj < kPrefetchTiles; ++pj) {
                prefetch_tile(cursor_tile(pre, it.pol, ilo32, ihi32));
                cursor_next(pl, pre);
            }
            for (int64_t j = 0; j < it.nt && ok; ++j) {
                const KvTile kt = cursor_tile(cur, it.pol, ilo32, ihi32);
                cursor_next(pl, cur);
                if (pj < it.nt) {
                    prefetch_tile(cursor_tile(pre, it.pol, ilo32, ihi32));
                    cursor_next(pl, pre);
                    ++pj;
                }
                for (int kv = 0; kv < 2; ++kv) {
                    const uint32_t st = L % NS, rd = L / NS;
                    if (rd > 0 && !mbar_wait(&kv_empty[st], (rd - 1) & 1, abort_flag, status)) { ok = false; break; }
                    stage_keys[st] = kt.nkeys;
                    uint8_t* dst = sKV + st * S::kKVBytes;
                    if (!kt.paged) {
                        mbar_arrive_expect_tx(&kv_full[st], S::kKVBytes);
                        const int32_t y = (int32_t)(it.key_row0 + (kt.start - it.n_b));
                        for (int hf = 0; hf < S::kHalves; ++hf)
                            tma_load_2d(dst + hf * S::kHalfBytes, kv ? &tmV : &tmK, &kv_full[st],
                                        it.kvh * D + hf * 64, y);
                    } else if (F8) {
                        // codes into the next slot; a converter warp turns them into
                        // bf16 rows of stage st and completes kv_full[st] itself
                        const int np = (kt.nkeys + P - 1) / P;
                        const uint32_t f = F & 1, fr = F >> 1;
                        if (fr > 0 && !mbar_wait(&f_empty[f], (fr - 1) & 1, abort_flag, status)) { ok = false; break; }
                        jobs[f] = make_int4((int)st, kv, it.kvh, np * P);
                        mbar_arrive_expect_tx(&f_full[f], np * P * 128);
                        for (int pg = 0; pg < np; ++pg) {
                            int32_t phys = it.ptab[kt.start / P + pg];
                            if (phys < 0 || phys >= g.num_pages) { atomicOr(status, kStatusBadPage); phys = 0; }
                            tma_load_2d(sF8 + f * S::kF8Slot + pg * P * 128, kv ? &tmVp : &tmKp,
                                        &f_full[f], 0, phys * P);
                        }
                        ++F;
                    } else {
                        const int np = (kt.nkeys + P - 1) / P;
                        mbar_arrive_expect_tx(&kv_full[st], np * P * 128 * S::kHalves);
                        for (int pg = 0; pg < np; ++pg) {
                            int32_t phys = it.ptab[kt.start / P + pg];
                            if (phys < 0 || phys >= g.num_pages) { atomicOr(status, kStatusBadPage); phys = 0; }
                            for (int hf = 0; hf < S::kHalves; ++hf)
                                tma_load_2d(dst + hf * S::kHalfBytes + pg * P * 128, kv ? &tmVp : &tmKp,
                                            &kv_full[st], hf * 64, phys * P);
                        }
                    }
                    ++L;
                }
            }
        }
        if (F8) {
            // no more conversion jobs: an empty job through the next slot
            const uint32_t f = F & 1, fr = F >> 1;
            if (fr == 0 || mbar_wait(&f_empty[f], (fr - 1) & 1, abort_flag, status)) {
                jobs[f] = make_int4(-1, 0, 0, 0);
                mbar_arrive(&f_full[f]);
            }
        }
        // drain: every copy issued has landed before the CTA may exit (FP8
        // stages complete when converted, after their codes landed)
        for (uint32_t s = 0; s < NS && s < L; ++s)
            mbar_wait(&kv_full[s], ((L - 1 - s) / NS) & 1, nullptr, nullptr);
        if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, nullptr, nullptr);
      } else if (lane == 0 && (warp == kMmaWarp || (two && warp == kMmaWarp2))) {
        // ------------------------------ MMA issuer ------------------------------
        const uint32_t q_addr = smem_u32(sQ), kv_addr = smem_u32(sKV);
        const uint32_t idesc_pv = idesc_bf16(128, D, true);
        // Descriptors are built once as 32-bit halves; stepping through a tile
        // only adds the byte offset >> 4 to the low half's start-address field
        // (no carry: every tile lies inside the 256 KB shared window).
        const uint64_t dq0 = sdesc_sw128(q_addr, 16, 1024);
        const uint64_t dk0 = sdesc_sw128(kv_addr, 16, 1024);
        const uint64_t dv0 = sdesc_sw128(kv_addr, S::kHalfBytes, 1024);
        const uint32_t q_lo = (uint32_t)dq0, k_lo = (uint32_t)dk0, v_lo = (uint32_t)dv0;
        const uint32_t kmaj_hi = (uint32_t)(dq0 >> 32), v_hi = (uint32_t)(dv0 >> 32);
        auto issue_qk = [&](int t, uint32_t st, int nkeys) {
            const uint32_t idesc = idesc_bf16(128, nkeys, false);
            const uint32_t a0 = q_lo + ((t * S::kQBytes) >> 4);
            const uint32_t b0 = k_lo + ((st * S::kKVBytes) >> 4);
            const uint32_t d = tmem + t * 128;
            tc_mma_first(d, a0, kmaj_hi, b0, kmaj_hi, idesc);
            #pragma unroll
            for (int ks = 1; ks < D / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * S::kHalfBytes + (ks & 3) * 32) >> 4;
                tc_mma_acc(d, a0 + off, kmaj_hi, b0 + off, kmaj_hi, idesc);
            }
        };
        // The same QK with `before_last` run kTurnEarly MMAs before its end.
        auto issue_qk_hook = [&](int t, uint32_t st, int nkeys, auto&& before_last) {
            const uint32_t idesc = idesc_bf16(128, nkeys, false);
            const uint32_t a0 = q_lo + ((t * S::kQBytes) >> 4);
            const uint32_t b0 = k_lo + ((st * S::kKVBytes) >> 4);
            const uint32_t d = tmem + t * 128;
            tc_mma_first(d, a0, kmaj_hi, b0, kmaj_hi, idesc);
            #pragma unroll
            for (int ks = 1; ks < D / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * S::kHalfBytes + (ks & 3) * 32) >> 4;
                if (ks == D / 16 - kTurnEarly) before_last();
                tc_mma_acc(d, a0 + off, kmaj_hi, b0 + off, kmaj_hi, idesc);
            }
        };
        // O_t (+)= P_t V: P_t sits in TMEM over the first 64 columns of S_t
        // (16 keys = 8 columns per K step), V from shared memory.  The tensor
        // core runs this thread's MMAs in issue order, so S_t of the next tile
        // (issued after this PV) cannot overwrite P_t before it is read.
        auto issue_pv = [&](int t, uint32_t st, int nkeys, bool acc) {
            const uint32_t a0 = tmem + t * 128;
            const uint32_t b0 = v_lo + ((st * S::kKVBytes) >> 4);
            const uint32_t d = tmem + 256 + t * D;
            tc_mma_ta(d, a0, b0, v_hi, idesc_pv, acc ? 1u : 0u);
            if (nkeys == 128) {
                #pragma unroll
                for (int ks = 1; ks < 8; ++ks)
                    tc_mma_ta_acc(d, a0 + ks * 8, b0 + ((ks * 2048) >> 4), v_hi, idesc_pv);
            } else {
                for (int ks = 1; ks * 16 < nkeys; ++ks)
                    tc_mma_ta_acc(d, a0 + ks * 8, b0 + ((ks * 2048) >> 4), v_hi, idesc_pv);
            }
        };
        auto issue_pv_full = [&](int t, uint32_t st, bool acc) {
            const uint32_t a0 = tmem + t * 128;
            const uint32_t b0 = v_lo + ((st * S::kKVBytes) >> 4);
            const uint32_t d = tmem + 256 + t * D;
            tc_mma_ta(d, a0, b0, v_hi, idesc_pv, acc ? 1u : 0u);
            #pragma unroll
            for (int ks = 1; ks < 8; ++ks)
                tc_mma_ta_acc(d, a0 + ks * 8, b0 + ((ks * 2048) >> 4), v_hi, idesc_pv);
        };
        // The MMA thread keeps no plan: the host put each item's tile count in
        // its work entry and the producer writes each stage's key width next to
        // the stage, so between two tiles this thread only waits and issues.
        uint32_t q_uses = 0, L = 0, e = 0, tiles = 0;   // both query tiles see every K/V tile
        bool ok = true;
        const int n_end = cta_off[cta + 1];
        if constexpr (TWO) {
        // One issuer per query tile.  The CTA's blocks (a tile's QK of an
        // item's first K tile, then per K/V tile its PV + next QK) alternate
        // between the issuers, tile 0 first: each starts its block only after
        // the other has issued all but the last kTurnEarly MMAs of the block
        // before (tokens), so the two tiles' MMAs meet in the tensor pipe only
        // at a block's tail and the pipe does not run dry at the hand-over,
        // while each issuer does its own commits and waits for its P and
        // stages as the other's block runs.  Stages and the Q buffer are
        // released when both issuers have committed.
        const int t = warp - kMmaWarp;
        uint32_t nb = 0;                               // blocks this issuer issued
        auto take_turn = [&]() -> bool {
            if (t == 0) return nb == 0 || mbar_wait(&tok[1], (nb - 1) & 1, abort_flag, status);
            return mbar_wait(&tok[0], nb & 1, abort_flag, status);
        };
        auto pass_turn = [&]() { mbar_arrive(&tok[t]); ++nb; };
        for (int n = cta_off[cta]; n < n_end && ok; ++n) {
            const int nt = items[n].w & 0xFFFFF;
            if (nt == 0) continue;
            if (!mbar_wait(q_full, q_uses & 1, abort_flag, status)) { ok = false; break; }
            ++q_uses;
            const uint32_t stK = L % NS;
            if (!mbar_wait(&kv_full[stK], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
            ++L;
            const int nk0 = stage_keys[stK];
            tc_fence_after();
            if (!take_turn()) { ok = false; break; }
            issue_qk_hook(t, stK, nk0, pass_turn);
            tc_commit(&s_full[t]);
            tc_commit(&kv_empty[stK]);
            if (nt == 1) tc_commit(q_empty);
            for (int j = 0; j < nt && ok; ++j) {
                const uint32_t stV = L % NS;
                if (!mbar_wait(&kv_full[stV], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
                ++L;
                const int nkv = stage_keys[stV];
                const bool more = j + 1 < nt;
                uint32_t stK2 = 0;
                int nk2 = 0;
                if (more) {
                    stK2 = L % NS;
                    if (!mbar_wait(&kv_full[stK2], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
                    ++L;
                    nk2 = stage_keys[stK2];
                }
                const bool first = j == 0 && e > 0;     // O_t still holds the last item
                if (!mbar_wait(&p_full[t], tiles & 1, abort_flag, status)) { ok = false; break; }
                if (first && !mbar_wait(&o_empty[t], (e - 1) & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                if (!take_turn()) { ok = false; break; }
                // the turn passes two MMAs before the block's end, so the
                // other issuer's first MMAs queue while this one's last run
                if (nkv == 128 && more) {
                    issue_pv_full(t, stV, j > 0);
                    tc_commit(&o_full[t]);
                    issue_qk_hook(t, stK2, nk2, pass_turn);
                    tc_commit(&s_full[t]);
                } else {
                    issue_pv(t, stV, nkv, j > 0);
                    tc_commit(&o_full[t]);
                    if (more) {
                        issue_qk_hook(t, stK2, nk2, pass_turn);
                        tc_commit(&s_full[t]);
                    } else {
                        pass_turn();
                    }
                }
                ++tiles;
                tc_commit(&kv_empty[stV]);
                if (more) {
                    tc_commit(&kv_empty[stK2]);
                    if (j + 2 == nt) tc_commit(q_empty);
                }
            }
            ++e;
        }
        } else {
        for (int n = cta_off[cta]; n < n_end && ok; ++n) {
            const int nt = items[n].w & 0xFFFFF;
            if (nt == 0) continue;
            if (!mbar_wait(q_full, q_uses & 1, abort_flag, status)) { ok = false; break; }
            ++q_uses;
            const uint32_t stK = L % NS;
            if (!mbar_wait(&kv_full[stK], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
            ++L;
            const int nk0 = stage_keys[stK];
            tc_fence_after();
            for (int t = 0; t < nq; ++t) { issue_qk(t, stK, nk0); tc_commit(&s_full[t]); }
            tc_commit(&kv_empty[stK]);
            if (nt == 1) tc_commit(q_empty);
            for (int j = 0; j < nt && ok; ++j) {
                const uint32_t stV = L % NS;
                if (!mbar_wait(&kv_full[stV], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
                ++L;
                const int nkv = stage_keys[stV];          // width of tile j
                const bool more = j + 1 < nt;
                uint32_t stK2 = 0;
                int nk2 = 0;
                if (more) {
                    stK2 = L % NS;
                    if (!mbar_wait(&kv_full[stK2], (L / NS) & 1, abort_flag, status)) { ok = false; break; }
                    ++L;
                    nk2 = stage_keys[stK2];                // width of tile j + 1
                }
                const bool first = j == 0 && e > 0;     // O_t still holds the last item
                const bool steady = nkv == 128 && more;
                // Per query tile: PV of this tile, then QK of the next.  In the
                // steady state the 16 MMAs and their commits are one straight
                // run of code: a branch between two MMAs costs the tensor core
                // tens of cycles of issue.
                auto step = [&](int t) -> bool {
                    if (!mbar_wait(&p_full[t], tiles & 1, abort_flag, status)) return false;
                    if (first && !mbar_wait(&o_empty[t], (e - 1) & 1, abort_flag, status)) return false;
                    tc_fence_after();
                    if (steady) {
                        issue_pv_full(t, stV, j > 0);
                        tc_commit(&o_full[t]);
                        issue_qk(t, stK2, nk2);
                        tc_commit(&s_full[t]);
                    } else {
                        issue_pv(t, stV, nkv, j > 0);
                        tc_commit(&o_full[t]);
                        if (more) { issue_qk(t, stK2, nk2); tc_commit(&s_full[t]); }
                    }
                    return true;
                };
                if (!step(0) || (nq > 1 && !step(1))) { ok = false; break; }
                ++tiles;
                tc_commit(&kv_empty[stV]);
                if (more) {
                    tc_commit(&kv_empty[stK2]);
                    if (j + 2 == nt) tc_commit(q_empty);
                }
            }
            ++e;
        }
        }
        // all MMAs issued by this thread complete before TMEM can be freed
        tc_commit(mma_done);
        mbar_wait(mma_done, 0, nullptr, nullptr);
      } else if (F8 && warp >= 10) {
        // ------------------ FP8 history: codes -> bf16 stage rows ------------------
        // 64 threads: thread (row r0 of each 8, 16-code chunk c16) writes
        // bf16(code * scale) of dims c16*16 .. +15 into the 128-byte-swizzled
        // K-major layout the MMA reads (two 64-dim halves per row).
        const int ct = threadIdx.x - 320;
        const int c16 = ct & 7, r0 = ct >> 3;
        uint32_t fj = 0;
        while (true) {
            const uint32_t f = fj & 1;
            const bool got = mbar_wait(&f_full[f], (fj >> 1) & 1, abort_flag, status);
            // The two warps decide together: either wait may give up on its
            // own (its time limit, or the abort flag raised by another role
            // while the codes land), and the barrier after the conversion
            // must be met by both.  So both leave if either gave up.
            if (meet_any<3>(64, !got)) break;
            const int4 jb = jobs[f];
            if (jb.x < 0) break;
            const float* scp = (jb.y ? p.meta.vscale : p.meta.kscale) +
                               ((int64_t)p.layer * g.hkv + jb.z) * D + c16 * 16;
            float sc[16];
            #pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 v4 = __ldg(reinterpret_cast<const float4*>(scp + e));
                sc[e] = v4.x; sc[e + 1] = v4.y; sc[e + 2] = v4.z; sc[e + 3] = v4.w;
            }
            const uint8_t* src = sF8 + f * S::kF8Slot;
            uint8_t* dst = sKV + jb.x * S::kKVBytes + (c16 >> 2) * S::kHalfBytes;
            const uint32_t ch = (c16 & 3) * 2;
            for (int r = r0; r < jb.w; r += 8) {
                const uint4 q4 = *reinterpret_cast<const uint4*>(src + sw128(r, c16));
                const uint32_t w[4] = {q4.x, q4.y, q4.z, q4.w};
                uint32_t o[8];
                #pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t h2 = f16x2_of_e4m3x2((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
                    const __half2 hv = *reinterpret_cast<const __half2*>(&h2);
                    o[e] = pack_bf16(__low2float(hv) * sc[2 * e], __high2float(hv) * sc[2 * e + 1]);
                }
                *reinterpret_cast<uint4*>(dst + sw128(r, ch)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4*>(dst + sw128(r, ch + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
            fence_async_smem();                       // rows visible to the tensor core
            asm volatile("bar.sync 2, 64;" ::: "memory");
            if (ct == 0) {
                mbar_arrive(&f_empty[f]);
                mbar_arrive(&kv_full[jb.x]);
            }
            ++fj;
        }
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kHighRegs));
        // --------------------------- softmax + epilogue ---------------------------
        const int t = warp >> 2;
        if (t < nq) {
            const int r = threadIdx.x - t * 128;                       // query row in the tile
            const uint32_t lane_off = ((uint32_t)(warp & 3) * 32u) << 16;
            const uint32_t tS = tmem + lane_off + t * 128;
            const uint32_t tO = tmem + lane_off + 256 + t * D;
            const float sl2 = p.scale_log2;
            uint32_t k = 0;
            bool ok = true;
            for (int n = cta_off[cta]; n < cta_off[cta + 1] && ok; ++n) {
                const Item it = load_item(p, items, n);
                const Plan pl = make_plan(it.pol, it.idx, it.n_b, it.i_lo, it.i_hi, P);
                const int head = it.h0 + t;
                const bool row_ok = r < it.rows;
                const int32_t i = (int32_t)(it.i_lo + r);
                __nv_bfloat16* orow = p.out + ((it.row_base + r) * g.hq + head) * D;
                if (it.nt == 0) {      // no visible key (never a piece of a split item)
                    if (row_ok) {
                        for (int c = 0; c < D; c += 8)
                            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
                        if (p.lse) p.lse[(it.row_base + r) * g.hq + head] = -INFINITY;
                    }
                    continue;
                }
                float m = -INFINITY, l = 0.f;
                TileCursor cur = cursor_at(pl, it.t0);
                for (int64_t j = 0; j < it.nt; ++j, ++k) {
                    const KvTile kt = cursor_tile(cur, it.pol, (int32_t)it.i_lo, (int32_t)it.i_hi);
                    cursor_next(pl, cur);
                    const bool masked = !kt.full;
                    int32_t tpos[4] = {-1, -1, -1, -1};
                    if (masked && kt.table && !kt.paged) {
                        #pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            tpos[q4] = (int32_t)tile_key_position(kt, it.pol, it.idx, it.n_b,
                                                                  lane + 32 * q4, P);
                    }
                    if (!mbar_wait(&s_full[t], k & 1, abort_flag, status)) { ok = false; break; }
                    tc_fence_after();
                    // Visibility bits of this row for columns 0..127.  Chunk tiles
                    // (affine positions p = start + c): c < nvalid, c <= i - start,
                    // and for LOCAL c < sink - start or c >= i - window + 1 - start.
                    // Table tiles: key_visible on the broadcast position table.
                    uint32_t vm[4];
                    if (!masked) {
                        #pragma unroll
                        for (int w = 0; w < 4; ++w) vm[w] = lowmask32(kt.nkeys - 32 * w);
                    } else if (!kt.table) {
                        const int32_t p0 = (int32_t)kt.start;
                        const int32_t up = min(kt.nvalid, i - p0 + 1);
                        #pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint32_t b = lowmask32(up - 32 * w);
                            if (it.pol.kind == kLocal)
                                b &= lowmask32(it.pol.sink - p0 - 32 * w) |
                                     ~lowmask32(i - it.pol.window + 1 - p0 - 32 * w);
                            vm[w] = b;
                        }
                    } else if (kt.paged) {
                        // history slots: arithmetic bits (sp_plan.h)
                        paged_row_mask(kt, it.pol, (int32_t)it.n_b, i, P, vm);
                    } else {
                        // RETRIEVAL chunk rows: the per-key position table
                        #pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint32_t b = 0;
                            #pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const int32_t tp = __shfl_sync(0xffffffffu, tpos[w], e);
                                if (key_visible<int32_t>(kt, it.pol, i, 32 * w + e, tp)) b |= 1u << e;
                            }
                            vm[w] = b;
                        }
                    }
                    // S row of this thread, all 128 columns at once (the softmax
                    // warpgroups hold 208 registers a thread).  Columns at or past
                    // nkeys were not written by this tile's MMA and hold stale
                    // values; their visibility bits are 0, so the select below
                    // turns them into -inf like any invisible key.  One code path
                    // for every tile width keeps the loop small.
                    uint32_t sr[128];
                    tmem_ld128(tS, sr);
                    const bool fast = !masked && kt.nkeys == 128;
                    if (!fast) {
                        // invisible or absent columns -> -inf, once (branch-free)
                        #pragma unroll
                        for (int c = 0; c < 128; ++c)
                            sr[c] = ((vm[c >> 5] >> (c & 31)) & 1u) ? sr[c] : 0xff800000u;
                    }
                    if constexpr (!SPEC) {
                        // row maximum (raw score units; the scale is positive): eight
                        // running maxima, two new columns each per three-input max
                        float tmax;
                        {
                            float m8[8];
                            #pragma unroll
                            for (int a = 0; a < 8; ++a) m8[a] = fmaxf(__uint_as_float(sr[a]), __uint_as_float(sr[8 + a]));
                            #pragma unroll
                            for (int e = 16; e < 128; e += 16)
                                #pragma unroll
                                for (int a = 0; a < 8; ++a)
                                    m8[a] = fmax3(m8[a], __uint_as_float(sr[e + a]), __uint_as_float(sr[e + 8 + a]));
                            tmax = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                         fmaxf(m8[6], m8[7])) * sl2;
                        }
                        // online softmax with lazy rescale
                        float alpha = 1.f;
                        bool resc = false;
                        const float m_new = fmaxf(m, tmax);
                        if (m == -INFINITY) {
                            m = m_new;
                        } else if (m_new > m + kRescaleLog2) {
                            alpha = fast_exp2(m - m_new);
                            m = m_new;
                            resc = true;
                        }
                        const float mb = m == -INFINITY ? 0.f : m;
                        // The previous tile's PV must be done before P is overwritten
                        // and before O is rescaled.  It is: this tile's S arrived
                        // through a tcgen05.commit issued after that PV, and a commit
                        // tracks every earlier tcgen05 operation of the issuing
                        // thread, so no separate wait on o_full is needed here (the
                        // epilogue still waits for the item's last PV).
                        if (__any_sync(0xffffffffu, resc)) {
                            #pragma unroll
                            for (int ch = 0; ch < D / 16; ++ch) {
                                uint32_t o[16];
                                tmem_ld16(tO + ch * 16, o);
                                #pragma unroll
                                for (int e2 = 0; e2 < 16; ++e2)
                                    o[e2] = __float_as_uint(__uint_as_float(o[e2]) * alpha);
                                tmem_st16(tO + ch * 16, o);
                            }
                            tmem_st_wait();
                        }
                        // exponentials, row sum, P row -> shared memory in the K-major
                        // 128-byte-swizzled operand layout (-inf columns give 0).  The
                        // scale-and-shift and the row sum use packed fp32x2 arithmetic.
                        uint64_t rsum2[4] = {0ull, 0ull, 0ull, 0ull};
                        const uint64_t sl2x2 = pack_f32x2(sl2, sl2), nmbx2 = pack_f32x2(-mb, -mb);
                        // P row as bf16 pairs (column j of the S tile = keys 2j, 2j+1),
                        // stored to TMEM 32 keys at a time
                        auto exp_group = [&](int g4) {
                            uint32_t pk[16];
                            #pragma unroll
                            for (int e2 = 0; e2 < 16; ++e2) {
                                const int c = g4 * 32 + 2 * e2;
                                const uint64_t x2 = fma_f32x2(pack_u32x2(sr[c], sr[c + 1]), sl2x2, nmbx2);
                                float x0, x1;
                                unpack_f32x2(x2, x0, x1);
                                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                                rsum2[e2 & 3] = add_f32x2(rsum2[e2 & 3], pack_f32x2(p0, p1));
                                pk[e2] = pack_bf16(p0, p1);
                            }
                            tmem_st16(tS + g4 * 16, pk);
                        };
                        // all four groups on every tile (no guards, so the compiler can
                        // interleave them): past nkeys the row is -inf, P is 0 there,
                        // and the PV MMA reads only the first nkeys / 2 columns
                        #pragma unroll
                        for (int g4 = 0; g4 < 4; ++g4) exp_group(g4);
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&p_full[t]);
                        // the row sum is not needed by the MMA: fold it after the arrive
                        float rsum[8];
                        #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) unpack_f32x2(rsum2[e2], rsum[2 * e2], rsum[2 * e2 + 1]);
                        const float rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) +
                                         ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
                        l = l * alpha + rs;
                    } else {
                        // Exponentials against the running max m straight away (the
                        // lazy rescale already lets a score exceed m by up to 2^8),
                        // with this tile's max taken alongside in the issue slots
                        // the MUFU-bound exponentials leave free.  Only where a row
                        // has no max yet (an item's first tiles) or its max grew by
                        // more than 2^8 is the online state updated, O rescaled and
                        // the row's exponentials taken again (warp-uniform).
                        uint64_t rsum2[4] = {0ull, 0ull, 0ull, 0ull};
                        const uint64_t sl2x2 = pack_f32x2(sl2, sl2);
                        // P row as bf16 pairs (column j of the S tile = keys 2j, 2j+1),
                        // stored to TMEM 32 keys at a time
                        auto exp_group = [&](int g4, uint64_t nmbx2) {
                            uint32_t pk[16];
                            #pragma unroll
                            for (int e2 = 0; e2 < 16; ++e2) {
                                const int c = g4 * 32 + 2 * e2;
                                const uint64_t x2 = fma_f32x2(pack_u32x2(sr[c], sr[c + 1]), sl2x2, nmbx2);
                                float x0, x1;
                                unpack_f32x2(x2, x0, x1);
                                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                                rsum2[e2 & 3] = add_f32x2(rsum2[e2 & 3], pack_f32x2(p0, p1));
                                pk[e2] = pack_bf16(p0, p1);
                            }
                            tmem_st16(tS + g4 * 16, pk);
                        };
                        // first pass: exponentials against m (0 while the row has
                        // none) and the row maximum (raw score units; the scale is
                        // positive): eight running maxima, two columns per
                        // three-input max per group of 16
                        float m8[8];
                        #pragma unroll
                        for (int a = 0; a < 8; ++a) m8[a] = -INFINITY;
                        {
                            const float mb0 = m == -INFINITY ? 0.f : m;
                            const uint64_t nmbx2 = pack_f32x2(-mb0, -mb0);
                            #pragma unroll
                            for (int g4 = 0; g4 < 4; ++g4) {
                                #pragma unroll
                                for (int e = g4 * 32; e < g4 * 32 + 32; e += 16)
                                    #pragma unroll
                                    for (int a = 0; a < 8; ++a)
                                        m8[a] = fmax3(m8[a], __uint_as_float(sr[e + a]), __uint_as_float(sr[e + 8 + a]));
                                exp_group(g4, nmbx2);
                            }
                        }
                        const float tmax = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                                                 fmaxf(m8[6], m8[7])) * sl2;
                        // online softmax with lazy rescale
                        float alpha = 1.f;
                        bool resc = false, redo = false;
                        if (m == -INFINITY) {
                            m = tmax;                 // stays -inf if nothing visible yet
                            redo = m != -INFINITY;
                        } else if (tmax > m + kRescaleLog2) {
                            alpha = fast_exp2(m - tmax);
                            m = tmax;
                            resc = redo = true;
                        }
                        if (__any_sync(0xffffffffu, redo)) {
                            // The previous tile's PV must be done before P is
                            // overwritten and before O is rescaled.  It is: this
                            // tile's S arrived through a tcgen05.commit issued after
                            // that PV, and a commit tracks every earlier tcgen05
                            // operation of the issuing thread, so no separate wait on
                            // o_full is needed here (the epilogue still waits for the
                            // item's last PV).
                            if (__any_sync(0xffffffffu, resc)) {
                                #pragma unroll
                                for (int ch = 0; ch < D / 16; ++ch) {
                                    uint32_t o[16];
                                    tmem_ld16(tO + ch * 16, o);
                                    #pragma unroll
                                    for (int e2 = 0; e2 < 16; ++e2)
                                        o[e2] = __float_as_uint(__uint_as_float(o[e2]) * alpha);
                                    tmem_st16(tO + ch * 16, o);
                                }
                                tmem_st_wait();
                            }
                            // second pass against the new m (rows that kept theirs
                            // recompute the same values)
                            #pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2) rsum2[e2] = 0ull;
                            const float mb = m == -INFINITY ? 0.f : m;
                            const uint64_t nmbx2 = pack_f32x2(-mb, -mb);
                            #pragma unroll
                            for (int g4 = 0; g4 < 4; ++g4) exp_group(g4, nmbx2);
                        }
                        // past nkeys the row is -inf, P is 0 there, and the PV MMA
                        // reads only the first nkeys / 2 columns
                        tmem_st_wait();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&p_full[t]);
                        // the row sum is not needed by the MMA: fold it after the arrive
                        float rsum[8];
                        #pragma unroll
                        for (int e2 = 0; e2 < 4; ++e2) unpack_f32x2(rsum2[e2], rsum[2 * e2], rsum[2 * e2 + 1]);
                        const float rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) +
                                         ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
                        l = l * alpha + rs;
                    }
                }
                if (!ok) break;
                // epilogue: O / l -> bf16 rows, LSE
                if (!mbar_wait(&o_full[t], (k - 1) & 1, abort_flag, status)) { ok = false; break; }
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                // The whole O row into registers first, then O_t is released at
                // once (the next item's first PV may overwrite it) and the row
                // is normalised and written with 32-byte stores.
                uint32_t orr[D];
                if constexpr (D == 128) tmem_ld128(tO, *reinterpret_cast<uint32_t(*)[128]>(orr));
                else tmem_ld64(tO, *reinterpret_cast<uint32_t(*)[64]>(orr));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty[t]);
                if (it.slot >= 0) {
                    // a piece of a split item: its unnormalised O and (m, l)
                    // for the merge (rows with no key seen keep m = -inf, l = 0)
                    if (row_ok) {
                        const int64_t sb = (int64_t)it.slot * 2 + t;
                        float4* po = p.split_o + sb * (D / 4) * 128 + r;
                        #pragma unroll
                        for (int c4 = 0; c4 < D / 4; ++c4)
                            po[c4 * 128] = make_float4(__uint_as_float(orr[4 * c4]), __uint_as_float(orr[4 * c4 + 1]),
                                                       __uint_as_float(orr[4 * c4 + 2]), __uint_as_float(orr[4 * c4 + 3]));
                        p.split_ml[sb * 128 + r] = make_float2(m, l);
                    }
                    continue;
                }
                if (row_ok) {
                    #pragma unroll
                    for (int c = 0; c < D; c += 16) {
                        uint32_t w[8];
                        #pragma unroll
                        for (int e2 = 0; e2 < 8; ++e2)
                            w[e2] = pack_bf16(__uint_as_float(orr[c + 2 * e2]) * inv,
                                              __uint_as_float(orr[c + 2 * e2 + 1]) * inv);
                        st_global_v8(orow + c, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                    }
                }
                if (row_ok && p.lse)
                    p.lse[(it.row_base + r) * g.hq + head] =
                        l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// |V(i)| as the tile plan and the mask see it (one thread per position).
__global__ void k_prefill_counts(Meta meta, Geo g, int seq, int layer, int h,
                                 const int64_t* pos, int npos, int32_t* out) {
    const int64_t urow = g.unit_row(seq, layer, h);
    const UnitPol pol = meta.pol[urow];
    const int32_t* idx = meta.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
    const int64_t held = meta.seqlen[(int64_t)seq * g.layers + layer];
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < npos; k += gridDim.x * blockDim.x) {
        const int64_t i = pos[k];
        if (i < held) continue;
        const int64_t i_lo = held + (i - held) / 128 * 128;
        const int64_t i_hi = i_lo + 127;
        const Plan pl = make_plan(pol, idx, held, i_lo, i_hi, g.page);
        int64_t cnt = 0;
        for (int64_t t = 0; t < pl.ntiles; ++t) {
            const KvTile kt = plan_tile(pl, pol, t, i_lo, i_hi);
            for (int c = 0; c < kt.nkeys; ++c) {
                const int64_t tp = kt.table ? tile_key_position(kt, pol, idx, held, c, g.page) : 0;
                cnt += key_visible<int64_t>(kt, pol, i, c, tp) ? 1 : 0;
            }
        }
        out[k] = (int32_t)cnt;
    }
}

// Pieces of split items -> final rows: per (item, query tile, 32 columns)
// block, one thread per row combines the pieces' (O, m, l): m* = max m, each piece
// weighted by 2^(m - m*), O = sum w O / sum w l, LSE = m* + log2(sum w l) in
// natural-log units.  A row no piece saw gives O = 0, LSE = -inf.
constexpr int kMaxMergeGroups = 1024;
constexpr int kMaxPieces = 8;
struct MergeParams {
    int32_t n_groups, hq;
    const float4* split_o;
    const float2* split_ml;
    __nv_bfloat16* out;
    float* lse;
    int4 groups[kMaxMergeGroups];   // {row_base, first query head, rows, first slot | pieces << 16}
};

template <int D>
__global__ void __launch_bounds__(128) k_prefill_merge(const __grid_constant__ MergeParams p) {
    // block (group, query tile, 32-column slice); thread = row
    const int4 gr = p.groups[blockIdx.x];
    const int t = blockIdx.y, c0 = blockIdx.z * 32, r = threadIdx.x;
    if (r >= gr.z) return;
    const int slot0 = gr.w & 0xFFFF, np = gr.w >> 16;
    float ms[kMaxPieces], wq[kMaxPieces], mx = -INFINITY;
    #pragma unroll
    for (int q = 0; q < kMaxPieces; ++q) {
        ms[q] = -INFINITY;
        wq[q] = 0.f;
        if (q < np) {
            const float2 ml = p.split_ml[((int64_t)(slot0 + q) * 2 + t) * 128 + r];
            ms[q] = ml.x;
            wq[q] = ml.y;
            mx = fmaxf(mx, ml.x);
        }
    }
    float L = 0.f;
    #pragma unroll
    for (int q = 0; q < kMaxPieces; ++q) {
        const float w = ms[q] != -INFINITY ? exp2f(ms[q] - mx) : 0.f;
        L += w * wq[q];
        wq[q] = w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float a[32];
    #pragma unroll
    for (int e = 0; e < 32; ++e) a[e] = 0.f;
    #pragma unroll
    for (int q = 0; q < kMaxPieces; ++q) {
        if (q < np) {
            const float4* po = p.split_o + ((int64_t)(slot0 + q) * 2 + t) * (D / 4) * 128 + r;
            #pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 x = po[(c0 / 4 + e4) * 128];
                a[4 * e4] += wq[q] * x.x; a[4 * e4 + 1] += wq[q] * x.y;
                a[4 * e4 + 2] += wq[q] * x.z; a[4 * e4 + 3] += wq[q] * x.w;
            }
        }
    }
    __nv_bfloat16* orow = p.out + ((int64_t)(gr.x + r) * p.hq + gr.y + t) * D + c0;
    #pragma unroll
    for (int e = 0; e < 32; e += 8)
        *reinterpret_cast<uint4*>(orow + e) =
            make_uint4(pack_bf16(a[e] * inv, a[e + 1] * inv), pack_bf16(a[e + 2] * inv, a[e + 3] * inv),
                       pack_bf16(a[e + 4] * inv, a[e + 5] * inv), pack_bf16(a[e + 6] * inv, a[e + 7] * inv));
    if (p.lse && blockIdx.z == 0)
        p.lse[(int64_t)(gr.x + r) * p.hq + gr.y + t] =
            L > 0.f ? (mx + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

static_assert(sizeof(MergeParams) <= 32764, "merge parameters exceed the kernel parameter space");

// the parameters (work list included) and the five tensor maps must fit the
// kernel parameter space (32,764 bytes)
static_assert(sizeof(PrefillParams) + 5 * sizeof(CUtensorMap) <= 32764,
              "prefill parameters exceed the kernel parameter space");

template <int D, int P, bool F8 = false, bool TWO = false, bool SPEC = false>
cudaError_t launch_prefill_t(sp_cache* c, const PrefillParams& p, int grid,
                             const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             cudaStream_t s) {
    using Sh = PfShape<D, F8>;
    bool& checked = c->prefill_checked[SPEC ? 4 : TWO ? 3 : F8 ? 2 : D == 128][P == 16 ? 0 : P == 32 ? 1 : P == 64 ? 2 : 3];
    if (!checked) {   // once per cache and kernel instance
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k_prefill<D, P, F8, TWO, SPEC>);
        if (e != cudaSuccess) return e;
        // The setmaxnreg split assumes exactly kLaunchRegs registers per thread
        // at launch; anything else could leave an increase waiting forever.
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(k_prefill<D, P, F8, TWO, SPEC>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::kSmem);
        if (e != cudaSuccess) return e;
        checked = true;
    }
    k_prefill<D, P, F8, TWO, SPEC><<<grid, kPfThreads, Sh::kSmem, s>>>(p, tq, tk, tv, c->tm_kpool, c->tm_vpool);
    return cudaGetLastError();
}

}  // namespace

int64_t prefill_max_tiles(const sp_config* c) {
    // work items plus room for the per-CTA offsets behind them
    return ((int64_t)c->max_tokens / 128 + c->max_batch + 1) * c->num_q_heads + 512;
}

sp_status prefill_impl(sp_cache* c, int32_t layer, const int32_t* seq_ids, int32_t n_seqs,
                       const int32_t* cu_q, const __nv_bfloat16* q, const __nv_bfloat16* k,
                       const __nv_bfloat16* v, __nv_bfloat16* out, float* lse,
                       cudaStream_t stream) {
    const int T = cu_q[n_seqs];
    if (T == 0) return SP_OK;
    std::unique_ptr<PrefillParams> pp(new PrefillParams());
    PrefillParams& p = *pp;
    p.meta = c->meta;
    p.geo = c->geo;
    p.layer = layer;
    const int group = c->geo.group;
    p.nq = (group % 2 == 0) ? 2 : 1;
    const int pairs = group / p.nq;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
    p.out = out;
    p.lse = lse;
    p.split_o = reinterpret_cast<float4*>(c->ws.split_o);
    p.split_ml = reinterpret_cast<float2*>(c->ws.split_ml);
    struct Cand { int64_t cost; int32_t unit; int4 item; };   // unit: call sequence * Hkv + KV head
    std::vector<Cand> whole;
    {
        size_t n_rb = 0;
        for (int b = 0; b < n_seqs; ++b) n_rb += (size_t)(cu_q[b + 1] - cu_q[b] + 127) / 128;
        whole.reserve(n_rb * c->cfg.num_kv_heads * pairs);
    }
    const int P = c->cfg.page_size;
    for (int b = 0; b < n_seqs; ++b) {
        const int seq = seq_ids[b];
        const int64_t n_b = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
        const int cb = cu_q[b + 1] - cu_q[b];
        p.seq[b] = seq;
        p.n_b[b] = (int32_t)n_b;
        p.cnt[b] = cb;
        p.row0[b] = cu_q[b];
        for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
            const size_t ui = ((size_t)seq * c->cfg.num_layers + layer) * c->cfg.num_kv_heads + h;
            const UnitPol& u = c->h_pol[ui];
            const int32_t* idx = c->h_idx[seq].data() + u.idx_off;
            for (int rb = 0; rb * 128 < cb; ++rb) {
                const int64_t i_lo = n_b + rb * 128;
                const int64_t i_hi = n_b + std::min(cb, rb * 128 + 128) - 1;
                const Plan pl = make_plan(u, idx, n_b, i_lo, i_hi, P);
                if (pl.ntiles >= (int64_t(1) << 20))
                    return fail(SP_ERR_UNSUPPORTED, "more than 2^20 key tiles for one row block");
                // Time model for the assignment, measured per CTA with clock64
                // traces: every K/V tile costs about the same whatever its
                // width (the softmax treats a whole tile), and an item adds the
                // pipeline fill, the epilogue and the hand-over to the next
                // item, about three tiles' worth.
                const int64_t cost = kTileCost * pl.ntiles + kItemCost;
                for (int pr = 0; pr < pairs; ++pr)
                    whole.push_back({cost, b * c->cfg.num_kv_heads + h,
                                     make_int4(b, h, pr | (rb << 8), (int)pl.ntiles)});
            }
        }
    }
    // An item much longer than a CTA's fair share of the call would set the
    // launch's end on its own (a GLOBAL head's row blocks over a long
    // history, next to short LOCAL ones).  Such items are split along their
    // key tiles into pieces of about half a share; each piece leaves its
    // unnormalised O and (m, l) in a workspace slot and k_prefill_merge
    // combines them.
    int64_t total = 0;
    for (const Cand& cd : whole) total += cd.cost;
    const double share = (double)total / std::max(1, c->num_sms);
    std::vector<Cand> cands;
    cands.reserve(whole.size() + kPrefillSplitSlots);
    std::vector<int4> groups;                  // merge: {row_base, first head, rows, slot | pieces << 16}
    int slots = 0;
    for (const Cand& cd : whole) {
        const int nt = cd.item.w;
        int np = 1;
        if ((double)cd.cost > 0.8 * share && nt >= 2 * kMinPieceTiles) {
            np = (int)std::ceil((double)cd.cost / (0.5 * share));
            np = std::min(std::min(np, kMaxPieces), nt / kMinPieceTiles);
            if (slots + np > kPrefillSplitSlots || (int)groups.size() >= kMaxMergeGroups) np = 1;
        }
        if (np <= 1) {
            cands.push_back(cd);
            continue;
        }
        const int b = cd.item.x, h = cd.item.y, pr = cd.item.z & 255, rb = cd.item.z >> 8;
        const int cb = cu_q[b + 1] - cu_q[b];
        groups.push_back(make_int4(cu_q[b] + rb * 128, h * group + pr * p.nq,
                                   std::min(128, cb - rb * 128), slots | (np << 16)));
        for (int q = 0; q < np; ++q) {
            const int t0 = (int)((int64_t)nt * q / np), t1 = (int)((int64_t)nt * (q + 1) / np);
            const int4 it = make_int4(b | (t0 << 10), h, cd.item.z, (t1 - t0) | ((slots + q + 1) << 20));
            cands.push_back({kTileCost * (t1 - t0) + kItemCost, cd.unit, it});
        }
        slots += np;
    }
    if ((int64_t)cands.size() + (c->num_sms + 4) / 4 > c->ws.max_tiles)
        return fail(SP_ERR_UNSUPPORTED, "prefill work list larger than the workspace");
    // Order.  When the call's K/V is larger than about half of L2: unit by
    // unit (units with the most work first), each unit's items longest
    // first, so all CTAs work through one unit's K/V at a time (a GLOBAL
    // head of a 128K sequence holds 67 MB of K and V) instead of every unit
    // whose items have similar lengths at once, which overflows L2 and reads
    // K/V tiles from HBM several times (measured: a 128K layer with two
    // GLOBAL heads reads 8.6 GB instead of 16.5 GB, in the same time).
    // Otherwise longest first over all items, which balances the CTAs'
    // end times a little better (3-9 % faster on 8K-token calls).
    const int n_units = n_seqs * c->cfg.num_kv_heads;
    std::vector<int32_t> rank(n_units, 0);
    int64_t kv_bytes = 0;
    for (int b = 0; b < n_seqs; ++b)
        kv_bytes += (int64_t)(p.n_b[b] + p.cnt[b]) * c->cfg.num_kv_heads * 2 * c->cfg.head_dim *
                    (c->geo.fp8 ? 1 : 2);
    if (kv_bytes > kL2UnitOrderBytes) {
        std::vector<int64_t> unit_cost(n_units, 0);
        for (const Cand& cd : cands) unit_cost[cd.unit] += cd.cost;
        std::vector<int32_t> by_cost(n_units);
        for (int u = 0; u < n_units; ++u) by_cost[u] = u;
        std::stable_sort(by_cost.begin(), by_cost.end(),
                         [&](int32_t a, int32_t b2) { return unit_cost[a] > unit_cost[b2]; });
        for (int r = 0; r < n_units; ++r) rank[by_cost[r]] = r;
    }
    // One sort of packed keys (unit rank, cost descending, candidate index:
    // a stable order); a comparison sort of the records when a field would
    // not fit its bits.
    const size_t n_items = cands.size();
    std::vector<uint32_t> order(n_items);
    if (n_units < (1 << 16) && n_items < (size_t(1) << 20)) {
        // cost = kTileCost * tiles + kItemCost < 2^28 for tiles < 2^20
        std::vector<uint64_t> key(n_items);
        for (size_t i = 0; i < n_items; ++i)
            key[i] = ((uint64_t)rank[cands[i].unit] << 48) |
                     ((uint64_t)((int64_t(1) << 28) - 1 - cands[i].cost) << 20) | (uint64_t)i;
        std::sort(key.begin(), key.end());
        for (size_t i = 0; i < n_items; ++i) order[i] = (uint32_t)(key[i] & 0xFFFFFu);
    } else {
        for (size_t i = 0; i < n_items; ++i) order[i] = (uint32_t)i;
        std::stable_sort(order.begin(), order.end(), [&](uint32_t a, uint32_t b2) {
            const Cand &x = cands[a], &y = cands[b2];
            return rank[x.unit] != rank[y.unit] ? rank[x.unit] < rank[y.unit] : x.cost > y.cost;
        });
    }
    // Greedy assignment in that order: each item goes to the CTA with the
    // least work so far (longest-processing-time rule within a unit; ties to
    // the lower CTA).
    const int grid = (int)std::min<int64_t>(c->num_sms, (int64_t)n_items);
    std::vector<int32_t> owner(n_items);
    std::vector<int32_t> fill(grid + 1, 0);
    {
        typedef std::pair<int64_t, int> LoadCta;
        std::vector<LoadCta> heap(grid);
        for (int g2 = 0; g2 < grid; ++g2) heap[g2] = LoadCta(0, g2);   // a valid min-heap
        const auto later = std::greater<LoadCta>();
        for (size_t k2 = 0; k2 < n_items; ++k2) {
            const uint32_t i = order[k2];
            std::pop_heap(heap.begin(), heap.end(), later);
            LoadCta& top = heap.back();
            owner[i] = top.second;
            ++fill[top.second + 1];
            top.first += cands[i].cost;
            std::push_heap(heap.begin(), heap.end(), later);
        }
    }
    // The items grouped by CTA (each CTA's in the sorted order), then the CTA
    // offsets: inside the kernel parameters when they fit, else one upload
    // through the next pinned staging buffer (asynchronous; waits only if
    // that buffer's previous copy has not run yet)
    const size_t words = n_items + (grid + 1 + 3) / 4;
    const bool inl = words <= (size_t)kInlineWords;
    int si = -1;
    int4* buf = inl ? p.inl : static_cast<int4*>(stage_acquire(c, words * sizeof(int4), &si));
    if (!buf) return fail(SP_ERR_CUDA, "prefill staging buffer");
    int32_t* off = reinterpret_cast<int32_t*>(buf + n_items);
    for (int g2 = 0; g2 < grid; ++g2) fill[g2 + 1] += fill[g2];
    for (int g2 = 0; g2 <= grid; ++g2) off[g2] = fill[g2];
    for (size_t k2 = 0; k2 < n_items; ++k2) {
        const uint32_t i = order[k2];
        buf[fill[owner[i]]++] = cands[i].item;
    }
    p.n_items = (int32_t)n_items;
    p.inline_words = inl ? (int32_t)words : 0;
    // One MMA issuer per query tile wherever the kernel has that instance:
    // bf16 K/V, head_dim 128, two query tiles per item (the single issuer
    // sits behind its own commits and waits while the other tile's P is
    // ready: 0.67 vs 0.73 of peak on 128K calls, 0.46 vs 0.50 on 8K).
    const bool two = !c->geo.fp8 && p.nq == 2 && c->cfg.head_dim == 128;
    // speculative exponentials (SPEC) for calls whose items average more
    // than kSpecTilesPerItem tiles
    bool spec = false;
    if (two) {
        int64_t tiles_total = 0;
        for (const Cand& cd : cands) tiles_total += cd.item.w & 0xFFFFF;
        spec = tiles_total > kSpecTilesPerItem * (int64_t)n_items;
    }
    cudaError_t e = cudaSuccess;
    if (!inl) {
        p.items = c->ws.tiles;
        p.cta_off = reinterpret_cast<const int32_t*>(c->ws.tiles + n_items);
        e = stage_copy(c, si, c->ws.tiles, words * sizeof(int4), stream);
        if (e != cudaSuccess) return cuda_fail(e, "prefill work list upload");
    }
    CUtensorMap tq, tk, tv;
    std::string err;
    const int D = c->cfg.head_dim;
    if (!encode_tmap_2d(&tq, q, (uint64_t)c->cfg.num_q_heads * D, T,
                        (uint64_t)c->cfg.num_q_heads * D * 2, 64, 128, true, &err) ||
        !encode_tmap_2d(&tk, k, (uint64_t)c->cfg.num_kv_heads * D, T,
                        (uint64_t)c->cfg.num_kv_heads * D * 2, 64, 128, true, &err) ||
        !encode_tmap_2d(&tv, v, (uint64_t)c->cfg.num_kv_heads * D, T,
                        (uint64_t)c->cfg.num_kv_heads * D * 2, 64, 128, true, &err))
        return fail(SP_ERR_CUDA, err);
    launch_mark_start(c, stream);
#define SP_PF(DD, PP) \
    if (D == DD && P == PP) e = launch_prefill_t<DD, PP>(c, p, grid, tq, tk, tv, stream); else
#define SP_PF2(PP) \
    if (P == PP) e = spec ? launch_prefill_t<128, PP, false, true, true>(c, p, grid, tq, tk, tv, stream) \
                          : launch_prefill_t<128, PP, false, true>(c, p, grid, tq, tk, tv, stream); else
#define SP_PF8(PP) \
    if (D == 128 && P == PP) e = launch_prefill_t<128, PP, true>(c, p, grid, tq, tk, tv, stream); else
    if (c->geo.fp8) {   // FP8 pages (head_dim 128, checked at create)
        SP_PF8(16) SP_PF8(32) SP_PF8(64) SP_PF8(128)
        e = cudaErrorInvalidValue;
    } else if (two) {   // head_dim 128, two query tiles
        SP_PF2(16) SP_PF2(32) SP_PF2(64) SP_PF2(128)
        e = cudaErrorInvalidValue;
    } else {
        SP_PF(64, 16) SP_PF(64, 32) SP_PF(64, 64) SP_PF(64, 128)
        SP_PF(128, 16) SP_PF(128, 32) SP_PF(128, 64) SP_PF(128, 128)
        e = cudaErrorInvalidValue;
    }
#undef SP_PF
#undef SP_PF2
#undef SP_PF8
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    if (!groups.empty()) {
        std::unique_ptr<MergeParams> mp(new MergeParams());
        mp->n_groups = (int32_t)groups.size();
        mp->hq = c->cfg.num_q_heads;
        mp->split_o = p.split_o;
        mp->split_ml = p.split_ml;
        mp->out = out;
        mp->lse = lse;
        std::copy(groups.begin(), groups.end(), mp->groups);
        const dim3 mg((unsigned)groups.size(), (unsigned)p.nq, (unsigned)(D / 32));
        if (D == 128) k_prefill_merge<128><<<mg, 128, 0, stream>>>(*mp);
        else k_prefill_merge<64><<<mg, 128, 0, stream>>>(*mp);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "prefill merge launch");
    }
    launch_mark_end(c, stream);
    return SP_OK;
}

cudaError_t launch_prefill_counts(const sp_cache* c, int seq, int layer, int h,
                                  const int64_t* pos, int n, int32_t* out, cudaStream_t s) {
    k_prefill_counts<<<(n + 127) / 128, 128, 0, s>>>(c->meta, c->geo, seq, layer, h, pos, n, out);
    return cudaGetLastError();
}

}  // namespace sp
