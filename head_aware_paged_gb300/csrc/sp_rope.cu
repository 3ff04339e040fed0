// sp_rope.cu -- RoPE realignment of stored K rows (the first step of the
// news summary's Elastic Sparsity recovery, "RoPE position alignment": a
// segment of KV computed at one position is reused at another, so the
// rotation baked into its keys must move with it).
//
// Rotary embedding with frequencies theta^(-2i/d), the "rotate half" pairing
// (element i with element i + d/2).  Moving a key by delta positions is the
// same plane rotation by delta * theta^(-2i/d) for every row, so the host
// computes the d/2 (cos, sin) pairs once in double precision and the kernel
// is a pure streaming rotation: read a row of K, rotate, write it back.  It
// is HBM-bound: 2 * 2d bytes per rotated row (read + write); V is untouched.
#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

namespace {

// Position held by unit slot us (the rule of slot_position in sp_rules.h, in
// 32-bit arithmetic: positions and slots are below 2^31).  held_idx is the
// number of RETRIEVAL indices below n.
__device__ __forceinline__ int32_t slot_pos32(const UnitPol& u, const int32_t* idx, int32_t us,
                                              int32_t n, int32_t held_idx, int P) {
    if (u.kind == kGlobal) return us < n ? us : -1;
    if (u.kind == kLocal) {
        const int32_t base = u.sink_pages * P;
        if (us < base) return us < min(n, u.sink) ? us : -1;
        const int32_t q = us - base, ring_slots = u.ring * P;
        if (q >= ring_slots) return -1;
        const int32_t newest = n - 1 - u.sink;       // largest offset t - sink written
        if (newest < q) return -1;
        return u.sink + q + ((newest - q) / ring_slots) * ring_slots;
    }
    return us < held_idx ? idx[us] : -1;
}

// 8 bf16 pairs (x: elements i .. i+7, y: elements i+d/2 .. i+d/2+7) rotated by
// the angles of frequencies i .. i+7.
__device__ __forceinline__ void rotate8(uint4& xa, uint4& yb, const float* cs, const float* sn) {
    uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w}, yw[4] = {yb.x, yb.y, yb.z, yb.w};
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&xw[e]);
        const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162*>(&yw[e]);
        const float x0 = __low2float(x), x1 = __high2float(x);
        const float y0 = __low2float(y), y1 = __high2float(y);
        const float c0 = cs[2 * e], s0 = sn[2 * e], c1 = cs[2 * e + 1], s1 = sn[2 * e + 1];
        xw[e] = pack_bf16(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
        yw[e] = pack_bf16(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
    }
    xa = make_uint4(xw[0], xw[1], xw[2], xw[3]);
    yb = make_uint4(yw[0], yw[1], yw[2], yw[3]);
}

// One block per (unit, page) of the call, grid-strided: the unit comes from
// a binary search of the page offsets.  A work item is 8 frequency pairs of
// one row: a 16-byte load from each half of the row, the rotation, two
// 16-byte stores.
__global__ void __launch_bounds__(256)
k_rope(const __grid_constant__ RopeParams p, __nv_bfloat16* kpool) {
    const Geo& g = p.geo;
    const int P = g.page, D = g.d, half = D / 2;
    const int chunks = half / 8;                     // work items per row
    const int items = P * chunks;
    const int32_t lo = (int32_t)min64(p.pos_lo, (int64_t)INT32_MAX);
    const int32_t hi = (int32_t)min64(p.pos_hi, (int64_t)INT32_MAX);
    const int32_t total = p.page_off[p.n_units];
    for (int32_t blk = blockIdx.x; blk < total; blk += gridDim.x) {
        int a = 0, z = p.n_units - 1;                // unit with page_off[u] <= blk < page_off[u+1]
        while (a < z) {
            const int mid = (a + z + 1) >> 1;
            if (p.page_off[mid] <= blk) a = mid; else z = mid - 1;
        }
        const int u = a, pg = blk - p.page_off[u];
        const int seq = p.unit_seq[u], h = p.unit_head[u];
        const int32_t n = p.unit_n[u];
        const int64_t urow = g.unit_row(seq, p.layer, h);
        const UnitPol pol = p.meta.pol[urow];
        const int32_t* idx = p.meta.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
        // RETRIEVAL: how many indices lie below n (the same for the whole block)
        const int32_t held_idx = pol.kind == kRetrieval ? (int32_t)count_below(idx, pol.n_idx, n) : 0;
        const int32_t phys = p.meta.ptab[urow * g.max_pages_unit + pg];
        if (phys < 0 || phys >= g.num_pages) {       // same for the whole block
            if (threadIdx.x == 0) atomicOr(p.meta.status, kStatusBadPage);
            continue;
        }
        for (int w = threadIdx.x; w < items; w += blockDim.x) {
            const int row = w / chunks, c = w - row * chunks;
            const int32_t pos = slot_pos32(pol, idx, pg * P + row, n, held_idx, P);
            if (pos < 0 || pos < lo || pos >= hi) continue;
            __nv_bfloat16* r = kpool + ((int64_t)phys * P + row) * D;
            const int i0 = c * 8;
            uint4* px = reinterpret_cast<uint4*>(r + i0);
            uint4* py = reinterpret_cast<uint4*>(r + half + i0);
            uint4 x = *px, y = *py;
            rotate8(x, y, p.cs + i0, p.sn + i0);
            *px = x;
            *py = y;
        }
    }
}

}  // namespace

static_assert(sizeof(RopeParams) <= 32000, "RopeParams must fit the kernel parameter space");

cudaError_t launch_rope(const sp_cache* c, const RopeParams& p, cudaStream_t s) {
    const int32_t total = p.page_off[p.n_units];
    if (total <= 0) return cudaSuccess;
    const int grid = total < 16 * c->num_sms ? total : 16 * c->num_sms;
    k_rope<<<grid, 256, 0, s>>>(p, c->kpool);
    return cudaGetLastError();
}

}  // namespace sp
