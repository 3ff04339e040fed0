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

// FP8 pages: 16 pairs held as e4m3 codes (x: elements i .. i+15, y: i+d/2 ..
// i+d/2+15).  Each element is dequantised with its channel's K scale, the
// pair rotated in fp32 with every product and sum rounded separately (no
// fused multiply-add, so the result is one fixed sequence of roundings) and
// requantised like a write: e4m3(v * fp32(1 / scale)), nearest even,
// saturating.
__device__ __forceinline__ float f32_of_e4m3(uint32_t code) {
    const uint32_t h2 = f16x2_of_e4m3x2(code & 0xFFu);
    return __half2float(*reinterpret_cast<const __half*>(&h2));
}
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void rotate16_fp8(uint4& xa, uint4& yb, const float* cs, const float* sn,
                                             const float* sx, const float* sy, const float* ix,
                                             const float* iy) {
    uint32_t xw[4] = {xa.x, xa.y, xa.z, xa.w}, yw[4] = {yb.x, yb.y, yb.z, yb.w};
    #pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t xo = 0, yo = 0;
        #pragma unroll
        for (int e = 0; e < 4; e += 2) {
            float xr[2], yr[2];
            #pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int k = 4 * w + e + t;
                const float x = __fmul_rn(f32_of_e4m3(xw[w] >> (8 * (e + t))), sx[k]);
                const float y = __fmul_rn(f32_of_e4m3(yw[w] >> (8 * (e + t))), sy[k]);
                const float xn = __fsub_rn(__fmul_rn(x, cs[k]), __fmul_rn(y, sn[k]));
                const float yn = __fadd_rn(__fmul_rn(y, cs[k]), __fmul_rn(x, sn[k]));
                xr[t] = __fmul_rn(xn, ix[k]);
                yr[t] = __fmul_rn(yn, iy[k]);
            }
            xo |= e4m3x2_of(xr[0], xr[1]) << (8 * e);
            yo |= e4m3x2_of(yr[0], yr[1]) << (8 * e);
        }
        xw[w] = xo;
        yw[w] = yo;
    }
    xa = make_uint4(xw[0], xw[1], xw[2], xw[3]);
    yb = make_uint4(yw[0], yw[1], yw[2], yw[3]);
}

// One block per (unit, page) of the call, grid-strided: the unit comes from
// a binary search of the page offsets.  A work item is 8 frequency pairs of
// one row (16 for FP8 pages): a 16-byte load from each half of the row, the
// rotation, two 16-byte stores.
template <bool F8>
__global__ void __launch_bounds__(256)
k_rope(const __grid_constant__ RopeParams p, void* kpool_) {
    const Geo& g = p.geo;
    const int P = g.page, D = g.d, half = D / 2;
    constexpr int kPairs = F8 ? 16 : 8;              // frequency pairs per work item
    const int chunks = half / kPairs;                // work items per row
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
            const int i0 = c * kPairs;
            if constexpr (F8) {
                uint8_t* r = static_cast<uint8_t*>(kpool_) + ((int64_t)phys * P + row) * D;
                uint4* px = reinterpret_cast<uint4*>(r + i0);
                uint4* py = reinterpret_cast<uint4*>(r + half + i0);
                uint4 x = *px, y = *py;
                const int64_t so = ((int64_t)p.layer * g.hkv + h) * D;
                rotate16_fp8(x, y, p.cs + i0, p.sn + i0, p.meta.kscale + so + i0,
                             p.meta.kscale + so + half + i0, p.meta.kinv + so + i0,
                             p.meta.kinv + so + half + i0);
                *px = x;
                *py = y;
            } else {
                __nv_bfloat16* r = static_cast<__nv_bfloat16*>(kpool_) + ((int64_t)phys * P + row) * D;
                uint4* px = reinterpret_cast<uint4*>(r + i0);
                uint4* py = reinterpret_cast<uint4*>(r + half + i0);
                uint4 x = *px, y = *py;
                rotate8(x, y, p.cs + i0, p.sn + i0);
                *px = x;
                *py = y;
            }
        }
    }
}

}  // namespace

static_assert(sizeof(RopeParams) <= 32000, "RopeParams must fit the kernel parameter space");

cudaError_t launch_rope(const sp_cache* c, const RopeParams& p, cudaStream_t s) {
    const int32_t total = p.page_off[p.n_units];
    if (total <= 0) return cudaSuccess;
    const int grid = total < 16 * c->num_sms ? total : 16 * c->num_sms;
    if (c->geo.fp8) k_rope<true><<<grid, 256, 0, s>>>(p, c->kpool);
    else k_rope<false><<<grid, 256, 0, s>>>(p, c->kpool);
    return cudaGetLastError();
}

}  // namespace sp
