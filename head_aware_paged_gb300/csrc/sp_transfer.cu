// sp_transfer.cu -- pack / unpack of one sequence's trimmed pages for a
// prefill/decode-disaggregated transfer (news summary, "system gains": in the
// PD-separated setting the head-aware layout cuts KV transfer bytes by up to
// 6.3x, because only the tokens each head keeps travel).
//
// The packed payload holds, for every (layer, KV head) unit in order, the
// unit's retained K rows then its retained V rows, each in position order;
// a header in front of it (written by the host) records the layout, the
// policies and per-unit row and block offsets.  One kernel copies in either
// direction between the page pool and the payload; it is HBM-bound
// (2 * 2d bytes moved per retained token per head, read + write).
#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

namespace {

// Position of the r-th retained row (position order) of a unit holding n
// tokens, and the unit slot that holds it.
__device__ __forceinline__ void row_slot(const UnitPol& u, const int32_t* idx, int32_t r,
                                         int32_t n, int32_t rows, int P, int32_t& pos,
                                         int32_t& slot) {
    if (u.kind == kGlobal) {
        pos = r;
        slot = r;
    } else if (u.kind == kLocal) {
        const int32_t a = min(n, u.sink);              // sink rows, then the newest rows
        pos = r < a ? r : n - (rows - a) + (r - a);
        slot = pos < u.sink ? pos : u.sink_pages * P + (pos - u.sink) % (u.ring * P);
    } else {
        pos = idx[r];
        slot = r;
    }
}

__global__ void __launch_bounds__(256)
k_transfer(const __grid_constant__ TransferParams p, __nv_bfloat16* kpool, __nv_bfloat16* vpool) {
    const Geo& g = p.geo;
    const int D = g.d, P = g.page;
    const int vec = D / 8;                             // 16-byte chunks per row
    for (int64_t blk = blockIdx.x; blk < p.total_blocks; blk += gridDim.x) {
        int a = 0, z = p.n_units - 1;                  // unit with blk_off[u] <= blk < blk_off[u+1]
        while (a < z) {
            const int mid = (a + z + 1) >> 1;
            if (p.units[mid].blk_off <= blk) a = mid; else z = mid - 1;
        }
        const PackUnit un = p.units[a];
        const int layer = a / g.hkv, h = a - layer * g.hkv;
        const int64_t urow = g.unit_row(p.seq, layer, h);
        const UnitPol pol = p.meta.pol[urow];
        const int32_t* idx = p.meta.idx + (int64_t)p.seq * g.max_idx_per_seq + pol.idx_off;
        const int32_t* ptab = p.meta.ptab + urow * g.max_pages_unit;
        const int32_t n = (int32_t)p.n_layer[layer];
        const int32_t rows = (int32_t)un.rows;
        const int32_t r0 = (int32_t)(blk - un.blk_off) * kTransferRows;
        const int32_t nr = min(kTransferRows, rows - r0);
        __nv_bfloat16* kblk = p.payload + 2 * un.row_off * D;     // the unit's K rows
        __nv_bfloat16* vblk = kblk + (int64_t)rows * D;           // then its V rows
        for (int w = threadIdx.x; w < nr * vec * 2; w += blockDim.x) {
            const int kv = w / (nr * vec);             // 0 = K, 1 = V
            const int rem = w - kv * nr * vec;
            const int rr = rem / vec, c = rem - rr * vec;
            const int32_t r = r0 + rr;
            int32_t pos, slot;
            row_slot(pol, idx, r, n, rows, P, pos, slot);
            const int32_t phys = ptab[slot / P];
            if (phys < 0 || phys >= g.num_pages) {
                atomicOr(p.meta.status, kStatusBadPage);
                continue;
            }
            __nv_bfloat16* pool = (kv ? vpool : kpool) + ((int64_t)phys * P + slot % P) * D + c * 8;
            __nv_bfloat16* pay = (kv ? vblk : kblk) + (int64_t)r * D + c * 8;
            if (p.unpack) *reinterpret_cast<uint4*>(pool) = *reinterpret_cast<const uint4*>(pay);
            else *reinterpret_cast<uint4*>(pay) = *reinterpret_cast<const uint4*>(pool);
        }
    }
}

}  // namespace

cudaError_t launch_transfer(const sp_cache* c, const TransferParams& p, cudaStream_t s) {
    if (p.total_blocks <= 0) return cudaSuccess;
    const int64_t cap = 16LL * c->num_sms;
    const int grid = (int)(p.total_blocks < cap ? p.total_blocks : cap);
    k_transfer<<<grid, 256, 0, s>>>(p, c->kpool, c->vpool);
    return cudaGetLastError();
}

}  // namespace sp
