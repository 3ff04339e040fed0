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
// (2 * 2d bytes per retained token per head and side, read + write; half
// that for FP8 pages).
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
k_transfer(const __grid_constant__ TransferParams p, uint8_t* kpool, uint8_t* vpool) {
    const Geo& g = p.geo;
    const int P = g.page;
    const int row_bytes = g.d * (g.fp8 ? 1 : 2);
    const int vec = row_bytes / 16;                    // 16-byte chunks per row
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
        uint8_t* kblk = p.payload + 2 * un.row_off * row_bytes;   // the unit's K rows
        uint8_t* vblk = kblk + (int64_t)rows * row_bytes;           // then its V rows
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
            uint8_t* pool = (kv ? vpool : kpool) + ((int64_t)phys * P + slot % P) * row_bytes + c * 16;
            uint8_t* pay = (kv ? vblk : kblk) + (int64_t)r * row_bytes + c * 16;
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
    k_transfer<<<grid, 256, 0, s>>>(p, reinterpret_cast<uint8_t*>(c->kpool),
                                    reinterpret_cast<uint8_t*>(c->vpool));
    return cudaGetLastError();
}

}  // namespace sp
