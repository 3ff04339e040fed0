// sp_storage.cu -- page-pool allocator, page-table builder and KV
// scatter/trim kernels (write-time layout, RedKnot SegPagedAttention runtime
// article section 3; section 5 notes the layout must be built when KV is
// written, not per attention call).
//
// Allocation is deterministic: one call pops pages from a device free stack in
// unit order (sequences in call order, then KV heads), unit k taking the
// entries below top - o_k where o_k is the exclusive prefix sum of the page
// demands; release pushes a sequence's pages back in (layer, KV head, page)
// order.  The host mirrors the stack height, so every capacity check happens
// before launch and the kernels never fail for lack of pages.
#include "sp_internal.h"
#include "sp_device.cuh"

namespace sp {

namespace {

constexpr int kAllocThreads = 1024;

// In-place exclusive scan of a[0..n) by one CTA; returns the total.
__device__ int32_t block_exclusive_scan(int32_t* a, int n, int32_t* warp_sums) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int32_t s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    // inclusive scan of s across the warp
    const int lane = tid & 31, warp = tid >> 5;
    int32_t x = s;
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = (nt + 31) >> 5;
        int32_t w = lane < nw ? warp_sums[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) warp_sums[lane] = w;   // inclusive per-warp totals
    }
    __syncthreads();
    int32_t off = (warp > 0 ? warp_sums[warp - 1] : 0) + x - s;
    const int32_t total = warp_sums[((nt + 31) >> 5) - 1];
    for (int i = lo; i < hi; ++i) {
        const int32_t v = a[i];
        a[i] = off;
        off += v;
    }
    __syncthreads();
    return total;
}

__global__ void k_init_stack(int32_t* fstack, int32_t num_pages) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < num_pages;
         i += (int64_t)gridDim.x * blockDim.x)
        fstack[i] = num_pages - 1 - (int32_t)i;
}

// Page demand, scan and pops for one append/build call (one CTA).
__global__ void __launch_bounds__(kAllocThreads)
k_alloc(Meta m, Geo g, CallSeqs cs, int layer, int32_t top) {
    extern __shared__ int32_t sm[];
    __shared__ int32_t warp_sums[32];
    const int n_units = cs.n * g.hkv;
    int32_t* dem = sm;             // demand, then offsets
    int32_t* onp = sm + n_units;   // pages held before the call
    for (int u = threadIdx.x; u < n_units; u += blockDim.x) {
        const int b = u / g.hkv, h = u % g.hkv;
        const int seq = cs.seq[b];
        const int64_t row = g.unit_row(seq, layer, h);
        const UnitPol pol = m.pol[row];
        const int32_t* idx = m.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
        const int64_t want = unit_pages(pol, idx, (int64_t)cs.n_old[b] + cs.cnt[b], g.page);
        const int32_t have = m.npages[row];
        dem[u] = (int32_t)(want - have);
        onp[u] = have;
        if (want < have || want > g.max_pages_unit) atomicOr(m.status, kStatusBadState);
    }
    __syncthreads();
    const int32_t total = block_exclusive_scan(dem, n_units, warp_sums);
    if (total > top) {                       // the host checked this; never expected
        if (threadIdx.x == 0) atomicOr(m.status, kStatusBadState);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int u = warp; u < n_units; u += nw) {
        const int b = u / g.hkv, h = u % g.hkv;
        const int64_t row = g.unit_row(cs.seq[b], layer, h);
        const int32_t off = dem[u];
        const int32_t cnt = (u + 1 < n_units ? dem[u + 1] : total) - off;
        int32_t* tab = m.ptab + row * g.max_pages_unit + onp[u];
        for (int j = lane; j < cnt; j += 32) tab[j] = m.fstack[top - 1 - (off + j)];
        if (lane == 0) m.npages[row] = onp[u] + cnt;
    }
    for (int b = threadIdx.x; b < cs.n; b += blockDim.x)
        m.seqlen[(int64_t)cs.seq[b] * g.layers + layer] = cs.n_old[b] + cs.cnt[b];
    if (threadIdx.x == 0) m.status[1] = top - total;
}

// 8 bf16 values (one 16-byte vector) -> 8 e4m3 codes of x * inv[i] (fp32
// product, then round to nearest even, saturated at +-448), in element order.
__device__ __forceinline__ uint2 quant_e4m3x8(int4 x, const float* inv) {
    const uint32_t w[4] = {(uint32_t)x.x, (uint32_t)x.y, (uint32_t)x.z, (uint32_t)x.w};
    uint32_t out[2] = {0u, 0u};
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
        const float lo = __low2float(p2) * __ldg(inv + 2 * e);
        const float hi = __high2float(p2) * __ldg(inv + 2 * e + 1);
        uint16_t code;   // first operand goes to the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(hi), "f"(lo));
        out[e >> 1] |= (uint32_t)code << (16 * (e & 1));
    }
    return make_uint2(out[0], out[1]);
}

// Copy the retained rows of each unit into its pages (16-byte vectors).
__global__ void __launch_bounds__(256)
k_scatter(Meta m, Geo g, CallSeqs cs, int layer, const __nv_bfloat16* __restrict__ k,
          const __nv_bfloat16* __restrict__ v, int64_t row_stride,
          __nv_bfloat16* __restrict__ kpool, __nv_bfloat16* __restrict__ vpool) {
    const int u = blockIdx.y;
    const int b = u / g.hkv, h = u % g.hkv;
    const int seq = cs.seq[b];
    const int64_t n_old = cs.n_old[b], n_new = n_old + cs.cnt[b];
    const int64_t row = g.unit_row(seq, layer, h);
    const UnitPol pol = m.pol[row];
    const int32_t* idx = m.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
    const ItemRanges r = retained_items(pol, idx, n_old, n_new, g.page);
    const int64_t n0 = r.hi[0] - r.lo[0], n1 = r.hi[1] - r.lo[1];
    const int vecs = g.d / 8;
    const int64_t total = (n0 + n1) * vecs;
    const int32_t* tab = m.ptab + row * g.max_pages_unit;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = e / vecs;
        const int c = (int)(e - j * vecs);
        const int64_t item = j < n0 ? r.lo[0] + j : r.lo[1] + (j - n0);
        int64_t t, us;
        if (pol.kind == kRetrieval) { t = idx[item]; us = item; }
        else { t = item; us = unit_slot(pol, idx, t, g.page); }
        const int32_t page = tab[us / g.page];
        if (page < 0 || page >= g.num_pages) { atomicOr(m.status, kStatusBadPage); continue; }
        const int64_t src = (cs.row0[b] + (t - n_old)) * row_stride + (int64_t)h * g.d + c * 8;
        const int64_t dst = ((int64_t)page * g.page + us % g.page) * g.d + c * 8;
        const int4 kv = __ldg(reinterpret_cast<const int4*>(k + src));
        const int4 vv = __ldg(reinterpret_cast<const int4*>(v + src));
        if (!g.fp8) {
            *reinterpret_cast<int4*>(kpool + dst) = kv;
            *reinterpret_cast<int4*>(vpool + dst) = vv;
        } else {
            // e4m3 codes of x * (1 / scale), channel by channel (8 bytes per side)
            const int64_t so = ((int64_t)layer * g.hkv + h) * g.d + c * 8;
            uint8_t* kp = reinterpret_cast<uint8_t*>(kpool) + dst;
            uint8_t* vp = reinterpret_cast<uint8_t*>(vpool) + dst;
            *reinterpret_cast<uint2*>(kp) = quant_e4m3x8(kv, m.kinv + so);
            *reinterpret_cast<uint2*>(vp) = quant_e4m3x8(vv, m.vinv + so);
        }
    }
}

// Push every page of one sequence back onto the free stack (one CTA).
__global__ void __launch_bounds__(kAllocThreads)
k_release(Meta m, Geo g, int seq, int32_t top) {
    extern __shared__ int32_t sm[];
    __shared__ int32_t warp_sums[32];
    const int n_units = g.layers * g.hkv;
    int32_t* cnt = sm;
    for (int u = threadIdx.x; u < n_units; u += blockDim.x)
        cnt[u] = m.npages[(int64_t)seq * n_units + u];
    __syncthreads();
    const int32_t total = block_exclusive_scan(cnt, n_units, warp_sums);
    if ((int64_t)top + total > g.num_pages) {
        if (threadIdx.x == 0) atomicOr(m.status, kStatusBadState);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int u = warp; u < n_units; u += nw) {
        const int64_t row = (int64_t)seq * n_units + u;
        const int32_t off = cnt[u];
        const int32_t np = (u + 1 < n_units ? cnt[u + 1] : total) - off;
        const int32_t* tab = m.ptab + row * g.max_pages_unit;
        for (int j = lane; j < np; j += 32) m.fstack[top + off + j] = tab[j];
        __syncwarp();
        if (lane == 0) m.npages[row] = 0;
    }
    for (int l = threadIdx.x; l < g.layers; l += blockDim.x)
        m.seqlen[(int64_t)seq * g.layers + l] = 0;
    if (threadIdx.x == 0) m.status[1] = top + total;
}

// Device view of one unit's table: page ids and the position of every slot.
__global__ void k_export(Meta m, Geo g, int seq, int layer, int h, int32_t* out_ids,
                         int32_t* out_pos) {
    const int64_t row = g.unit_row(seq, layer, h);
    const UnitPol pol = m.pol[row];
    const int32_t* idx = m.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
    const int32_t np = m.npages[row];
    const int64_t n = m.seqlen[(int64_t)seq * g.layers + layer];
    for (int j = threadIdx.x; j < np; j += blockDim.x)
        out_ids[j] = m.ptab[row * g.max_pages_unit + j];
    for (int64_t us = threadIdx.x; us < (int64_t)np * g.page; us += blockDim.x)
        out_pos[us] = (int32_t)slot_position(pol, idx, us, n, g.page);
}

// For positions i = n - 1 (a decode query): count the slots the decode kernel
// streams whose stored token is in V(i); -1 for other positions.
__global__ void k_decode_counts(Meta m, Geo g, int seq, int layer, int h,
                                const int64_t* pos, int npos, int32_t* out) {
    const int64_t row = g.unit_row(seq, layer, h);
    const UnitPol pol = m.pol[row];
    const int32_t* idx = m.idx + (int64_t)seq * g.max_idx_per_seq + pol.idx_off;
    const int64_t n = m.seqlen[(int64_t)seq * g.layers + layer];
    const int32_t np = m.npages[row];
    for (int k = threadIdx.x; k < npos; k += blockDim.x) {
        const int64_t i = pos[k];
        if (i != n - 1) { out[k] = -1; continue; }
        const SlotRanges r = decode_ranges(pol, idx, i, g.page);
        int32_t c = 0;
        for (int q = 0; q < r.count; ++q)
            for (int64_t us = r.lo[q]; us < r.hi[q]; ++us) {
                if (us >= (int64_t)np * g.page) { c = -2; break; }
                const int64_t p = slot_position(pol, idx, us, n, g.page);
                bool vis = p >= 0 && p <= i;
                if (pol.kind == kLocal) vis = vis && (p < pol.sink || p > i - pol.window);
                c += vis ? 1 : 0;
            }
        out[k] = c;
    }
}

}  // namespace

cudaError_t launch_init_meta(const sp_cache* c, cudaStream_t s) {
    k_init_stack<<<256, 256, 0, s>>>(c->meta.fstack, c->cfg.num_pages);
    return cudaGetLastError();
}

cudaError_t launch_alloc(const sp_cache* c, const CallSeqs& cs, int layer, int32_t top,
                         cudaStream_t s) {
    const size_t smem = (size_t)cs.n * c->geo.hkv * 2 * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_alloc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    k_alloc<<<1, kAllocThreads, smem, s>>>(c->meta, c->geo, cs, layer, top);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const sp_cache* c, const CallSeqs& cs, int layer,
                           const __nv_bfloat16* k, const __nv_bfloat16* v,
                           int64_t row_stride, int64_t max_items, cudaStream_t s) {
    const int64_t work = max_items * (c->geo.d / 8);
    if (work <= 0) return cudaSuccess;
    int64_t gx = (work + 255) / 256;
    if (gx > 4096) gx = 4096;
    dim3 grid((unsigned)gx, (unsigned)(cs.n * c->geo.hkv));
    k_scatter<<<grid, 256, 0, s>>>(c->meta, c->geo, cs, layer, k, v, row_stride,
                                   c->kpool, c->vpool);
    return cudaGetLastError();
}

cudaError_t launch_release(const sp_cache* c, int seq, int32_t top, cudaStream_t s) {
    const size_t smem = (size_t)c->geo.layers * c->geo.hkv * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_release, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    k_release<<<1, kAllocThreads, smem, s>>>(c->meta, c->geo, seq, top);
    return cudaGetLastError();
}

cudaError_t launch_export(const sp_cache* c, int seq, int layer, int h, int32_t* out_ids,
                          int32_t* out_pos, cudaStream_t s) {
    k_export<<<1, 256, 0, s>>>(c->meta, c->geo, seq, layer, h, out_ids, out_pos);
    return cudaGetLastError();
}

cudaError_t launch_decode_counts(const sp_cache* c, int seq, int layer, int h,
                                 const int64_t* pos, int n, int32_t* out, cudaStream_t s) {
    k_decode_counts<<<1, 256, 0, s>>>(c->meta, c->geo, seq, layer, h, pos, n, out);
    return cudaGetLastError();
}

}  // namespace sp
