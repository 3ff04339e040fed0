// sp_api.cu -- host side of the C ABI declared in include/segpaged.h:
// argument validation, the host mirror of lengths / page counts / policies,
// device-memory layout over the caller's buffers, and kernel launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <mutex>

#include "sp_device.cuh"
#include "sp_internal.h"
#include "sp_prefill.h"

namespace sp {

namespace {
thread_local std::string g_last_error;
constexpr int kMaxDecodeCtas = 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    int32_t max_pages_unit = 0;
    size_t pol = 0, npages = 0, seqlen = 0, ptab = 0, idx = 0, fstack = 0, status = 0,
           scales = 0, meta_total = 0;
    size_t tiles = 0, tile_ctr = 0, part_o = 0, part_ml = 0, counters = 0, scratch = 0,
           split_o = 0, split_ml = 0, ws_total = 0;
    int64_t max_tiles = 0, max_parts = 0, max_counter_units = 0, scratch_ints = 0;
    size_t pool_total = 0;
};

sp_status check_config(const sp_config* c) {
    if (!c) return fail(SP_ERR_INVALID_ARG, "config is null");
    if (c->num_layers < 1 || c->num_q_heads < 1 || c->num_kv_heads < 1)
        return fail(SP_ERR_INVALID_ARG, "num_layers, num_q_heads and num_kv_heads must be >= 1");
    if (c->num_q_heads % c->num_kv_heads != 0)
        return fail(SP_ERR_INVALID_ARG, "num_q_heads must be a multiple of num_kv_heads");
    if (c->num_q_heads / c->num_kv_heads > 16)
        return fail(SP_ERR_UNSUPPORTED, "more than 16 query heads per KV head");
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(SP_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128)
        return fail(SP_ERR_UNSUPPORTED, "page_size must be 16, 32, 64 or 128");
    if (c->max_seqs < 1 || c->max_seq_len < 1 || c->num_pages < 1 || c->max_tokens < 1 ||
        c->max_batch < 1 || c->max_idx_per_seq < 0)
        return fail(SP_ERR_INVALID_ARG, "capacities must be positive");
    if ((int64_t)c->num_pages * c->page_size >= (int64_t(1) << 31))
        return fail(SP_ERR_UNSUPPORTED, "num_pages * page_size must stay below 2^31 rows");
    if (c->max_batch > kMaxCallSeqs)
        return fail(SP_ERR_UNSUPPORTED, "max_batch above 512");
    if ((int64_t)c->max_batch * c->num_kv_heads > kMaxDecodeUnits)
        return fail(SP_ERR_UNSUPPORTED, "max_batch * num_kv_heads above 4096");
    if ((int64_t)c->num_layers * c->num_kv_heads > kMaxPolicyUnits)
        return fail(SP_ERR_UNSUPPORTED, "num_layers * num_kv_heads above 8192");
    if (c->kv_dtype != SP_KV_BF16 && c->kv_dtype != SP_KV_FP8_E4M3)
        return fail(SP_ERR_INVALID_ARG, "unknown kv_dtype");
    if (c->kv_dtype == SP_KV_FP8_E4M3 && c->head_dim != 128)
        return fail(SP_ERR_UNSUPPORTED, "FP8 pages need head_dim 128");
    return SP_OK;
}

Layout make_layout(const sp_config* c) {
    Layout L;
    const int64_t S = c->max_seqs, NL = c->num_layers, H = c->num_kv_heads;
    const int64_t units = S * NL * H;
    L.max_pages_unit = (int32_t)((c->max_seq_len + c->page_size - 1) / c->page_size + 1);
    size_t o = 0;
    L.pol = o;     o = align_up(o + units * sizeof(UnitPol), 256);
    L.npages = o;  o = align_up(o + units * 4, 256);
    L.seqlen = o;  o = align_up(o + S * NL * 4, 256);
    L.ptab = o;    o = align_up(o + units * (size_t)L.max_pages_unit * 4, 256);
    L.idx = o;     o = align_up(o + S * (size_t)std::max(c->max_idx_per_seq, 1) * 4, 256);
    L.fstack = o;  o = align_up(o + (size_t)c->num_pages * 4, 256);
    L.status = o;  o = align_up(o + 64, 256);
    // FP8 scales and their reciprocals: k, v, 1/k, 1/v, each [layers][hkv][d] fp32
    L.scales = o;  o = align_up(o + 4 * (size_t)NL * H * c->head_dim * 4, 256);
    L.meta_total = o;
    const int group = c->num_q_heads / c->num_kv_heads;
    L.max_tiles = prefill_max_tiles(c);
    L.max_counter_units = (int64_t)c->max_batch * H;
    L.max_parts = L.max_counter_units + kMaxDecodeCtas;
    L.scratch_ints = std::max<int64_t>((int64_t)L.max_pages_unit * (1 + c->page_size), 3 * 65536);
    o = 0;
    L.tiles = o;    o = align_up(o + L.max_tiles * sizeof(int4), 256);
    L.tile_ctr = o; o = align_up(o + 64, 256);
    L.part_o = o;   o = align_up(o + L.max_parts * group * (size_t)c->head_dim * 4, 256);
    L.part_ml = o;  o = align_up(o + L.max_parts * group * 2 * 4, 256);
    L.counters = o; o = align_up(o + L.max_counter_units * 4, 256);
    L.scratch = o;  o = align_up(o + L.scratch_ints * 4, 256);
    L.split_o = o;  o = align_up(o + (size_t)kPrefillSplitSlots * 2 * 128 * c->head_dim * 4, 256);
    L.split_ml = o; o = align_up(o + (size_t)kPrefillSplitSlots * 2 * 128 * 2 * 4, 256);
    L.ws_total = o;
    L.pool_total = 2 * (size_t)c->num_pages * c->page_size * c->head_dim *
                   (c->kv_dtype == SP_KV_FP8_E4M3 ? 1 : 2);
    return L;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool valid_seq(const sp_cache* c, int32_t seq) { return seq >= 0 && seq < c->cfg.max_seqs; }

size_t unit_index(const sp_cache* c, int seq, int layer, int h) {
    return ((size_t)seq * c->cfg.num_layers + layer) * c->cfg.num_kv_heads + h;
}

const int32_t* host_idx(const sp_cache* c, int seq, const UnitPol& u) {
    return c->h_idx[seq].data() + u.idx_off;
}

// Shared by build and append: validate lengths, check pool capacity against
// the host mirror, then launch the allocator and the scatter kernel.
// Allocate pages for `counts[b]` new tokens of each listed sequence in
// `layer` (page-table build on the device) and advance the host mirror; the
// caller then launches the kernel that fills the new slots.  cs / max_items
// describe the call for that kernel.
sp_status alloc_tokens(sp_cache* c, int32_t layer, const int32_t* seqs, int32_t n_seqs,
                       const int64_t* counts, cudaStream_t stream, CallSeqs& cs,
                       int64_t& max_items, int64_t& rows) {
    std::memset(&cs, 0, sizeof(cs));
    cs.n = n_seqs;
    int64_t demand = 0;
    rows = 0;
    max_items = 0;
    for (int b = 0; b < n_seqs; ++b) {
        const int seq = seqs[b];
        const int64_t n_old = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
        const int64_t n_new = n_old + counts[b];
        if (n_new > c->cfg.max_seq_len)
            return fail(SP_ERR_INVALID_ARG, "sequence " + std::to_string(seq) +
                                                " would exceed max_seq_len");
        cs.seq[b] = seq;
        cs.n_old[b] = (int32_t)n_old;
        cs.cnt[b] = (int32_t)counts[b];
        cs.row0[b] = (int32_t)rows;
        rows += counts[b];
        for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
            const UnitPol& u = c->h_pol[unit_index(c, seq, layer, h)];
            const int32_t* idx = host_idx(c, seq, u);
            demand += unit_pages(u, idx, n_new, c->cfg.page_size) -
                      unit_pages(u, idx, n_old, c->cfg.page_size);
            const ItemRanges r = retained_items(u, idx, n_old, n_new, c->cfg.page_size);
            max_items = std::max(max_items, (r.hi[0] - r.lo[0]) + (r.hi[1] - r.lo[1]));
        }
    }
    if (demand > c->h_free)
        return fail(SP_ERR_OUT_OF_PAGES, "call needs " + std::to_string(demand) +
                                             " pages, " + std::to_string(c->h_free) + " free");
    if (rows == 0) return SP_OK;
    cudaError_t e = launch_alloc(c, cs, layer, (int32_t)c->h_free, stream);
    if (e != cudaSuccess) return cuda_fail(e, "allocator launch");
    c->h_free -= demand;
    for (int b = 0; b < n_seqs; ++b) {
        const int seq = seqs[b];
        c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer] += (int32_t)counts[b];
        for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
            const size_t ui = unit_index(c, seq, layer, h);
            const UnitPol& u = c->h_pol[ui];
            c->h_npages[ui] = (int32_t)unit_pages(u, host_idx(c, seq, u),
                                                  c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer],
                                                  c->cfg.page_size);
        }
    }
    return SP_OK;
}

sp_status write_tokens(sp_cache* c, int32_t layer, const int32_t* seqs, int32_t n_seqs,
                       const int64_t* counts, const __nv_bfloat16* k, const __nv_bfloat16* v,
                       int64_t row_stride, cudaStream_t stream) {
    CallSeqs cs;
    int64_t max_items = 0, rows = 0;
    sp_status s = alloc_tokens(c, layer, seqs, n_seqs, counts, stream, cs, max_items, rows);
    if (s != SP_OK || rows == 0) return s;
    cudaError_t e = launch_scatter(c, cs, layer, k, v, row_stride, max_items, stream);
    if (e != cudaSuccess) return cuda_fail(e, "scatter launch");
    return SP_OK;
}

// Rows a unit holding n tokens keeps (the retained set of the slot rules):
// GLOBAL every token, LOCAL the sink and the newest ring's worth, RETRIEVAL
// its listed positions below n.
int64_t retained_rows(const UnitPol& u, const int32_t* idx, int64_t n, int P) {
    if (n <= 0) return 0;
    if (u.kind == kGlobal) return n;
    if (u.kind == kLocal)
        return std::min<int64_t>(n, u.sink) + std::min<int64_t>(std::max<int64_t>(n - u.sink, 0),
                                                                (int64_t)u.ring * P);
    return count_below(idx, u.n_idx, n);
}

// UnitPol of a LOCAL / GLOBAL / RETRIEVAL class, as sp_set_policy encodes it.
UnitPol encode_unit(int64_t kind, int64_t sink, int64_t window, int32_t idx_off, int32_t n_idx,
                    int P) {
    UnitPol r{};
    r.kind = (int32_t)kind;
    if (kind == kLocal) {
        r.sink = (int32_t)sink;
        r.window = (int32_t)window;
        r.ring = (int32_t)((window + P - 1) / P + 1);
        r.sink_pages = (int32_t)((sink + P - 1) / P);
    } else if (kind == kRetrieval) {
        r.idx_off = idx_off;
        r.n_idx = n_idx;
    }
    return r;
}

size_t align_to(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

bool valid_layer(const sp_cache* c, int32_t l) { return l >= 0 && l < c->cfg.num_layers; }

sp_status check_seq_list(const sp_cache* c, const int32_t* seq_ids, int32_t n_seqs) {
    if (!seq_ids || n_seqs < 1) return fail(SP_ERR_INVALID_ARG, "empty sequence list");
    if (n_seqs > c->cfg.max_batch) return fail(SP_ERR_INVALID_ARG, "more sequences than max_batch");
    // duplicates through a sorted copy on the stack (n_seqs <= max_batch <=
    // kMaxCallSeqs): the check allocates nothing
    int32_t sorted[kMaxCallSeqs];
    for (int b = 0; b < n_seqs; ++b) {
        const int s = seq_ids[b];
        if (!valid_seq(c, s)) return fail(SP_ERR_INVALID_ARG, "sequence id out of range");
        if (!c->h_policy_set[s]) return fail(SP_ERR_INVALID_ARG, "sequence has no policy");
        sorted[b] = s;
    }
    std::sort(sorted, sorted + n_seqs);
    for (int b = 1; b < n_seqs; ++b)
        if (sorted[b] == sorted[b - 1]) return fail(SP_ERR_INVALID_ARG, "sequence listed twice");
    return SP_OK;
}

void* stage_acquire(sp_cache* c, size_t bytes, int* slot) {
    if (bytes > c->stage_bytes) return nullptr;
    const int si = c->stage_next;
    c->stage_next = (si + 1) % sp_cache::kStaging;
    if (cudaEventSynchronize(c->stage_ev[si]) != cudaSuccess) return nullptr;
    *slot = si;
    return c->stage_buf[si];
}

namespace {
// Staging buffer -> device memory, read by the SMs through the mapped host
// address: no copy engine is involved, so the upload never queues behind the
// caller's own large host<->device transfers on the copy engines.
__global__ void k_stage_copy(const int4* __restrict__ src, int4* __restrict__ dst, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}
}  // namespace

cudaError_t stage_copy(sp_cache* c, int slot, void* dst, size_t bytes, cudaStream_t s) {
    if (bytes % sizeof(int4) != 0 || (reinterpret_cast<uintptr_t>(dst) & 15)) return cudaErrorInvalidValue;
    const size_t n = bytes / sizeof(int4);
    if (n > 0) {
        const size_t blocks = std::min<size_t>((n + 255) / 256, (size_t)4 * c->num_sms);
        k_stage_copy<<<(unsigned)blocks, 256, 0, s>>>(c->stage_dev[slot], static_cast<int4*>(dst), n);
    }
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventRecord(c->stage_ev[slot], s);
    return e;
}

sp_status fail(sp_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

sp_status cuda_fail(cudaError_t e, const char* what) {
    g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
    return SP_ERR_CUDA;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128,
                    std::string* err, bool bytes) {
    auto fn = get_encode();
    if (!fn) { *err = "cuTensorMapEncodeTiled unavailable (no CUDA driver)"; return false; }
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { *err = "cuTensorMapEncodeTiled failed, code " + std::to_string((int)r); return false; }
    return true;
}

}  // namespace sp

using namespace sp;

extern "C" {

const char* sp_last_error(void) { return g_last_error.c_str(); }

sp_status sp_required_bytes(const sp_config* cfg, size_t* pool_bytes, size_t* meta_bytes,
                            size_t* ws_bytes) {
    sp_status s = check_config(cfg);
    if (s != SP_OK) return s;
    if (!pool_bytes || !meta_bytes || !ws_bytes) return fail(SP_ERR_INVALID_ARG, "null output");
    const Layout L = make_layout(cfg);
    *pool_bytes = L.pool_total;
    *meta_bytes = L.meta_total;
    *ws_bytes = L.ws_total;
    return SP_OK;
}

sp_status sp_cache_create(const sp_config* cfg, void* pool, void* meta, void* ws, sp_cache** out) {
    sp_status s = check_config(cfg);
    if (s != SP_OK) return s;
    if (!out) return fail(SP_ERR_INVALID_ARG, "null output handle");
    *out = nullptr;
    if (!pool || !meta || !ws) return fail(SP_ERR_INVALID_ARG, "null device buffer");
    if ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(meta) |
         reinterpret_cast<uintptr_t>(ws)) & 1023)
        return fail(SP_ERR_INVALID_ARG, "device buffers must be 1024-byte aligned");
    const Layout L = make_layout(cfg);
    sp_cache* c = new sp_cache();
    c->cfg = *cfg;
    Geo& g = c->geo;
    g.layers = cfg->num_layers; g.hq = cfg->num_q_heads; g.hkv = cfg->num_kv_heads;
    g.group = cfg->num_q_heads / cfg->num_kv_heads; g.d = cfg->head_dim; g.page = cfg->page_size;
    g.max_seqs = cfg->max_seqs; g.max_pages_unit = L.max_pages_unit;
    g.max_idx_per_seq = std::max(cfg->max_idx_per_seq, 1); g.num_pages = cfg->num_pages;
    g.fp8 = cfg->kv_dtype == SP_KV_FP8_E4M3 ? 1 : 0;
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) { delete c; return cuda_fail(e, "device query"); }
    // FP8 decode runs two CTAs per SM
    c->decode_ctas = std::min(c->num_sms * (g.fp8 ? 2 : 1), kMaxDecodeCtas);
    const size_t pool_half = (size_t)cfg->num_pages * cfg->page_size * cfg->head_dim;
    // (FP8 pages: the same pointers address bytes; kernels cast them)
    c->kpool = static_cast<__nv_bfloat16*>(pool);
    c->vpool = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(pool) + pool_half * (g.fp8 ? 1 : 2));
    uint8_t* mb = static_cast<uint8_t*>(meta);
    c->meta.pol = reinterpret_cast<UnitPol*>(mb + L.pol);
    c->meta.npages = reinterpret_cast<int32_t*>(mb + L.npages);
    c->meta.seqlen = reinterpret_cast<int32_t*>(mb + L.seqlen);
    c->meta.ptab = reinterpret_cast<int32_t*>(mb + L.ptab);
    c->meta.idx = reinterpret_cast<int32_t*>(mb + L.idx);
    c->meta.fstack = reinterpret_cast<int32_t*>(mb + L.fstack);
    c->meta.status = reinterpret_cast<int32_t*>(mb + L.status);
    {
        const size_t nsc = (size_t)cfg->num_layers * cfg->num_kv_heads * cfg->head_dim;
        float* sc = reinterpret_cast<float*>(mb + L.scales);
        c->meta.kscale = sc;
        c->meta.vscale = sc + nsc;
        c->meta.kinv = sc + 2 * nsc;
        c->meta.vinv = sc + 3 * nsc;
    }
    uint8_t* wb = static_cast<uint8_t*>(ws);
    c->ws.base = ws; c->ws.bytes = L.ws_total;
    c->ws.tiles = reinterpret_cast<int4*>(wb + L.tiles); c->ws.max_tiles = L.max_tiles;
    c->ws.tile_ctr = reinterpret_cast<int32_t*>(wb + L.tile_ctr);
    c->ws.part_o = reinterpret_cast<float*>(wb + L.part_o);
    c->ws.part_ml = reinterpret_cast<float*>(wb + L.part_ml);
    c->ws.max_parts = L.max_parts;
    c->ws.counters = reinterpret_cast<int32_t*>(wb + L.counters);
    c->ws.max_counter_units = L.max_counter_units;
    c->ws.scratch = reinterpret_cast<int32_t*>(wb + L.scratch);
    c->ws.scratch_ints = L.scratch_ints;
    c->ws.split_o = reinterpret_cast<float*>(wb + L.split_o);
    c->ws.split_ml = reinterpret_cast<float*>(wb + L.split_ml);
    std::string err;
    const uint64_t rows = (uint64_t)cfg->num_pages * cfg->page_size;
    // bf16: boxes of 64 elements (one 128-byte swizzle row); FP8: a 128-element
    // row is 128 bytes, one swizzle row
    const uint32_t box = g.fp8 ? (uint32_t)cfg->head_dim : 64u;
    const uint64_t rowb = (uint64_t)cfg->head_dim * (g.fp8 ? 1 : 2);
    if (!encode_tmap_2d(&c->tm_kpool, c->kpool, cfg->head_dim, rows, rowb, box,
                        cfg->page_size, true, &err, g.fp8) ||
        !encode_tmap_2d(&c->tm_vpool, c->vpool, cfg->head_dim, rows, rowb, box,
                        cfg->page_size, true, &err, g.fp8)) {
        delete c;
        return fail(SP_ERR_CUDA, err);
    }
    if (g.fp8 && cfg->page_size >= 64 &&
        (!encode_tmap_2d(&c->tm_kpool_half, c->kpool, cfg->head_dim, rows, rowb, box,
                         cfg->page_size / 2, true, &err, true) ||
         !encode_tmap_2d(&c->tm_vpool_half, c->vpool, cfg->head_dim, rows, rowb, box,
                         cfg->page_size / 2, true, &err, true))) {
        delete c;
        return fail(SP_ERR_CUDA, err);
    }
    // Device state: every page free, all units empty, the pool zeroed (slots
    // past a page's valid range are read by the kernels and multiplied by a
    // zero weight, so they must hold finite values).
    // pinned host staging ring for the prefill work list (host memory: the
    // device buffers stay the caller's)
    // (also the header of a packed sequence, see sp_pack_seq)
    c->stage_bytes = std::max((size_t)L.max_tiles * sizeof(int4),
                              align_to(sizeof(PackHeader) + 8 * (size_t)cfg->num_layers +
                                           sizeof(PackUnit) * (size_t)cfg->num_layers * cfg->num_kv_heads +
                                           4 * (size_t)std::max(cfg->max_idx_per_seq, 1), 256));
    for (int i = 0; i < sp_cache::kStaging && e == cudaSuccess; ++i) {
        e = cudaHostAlloc(reinterpret_cast<void**>(&c->stage_buf[i]), c->stage_bytes,
                          cudaHostAllocMapped);
        void* dp = nullptr;
        if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dp, c->stage_buf[i], 0);
        c->stage_dev[i] = static_cast<const int4*>(dp);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->stage_ev[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) { delete c; return cuda_fail(e, "pinned staging buffers"); }
    e = cudaMemset(meta, 0, L.meta_total);
    if (e == cudaSuccess) e = cudaMemset(ws, 0, L.ws_total);
    if (e == cudaSuccess) e = cudaMemset(pool, 0, L.pool_total);
    if (e == cudaSuccess) e = launch_init_meta(c, 0);
    if (e == cudaSuccess) {   // FP8 scales and reciprocals start at 1
        const std::vector<float> ones(4 * (size_t)cfg->num_layers * cfg->num_kv_heads * cfg->head_dim, 1.f);
        e = cudaMemcpy(c->meta.kscale, ones.data(), ones.size() * 4, cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { delete c; return cuda_fail(e, "cache initialisation"); }
    const size_t units = (size_t)cfg->max_seqs * cfg->num_layers * cfg->num_kv_heads;
    c->h_pol.assign(units, UnitPol{});
    c->h_idx.assign(cfg->max_seqs, std::vector<int32_t>(1, 0));
    c->h_policy_set.assign(cfg->max_seqs, 0);
    c->h_seqlen.assign((size_t)cfg->max_seqs * cfg->num_layers, 0);
    c->h_npages.assign(units, 0);
    c->h_free = cfg->num_pages;
    *out = c;
    return SP_OK;
}

sp_cache::~sp_cache() {
    for (int i = 0; i < kStaging; ++i) {
        if (stage_ev[i]) {
            cudaEventSynchronize(stage_ev[i]);   // no copy may still read the buffer
            cudaEventDestroy(stage_ev[i]);
        }
        if (stage_buf[i]) cudaFreeHost(stage_buf[i]);
    }
}

sp_status sp_cache_destroy(sp_cache* cache) {
    if (!cache) return fail(SP_ERR_INVALID_ARG, "null handle");
    delete cache;
    return SP_OK;
}

sp_status sp_set_policy(sp_cache* c, int32_t seq, const sp_head_policy* p, void* stream) {
    if (!c || !p) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq)) return fail(SP_ERR_INVALID_ARG, "sequence id out of range");
    for (int l = 0; l < c->cfg.num_layers; ++l)
        if (c->h_seqlen[(size_t)seq * c->cfg.num_layers + l] != 0)
            return fail(SP_ERR_INVALID_ARG, "sequence holds tokens; release it first");
    const int NU = c->cfg.num_layers * c->cfg.num_kv_heads, P = c->cfg.page_size;
    std::vector<UnitPol> recs(NU);
    std::vector<int32_t> idx;
    for (int u = 0; u < NU; ++u) {
        const sp_head_policy& hp = p[u];
        UnitPol r{};
        r.kind = hp.kind;
        if (hp.kind == SP_GLOBAL) {
        } else if (hp.kind == SP_LOCAL) {
            if (hp.sink < 0 || hp.window < 1)
                return fail(SP_ERR_INVALID_ARG, "LOCAL needs sink >= 0 and window >= 1");
            if ((int64_t)hp.window > c->cfg.max_seq_len + (int64_t)P)
                return fail(SP_ERR_INVALID_ARG, "LOCAL window longer than max_seq_len");
            r.sink = hp.sink;
            r.window = hp.window;
            r.ring = (hp.window + P - 1) / P + 1;
            r.sink_pages = (hp.sink + P - 1) / P;
            if ((int64_t)r.sink_pages + r.ring > (c->cfg.max_seq_len + P - 1) / P + 1 &&
                (int64_t)hp.sink > c->cfg.max_seq_len)
                return fail(SP_ERR_INVALID_ARG, "LOCAL sink longer than max_seq_len");
        } else if (hp.kind == SP_RETRIEVAL) {
            if (hp.n_idx < 0 || (hp.n_idx > 0 && !hp.idx))
                return fail(SP_ERR_INVALID_ARG, "RETRIEVAL list missing");
            for (int k = 0; k < hp.n_idx; ++k) {
                if (hp.idx[k] < 0 || (k > 0 && hp.idx[k] <= hp.idx[k - 1]))
                    return fail(SP_ERR_INVALID_ARG, "RETRIEVAL indices must be >= 0 and strictly ascending");
            }
            r.idx_off = (int32_t)idx.size();
            r.n_idx = hp.n_idx;
            idx.insert(idx.end(), hp.idx, hp.idx + hp.n_idx);
            if ((int64_t)idx.size() > c->cfg.max_idx_per_seq)
                return fail(SP_ERR_INVALID_ARG, "retrieval lists exceed max_idx_per_seq");
        } else {
            return fail(SP_ERR_INVALID_ARG, "unknown head class " + std::to_string(hp.kind));
        }
        recs[u] = r;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t base = unit_index(c, seq, 0, 0);
    cudaError_t e = cudaMemcpyAsync(c->meta.pol + base, recs.data(), NU * sizeof(UnitPol),
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !idx.empty())
        e = cudaMemcpyAsync(c->meta.idx + (size_t)seq * c->geo.max_idx_per_seq, idx.data(),
                            idx.size() * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // host staging buffers go out of scope
    if (e != cudaSuccess) return cuda_fail(e, "policy upload");
    std::copy(recs.begin(), recs.end(), c->h_pol.begin() + base);
    if (idx.empty()) idx.push_back(0);
    c->h_idx[seq] = std::move(idx);
    c->h_policy_set[seq] = 1;
    return SP_OK;
}

sp_status sp_build_cache(sp_cache* c, int32_t seq, int32_t layer, const void* k, const void* v,
                         int64_t n_tokens, int64_t row_stride, void* stream) {
    if (!c || !k || !v) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq) || !valid_layer(c, layer))
        return fail(SP_ERR_INVALID_ARG, "sequence or layer out of range");
    if (!c->h_policy_set[seq]) return fail(SP_ERR_INVALID_ARG, "sequence has no policy");
    if (c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer] != 0)
        return fail(SP_ERR_INVALID_ARG, "build needs an empty (sequence, layer)");
    if (n_tokens < 0 || n_tokens > c->cfg.max_seq_len)
        return fail(SP_ERR_INVALID_ARG, "n_tokens outside [0, max_seq_len]");
    if (row_stride < (int64_t)c->cfg.num_kv_heads * c->cfg.head_dim || row_stride % 8 != 0)
        return fail(SP_ERR_INVALID_ARG, "row_stride must be >= kv_heads*head_dim and a multiple of 8");
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
        return fail(SP_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    const int64_t cnt = n_tokens;
    return write_tokens(c, layer, &seq, 1, &cnt, static_cast<const __nv_bfloat16*>(k),
                        static_cast<const __nv_bfloat16*>(v), row_stride,
                        static_cast<cudaStream_t>(stream));
}

sp_status sp_append_kv(sp_cache* c, int32_t layer, const int32_t* seq_ids, int32_t n_seqs,
                       const int32_t* cu_new, const void* k, const void* v, void* stream) {
    if (!c || !cu_new || !k || !v) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    sp_status s = check_seq_list(c, seq_ids, n_seqs);
    if (s != SP_OK) return s;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
        return fail(SP_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    if (cu_new[0] != 0) return fail(SP_ERR_INVALID_ARG, "cu_new[0] must be 0");
    std::vector<int64_t> counts(n_seqs);
    for (int b = 0; b < n_seqs; ++b) {
        counts[b] = (int64_t)cu_new[b + 1] - cu_new[b];
        if (counts[b] < 0) return fail(SP_ERR_INVALID_ARG, "cu_new must be non-decreasing");
    }
    if (cu_new[n_seqs] > c->cfg.max_tokens)
        return fail(SP_ERR_INVALID_ARG, "more new tokens than max_tokens");
    return write_tokens(c, layer, seq_ids, n_seqs, counts.data(),
                        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                        (int64_t)c->cfg.num_kv_heads * c->cfg.head_dim,
                        static_cast<cudaStream_t>(stream));
}

sp_status sp_attention_prefill(sp_cache* c, int32_t layer, const int32_t* seq_ids,
                               int32_t n_seqs, const int32_t* cu_q, const void* q,
                               const void* k, const void* v, void* out, float* lse,
                               void* stream) {
    if (!c || !cu_q || !q || !k || !v || !out) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    sp_status s = check_seq_list(c, seq_ids, n_seqs);
    if (s != SP_OK) return s;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v)) & 15)
        return fail(SP_ERR_INVALID_ARG, "q, k and v must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(out) & 31)   // the epilogue writes 32-byte vectors
        return fail(SP_ERR_INVALID_ARG, "out must be 32-byte aligned");
    if (cu_q[0] != 0) return fail(SP_ERR_INVALID_ARG, "cu_q[0] must be 0");
    for (int b = 0; b < n_seqs; ++b) {
        if (cu_q[b + 1] < cu_q[b]) return fail(SP_ERR_INVALID_ARG, "cu_q must be non-decreasing");
        const int64_t n = c->h_seqlen[(size_t)seq_ids[b] * c->cfg.num_layers + layer];
        if (n + (cu_q[b + 1] - cu_q[b]) > c->cfg.max_seq_len)
            return fail(SP_ERR_INVALID_ARG, "chunk would pass max_seq_len");
    }
    if (cu_q[n_seqs] > c->cfg.max_tokens) return fail(SP_ERR_INVALID_ARG, "more rows than max_tokens");
    return prefill_impl(c, layer, seq_ids, n_seqs, cu_q, static_cast<const __nv_bfloat16*>(q),
                        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                        static_cast<__nv_bfloat16*>(out), lse, static_cast<cudaStream_t>(stream));
}

sp_status sp_attention_decode(sp_cache* c, int32_t layer, const int32_t* seq_ids, int32_t n_seqs,
                              const void* q, void* out, float* lse, void* stream) {
    if (!c || !q || !out) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    sp_status s = check_seq_list(c, seq_ids, n_seqs);
    if (s != SP_OK) return s;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 3)
        return fail(SP_ERR_INVALID_ARG, "q and out must be 4-byte aligned");
    DecodeParams* p = new DecodeParams();   // large; keep it off the host stack
    std::unique_ptr<DecodeParams> guard(p);
    p->meta = c->meta;
    p->geo = c->geo;
    p->layer = layer;
    p->n_seqs = n_seqs;
    p->n_units = n_seqs * c->cfg.num_kv_heads;
    p->item_off[0] = 0;
    int64_t total = 0;
    const int P = c->cfg.page_size;
    for (int b = 0; b < n_seqs; ++b) {
        const int seq = seq_ids[b];
        const int64_t n = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
        if (n < 1) return fail(SP_ERR_INVALID_ARG, "decode needs the query's own token appended first");
        p->seq[b] = seq;
        p->tq[b] = (int32_t)(n - 1);
        for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
            const UnitPol& u = c->h_pol[unit_index(c, seq, layer, h)];
            total += decode_items(decode_ranges(u, host_idx(c, seq, u), n - 1, P), P);
            p->item_off[b * c->cfg.num_kv_heads + h + 1] = (int32_t)total;
        }
    }
    if (total >= (int64_t(1) << 31)) return fail(SP_ERR_UNSUPPORTED, "too many pages in one call");
    p->total_items = total;
    p->q = static_cast<const __nv_bfloat16*>(q);
    p->out = static_cast<__nv_bfloat16*>(out);
    p->lse = lse;
    p->part_o = c->ws.part_o;
    p->part_ml = c->ws.part_ml;
    p->counters = c->ws.counters;
    p->scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->cfg.head_dim));
    launch_mark_start(c, static_cast<cudaStream_t>(stream));
    cudaError_t e = launch_decode(c, *p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    launch_mark_end(c, static_cast<cudaStream_t>(stream));
    return SP_OK;
}

sp_status sp_set_launch_events(sp_cache* c, void* start_event, void* end_event) {
    if (!c) return fail(SP_ERR_INVALID_ARG, "null handle");
    if ((start_event == nullptr) != (end_event == nullptr))
        return fail(SP_ERR_INVALID_ARG, "give both events or neither");
    c->launch_ev[0] = static_cast<cudaEvent_t>(start_event);
    c->launch_ev[1] = static_cast<cudaEvent_t>(end_event);
    return SP_OK;
}

sp_status sp_release_seq(sp_cache* c, int32_t seq, void* stream) {
    if (!c) return fail(SP_ERR_INVALID_ARG, "null handle");
    if (!valid_seq(c, seq)) return fail(SP_ERR_INVALID_ARG, "sequence id out of range");
    int64_t held = 0;
    const size_t base = unit_index(c, seq, 0, 0);
    const int NU = c->cfg.num_layers * c->cfg.num_kv_heads;
    for (int u = 0; u < NU; ++u) held += c->h_npages[base + u];
    cudaError_t e = launch_release(c, seq, (int32_t)c->h_free, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "release launch");
    c->h_free += held;
    for (int u = 0; u < NU; ++u) c->h_npages[base + u] = 0;
    for (int l = 0; l < c->cfg.num_layers; ++l) c->h_seqlen[(size_t)seq * c->cfg.num_layers + l] = 0;
    return SP_OK;
}

sp_status sp_set_kv_scales(sp_cache* c, int32_t layer, const float* k_scale, const float* v_scale,
                           void* stream) {
    if (!c || !k_scale || !v_scale) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!c->geo.fp8) return fail(SP_ERR_INVALID_ARG, "scales apply to FP8 pages only");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    for (int s = 0; s < c->cfg.max_seqs; ++s)
        if (c->h_seqlen[(size_t)s * c->cfg.num_layers + layer] != 0)
            return fail(SP_ERR_INVALID_ARG, "layer holds tokens; scales are fixed once a page is written");
    const size_t n = (size_t)c->cfg.num_kv_heads * c->cfg.head_dim;
    std::vector<float> ks(k_scale, k_scale + n), vs(v_scale, v_scale + n), ki(n), vi(n);
    for (size_t i = 0; i < n; ++i) {
        // f16 decode: the scale stays a normal f16 and 448 * scale stays finite
        const float lo = 1.0f / 16384.0f, hi = 128.0f;
        if (!(ks[i] >= lo && ks[i] <= hi) || !(vs[i] >= lo && vs[i] <= hi))
            return fail(SP_ERR_INVALID_ARG, "scales must lie in [2^-14, 128]");
        ki[i] = 1.0f / ks[i];     // fp32 reciprocals: the quantiser multiplies by these
        vi[i] = 1.0f / vs[i];
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t off = (size_t)layer * n;
    cudaError_t e = cudaMemcpyAsync(c->meta.kscale + off, ks.data(), n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->meta.vscale + off, vs.data(), n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->meta.kinv + off, ki.data(), n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->meta.vinv + off, vi.data(), n * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "scale upload");
    return SP_OK;
}

sp_status sp_rope_realign(sp_cache* c, int32_t layer, const int32_t* seq_ids, int32_t n_seqs,
                          int32_t kv_head, int64_t pos_lo, int64_t pos_hi, int64_t delta,
                          double rope_theta, void* stream) {
    if (!c) return fail(SP_ERR_INVALID_ARG, "null handle");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    sp_status s = check_seq_list(c, seq_ids, n_seqs);
    if (s != SP_OK) return s;
    if (kv_head < -1 || kv_head >= c->cfg.num_kv_heads) return fail(SP_ERR_INVALID_ARG, "kv_head out of range");
    if (pos_lo < 0 || pos_hi < pos_lo) return fail(SP_ERR_INVALID_ARG, "need 0 <= pos_lo <= pos_hi");
    if (!(rope_theta > 0.0) || !std::isfinite(rope_theta))
        return fail(SP_ERR_INVALID_ARG, "rope_theta must be positive and finite");
    if (delta < -(int64_t(1) << 40) || delta > (int64_t(1) << 40))
        return fail(SP_ERR_INVALID_ARG, "delta out of range (|delta| <= 2^40)");
    if (pos_lo == pos_hi || delta == 0) return SP_OK;   // nothing moves
    std::unique_ptr<RopeParams> pp(new RopeParams());
    RopeParams& p = *pp;
    p.meta = c->meta;
    p.geo = c->geo;
    p.layer = layer;
    p.pos_lo = pos_lo;
    p.pos_hi = pos_hi;
    const int d = c->cfg.head_dim;
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < d / 2; ++i) {
        // angle delta * theta^(-2i/d), reduced in double before the cos / sin
        const double ang = std::fmod((double)delta * std::pow(rope_theta, -2.0 * i / d), two_pi);
        p.cs[i] = (float)std::cos(ang);
        p.sn[i] = (float)std::sin(ang);
    }
    const int h0 = kv_head < 0 ? 0 : kv_head;
    const int h1 = kv_head < 0 ? c->cfg.num_kv_heads : kv_head + 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // units in launches of at most kMaxRopeUnits, each with its page offsets
    p.n_units = 0;
    p.page_off[0] = 0;
    auto flush = [&]() -> cudaError_t {
        if (p.n_units == 0) return cudaSuccess;
        cudaError_t e = launch_rope(c, p, st);
        p.n_units = 0;
        p.page_off[0] = 0;
        return e;
    };
    for (int b = 0; b < n_seqs; ++b) {
        const int32_t n = c->h_seqlen[(size_t)seq_ids[b] * c->cfg.num_layers + layer];
        for (int h = h0; h < h1; ++h) {
            const int32_t np = c->h_npages[unit_index(c, seq_ids[b], layer, h)];
            if (np == 0) continue;
            const int u = p.n_units++;
            p.unit_seq[u] = seq_ids[b];
            p.unit_head[u] = (int16_t)h;
            p.unit_n[u] = n;
            p.page_off[u + 1] = p.page_off[u] + np;
            if (p.n_units == kMaxRopeUnits) {
                cudaError_t e = flush();
                if (e != cudaSuccess) return cuda_fail(e, "rope launch");
            }
        }
    }
    cudaError_t e = flush();
    if (e != cudaSuccess) return cuda_fail(e, "rope launch");
    return SP_OK;
}

sp_status sp_pack_seq(sp_cache* c, int32_t seq, void* dst, size_t dst_bytes, size_t* packed_bytes,
                      void* stream) {
    if (!c || !packed_bytes) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq)) return fail(SP_ERR_INVALID_ARG, "sequence id out of range");
    if (!c->h_policy_set[seq]) return fail(SP_ERR_INVALID_ARG, "sequence has no policy");
    const int L = c->cfg.num_layers, H = c->cfg.num_kv_heads, d = c->cfg.head_dim;
    const int P = c->cfg.page_size, U = L * H;
    int64_t idx_total = 0;
    for (int u = 0; u < U; ++u) {
        const UnitPol& up = c->h_pol[unit_index(c, seq, u / H, u % H)];
        if (up.kind == kRetrieval) idx_total += up.n_idx;
    }
    const size_t off_n = sizeof(PackHeader), off_units = off_n + 8 * (size_t)L;
    const size_t off_idx = off_units + sizeof(PackUnit) * (size_t)U;
    const size_t payload_off = align_to(off_idx + 4 * (size_t)idx_total, 256);
    int slot = -1;
    uint8_t* head = dst ? static_cast<uint8_t*>(stage_acquire(c, payload_off, &slot)) : nullptr;
    std::vector<uint8_t> scratch;
    if (!head) {                                       // size query, or a header too large to stage
        if (dst && payload_off <= c->stage_bytes) return fail(SP_ERR_CUDA, "pinned staging buffer");
        scratch.assign(payload_off, 0);
        head = scratch.data();
    } else {
        std::memset(head, 0, payload_off);
    }
    PackHeader* ph = reinterpret_cast<PackHeader*>(head);
    int64_t* nl = reinterpret_cast<int64_t*>(head + off_n);
    PackUnit* pu = reinterpret_cast<PackUnit*>(head + off_units);
    int32_t* pidx = reinterpret_cast<int32_t*>(head + off_idx);
    int64_t row_off = 0, blk_off = 0, io = 0;
    for (int l = 0; l < L; ++l) nl[l] = c->h_seqlen[(size_t)seq * L + l];
    for (int u = 0; u < U; ++u) {
        const UnitPol& up = c->h_pol[unit_index(c, seq, u / H, u % H)];
        const int32_t* idx = host_idx(c, seq, up);
        const int64_t rows = retained_rows(up, idx, nl[u / H], P);
        pu[u] = PackUnit{up.kind, up.sink, up.window, up.kind == kRetrieval ? up.n_idx : 0, rows,
                         row_off, blk_off};
        if (up.kind == kRetrieval)
            for (int k = 0; k < up.n_idx; ++k) pidx[io++] = idx[k];
        row_off += rows;
        blk_off += (rows + kTransferRows - 1) / kTransferRows;
    }
    const size_t payload_bytes = (size_t)row_off * 2 * d * (c->geo.fp8 ? 1 : 2);
    *ph = PackHeader{kPackMagic, 1, L, H, d, P, U, idx_total, (int64_t)payload_off,
                     (int64_t)payload_bytes, (int64_t)(payload_off + payload_bytes),
                     (int64_t)c->cfg.kv_dtype};
    *packed_bytes = payload_off + payload_bytes;
    if (!dst) return SP_OK;                            // size query
    if (dst_bytes < *packed_bytes) return fail(SP_ERR_INVALID_ARG, "dst smaller than the packed size");
    if (reinterpret_cast<uintptr_t>(dst) & 255) return fail(SP_ERR_INVALID_ARG, "dst must be 256-byte aligned");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (slot >= 0) {
        e = stage_copy(c, slot, dst, payload_off, st);  // asynchronous, from pinned memory
    } else {
        e = cudaMemcpyAsync(dst, head, payload_off, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // the host header goes out of scope
    }
    if (e != cudaSuccess) return cuda_fail(e, "pack header upload");
    uint8_t* db = static_cast<uint8_t*>(dst);
    TransferParams tp{};
    tp.meta = c->meta;
    tp.geo = c->geo;
    tp.seq = seq;
    tp.unpack = 0;
    tp.n_units = U;
    tp.total_blocks = blk_off;
    tp.n_layer = reinterpret_cast<const int64_t*>(db + off_n);
    tp.units = reinterpret_cast<const PackUnit*>(db + off_units);
    tp.payload = db + payload_off;
    e = launch_transfer(c, tp, st);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    return SP_OK;
}

sp_status sp_unpack_seq(sp_cache* c, int32_t seq, const void* src, size_t src_bytes, void* stream) {
    if (!c || !src) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq)) return fail(SP_ERR_INVALID_ARG, "sequence id out of range");
    if (reinterpret_cast<uintptr_t>(src) & 255) return fail(SP_ERR_INVALID_ARG, "src must be 256-byte aligned");
    for (int l = 0; l < c->cfg.num_layers; ++l)
        if (c->h_seqlen[(size_t)seq * c->cfg.num_layers + l] != 0)
            return fail(SP_ERR_INVALID_ARG, "sequence holds tokens; release it first");
    if (src_bytes < sizeof(PackHeader)) return fail(SP_ERR_INVALID_ARG, "src shorter than a header");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PackHeader ph;
    cudaError_t e = cudaMemcpyAsync(&ph, src, sizeof(ph), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "unpack header read");
    const int L = c->cfg.num_layers, H = c->cfg.num_kv_heads, P = c->cfg.page_size;
    const int U = L * H;
    if (ph.magic != kPackMagic || ph.version != 1) return fail(SP_ERR_INVALID_ARG, "not a packed sequence");
    if (ph.layers != L || ph.hkv != H || ph.head_dim != c->cfg.head_dim || ph.page_size != P ||
        ph.n_units != U || ph.kv_dtype != c->cfg.kv_dtype)
        return fail(SP_ERR_INVALID_ARG, "packed sequence has another layer count, head count, "
                                        "head_dim, page_size or page type");
    const size_t off_n = sizeof(PackHeader), off_units = off_n + 8 * (size_t)L;
    const size_t off_idx = off_units + sizeof(PackUnit) * (size_t)U;
    if (ph.idx_total < 0 || ph.payload_off != (int64_t)align_to(off_idx + 4 * (size_t)ph.idx_total, 256) ||
        ph.total_bytes != ph.payload_off + ph.payload_bytes || (size_t)ph.total_bytes > src_bytes)
        return fail(SP_ERR_INVALID_ARG, "packed header inconsistent with its size");
    std::vector<uint8_t> head(ph.payload_off);
    e = cudaMemcpyAsync(head.data(), src, head.size(), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "unpack header read");
    const int64_t* nl = reinterpret_cast<const int64_t*>(head.data() + off_n);
    const PackUnit* pu = reinterpret_cast<const PackUnit*>(head.data() + off_units);
    const int32_t* pidx = reinterpret_cast<const int32_t*>(head.data() + off_idx);
    // policies and capacity first: a refused unpack changes nothing
    std::vector<sp_head_policy> pols(U);
    int64_t io = 0, demand = 0, rows_total = 0, blocks = 0;
    for (int u = 0; u < U; ++u) {
        const PackUnit& x = pu[u];
        if (x.kind < kGlobal || x.kind > kRetrieval || x.n_idx < 0 || io + x.n_idx > ph.idx_total)
            return fail(SP_ERR_INVALID_ARG, "packed unit record out of range");
        pols[u] = sp_head_policy{(int32_t)x.kind, (int32_t)x.sink, (int32_t)x.window,
                                 (int32_t)x.n_idx, x.n_idx ? pidx + io : nullptr};
        const int64_t n = nl[u / H];
        if (n < 0 || n > c->cfg.max_seq_len) return fail(SP_ERR_INVALID_ARG, "packed length out of range");
        const UnitPol r = encode_unit(x.kind, x.sink, x.window, 0, (int32_t)x.n_idx, P);
        const int32_t* idx = x.kind == kRetrieval ? pidx + io : nullptr;
        if (x.rows != retained_rows(r, idx, n, P) || x.row_off != rows_total || x.blk_off != blocks)
            return fail(SP_ERR_INVALID_ARG, "packed unit layout does not follow its policy");
        demand += unit_pages(r, idx, n, P);
        rows_total += x.rows;
        blocks += (x.rows + kTransferRows - 1) / kTransferRows;
        io += x.n_idx;
    }
    if (ph.payload_bytes != rows_total * 2 * c->cfg.head_dim * (c->geo.fp8 ? 1 : 2))
        return fail(SP_ERR_INVALID_ARG, "packed payload size does not match its units");
    if (demand > c->h_free)
        return fail(SP_ERR_OUT_OF_PAGES, "unpack needs " + std::to_string(demand) + " pages, " +
                                             std::to_string(c->h_free) + " free");
    sp_status s = sp_set_policy(c, seq, pols.data(), stream);
    if (s != SP_OK) return s;
    for (int l = 0; l < L; ++l) {
        if (nl[l] == 0) continue;
        CallSeqs cs;
        int64_t max_items = 0, rows = 0;
        const int64_t cnt = nl[l];
        s = alloc_tokens(c, l, &seq, 1, &cnt, st, cs, max_items, rows);
        if (s != SP_OK) return s;
    }
    const uint8_t* sb = static_cast<const uint8_t*>(src);
    TransferParams tp{};
    tp.meta = c->meta;
    tp.geo = c->geo;
    tp.seq = seq;
    tp.unpack = 1;
    tp.n_units = U;
    tp.total_blocks = blocks;
    tp.n_layer = reinterpret_cast<const int64_t*>(sb + off_n);
    tp.units = reinterpret_cast<const PackUnit*>(sb + off_units);
    tp.payload = const_cast<uint8_t*>(sb + ph.payload_off);
    e = launch_transfer(c, tp, st);
    if (e != cudaSuccess) return cuda_fail(e, "unpack launch");
    return SP_OK;
}

sp_status sp_export_table(sp_cache* c, int32_t seq, int32_t layer, int32_t kv_head,
                          int32_t* npages, int32_t* page_ids, int32_t* slot_pos, int32_t cap,
                          void* stream) {
    if (!c || !npages || !page_ids || !slot_pos) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq) || !valid_layer(c, layer) || kv_head < 0 || kv_head >= c->cfg.num_kv_heads)
        return fail(SP_ERR_INVALID_ARG, "unit out of range");
    const int32_t np = c->h_npages[unit_index(c, seq, layer, kv_head)];
    *npages = np;
    if (np > cap) return fail(SP_ERR_INVALID_ARG, "cap smaller than the unit's page count");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* d_ids = c->ws.scratch;
    int32_t* d_pos = c->ws.scratch + c->geo.max_pages_unit;
    cudaError_t e = launch_export(c, seq, layer, kv_head, d_ids, d_pos, st);
    if (e == cudaSuccess && np > 0)
        e = cudaMemcpyAsync(page_ids, d_ids, (size_t)np * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && np > 0)
        e = cudaMemcpyAsync(slot_pos, d_pos, (size_t)np * c->cfg.page_size * 4,
                            cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "export");
    return SP_OK;
}

sp_status sp_visible_count(sp_cache* c, int32_t seq, int32_t layer, int32_t kv_head,
                           const int64_t* positions, int32_t n, int32_t* counts, void* stream) {
    if (!c || !positions || !counts) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq) || !valid_layer(c, layer) || kv_head < 0 || kv_head >= c->cfg.num_kv_heads)
        return fail(SP_ERR_INVALID_ARG, "unit out of range");
    if (n < 0 || n > 65536) return fail(SP_ERR_INVALID_ARG, "between 0 and 65536 positions");
    if (n == 0) return SP_OK;
    const int64_t held = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
    for (int k = 0; k < n; ++k)
        if (positions[k] < held - 1 || positions[k] >= held + c->cfg.max_tokens)
            return fail(SP_ERR_INVALID_ARG, "position outside [held-1, held+max_tokens)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int64_t* d_pos = reinterpret_cast<int64_t*>(c->ws.scratch);
    int32_t* d_out = c->ws.scratch + 2 * 65536;
    cudaError_t e = cudaMemcpyAsync(d_pos, positions, (size_t)n * 8, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = launch_decode_counts(c, seq, layer, kv_head, d_pos, n, d_out, st);
    if (e == cudaSuccess) e = launch_prefill_counts(c, seq, layer, kv_head, d_pos, n, d_out, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(counts, d_out, (size_t)n * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "visible count");
    return SP_OK;
}

sp_status sp_seq_len(const sp_cache* c, int32_t seq, int32_t layer, int32_t* n) {
    if (!c || !n) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq) || !valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "out of range");
    *n = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
    return SP_OK;
}

sp_status sp_free_pages(const sp_cache* c, int32_t* n) {
    if (!c || !n) return fail(SP_ERR_INVALID_ARG, "null argument");
    *n = (int32_t)c->h_free;
    return SP_OK;
}

sp_status sp_count_prefill_pairs(const sp_cache* c, int32_t seq, int32_t layer, int64_t n0,
                                 int64_t cnt, int64_t* pairs) {
    if (!c || !pairs) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_seq(c, seq) || !valid_layer(c, layer) || n0 < 0 || cnt < 0)
        return fail(SP_ERR_INVALID_ARG, "out of range");
    if (!c->h_policy_set[seq]) return fail(SP_ERR_INVALID_ARG, "sequence has no policy");
    int64_t total = 0;
    for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
        const UnitPol& u = c->h_pol[unit_index(c, seq, layer, h)];
        const int32_t* idx = host_idx(c, seq, u);
        int64_t s = 0;
        if (u.kind == kGlobal) {
            // sum_{i=n0}^{n0+cnt-1} (i + 1)
            s = (n0 + 1 + n0 + cnt) * cnt / 2;
        } else {
            for (int64_t i = n0; i < n0 + cnt; ++i) s += visible_count(u, idx, i);
        }
        total += s * c->geo.group;
    }
    *pairs = total;
    return SP_OK;
}

sp_status sp_count_decode_bytes(const sp_cache* c, int32_t layer, const int32_t* seq_ids,
                                int32_t n_seqs, const int64_t* t, int64_t* bytes) {
    if (!c || !seq_ids || !t || !bytes) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    int64_t total = 0;
    for (int b = 0; b < n_seqs; ++b) {
        if (!valid_seq(c, seq_ids[b]) || !c->h_policy_set[seq_ids[b]])
            return fail(SP_ERR_INVALID_ARG, "bad sequence");
        for (int h = 0; h < c->cfg.num_kv_heads; ++h) {
            const UnitPol& u = c->h_pol[unit_index(c, seq_ids[b], layer, h)];
            total += visible_count(u, host_idx(c, seq_ids[b], u), t[b]);
        }
    }
    *bytes = total * 2 * c->cfg.head_dim * (c->geo.fp8 ? 1 : 2);   // K + V rows of the page type
    return SP_OK;
}

sp_status sp_get_status(sp_cache* c, void* stream, int32_t* word) {
    if (!c) return fail(SP_ERR_INVALID_ARG, "null handle");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t w = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemcpy(&w, c->meta.status, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && w != 0) e = cudaMemset(c->meta.status, 0, 4);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (word) *word = w;
    if (w & kStatusTimeout) return fail(SP_ERR_TIMEOUT, "a device wait timed out");
    if (w != 0) return fail(SP_ERR_DEVICE_STATUS, "device status flags " + std::to_string(w));
    return SP_OK;
}

}  // extern "C"
