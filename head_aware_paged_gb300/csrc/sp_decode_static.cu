// sp_decode_static.cu -- decode whose split-KV scratch lives in a fixed device
// array compiled into this library, for callers that cannot allocate device
// memory when they decode.
//
// Who needs it: a host that links libsegpaged.so from plain C and has no
// device allocator of its own, or a serving loop that must not call
// cudaMalloc mid-step (cudaMalloc can synchronise the device and stall every
// other stream, and a fixed-memory deployment may forbid new allocations
// after start-up).  Such a caller still passes the cache, q and the outputs;
// only the decode's scratch (unnormalised split partials, their (m, l) and
// the merge tickets) comes from here instead of the cache's workspace.
//
// The array (kStaticScratchBytes) is held by every GPU that loads the
// library until the process exits.  Host code must not pass the array's name
// to a kernel (in host code it names a host-side stand-in, not device memory):
// the first call on each device looks up its device address with
// cudaGetSymbolAddress while that device is current, so make that first call
// before any stream capture.  All calls share the one array: the ticket
// counters are cleared at the start of every call, and two calls that overlap
// on the GPU (different streams, or different caches, at the same time) race
// on it.
#include <cmath>
#include <mutex>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_mu;                          // guards the table and the parameter block
void* g_scratch_addr[kMaxDevices];        // device address per device (static storage)
DecodeParams g_params;                    // reused by every call: no per-call allocation

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

}  // namespace sp

using namespace sp;

extern "C" sp_status sp_attention_decode_static_scratch(sp_cache* c, int32_t layer,
                                                       const int32_t* seq_ids, int32_t n_seqs,
                                                       const void* q, void* out, float* lse,
                                                       void* stream) {
    if (!c || !q || !out) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (!valid_layer(c, layer)) return fail(SP_ERR_INVALID_ARG, "layer out of range");
    sp_status s = check_seq_list(c, seq_ids, n_seqs);
    if (s != SP_OK) return s;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 3)
        return fail(SP_ERR_INVALID_ARG, "q and out must be 4-byte aligned");
    for (int b = 0; b < n_seqs; ++b)
        if (c->h_seqlen[(size_t)seq_ids[b] * c->cfg.num_layers + layer] < 1)
            return fail(SP_ERR_INVALID_ARG, "decode needs the query's own token appended first");
    const int hkv = c->cfg.num_kv_heads, group = c->geo.group, d = c->cfg.head_dim;
    const int64_t n_units = (int64_t)n_seqs * hkv;
    // scratch layout: partial outputs, partial (m, l), tickets -- sized for the
    // largest grid the decode launch may use
    const int64_t parts = n_units + c->decode_ctas;
    const size_t o_bytes = up256((size_t)parts * group * d * sizeof(float));
    const size_t ml_bytes = up256((size_t)parts * group * 2 * sizeof(float));
    const size_t ctr_bytes = up256((size_t)n_units * sizeof(int32_t));
    if (o_bytes + ml_bytes + ctr_bytes > kStaticScratchBytes)
        return fail(SP_ERR_UNSUPPORTED,
                    "decode needs " + std::to_string(o_bytes + ml_bytes + ctr_bytes) +
                        " bytes of scratch; the built-in array holds " +
                        std::to_string(kStaticScratchBytes) + " (use sp_attention_decode)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return fail(SP_ERR_INVALID_ARG, "current device is not the cache's device");
    if (dev < 0 || dev >= kMaxDevices) return fail(SP_ERR_UNSUPPORTED, "device index above 63");

    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        // once per device, with that device current: the array's device address
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess || !ptr) return cuda_fail(e, "cudaGetSymbolAddress of the decode scratch");
        g_scratch_addr[dev] = ptr;
    }
    unsigned char* base = static_cast<unsigned char*>(g_scratch_addr[dev]);
    DecodeParams& p = g_params;
    p.meta = c->meta;
    p.geo = c->geo;
    p.layer = layer;
    p.n_seqs = n_seqs;
    p.n_units = (int32_t)n_units;
    p.item_off[0] = 0;
    int64_t total = 0;
    const int P = c->cfg.page_size;
    for (int b = 0; b < n_seqs; ++b) {
        const int seq = seq_ids[b];
        const int64_t n = c->h_seqlen[(size_t)seq * c->cfg.num_layers + layer];
        p.seq[b] = seq;
        p.tq[b] = (int32_t)(n - 1);
        for (int h = 0; h < hkv; ++h) {
            const UnitPol& u = c->h_pol[((size_t)seq * c->cfg.num_layers + layer) * hkv + h];
            total += decode_items(decode_ranges(u, c->h_idx[seq].data() + u.idx_off, n - 1, P), P);
            p.item_off[b * hkv + h + 1] = (int32_t)total;
        }
    }
    if (total >= (int64_t(1) << 31)) return fail(SP_ERR_UNSUPPORTED, "too many pages in one call");
    p.total_items = total;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.part_o = reinterpret_cast<float*>(base);
    p.part_ml = reinterpret_cast<float*>(base + o_bytes);
    p.counters = reinterpret_cast<int32_t*>(base + o_bytes + ml_bytes);
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the merge tickets must start at zero in every call
    e = cudaMemsetAsync(p.counters, 0, (size_t)n_units * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the decode tickets");
    launch_mark_start(c, st);
    e = launch_decode(c, p, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    launch_mark_end(c, st);
    return SP_OK;
}
