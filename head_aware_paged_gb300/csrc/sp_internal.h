// sp_internal.h -- handle, device-memory layout and launcher declarations
// shared by the host API (sp_api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "segpaged.h"
#include "sp_rules.h"

namespace sp {

constexpr int kMaxCallSeqs = 512;     // sequences in one call (kernel parameters)
constexpr int kMaxDecodeUnits = 4096; // (sequence, KV head) units in one decode call
constexpr int kMaxPolicyUnits = 8192; // layers * kv heads

// Device pointers into the caller's meta buffer.
struct Meta {
    UnitPol* pol;        // [max_seqs][layers][hkv]
    int32_t* npages;     // [max_seqs][layers][hkv]
    int32_t* seqlen;     // [max_seqs][layers]
    int32_t* ptab;       // [max_seqs][layers][hkv][max_pages_unit]
    int32_t* idx;        // [max_seqs][max_idx_per_seq]
    int32_t* fstack;     // [num_pages] free-page stack
    int32_t* status;     // [8]: 0 = status word, 1 = stack top (debug mirror)
    float* kscale;       // FP8 pages: [layers][hkv][d] per-channel scales of K
    float* vscale;       //            ... of V
    float* kinv;         //            fp32 reciprocals used to quantise
    float* vinv;
};

// Geometry every kernel needs.
struct Geo {
    int32_t layers, hq, hkv, group, d, page, max_seqs, max_pages_unit,
            max_idx_per_seq, num_pages;
    int32_t fp8;         // pages hold e4m3 codes (1 byte) instead of bf16
    __host__ __device__ int64_t unit_row(int seq, int layer, int h) const {
        return ((int64_t)seq * layers + layer) * hkv + h;
    }
};

// Per-call list of sequences (kernel parameter).
struct CallSeqs {
    int32_t n;
    int32_t seq[kMaxCallSeqs];   // sequence slot
    int32_t n_old[kMaxCallSeqs]; // tokens held before the call
    int32_t cnt[kMaxCallSeqs];   // new tokens / query rows
    int32_t row0[kMaxCallSeqs];  // first row in the call's packed tensors
};

struct DecodeParams {
    Meta meta;
    Geo geo;
    int32_t layer;
    int32_t n_seqs;
    int32_t n_units;             // n_seqs * hkv
    int64_t total_items;         // pages streamed, all units
    int32_t seq[kMaxCallSeqs];
    int32_t tq[kMaxCallSeqs];    // query position per sequence
    int32_t item_off[kMaxDecodeUnits + 1];
    const __nv_bfloat16* q;
    __nv_bfloat16* out;
    float* lse;
    float* part_o;               // [(n_units + grid)][group][d]
    float* part_ml;              // [(n_units + grid)][group][2]
    int32_t* counters;           // [n_units], zero between calls
    float scale_log2;            // log2(e) / sqrt(d)
    int32_t nst;                 // pipeline stages (set by the launcher)
    int32_t owners;              // consumer warps that own stages (divides nst)
    int32_t merge_floats;        // merge buffer floats (set by the launcher)
};

// RoPE realignment of stored K rows (sp_rope.cu), one launch per call.
constexpr int kMaxRopeUnits = 2048;   // (sequence, KV head) units in one rope launch
struct RopeParams {
    Meta meta;
    Geo geo;
    int32_t layer;
    int32_t n_units;
    int64_t pos_lo, pos_hi;       // rotate rows whose position is in [pos_lo, pos_hi)
    float cs[64], sn[64];         // cos / sin of delta * theta^(-2i/d), i < d/2
    int32_t unit_seq[kMaxRopeUnits];
    int16_t unit_head[kMaxRopeUnits];
    int32_t unit_n[kMaxRopeUnits];         // tokens the unit's (sequence, layer) holds
    int32_t page_off[kMaxRopeUnits + 1];   // prefix of the units' page counts
};

// Packed-sequence layout (sp_pack_seq / sp_unpack_seq).  The buffer starts
// with PackHeader, then int64 n[layers] (tokens per layer), then
// PackUnit[layers * hkv] in (layer, KV head) order, then the int32 retrieval
// indices of every unit in the same order, then (at payload_off, 256-byte
// aligned) the payload: for each unit its retained K rows then its V rows,
// [rows][head_dim] elements of the page type (bf16, or e4m3 bytes), in
// position order.
constexpr int64_t kPackMagic = 0x3156504B50535053LL;   // "SPSPKPV1" little-endian
constexpr int kTransferRows = 32;                        // rows per copy block
struct PackHeader {
    int64_t magic, version, layers, hkv, head_dim, page_size, n_units, idx_total,
            payload_off, payload_bytes, total_bytes, kv_dtype;
};
struct PackUnit {
    int64_t kind, sink, window, n_idx, rows, row_off, blk_off;
};
struct TransferParams {
    Meta meta;
    Geo geo;
    int32_t seq;
    int32_t unpack;               // 0: pool -> payload, 1: payload -> pool
    int32_t n_units;
    int64_t total_blocks;
    const int64_t* n_layer;       // device: tokens per layer (in the packed buffer)
    const PackUnit* units;        // device: per-unit layout (in the packed buffer)
    uint8_t* payload;             // device
};

struct Workspace {
    void* base;
    size_t bytes;
    // regions
    int4* tiles;          int64_t max_tiles;
    int32_t* tile_ctr;
    float* part_o;        float* part_ml;  int64_t max_parts;
    int32_t* counters;    int64_t max_counter_units;
    float* split_o;       float* split_ml;        // prefill pieces of split items
    int32_t* scratch;     int64_t scratch_ints;   // export / visible-count staging
};

}  // namespace sp

struct sp_cache {
    sp_config cfg;
    sp::Geo geo;
    int device = 0;
    int num_sms = 0;
    int decode_ctas = 0;
    __nv_bfloat16* kpool = nullptr;
    __nv_bfloat16* vpool = nullptr;
    sp::Meta meta;
    sp::Workspace ws;
    CUtensorMap tm_kpool;   // [num_pages*P rows][d], box {64 or d, P}, 128B swizzle
    CUtensorMap tm_vpool;
    CUtensorMap tm_kpool_half;   // FP8 pages of P >= 64: the same with box {d, P / 2}
    CUtensorMap tm_vpool_half;   // (the decode streams such pages in halves)
    // host mirror (authoritative for lengths, page counts and policies)
    std::vector<sp::UnitPol> h_pol;              // [max_seqs][layers][hkv]
    std::vector<std::vector<int32_t>> h_idx;     // per sequence, CSR by unit
    std::vector<uint8_t> h_policy_set;           // per sequence
    std::vector<int32_t> h_seqlen;               // [max_seqs][layers]
    std::vector<int32_t> h_npages;               // [max_seqs][layers][hkv]
    int64_t h_free = 0;
    // Pinned host staging for the per-call prefill work list, so its upload is
    // an asynchronous copy and the host never waits for the device.  A ring:
    // a buffer is refilled only after the copy that last read it has run.
    static constexpr int kStaging = 4;
    int4* stage_buf[kStaging] = {};
    const int4* stage_dev[kStaging] = {};        // the same buffers as device addresses (mapped)
    cudaEvent_t stage_ev[kStaging] = {};
    size_t stage_bytes = 0;                       // size of each buffer
    int stage_next = 0;
    bool prefill_checked[5][4] = {};             // [speculative ? 4 : two issuers ? 3 : FP8 ? 2 : D == 128][log2(P) - 4]: attributes set
    // Caller's event pair armed by sp_set_launch_events for the next
    // attention call (both null when not armed).
    cudaEvent_t launch_ev[2] = {};
    ~sp_cache();
};

namespace sp {

// Pinned staging ring (sp_api.cu): stage_acquire returns the next buffer once
// the copy that last read it has run (nullptr if `bytes` does not fit);
// stage_copy issues its asynchronous upload to `dst` and records its event.
void* stage_acquire(sp_cache* c, size_t bytes, int* slot);
cudaError_t stage_copy(sp_cache* c, int slot, void* dst, size_t bytes, cudaStream_t s);

// Argument checks shared by the entry points (sp_api.cu); they allocate
// nothing.  check_seq_list: 1..max_batch ids, each in range, with a policy,
// none listed twice.
bool valid_layer(const sp_cache* c, int32_t layer);
sp_status check_seq_list(const sp_cache* c, const int32_t* seq_ids, int32_t n_seqs);

// Armed launch events (sp_set_launch_events): the start is recorded right
// before an attention call's first kernel, the end right after its last,
// which also disarms the pair.
inline void launch_mark_start(sp_cache* c, cudaStream_t s) {
    if (c->launch_ev[0]) cudaEventRecord(c->launch_ev[0], s);
}
inline void launch_mark_end(sp_cache* c, cudaStream_t s) {
    if (c->launch_ev[1]) cudaEventRecord(c->launch_ev[1], s);
    c->launch_ev[0] = c->launch_ev[1] = nullptr;
}

// Error plumbing (sp_api.cu).
sp_status fail(sp_status s, const std::string& msg);
sp_status cuda_fail(cudaError_t e, const char* what);
bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                    bool swizzle128, std::string* err, bool bytes = false);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_init_meta(const sp_cache* c, cudaStream_t s);
cudaError_t launch_alloc(const sp_cache* c, const CallSeqs& cs, int layer, int32_t top,
                         cudaStream_t s);
cudaError_t launch_scatter(const sp_cache* c, const CallSeqs& cs, int layer,
                           const __nv_bfloat16* k, const __nv_bfloat16* v,
                           int64_t row_stride, int64_t max_items, cudaStream_t s);
cudaError_t launch_release(const sp_cache* c, int seq, int32_t top, cudaStream_t s);
cudaError_t launch_export(const sp_cache* c, int seq, int layer, int h, int32_t* out_ids,
                          int32_t* out_pos, cudaStream_t s);
cudaError_t launch_decode_counts(const sp_cache* c, int seq, int layer, int h,
                                 const int64_t* pos, int n, int32_t* out, cudaStream_t s);
cudaError_t launch_decode(const sp_cache* c, DecodeParams& p, cudaStream_t s);
cudaError_t launch_rope(const sp_cache* c, const RopeParams& p, cudaStream_t s);
cudaError_t launch_transfer(const sp_cache* c, const TransferParams& p, cudaStream_t s);

}  // namespace sp
