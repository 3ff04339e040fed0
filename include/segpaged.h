/*
 * segpaged.h -- C ABI of libsegpaged.so, a head-aware paged KV cache with
 * mask-free attention for one GB300 GPU (sm_103a).
 *
 * Method: RedKnot SegPagedAttention, as described in the runtime article
 * "How different attention heads see different context" (section 1: why heads
 * may see different context; section 2: the per-(layer, KV head) head
 * classes; section 3: per-head page tables over one physical page pool, local
 * heads trimmed at KV-write time; section 4: one mask-free fused varlen
 * attention over every (query head, KV head) pair's own visible tokens; section
 * 5: the page layout must be built at write time and reused, never rebuilt per
 * attention call) and in the RedKnot news summary (head-class sparsification:
 * globals about 12-15 % of heads; the BUILDSTATE / SELECTVISIBLESTATE /
 * EXECUTE split of the runtime).
 *
 * Conventions for every call
 *   - Every function returns an sp_status; nothing else crosses the ABI.  On
 *     any status other than SP_OK, sp_last_error() holds a one-line message
 *     (thread-local) and, for argument or capacity errors, nothing was
 *     modified and nothing was launched.
 *   - Device memory belongs to the caller.  The library never allocates
 *     device memory: the caller allocates the pool, metadata and workspace
 *     buffers sized by sp_required_bytes() and keeps them alive until
 *     sp_cache_destroy().  Tensor arguments are borrowed until the
 *     stream-ordered work of the call has completed.
 *   - `stream` is a cudaStream_t (0 = legacy default stream).  Calls are
 *     asynchronous unless marked "synchronous".  All calls that touch one
 *     cache must be issued in stream order (one stream, or with events).
 *   - One cache handle must not be used from two host threads at once.
 *   - Tensors are bf16 (2-byte elements), row-major and contiguous unless a
 *     stride is given:  q / out [tokens][num_q_heads][head_dim];
 *     k / v [tokens][num_kv_heads][head_dim]; lse [tokens][num_q_heads] fp32
 *     (natural logarithm of the softmax denominator incl. the max shift;
 *     -inf for a query with no visible token, whose output row is 0).
 *   - Query head h belongs to KV head h / (num_q_heads / num_kv_heads)
 *     (grouped-query attention, KV-cache tutorial section 5.3, 0-indexed).
 *   - Per call order for one layer and chunk: sp_attention_prefill (history
 *     pages + the chunk itself) then sp_append_kv (the chunk); for decode:
 *     sp_append_kv (the new token) then sp_attention_decode.
 */
#ifndef SEGPAGED_H
#define SEGPAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sp_status {
    SP_OK = 0,
    SP_ERR_INVALID_ARG = 1,    /* bad argument; nothing modified            */
    SP_ERR_OUT_OF_PAGES = 2,   /* pool too small for this call; nothing modified */
    SP_ERR_UNSUPPORTED = 3,    /* shape or size this build does not handle  */
    SP_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed          */
    SP_ERR_DEVICE_STATUS = 5,  /* a kernel flagged an impossible state       */
    SP_ERR_TIMEOUT = 6         /* a bounded device wait gave up              */
} sp_status;

/* Head classes (runtime article section 2).  DENSE attends like GLOBAL; its
 * difference (full re-prefill on reuse) lies outside attention. */
typedef enum sp_kind { SP_GLOBAL = 0, SP_LOCAL = 1, SP_RETRIEVAL = 2 } sp_kind;

/* One (layer, KV head) policy.
 *   GLOBAL:        query i sees positions 0..i.
 *   LOCAL:         query i sees [0, min(sink, i+1)) and [max(0, i-window+1), i];
 *                  sink >= 0, window >= 1.
 *   RETRIEVAL:     query i sees idx[k] <= i; idx strictly ascending, >= 0,
 *                  n_idx >= 0; idx is a host pointer read during the call. */
typedef struct sp_head_policy {
    int32_t kind;
    int32_t sink;
    int32_t window;
    int32_t n_idx;
    const int32_t* idx;
} sp_head_policy;

typedef struct sp_config {
    int32_t num_layers;
    int32_t num_q_heads;
    int32_t num_kv_heads;      /* num_q_heads % num_kv_heads == 0, group <= 16 */
    int32_t head_dim;          /* 64 or 128 */
    int32_t page_size;         /* tokens per page: 16, 32, 64 or 128 */
    int32_t max_seqs;          /* sequence slots 0 .. max_seqs-1 */
    int32_t max_seq_len;       /* longest context a sequence may reach */
    int32_t num_pages;         /* physical pages in the pool (all units share it) */
    int32_t max_idx_per_seq;   /* RETRIEVAL index capacity per sequence (all its units) */
    int32_t max_tokens;        /* most query rows in one prefill / append call */
    int32_t max_batch;         /* most sequences in one call */
    int32_t kv_dtype;          /* sp_kv_dtype of the pages (0 = bf16) */
} sp_config;

/* Element type of the K/V pages.  SP_KV_FP8_E4M3 stores one byte per element
 * (the KV-cache tutorial's quantisation section: FP8 halves the KV cache,
 * per-channel scales keep outlier channels from dominating the range): code =
 * e4m3(x * inv_scale), rounded to nearest even and saturated at +-448, with a
 * scale per (layer, KV head, dimension) for K and for V set by
 * sp_set_kv_scales (1.0 until set); the stored value is code * scale.
 * FP8 pages need head_dim 128.  Decode and prefill read them: decode with
 * f16 MMAs (see sp_set_kv_scales), prefill by turning each history tile into
 * bf16(code * scale) rows in shared memory before its bf16 MMAs (a chunk's
 * own rows enter its attention as the caller's bf16 values).
 * sp_rope_realign on FP8 pages dequantises each key with its channel
 * scales, rotates in fp32 (every product and sum rounded once) and writes
 * the codes again as a write would. */
typedef enum { SP_KV_BF16 = 0, SP_KV_FP8_E4M3 = 1 } sp_kv_dtype;

typedef struct sp_cache sp_cache;  /* opaque host handle */

/* Bytes of the three caller-owned device buffers for cfg (host only, no GPU).
 *   pool: K pages then V pages, each [num_pages][page_size][head_dim] elements
 *         of kv_dtype (bf16, or one byte for FP8).
 *   meta: page tables, policies, retrieval lists, free-page stack, status.
 *   ws:   per-call scratch (prefill work list, decode split partials). */
sp_status sp_required_bytes(const sp_config* cfg, size_t* pool_bytes,
                            size_t* meta_bytes, size_t* ws_bytes);

/* Create a handle over caller-owned buffers (each 1024-byte aligned, at least
 * the sizes above, on the current CUDA device).  Initialises meta (all units
 * empty, every page free) and waits for that to finish: synchronous.  The
 * handle owns a few small pinned HOST buffers (4 x the prefill work list, at
 * most a few MB) so that sp_attention_prefill uploads its work list without
 * blocking the host; sp_cache_destroy waits for their last copies and frees
 * them.  No device memory is allocated. */
sp_status sp_cache_create(const sp_config* cfg, void* pool, void* meta, void* ws,
                          sp_cache** out);

/* Free the host handle only; the caller frees its device buffers. */
sp_status sp_cache_destroy(sp_cache* cache);

/* BUILDSTATE, step 1 (runtime article section 2): set the policy of every
 * (layer, KV head) of sequence `seq`; p has num_layers * num_kv_heads entries,
 * layer-major.  The sequence must hold no tokens (fresh or released).  Copies
 * the retrieval lists to the device on `stream`. */
sp_status sp_set_policy(sp_cache* cache, int32_t seq, const sp_head_policy* p,
                        void* stream);

/* BUILDSTATE, step 2 (runtime article section 3, build from dense K/V, trimming
 * local heads to their visible tokens): write positions 0 .. n_tokens-1 of
 * (seq, layer) from dense k, v laid out [n_tokens][num_kv_heads][head_dim]
 * with `row_stride` elements between consecutive tokens (>= kv_heads*head_dim,
 * multiple of 8).  The (seq, layer) must be empty.  Pages are allocated in
 * this call; only retained rows are copied. */
sp_status sp_build_cache(sp_cache* cache, int32_t seq, int32_t layer,
                         const void* k, const void* v, int64_t n_tokens,
                         int64_t row_stride, void* stream);

/* Append cu_new[b+1] - cu_new[b] new tokens to (seq_ids[b], layer) for
 * b < n_seqs; k, v [cu_new[n_seqs]][num_kv_heads][head_dim] contiguous.
 * GLOBAL heads store every token, LOCAL heads write sink slots or overwrite the
 * oldest ring slot, RETRIEVAL heads store only listed positions.  seq_ids and
 * cu_new are host arrays; sequences must be distinct. */
sp_status sp_append_kv(sp_cache* cache, int32_t layer, const int32_t* seq_ids,
                       int32_t n_seqs, const int32_t* cu_new, const void* k,
                       const void* v, void* stream);

/* EXECUTE, prefill (runtime article section 4): causal attention of a chunk.
 * Rows cu_q[b] .. cu_q[b+1]-1 of q belong to sequence seq_ids[b] and sit at
 * absolute positions n_b .. n_b + c_b - 1, where n_b is what (seq, layer)
 * already holds; keys below n_b come from the cache pages, the rest from the
 * chunk's own k, v (same row layout as q's rows, num_kv_heads heads).  Each
 * query head attends over exactly its KV head's visible set; no mask tensor.
 * out [cu_q[n_seqs]][num_q_heads][head_dim] bf16; lse nullable.  q, k and v
 * must be 16-byte aligned and out 32-byte aligned (SP_ERR_INVALID_ARG
 * otherwise).  Does not modify the cache: call sp_append_kv with the same
 * k, v afterwards. */
sp_status sp_attention_prefill(sp_cache* cache, int32_t layer,
                               const int32_t* seq_ids, int32_t n_seqs,
                               const int32_t* cu_q, const void* q,
                               const void* k, const void* v, void* out,
                               float* lse, void* stream);

/* EXECUTE, decode: one query per sequence at position t = n - 1, where n is
 * what (seq_ids[b], layer) holds (its own token was appended first).
 * q, out [n_seqs][num_q_heads][head_dim]; lse [n_seqs][num_q_heads] nullable.
 * Split-KV: the visible pages of all units are streamed by persistent CTAs;
 * partial results are merged in the same launch. */
sp_status sp_attention_decode(sp_cache* cache, int32_t layer,
                              const int32_t* seq_ids, int32_t n_seqs,
                              const void* q, void* out, float* lse, void* stream);

/* Decode without any device allocation by the caller for scratch: the same
 * computation as sp_attention_decode, but the split-KV scratch (partial
 * outputs, their max / sum and the merge tickets) lives in a fixed 4 MiB
 * device array compiled into this library instead of the cache's workspace.
 * (The method's sources have no counterpart; this entry point is for
 * callers that cannot allocate device memory when they decode: a plain C host
 * without a device allocator, or a serving loop that must not call cudaMalloc
 * mid-step because it can synchronise the device or is forbidden after
 * start-up.)
 *   - The caller still passes the cache, q, out and lse, as for
 *     sp_attention_decode.
 *   - Limit: (n_seqs * num_kv_heads + SM count) * group * (head_dim + 2) * 4
 *     bytes plus the tickets must fit in 4 MiB; larger calls return
 *     SP_ERR_UNSUPPORTED before any launch (use sp_attention_decode).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The current device must be the cache's.
 *   - Every call shares the one array; the tickets are cleared at the start of
 *     each call.  Calls that overlap on the GPU (other streams, other caches)
 *     race on the array and must not be issued concurrently.
 *   - Every GPU that loads the library holds the array until the process
 *     exits. */
sp_status sp_attention_decode_static_scratch(sp_cache* cache, int32_t layer,
                                             const int32_t* seq_ids, int32_t n_seqs,
                                             const void* q, void* out, float* lse,
                                             void* stream);

/* FP8 pages: the per-channel scales of `layer`.  k_scale, v_scale are host
 * arrays [num_kv_heads][head_dim] of floats in [2^-14, 128]; the pages store
 * e4m3(x * (1 / scale)) with the reciprocal taken in fp32.  Decode rebuilds
 * each element as code * scale in f16 (the scale rounded to f16 first), so the
 * range keeps scales normal in f16 and 448 * scale below the f16 maximum;
 * q and P enter the decode MMAs as f16 as well.  Only while no sequence holds
 * tokens in `layer` (SP_ERR_INVALID_ARG otherwise); for a bf16 cache or a
 * scale outside the range SP_ERR_INVALID_ARG.  Synchronous. */
sp_status sp_set_kv_scales(sp_cache* cache, int32_t layer, const float* k_scale,
                           const float* v_scale, void* stream);

/* RoPE realignment of reused keys (news summary, "Elastic Sparsity": the
 * first recovery step is RoPE position alignment).  For every listed sequence
 * and KV head kv_head (-1 = all KV heads) of `layer`, rotates in place every
 * STORED K row whose token position p satisfies pos_lo <= p < pos_hi by
 * `delta` positions of rotary embedding: with a_i = delta * rope_theta^(-2i/d)
 * for i < d/2 (the "rotate half" pairing of element i with element i + d/2),
 *     k'[i]       = k[i] cos a_i - k[i + d/2] sin a_i
 *     k'[i + d/2] = k[i + d/2] cos a_i + k[i] sin a_i.
 * The angles are formed and reduced modulo 2 pi in double precision on the
 * host; the rotation runs in fp32 and rounds to bf16 (at most one bf16 ulp
 * from the exact rotation of the stored value).  FP8 pages: each code is
 * dequantised with its channel's K scale, the pair rotated in fp32 with
 * every product and sum rounded once, and the results written as new codes
 * like a write (e4m3(v * fp32(1 / scale)), saturating).  V and the recorded positions
 * are not changed: a caller reusing KV computed at other positions stores it
 * at its new positions and calls this with delta = new - old.  Rows outside
 * [pos_lo, pos_hi), rows a policy does not store, and other heads are left
 * untouched.  SP_ERR_INVALID_ARG for a bad list or head, pos_lo > pos_hi,
 * rope_theta <= 0 or |delta| > 2^40.  The news summary names no such entry
 * point; this is its RoPE-alignment step applied to the paged layout. */
sp_status sp_rope_realign(sp_cache* cache, int32_t layer, const int32_t* seq_ids,
                          int32_t n_seqs, int32_t kv_head, int64_t pos_lo,
                          int64_t pos_hi, int64_t delta, double rope_theta,
                          void* stream);

/* On-device retrieval selection, heavy hitters (runtime article section 2:
 * retrieval heads see "the top-p important tokens"; section 5 measures an
 * H2O heavy-hitter decode scenario).  No cache is involved: run it on the
 * prompt's dense q / k before setting a RETRIEVAL(I) policy.
 *   q_obs [n_obs][num_q_heads][head_dim] bf16: the observation rows, the last
 *         n_obs query rows of the prompt (positions n - n_obs .. n - 1);
 *   k     [n][num_kv_heads][head_dim] bf16: the prompt's keys (positions 0..n-1).
 * For KV head h the score of key j is the causal softmax probability
 * (scale 1/sqrt(head_dim), visible keys j <= position of the row) summed over
 * h's query heads (grouped-query attention, query head q belongs to KV head
 * q / (num_q_heads / num_kv_heads)) and over the observation rows.  The
 * selection of head h is the topk highest scores among keys j < n - recent
 * (ties: lower j first), then the recent window n - recent .. n - 1, all in
 * ascending order.
 * Outputs (device): idx [num_kv_heads][topk + recent] int32, row h holding
 * min(topk, n - recent) + min(recent, n) indices followed by -1; counts
 * [num_kv_heads] int32 (nullable); scores [num_kv_heads][n] fp32 (nullable).
 * workspace: device scratch of sp_select_workspace_bytes(...) bytes, 256-byte
 * aligned.  Asynchronous on `stream`.  The runtime article names no such
 * entry point; it is the selection step its retrieval heads assume. */
sp_status sp_select_workspace_bytes(int32_t n_obs, int32_t n, int32_t num_q_heads,
                                    int32_t num_kv_heads, size_t* bytes);
sp_status sp_select_heavy_hitters(const void* q_obs, int32_t n_obs, const void* k, int32_t n,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t topk, int32_t recent, int32_t* idx, int32_t* counts,
                                  float* scores, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* The "top-p" form of the same selection (runtime article section 2, "the
 * top-p important tokens"), with the same scores, outputs and workspace:
 * for head h the candidates j < n - recent are ranked by score (descending;
 * ties: lower j first) and the shortest prefix whose summed score reaches
 * top_p times the candidates' total score is kept, at most max_keys keys
 * (the page budget the caller sizes the RETRIEVAL pages for; none when the
 * total is 0), then the recent window.  idx rows are max_keys + recent wide.
 * The sums are taken in float64, so a count whose exact prefix mass lies
 * within a few float64 roundings of the boundary may come out one higher or
 * lower than exact arithmetic would give.  SP_ERR_INVALID_ARG unless
 * 0 < top_p <= 1, as well as for the arguments sp_select_heavy_hitters
 * refuses. */
sp_status sp_select_heavy_hitters_top_p(const void* q_obs, int32_t n_obs, const void* k, int32_t n,
                                        int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, float top_p, int32_t max_keys,
                                        int32_t recent, int32_t* idx, int32_t* counts,
                                        float* scores, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* Pack / unpack one sequence for a prefill/decode-disaggregated transfer (news
 * summary, "system gains": in the PD-separated setting only the tokens each
 * head keeps travel, up to 6.3x fewer KV bytes).  The summary names no such
 * entry points; these carry its trimmed per-head layout across.
 *
 * sp_pack_seq writes into the device buffer dst (256-byte aligned) a header
 * (layer count, KV heads, head_dim, page_size, tokens per layer, every unit's
 * policy and retrieval list, per-unit row offsets) followed by the payload:
 * for each (layer, KV head) unit in order, its retained K rows then its
 * retained V rows, [rows][head_dim] elements of the page type each (bf16, or
 * e4m3 bytes for FP8 pages), in position order (GLOBAL
 * every token, LOCAL the sink then the newest ring's worth, RETRIEVAL its
 * listed positions).  *packed_bytes receives the total size; with dst NULL the
 * call only returns that size (no GPU work).  SP_ERR_INVALID_ARG if
 * dst_bytes is smaller.  The header upload is synchronous; the copy runs on
 * `stream`.
 *
 * sp_unpack_seq restores such a buffer into sequence slot `seq` of this cache,
 * which must hold no tokens and have the same layer count, KV heads, head_dim,
 * page_size and page type (FP8 scales are the receiver's own: set them equal
 * before unpacking): it sets the packed policy, allocates pages for every layer
 * and copies the rows into their slots, so the tables, visible sets and
 * attention results equal the source's.  It reads the header (synchronous),
 * checks it against its own size and policies, and checks page capacity
 * before changing anything (SP_ERR_INVALID_ARG / SP_ERR_OUT_OF_PAGES). */
sp_status sp_pack_seq(sp_cache* cache, int32_t seq, void* dst, size_t dst_bytes,
                      size_t* packed_bytes, void* stream);
sp_status sp_unpack_seq(sp_cache* cache, int32_t seq, const void* src, size_t src_bytes,
                        void* stream);

/* Return every page of `seq` (all layers) to the free stack and empty it; the
 * policy stays set. */
sp_status sp_release_seq(sp_cache* cache, int32_t seq, void* stream);

/* SELECTVISIBLESTATE, for tests: the device page table of one unit.
 * Synchronous.  Writes *npages, page_ids[npages] (physical page ids) and
 * slot_pos[npages * page_size] (token position held by each slot, -1 if
 * empty), as the device-side slot rules see them.  cap bounds both arrays
 * (in pages); SP_ERR_INVALID_ARG if the unit holds more. */
sp_status sp_export_table(sp_cache* cache, int32_t seq, int32_t layer,
                          int32_t kv_head, int32_t* npages, int32_t* page_ids,
                          int32_t* slot_pos, int32_t cap, void* stream);

/* For tests: |V(i)| of one unit for n host positions, computed on the device
 * by the same visible-range functions the attention kernels use.  A position
 * must be below what the unit holds plus max_tokens.  Synchronous. */
sp_status sp_visible_count(sp_cache* cache, int32_t seq, int32_t layer,
                           int32_t kv_head, const int64_t* positions, int32_t n,
                           int32_t* counts, void* stream);

/* Host-side mirrors, no GPU work: tokens held by (seq, layer); free pages. */
sp_status sp_seq_len(const sp_cache* cache, int32_t seq, int32_t layer, int32_t* n);
sp_status sp_free_pages(const sp_cache* cache, int32_t* n);

/* Work accounting from the host policy mirror (no GPU work):
 *   visible (query, key) pairs of a prefill of rows n0 .. n0+c-1 of (seq, layer),
 *   summed over query heads (FLOP = 4 * head_dim * pairs);
 *   visible K+V bytes one decode query at position t of each listed sequence
 *   reads in `layer` (head_dim elements of the page type per row). */
sp_status sp_count_prefill_pairs(const sp_cache* cache, int32_t seq, int32_t layer,
                                 int64_t n0, int64_t c, int64_t* pairs);
sp_status sp_count_decode_bytes(const sp_cache* cache, int32_t layer,
                                const int32_t* seq_ids, int32_t n_seqs,
                                const int64_t* t, int64_t* bytes);

/* Synchronise `stream` and read the device status word: SP_OK, or
 * SP_ERR_DEVICE_STATUS / SP_ERR_TIMEOUT if a kernel flagged a problem (the
 * word is then cleared).  *word (nullable) receives the raw flags. */
sp_status sp_get_status(sp_cache* cache, void* stream, int32_t* word);

/* Check of the bounded waits every kernel uses (no fault, no hang): one
 * warp waits on a shared-memory mbarrier for at most limit_cycles
 * ([1000, 2e9] clock cycles).  mode 0: nothing arrives, the wait gives up and
 * raises the timeout flag of the cache's status word, so the next
 * sp_get_status returns SP_ERR_TIMEOUT (and clears it); mode 1: a second
 * warp arrives after limit_cycles / 8 and the status stays clear; mode 2:
 * two warps that must leave together (the pattern of the prefill's FP8
 * converter pair) each wait on their own barrier, one completes and one
 * never does; both leave after the limit (SP_ERR_TIMEOUT as in mode 0) and
 * neither is left at a named barrier.
 * Asynchronous on `stream`; SP_ERR_INVALID_ARG for other arguments. */
sp_status sp_selftest_bounded_wait(sp_cache* cache, int64_t limit_cycles, int32_t mode,
                                   void* stream);

/* Instrumentation for profilers and benchmarks (the pages have no
 * counterpart).  Arms one pair of caller-created CUDA events (cudaEvent_t
 * handles passed as void*) for the next attention call on this cache
 * (sp_attention_prefill, sp_attention_decode or
 * sp_attention_decode_static_scratch): that call records start_event on its
 * stream immediately before its first kernel launch and end_event
 * immediately after its last one (the prefill's merge included), so the
 * interval between them is the device time of the call's kernels without
 * the host's planning, which otherwise shows in events recorded around the
 * call whenever the device is idle while the host plans.  The pair is used
 * by one call and then disarmed (a call that fails may leave it armed).
 * Both null disarms.  The events stay owned by the caller and
 * must stay alive until that call has been made.
 * SP_ERR_INVALID_ARG for a null cache or exactly one null event. */
sp_status sp_set_launch_events(sp_cache* cache, void* start_event, void* end_event);

/* Message of the last failing call on this thread ("" if none). */
const char* sp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SEGPAGED_H */
