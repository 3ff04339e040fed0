// sp_select.cu -- on-device retrieval selection (heavy hitters).
//
// The runtime article gives retrieval heads "the top-p important tokens" and
// measures an H2O (heavy-hitter) decode scenario; H2O keeps the keys with the
// largest accumulated attention.  Here, for each KV head h, the score of key
// j is the causal softmax probability it receives, summed over the query
// heads of h and over an observation window (the last n_obs rows of the
// prompt); the selection is the topk highest scores among keys outside a
// recent window (ties: lower position first), united with that window, in
// ascending order -- a RETRIEVAL(I) index list.
//
// Passes (QK^T on mma.sync bf16 tiles of 64 keys, fp32 accumulate):
//   1. k_hh_tile<0>: per key tile and observation row, the tile's max and
//      sum of exponentials (log2 units);
//   2. k_hh_rows: per row, the softmax max and denominator over all tiles;
//   3. k_hh_tile<1>: per key tile, the column sums of the normalised
//      probabilities over every row of the group (no atomics: a block owns
//      its keys);
//   4. k_hh_topk: per KV head, a radix select of the topk-th largest score
//      (scores are >= 0, so their bit patterns order like the values), then
//      the selected indices compacted in index order.
// The top-p form (sp_select_heavy_hitters_top_p) first runs k_hh_topp_count:
// per KV head, how many of the highest-ranked candidates (score descending,
// index ascending) it takes for their summed score to reach top_p times the
// candidates' total (at most max_keys), found by the same digit-by-digit
// descent with each bucket's score mass summed in float64; k_hh_topk then
// selects that many keys per head.
#include <cmath>
#include <memory>

#include "sp_device.cuh"
#include "sp_internal.h"

namespace sp {

namespace {

constexpr int kHhKeys = 64;            // keys per tile
constexpr int kHhRows = 64;            // observation rows per chunk (4 warps x 16)
constexpr int kHhTopkThreads = 1024;

struct HhParams {
    const __nv_bfloat16* q;            // [n_obs][hq][d]
    const __nv_bfloat16* k;            // [n][hkv][d]
    int32_t n, n_obs, hq, hkv, group, d, ntiles;
    float scale_log2;
    float* part_m;                     // [hq][n_obs][ntiles]
    float* part_l;
    float* row_m;                      // [hq][n_obs]
    float* row_l;
    float* scores;                     // [hkv][n]
};

// S tile (kHhRows rows x kHhKeys keys) of one chunk of observation rows for
// one warp: rows warp*16 .. +15 of the chunk, keys 0..63 of the tile.
template <int D>
__device__ __forceinline__ void qk_tile(uint32_t qb, uint32_t kb, int warp, int lane,
                                        float (&sc)[8][4]) {
    constexpr int kStride = (D + 8) * 2;           // padded smem row, bytes
    #pragma unroll
    for (int nt = 0; nt < 8; ++nt)
        #pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
    const int mi = lane >> 3;
    #pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        {   // A: 16 rows x 16 dims
            const int row = warp * 16 + (lane & 15);
            const int col = kk * 16 + (lane >> 4) * 8;
            ldsm_x4(qb + row * kStride + col * 2, a[0], a[1], a[2], a[3]);
        }
        #pragma unroll
        for (int np = 0; np < 4; ++np) {            // two n-tiles of 8 keys per ldmatrix
            const int key = np * 16 + (lane & 7) + (mi >= 2 ? 8 : 0);
            const int col = kk * 16 + (mi & 1) * 8;
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + key * kStride + col * 2, r0, r1, r2, r3);
            mma_bf16_16816(sc[2 * np], a, r0, r1);
            mma_bf16_16816(sc[2 * np + 1], a, r2, r3);
        }
    }
}

// PASS 0: per-row tile statistics; PASS 1: column sums of probabilities.
template <int D, int PASS>
__global__ void __launch_bounds__(128)
k_hh_tile(const __grid_constant__ HhParams p) {
    constexpr int kStride = (D + 8) * 2;
    extern __shared__ __align__(16) uint8_t sm[];
    uint8_t* sK = sm;                              // [64][D + 8] bf16
    uint8_t* sQ = sm + kHhKeys * kStride;          // [64][D + 8] bf16
    float* colsum = reinterpret_cast<float*>(sQ + kHhRows * kStride);   // [4 warps][64]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, h = blockIdx.y;
    const int key0 = tile * kHhKeys;
    // K tile (keys past n read as 0 and are masked below)
    for (int e = threadIdx.x; e < kHhKeys * (D / 8); e += blockDim.x) {
        const int r = e / (D / 8), c = e % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (key0 + r < p.n) v = *reinterpret_cast<const uint4*>(p.k + ((int64_t)(key0 + r) * p.hkv + h) * D + c * 8);
        *reinterpret_cast<uint4*>(sK + r * kStride + c * 16) = v;
    }
    float csum[8][2];
    #pragma unroll
    for (int nt = 0; nt < 8; ++nt) csum[nt][0] = csum[nt][1] = 0.f;
    const int rows = p.group * p.n_obs;            // (query head in group, observation row)
    const int g = lane >> 2, t = lane & 3;
    for (int r0 = 0; r0 < rows; r0 += kHhRows) {
        __syncthreads();                           // previous Q chunk consumed, K tile stored
        for (int e = threadIdx.x; e < kHhRows * (D / 8); e += blockDim.x) {
            const int r = e / (D / 8), c = e % (D / 8);
            const int row = r0 + r;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row < rows) {
                const int gi = row / p.n_obs, oi = row % p.n_obs;
                v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)oi * p.hq + h * p.group + gi) * D + c * 8);
            }
            *reinterpret_cast<uint4*>(sQ + r * kStride + c * 16) = v;
        }
        __syncthreads();
        float sc[8][4];
        qk_tile<D>(smem_u32(sQ), smem_u32(sK), warp, lane, sc);
        // this thread's two rows of the chunk
        #pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = r0 + warp * 16 + g + half * 8;
            const bool row_ok = row < rows;
            const int gi = row_ok ? row / p.n_obs : 0, oi = row_ok ? row % p.n_obs : 0;
            const int pos = p.n - p.n_obs + oi;        // query position
            const int qh = h * p.group + gi;
            if (PASS == 0) {
                float mx = -INFINITY;
                #pragma unroll
                for (int nt = 0; nt < 8; ++nt)
                    #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = key0 + nt * 8 + 2 * t + e;
                        if (key <= pos && key < p.n) mx = fmaxf(mx, sc[nt][half * 2 + e] * p.scale_log2);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                float sum = 0.f;
                if (mx != -INFINITY) {
                    #pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int key = key0 + nt * 8 + 2 * t + e;
                            if (key <= pos && key < p.n) sum += fast_exp2(sc[nt][half * 2 + e] * p.scale_log2 - mx);
                        }
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (row_ok && t == 0) {
                    const int64_t o = ((int64_t)qh * p.n_obs + oi) * p.ntiles + tile;
                    p.part_m[o] = mx;
                    p.part_l[o] = sum;
                }
            } else {
                const float M = row_ok ? p.row_m[(int64_t)qh * p.n_obs + oi] : 0.f;
                const float Lr = row_ok ? p.row_l[(int64_t)qh * p.n_obs + oi] : 0.f;
                const float inv = (row_ok && Lr > 0.f) ? 1.f / Lr : 0.f;
                #pragma unroll
                for (int nt = 0; nt < 8; ++nt)
                    #pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = key0 + nt * 8 + 2 * t + e;
                        if (row_ok && key <= pos && key < p.n)
                            csum[nt][e] += fast_exp2(sc[nt][half * 2 + e] * p.scale_log2 - M) * inv;
                    }
            }
        }
    }
    if (PASS == 1) {
        // column sums: over the 8 lanes that share t (rows g), then over warps
        #pragma unroll
        for (int nt = 0; nt < 8; ++nt)
            #pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = csum[nt][e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                csum[nt][e] = v;
            }
        __syncthreads();
        if (g == 0) {
            #pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                #pragma unroll
                for (int e = 0; e < 2; ++e) colsum[warp * kHhKeys + nt * 8 + 2 * t + e] = csum[nt][e];
        }
        __syncthreads();
        if (threadIdx.x < kHhKeys) {
            const int key = key0 + threadIdx.x;
            const float s = colsum[threadIdx.x] + colsum[kHhKeys + threadIdx.x] +
                            colsum[2 * kHhKeys + threadIdx.x] + colsum[3 * kHhKeys + threadIdx.x];
            if (key < p.n) p.scores[(int64_t)h * p.n + key] = s;
        }
    }
}

// Softmax max and denominator of every (query head, observation row).
__global__ void k_hh_rows(const __grid_constant__ HhParams p) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= (int64_t)p.hq * p.n_obs) return;
    const float* pm = p.part_m + r * p.ntiles;
    const float* pl = p.part_l + r * p.ntiles;
    float M = -INFINITY;
    for (int t = 0; t < p.ntiles; ++t) M = fmaxf(M, pm[t]);
    float L = 0.f;
    if (M != -INFINITY)
        for (int t = 0; t < p.ntiles; ++t)
            if (pm[t] != -INFINITY) L += pl[t] * fast_exp2(pm[t] - M);
    p.row_m[r] = M;
    p.row_l[r] = L;
}

// Top-p count per KV head: the smallest m such that the m highest-ranked
// candidates (j < n - recent; score descending, index ascending) hold at
// least top_p times the candidates' total score, capped at max_keys; 0 when
// that target is 0.  The threshold score T is found digit by digit from the
// top (8 bits at a time) with each bucket's key count and float64 score mass;
// the keys above T are all taken, then as many keys equal to T as the target
// still needs.
__global__ void __launch_bounds__(kHhTopkThreads)
k_hh_topp_count(const float* scores, int32_t n, float top_p, int32_t max_keys, int32_t recent,
                int32_t* kk_out) {
    const int h = blockIdx.x;
    const float* sc = scores + (int64_t)h * n;
    const uint32_t* key = reinterpret_cast<const uint32_t*>(sc);
    const int ncand = max(n - recent, 0);
    __shared__ double wsum[kHhTopkThreads / 32];
    __shared__ uint32_t hcnt[256];
    __shared__ double hmass[256];
    __shared__ uint32_t s_prefix, s_cabove;
    __shared__ double s_above, s_target;
    // the candidates' total score (fixed reduction order)
    double t = 0.0;
    for (int j = threadIdx.x; j < ncand; j += blockDim.x) t += (double)sc[j];
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += wsum[w];
        s_target = (double)top_p * tot;
    }
    __syncthreads();
    const double target = s_target;
    if (ncand == 0 || !(target > 0.0)) {
        if (threadIdx.x == 0) kk_out[h] = 0;
        return;
    }
    uint32_t prefix = 0, mask = 0, cabove = 0;   // keys above the current prefix range
    double above = 0.0;                          // and their score mass
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) { hcnt[b] = 0; hmass[b] = 0.0; }
        __syncthreads();
        for (int j = threadIdx.x; j < ncand; j += blockDim.x) {
            const uint32_t v = key[j];
            if ((v & mask) == prefix) {
                const uint32_t b = (v >> shift) & 255u;
                atomicAdd(&hcnt[b], 1u);
                atomicAdd(&hmass[b], (double)__uint_as_float(v));
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            // the highest bucket at which the running mass reaches the target
            // (bucket 0 takes whatever is left)
            double acc = above;
            uint32_t cacc = cabove;
            int b = 255;
            for (; b > 0; --b) {
                if (hcnt[b] && acc + hmass[b] >= target) break;
                acc += hmass[b];
                cacc += hcnt[b];
            }
            s_prefix = prefix | ((uint32_t)b << shift);
            s_above = acc;
            s_cabove = cacc;
        }
        __syncthreads();
        prefix = s_prefix;
        above = s_above;
        cabove = s_cabove;
        mask |= 255u << shift;
    }
    if (threadIdx.x == 0) {
        const uint32_t ceq = hcnt[prefix & 255u];          // keys equal to T
        const double T = (double)__uint_as_float(prefix);
        int64_t m = ceq;                                    // all of them if the target is not met
        if (T > 0.0 && above + (double)ceq * T >= target) {
            m = (int64_t)ceil((target - above) / T);
            m = m < 1 ? 1 : (m > (int64_t)ceq ? (int64_t)ceq : m);
        }
        int64_t kk = (int64_t)cabove + m;
        kk = kk > max_keys ? max_keys : kk;
        kk_out[h] = (int32_t)(kk > ncand ? ncand : kk);
    }
}

// Top-k per KV head: radix select on the score bits, compaction in index
// order.  kk_head (nullable): a count per head instead of topk (the top-p
// counts); the output row width stays topk + recent.
__global__ void __launch_bounds__(kHhTopkThreads)
k_hh_topk(const float* scores, int32_t n, int32_t topk, const int32_t* kk_head, int32_t recent,
          int32_t* idx, int32_t* counts) {
    const int h = blockIdx.x;
    const uint32_t* key = reinterpret_cast<const uint32_t*>(scores + (int64_t)h * n);
    const int ncand = max(n - recent, 0);
    const int kk = min(kk_head ? min(kk_head[h], topk) : topk, ncand);
    const int width = topk + recent;
    int32_t* out = idx + (int64_t)h * width;
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix, s_need;
    __shared__ int32_t warp_tot[kHhTopkThreads / 32];
    __shared__ int32_t s_base;
    // threshold T: the kk-th largest key, digit by digit from the top
    uint32_t prefix = 0, mask = 0;
    uint32_t need = (uint32_t)kk;                  // still to take at or below the current prefix
    for (int shift = 24; shift >= 0 && kk > 0; shift -= 8) {
        for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < ncand; j += blockDim.x) {
            const uint32_t v = key[j];
            if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t acc = 0;
            int b = 255;
            for (; b > 0; --b) {
                if (acc + hist[b] >= need) break;
                acc += hist[b];
            }
            s_prefix = prefix | ((uint32_t)b << shift);
            s_need = need - acc;
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
        mask |= 255u << shift;
    }
    // selected: key > T, then the first `need` (lowest index) keys == T
    const uint32_t T = prefix;
    int32_t eq_seen = 0;                            // keys == T before the current chunk
    if (threadIdx.x == 0) s_base = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int c0 = 0; c0 < ncand && kk > 0; c0 += blockDim.x) {
        const int j = c0 + threadIdx.x;
        const uint32_t v = j < ncand ? key[j] : 0u;
        const bool gt = j < ncand && v > T;
        const bool eq = j < ncand && v == T;
        // rank among the chunk's equal keys (index order)
        const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
        int eq_rank = __popc(eqb & ((1u << lane) - 1u));
        __shared__ int32_t weq[kHhTopkThreads / 32];
        if (lane == 0) weq[wid] = __popc(eqb);
        __syncthreads();
        int eq_before = 0;
        for (int w = 0; w < wid; ++w) eq_before += weq[w];
        int eq_chunk = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) eq_chunk += weq[w];
        const bool take = gt || (eq && eq_seen + eq_before + eq_rank < (int)need);
        const uint32_t tb = __ballot_sync(0xffffffffu, take);
        const int t_rank = __popc(tb & ((1u << lane) - 1u));
        if (lane == 0) warp_tot[wid] = __popc(tb);
        __syncthreads();
        int before = 0, chunk_tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            if (w < wid) before += warp_tot[w];
            chunk_tot += warp_tot[w];
        }
        const int slot = s_base + before + t_rank;
        if (take && slot < kk) out[slot] = j;          // never past the head's row
        __syncthreads();
        if (threadIdx.x == 0) s_base += chunk_tot;
        eq_seen += eq_chunk;
        __syncthreads();
    }
    // the recent window, then -1 padding
    const int nrec = min(recent, n);
    for (int i = threadIdx.x; i < width - kk; i += blockDim.x)
        out[kk + i] = i < nrec ? ncand + i : -1;
    if (threadIdx.x == 0 && counts) counts[h] = kk + nrec;
}

// Workspace: per-tile and per-row softmax statistics, the scores unless the
// caller keeps them, then the per-head top-p counts.
size_t hh_workspace(int32_t n_obs, int32_t n, int32_t hq, int32_t hkv, bool own_scores) {
    const int64_t ntiles = (n + kHhKeys - 1) / kHhKeys;
    size_t b = 2 * (size_t)hq * n_obs * ntiles * 4 + 2 * (size_t)hq * n_obs * 4;
    if (own_scores) b += (size_t)hkv * n * 4;
    b = (b + 15) & ~size_t(15);
    return b + (size_t)hkv * 4 + 256;
}

// top_p > 0: per-head counts from the top-p rule (at most topk) into kk_buf
template <int D>
cudaError_t launch_hh(const HhParams& p, int32_t topk, float top_p, int32_t* kk_buf,
                      int32_t recent, int32_t* idx, int32_t* counts, cudaStream_t s) {
    constexpr int smem = (kHhKeys + kHhRows) * (D + 8) * 2 + 4 * kHhKeys * 4;
    const dim3 grid(p.ntiles, p.hkv);
    k_hh_tile<D, 0><<<grid, 128, smem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.hq * p.n_obs;
    k_hh_rows<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(p);
    k_hh_tile<D, 1><<<grid, 128, smem, s>>>(p);
    if (top_p > 0.f)
        k_hh_topp_count<<<p.hkv, kHhTopkThreads, 0, s>>>(p.scores, p.n, top_p, topk, recent, kk_buf);
    k_hh_topk<<<p.hkv, kHhTopkThreads, 0, s>>>(p.scores, p.n, topk, top_p > 0.f ? kk_buf : nullptr,
                                                recent, idx, counts);
    return cudaGetLastError();
}

sp_status select_impl(const void* q_obs, int32_t n_obs, const void* k, int32_t n, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t topk, float top_p,
                      int32_t recent, int32_t* idx, int32_t* counts, float* scores, void* workspace,
                      size_t workspace_bytes, void* stream) {
    if (!q_obs || !k || !idx || !workspace) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (n < 1 || n_obs < 1 || n_obs > n) return fail(SP_ERR_INVALID_ARG, "need 1 <= n_obs <= n");
    if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads)
        return fail(SP_ERR_INVALID_ARG, "num_q_heads must be a positive multiple of num_kv_heads");
    if (head_dim != 64 && head_dim != 128) return fail(SP_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (topk < 0 || recent < 0 || (int64_t)topk + recent > INT32_MAX)
        return fail(SP_ERR_INVALID_ARG, "topk and recent must be >= 0");
    if ((reinterpret_cast<uintptr_t>(q_obs) | reinterpret_cast<uintptr_t>(k)) & 15)
        return fail(SP_ERR_INVALID_ARG, "q_obs and k must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(workspace) & 255)
        return fail(SP_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < hh_workspace(n_obs, n, num_q_heads, num_kv_heads, scores == nullptr))
        return fail(SP_ERR_INVALID_ARG, "workspace smaller than sp_select_workspace_bytes");
    HhParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q_obs);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.n = n;
    p.n_obs = n_obs;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.d = head_dim;
    p.ntiles = (n + kHhKeys - 1) / kHhKeys;
    p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const size_t part = (size_t)num_q_heads * n_obs * p.ntiles * 4;
    p.part_m = reinterpret_cast<float*>(w);
    p.part_l = reinterpret_cast<float*>(w + part);
    p.row_m = reinterpret_cast<float*>(w + 2 * part);
    p.row_l = p.row_m + (size_t)num_q_heads * n_obs;
    p.scores = scores ? scores : p.row_l + (size_t)num_q_heads * n_obs;
    size_t used = 2 * part + 2 * (size_t)num_q_heads * n_obs * 4 +
                  (scores ? 0 : (size_t)num_kv_heads * n * 4);
    used = (used + 15) & ~size_t(15);
    int32_t* kk_buf = reinterpret_cast<int32_t*>(w + used);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        head_dim == 128 ? launch_hh<128>(p, topk, top_p, kk_buf, recent, idx, counts, st)
                        : launch_hh<64>(p, topk, top_p, kk_buf, recent, idx, counts, st);
    if (e != cudaSuccess) return cuda_fail(e, "selection launch");
    return SP_OK;
}

}  // namespace

}  // namespace sp

using namespace sp;

extern "C" sp_status sp_select_workspace_bytes(int32_t n_obs, int32_t n, int32_t num_q_heads,
                                               int32_t num_kv_heads, size_t* bytes) {
    if (!bytes) return fail(SP_ERR_INVALID_ARG, "null argument");
    if (n < 1 || n_obs < 1 || n_obs > n || num_q_heads < 1 || num_kv_heads < 1)
        return fail(SP_ERR_INVALID_ARG, "need 1 <= n_obs <= n and positive head counts");
    *bytes = hh_workspace(n_obs, n, num_q_heads, num_kv_heads, true);
    return SP_OK;
}

extern "C" sp_status sp_select_heavy_hitters(const void* q_obs, int32_t n_obs, const void* k,
                                             int32_t n, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t topk, int32_t recent,
                                             int32_t* idx, int32_t* counts, float* scores,
                                             void* workspace, size_t workspace_bytes, void* stream) {
    return select_impl(q_obs, n_obs, k, n, num_q_heads, num_kv_heads, head_dim, topk, 0.f, recent,
                       idx, counts, scores, workspace, workspace_bytes, stream);
}

extern "C" sp_status sp_select_heavy_hitters_top_p(const void* q_obs, int32_t n_obs, const void* k,
                                                   int32_t n, int32_t num_q_heads,
                                                   int32_t num_kv_heads, int32_t head_dim, float top_p,
                                                   int32_t max_keys, int32_t recent, int32_t* idx,
                                                   int32_t* counts, float* scores, void* workspace,
                                                   size_t workspace_bytes, void* stream) {
    if (!(top_p > 0.f && top_p <= 1.f)) return fail(SP_ERR_INVALID_ARG, "top_p must lie in (0, 1]");
    return select_impl(q_obs, n_obs, k, n, num_q_heads, num_kv_heads, head_dim, max_keys, top_p,
                       recent, idx, counts, scores, workspace, workspace_bytes, stream);
}
