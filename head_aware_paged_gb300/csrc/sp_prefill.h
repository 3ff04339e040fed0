// sp_prefill.h -- prefill entry points used by the host API.
#pragma once
#include "sp_internal.h"

namespace sp {

// Upper bound on prefill work items of one call (sizes the workspace list).
int64_t prefill_max_tiles(const sp_config* c);

// Workspace slots for the pieces of prefill items split along their keys
// (one slot: unnormalised O and (m, l) of 128 rows of two query tiles).
constexpr int kPrefillSplitSlots = 256;

// Plan, upload and launch one prefill call (arguments already validated).
sp_status prefill_impl(sp_cache* c, int32_t layer, const int32_t* seq_ids, int32_t n_seqs,
                       const int32_t* cu_q, const __nv_bfloat16* q, const __nv_bfloat16* k,
                       const __nv_bfloat16* v, __nv_bfloat16* out, float* lse,
                       cudaStream_t stream);

// For positions i >= held: |V(i)| as the prefill kernel's tile plan and mask
// see it, for a chunk starting at the unit's current length (entries with
// i < held are left untouched).
cudaError_t launch_prefill_counts(const sp_cache* c, int seq, int layer, int h,
                                  const int64_t* pos, int n, int32_t* out, cudaStream_t s);

}  // namespace sp
