// args_prefill.h -- launch interface of the prefill kernels (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

// ------------------------------------------------------------------ prefill
struct PrefillArgs {
    const __nv_bfloat16* q;  // [T, Hq, 64]
    const __nv_bfloat16* k;  // [T, Hkv, 64]
    const __nv_bfloat16* v;  // [T, Hkv, 64]
    const int32_t* cu_seqlens;  // [N+1]
    const float* sinks;         // [Hq]
    __nv_bfloat16* out;         // [T, Hq, 64]
    float* lse;                 // [T, Hq] or null
    unsigned* err;
    int N, T, max_seqlen, Hq, Hkv, G, causal;
    float scale_log2;
    // paged cache (sinkattn_prefill_paged only): k / v come from [P, Hkv, 16, 64] pools
    const int32_t* page_table;  // [N, max_pages]
    const int32_t* start_pos;   // [N] cache position of each sequence's first new token
    int num_pages, max_pages;
};
// Tensor-core (tcgen05) prefill; the tensor maps are built by the caller.
cudaError_t prefill_tc_launch(const PrefillArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, cudaStream_t stream);
// tcgen05 prefill over two query heads of one KV group per CTA (group size must be even).
cudaError_t prefill_pp_launch(const PrefillArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, cudaStream_t stream);
// Chunked prefill over a paged cache (one-head tcgen05 kernel, K / V gathered page by page).
cudaError_t prefill_paged_launch(const PrefillArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                 const CUtensorMap& tmap_v, cudaStream_t stream);
// The same over two query heads of one KV group per CTA (group size must be even).
cudaError_t prefill_pp_paged_launch(const PrefillArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                    const CUtensorMap& tmap_v, cudaStream_t stream);

}  // namespace sinkattn
