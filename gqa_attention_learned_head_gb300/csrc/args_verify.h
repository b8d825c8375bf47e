// args_verify.h -- launch interface of the verification of drafted tokens (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

// ------------------------------------------------------------------ draft verification
constexpr int kVerifyMaxRows = 64;  // q_len * G query rows of one (request, KV head)
constexpr int kVerifyMinTiles = 4;  // automatic split: never cut shares finer than this many key tiles
struct VerifyArgs {
    const __nv_bfloat16* q;     // [B, QL, Hq, 64]
    const int32_t* page_table;  // [B, max_pages]
    const int32_t* kv_lens;     // [B], counting the QL drafted tokens
    const float* sinks;         // [Hq]
    const unsigned long long* tree_mask;  // [B, QL] draft tree masks, or null for a linear draft
    __nv_bfloat16* out;         // [B, QL, Hq, 64]
    float* lse;                 // [B, QL, Hq] or null
    float* part_o;              // [slots, R, 64]
    float* part_lse;            // [slots, R], base-2 log-sum-exp
    int2* merge_list;           // [grid]: (segment, pieces) whose first piece the CTA holds without
                                // completing it, or (-1, 0); null when no segment can be split
    unsigned* err;
    int B, QL, Hq, Hkv, G, R, num_pages, max_pages;  // R = QL * G rows per segment
    int fixed_workers;  // 1: exactly tc_grid shares (the caller's num_workers)
    long long tc_grid;  // shares of the (request, KV head, 128-key tile) units, one CTA each
    float scale_log2;
};
struct VerifyPlan {
    long long tc_grid;                         // shares (CTAs)
    size_t slots, merge_list_offset, ws_bytes;  // workspace: partials per slot, then the merge list
};
cudaError_t verify_plan(int B, int QL, int Hq, int Hkv, int num_workers, VerifyPlan* plan);
// tmap_q covers q as [B * q_len tokens, Hq, 64] with a box of 64 x G heads x q_len tokens.
cudaError_t verify_tc_occupancy(int* per_sm);
// may_split = false: one share, so no segment is cut and no merge kernel is launched.
cudaError_t verify_tc_launch(const VerifyArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                             const CUtensorMap& tmap_v, bool may_split, cudaStream_t stream);
// An empty page pool: every request's cached tokens are absent (out = 0, lse = sink); a request
// with kv_len > 0 raises the bad-page error, one outside [0, max_pages * 16] the bad-length one.
cudaError_t verify_empty_pool_launch(const VerifyArgs& args, cudaStream_t stream);

}  // namespace sinkattn
