// args_verify.h -- launch interface of the verification of drafted tokens (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

// ------------------------------------------------------------------ draft verification
constexpr int kVerifyMaxRows = 64;  // q_len * G query rows of one (request, KV head)
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
    unsigned long long* counters;  // [B*Hkv]: (call epoch << 24) | pieces arrived
    unsigned long long epoch;      // this call's epoch, in [1, 2^40)
    unsigned* err;
    int B, QL, Hq, Hkv, G, R, num_pages, max_pages;  // R = QL * G rows per segment
    int workers, min_pages_per_worker, fixed_workers;  // the mma.sync kernel's split
    long long tc_grid;  // the tcgen05 kernel's shares (one CTA each); fixed_workers: exactly that many
    float scale_log2;
};
struct VerifyPlan {
    bool tc;  // the tcgen05 kernel runs (else the mma.sync kernel)
    int grid, warps, stages;  // mma.sync kernel
    long long tc_grid;  // tcgen05 kernel: shares
    size_t smem, slots, counters_offset, ws_bytes;  // workspace: enough for either kernel
};
// use_tc: -1 = the library's choice, 0 = the mma.sync kernel, 1 = the tcgen05 kernel
cudaError_t verify_plan(int B, int QL, int Hq, int Hkv, int num_workers, int use_tc, VerifyPlan* plan);
cudaError_t verify_launch(const VerifyArgs& args, const VerifyPlan& plan, const CUtensorMap& tmap_k,
                          const CUtensorMap& tmap_v, cudaStream_t stream);
// tcgen05 kernel (verify_tc.cu); tmap_q covers q as [B * q_len tokens, Hq, 64] with a box of
// 64 x G heads x q_len tokens.
cudaError_t verify_tc_occupancy(int* per_sm);
cudaError_t verify_tc_launch(const VerifyArgs& args, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                             const CUtensorMap& tmap_v, cudaStream_t stream);

}  // namespace sinkattn
