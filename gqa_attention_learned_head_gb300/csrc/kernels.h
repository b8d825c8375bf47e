// kernels.h -- host-side launch interface between the C ABI layer (api.cu)
// and the kernel translation units.  Internal to libsinkattn.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sinkattn {

constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;

// ------------------------------------------------------------------ decode
struct DecodeArgs {
    const __nv_bfloat16* q;   // [B, Hq, 64]
    const int32_t* page_table;  // [B, max_pages]
    const int32_t* kv_lens;     // [B]
    const float* sinks;         // [Hq]
    __nv_bfloat16* out;         // [B, Hq, 64]
    float* lse;                 // [B, Hq] or null
    float* part_o;              // [slots, G, 64]
    float* part_lse;            // [slots, G], base-2 log-sum-exp
    unsigned long long* counters;  // [B*Hkv]: (call epoch << 24) | pieces arrived
    unsigned long long epoch;      // this call's epoch, in [1, 2^40)
    unsigned* err;              // device error word
    int B, Hq, Hkv, G, num_pages, max_pages;
    int workers;                // number of worker warps sharing the work
    int min_pages_per_worker;   // automatic mode: never cut shares finer than this
    int fixed_workers;          // 1: `workers` shares exactly (capped at the page count)
    float scale_log2;           // scale * log2(e)
};

struct DecodePlan {
    int grid;            // CTAs of the split kernel
    int workers;         // worker warps
    int min_pages;       // automatic mode: never cut shares finer than this many pages
    size_t smem;         // dynamic shared memory of the split kernel
    size_t slots;            // partial-result slots the workspace must hold
    size_t counters_offset;  // byte offset of the per-segment arrival counters
    size_t ws_bytes;         // workspace bytes
};

// Plan the decode launch for the current device (no device memory touched).
cudaError_t decode_plan(int B, int Hq, int Hkv, int num_workers, DecodePlan* plan);
cudaError_t decode_launch(const DecodeArgs& args, const DecodePlan& plan, const CUtensorMap& tmap_k,
                          const CUtensorMap& tmap_v, cudaStream_t stream);

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
    int workers, min_pages_per_worker, fixed_workers;
    float scale_log2;
};
struct VerifyPlan {
    int grid, warps, stages;
    size_t smem, slots, counters_offset, ws_bytes;
};
cudaError_t verify_plan(int B, int QL, int Hq, int Hkv, int num_workers, VerifyPlan* plan);
cudaError_t verify_launch(const VerifyArgs& args, const VerifyPlan& plan, const CUtensorMap& tmap_k,
                          const CUtensorMap& tmap_v, cudaStream_t stream);

// ------------------------------------------------------------------ paged cache: append
struct AppendArgs {
    const __nv_bfloat16* k;     // [T, Hkv, 64] new tokens, packed by cu_seqlens
    const __nv_bfloat16* v;     // [T, Hkv, 64]
    const int32_t* cu_seqlens;  // [N+1]
    const int32_t* start_pos;   // [N] cache position of each sequence's first new token
    const int32_t* page_table;  // [N, max_pages]
    __nv_bfloat16* k_pages;     // [P, Hkv, 16, 64]
    __nv_bfloat16* v_pages;
    unsigned* err;
    int N, T, Hkv, num_pages, max_pages;
};
cudaError_t kv_append_launch(const AppendArgs& args, cudaStream_t stream);

// ------------------------------------------------------------------ pre-attention prologue
struct PrologueArgs {
    const __nv_bfloat16* qkv;   // [T, (Hq + 2 Hkv) * 64]: q heads, k heads, v heads
    const __nv_bfloat16* bias;  // [(Hq + 2 Hkv) * 64] or null
    const int32_t* cu_seqlens;  // [N+1] new tokens
    const int32_t* start_pos;   // [N]
    const int32_t* page_table;  // [N, max_pages]
    __nv_bfloat16* q_out;       // [T, Hq, 64]
    __nv_bfloat16* k_pages;     // [P, Hkv, 16, 64]
    __nv_bfloat16* v_pages;
    unsigned* err;
    int N, T, Hq, Hkv, num_pages, max_pages, interleaved;
    float mscale;                   // multiplier of rotated q and k
    double inv_freq[kHeadDim / 2];  // rotation angle per position of each pair
};
cudaError_t qkv_prologue_launch(const PrologueArgs& args, cudaStream_t stream);

// ------------------------------------------------------------------ merge
struct MergeArgs {
    const float* part_o;    // [S, R, H, 64]
    const float* part_lse;  // [S, R, H]
    const float* sinks;     // [H] or null
    __nv_bfloat16* out;     // [R, H, 64]
    float* lse;             // [R, H] or null
    int S, R, H;
};
cudaError_t merge_launch(const MergeArgs& args, cudaStream_t stream);

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
// Warp-level mma.sync prefill, kept as the legacy-tensor-path baseline.
cudaError_t prefill_mma_launch(const PrefillArgs& args, cudaStream_t stream);

}  // namespace sinkattn
