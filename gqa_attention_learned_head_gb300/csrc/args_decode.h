// args_decode.h -- launch interface of the paged split-KV decode (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

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
    int2* merge_list;           // [grid]: (segment, pieces) whose page 0 the CTA holds, or (-1, 0);
                                // null when no segment can be split (no merge kernel then)
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
    size_t slots;              // partial-result slots the workspace must hold
    size_t merge_list_offset;  // byte offset of the per-CTA merge list
    size_t ws_bytes;           // workspace bytes
};

// Plan the decode launch for the current device (no device memory touched).
cudaError_t decode_plan(int B, int Hq, int Hkv, int num_workers, DecodePlan* plan);
// may_split = false: the host knows that no segment can be cut (one share), so the merge kernel
// is not launched.
cudaError_t decode_launch(const DecodeArgs& args, const DecodePlan& plan, const CUtensorMap& tmap_k,
                          const CUtensorMap& tmap_v, bool may_split, cudaStream_t stream);

}  // namespace sinkattn
