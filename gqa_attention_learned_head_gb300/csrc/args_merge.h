// args_merge.h -- launch interface of the log-sum-exp merge of caller partials (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

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

}  // namespace sinkattn
