// args_merge.h -- launch interfaces of the log-sum-exp merges: of caller partials (sinkattn_merge)
// and of the split segments that the decode and verification kernels leave in their workspace.
// Internal to libsinkattn.
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

// ------------------------------------------------------------------ split segments
// A decode or verification grid of `listed` CTAs cuts the (request b, KV head g) segments into
// pieces; CTA c lists in list[c] the segment whose first piece it holds but does not complete, as
// (b * Hkv + g, pieces), or (-1, 0).  The pieces' normalised partials sit in slots c + seg ..
// c + pieces - 1 + seg of part_o [slots, R, 64] and part_lse [slots, R] (base-2 lse), with
// R = QL * G rows per segment, row r = i * G + h (drafted token i, query head g * G + h; QL = 1
// for decode).
struct SplitMergeArgs {
    const float* part_o;
    const float* part_lse;
    const int2* list;
    __nv_bfloat16* out;  // [B, QL, Hq, 64]
    float* lse;          // [B, QL, Hq] or null
    int listed, R, G, QL, Hq, Hkv;
};
// Launched as a programmatic dependent of the kernel just enqueued on `stream` (which must have
// written everything it reads before it completes): its launch overlaps that kernel, and it waits
// for it before reading.
cudaError_t split_merge_launch(const SplitMergeArgs& args, cudaStream_t stream);

}  // namespace sinkattn
