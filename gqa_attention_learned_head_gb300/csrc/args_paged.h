// args_paged.h -- launch interface of the writing new tokens into pages and the fused pre-attention prologue (between the C ABI
// layer, api.cu, and the kernel translation unit).  Internal to libsinkattn.
#pragma once
#include "args_common.h"

namespace sinkattn {

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

}  // namespace sinkattn
