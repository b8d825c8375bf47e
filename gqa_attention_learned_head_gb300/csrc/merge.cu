// merge.cu -- log-sum-exp merge of split partial results, sink counted once.
//
// Source: "GPT-OSS on day 0" (Perplexity), section "Kernels for GPT-OSS / Sink
// Attention": when attention is cut into blocks along the sequence, the sink
// must enter the softmax in one block only.  Here the caller either already
// put it in one split (sinks == null) or hands it to the merge, which adds
// exp(sink) exactly once.
//
// One warp per (row, head); lane l owns head-dims 2l and 2l+1, so the 64-wide
// fp32 partial rows are read with coalesced 8-byte loads and the bf16 output
// row is written as one 128-byte line.  HBM-bound and tiny next to the decode
// pass that produces the partials.
#include "args_merge.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();

__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // r * H + h
    const long long RH = (long long)a.R * a.H;
    if (row >= RH) return;
    const int h = (int)(row % a.H);
    const bool has_sink = a.sinks != nullptr;
    const float sink = has_sink ? __ldg(&a.sinks[h]) : kNegInf;

    float M = sink;
    for (int c = 0; c < a.S; ++c) M = fmaxf(M, __ldg(&a.part_lse[c * RH + row]));
    __nv_bfloat162* out2 = reinterpret_cast<__nv_bfloat162*>(a.out + row * kHeadDim) + lane;
    if (M == kNegInf) {  // nothing at all: empty softmax
        *out2 = __floats2bfloat162_rn(0.f, 0.f);
        if (lane == 0 && a.lse) a.lse[row] = kNegInf;
        return;
    }
    float sum = has_sink ? __expf(sink - M) : 0.f;
    float ox = 0.f, oy = 0.f;
    for (int c = 0; c < a.S; ++c) {
        const float w = __expf(__ldg(&a.part_lse[c * RH + row]) - M);
        if (w == 0.f) continue;  // empty split: its o_c is never read
        sum += w;
        const float2 v = __ldg(reinterpret_cast<const float2*>(a.part_o + (c * RH + row) * kHeadDim) + lane);
        ox += w * v.x;
        oy += w * v.y;
    }
    const float inv = 1.f / sum;
    *out2 = __floats2bfloat162_rn(ox * inv, oy * inv);
    if (lane == 0 && a.lse) a.lse[row] = M + logf(sum);
}

}  // namespace

cudaError_t merge_launch(const MergeArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.R * a.H;
    if (rows == 0) return cudaSuccess;
    merge_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
