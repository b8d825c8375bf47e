// merge.cu -- log-sum-exp merge of split partial results, sink counted once.
//
// Source: "GPT-OSS on day 0" (Perplexity), section "Kernels for GPT-OSS / Sink
// Attention": when attention is cut into blocks along the sequence, the sink
// must enter the softmax in one block only.  Here the caller either already
// put it in one split (sinks == null) or hands it to the merge, which adds
// exp(sink) exactly once.
//
// sinkattn_merge: one warp per (row, head); lane l owns head-dims 2l and 2l+1,
// so the 64-wide fp32 partial rows are read with coalesced 8-byte loads and
// the bf16 output row is written as one 128-byte line.  HBM-bound and tiny next
// to the pass that produces the partials.  The decode and verification kernels'
// own split segments are merged by split_merge_kernel, launched right behind
// them.
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

constexpr int kSplitThreads = 256;  // 16 half-warps, one (listed segment, row) each

// Log-sum-exp merge of the split segments: half-warp per (listed segment, row); lane l of the
// half-warp owns head-dims 4l..4l+3.  Pieces are taken 8 at a time with all loads issued together
// and combined online (base-2 partial lse).  Waits for the kernel that wrote the partials first,
// then lets the next kernel on the stream start launching.
__global__ void __launch_bounds__(kSplitThreads) split_merge_kernel(const SplitMergeArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kChunk = 8;
    const int R = a.R, hl = threadIdx.x & 15;
    const long long item = (long long)blockIdx.x * (kSplitThreads / 16) + (threadIdx.x >> 4);
    if (item >= (long long)a.listed * R) return;
    const int c = (int)(item / R), r = (int)(item % R);
    const int2 e = __ldcg(&a.list[c]);
    if (e.x < 0) return;
    const int seg = e.x, pieces = e.y;
    const long long slot0 = (long long)c + seg;
    const float* lp = a.part_lse + slot0 * R + r;
    const float* op = a.part_o + (slot0 * R + r) * kHeadDim + 4 * hl;
    float M = kNegInf, sum = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < pieces; c0 += kChunk) {
        float l[kChunk];
        float4 v[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool in = c0 + i < pieces;
            l[i] = in ? __ldcg(lp + (long long)(c0 + i) * R) : kNegInf;
            v[i] = in ? __ldcg(reinterpret_cast<const float4*>(op + (long long)(c0 + i) * R * kHeadDim))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mc = M;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) Mc = fmaxf(Mc, l[i]);
        if (Mc == kNegInf) continue;
        const float rs = M == kNegInf ? 0.f : exp2f(M - Mc);
        sum *= rs;
        o.x *= rs;
        o.y *= rs;
        o.z *= rs;
        o.w *= rs;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const float w = l[i] == kNegInf ? 0.f : exp2f(l[i] - Mc);
            sum += w;
            o.x += w * v[i].x;
            o.y += w * v[i].y;
            o.z += w * v[i].z;
            o.w += w * v[i].w;
        }
        M = Mc;
    }
    const int b = seg / a.Hkv, g = seg - b * a.Hkv;
    const long long row = ((long long)b * a.QL + r / a.G) * a.Hq + g * a.G + r % a.G;
    uint2* dst = reinterpret_cast<uint2*>(a.out + row * kHeadDim) + hl;
    if (M == kNegInf) {  // no live key and no finite sink in any piece
        *dst = make_uint2(0u, 0u);
        if (hl == 0 && a.lse) a.lse[row] = kNegInf;
        return;
    }
    const float inv = 1.f / sum;
    *dst = make_uint2(pack_bf16(o.x * inv, o.y * inv), pack_bf16(o.z * inv, o.w * inv));
    if (hl == 0 && a.lse) a.lse[row] = (M + log2f(sum)) * 0.6931471805599453f;
}

}  // namespace

cudaError_t split_merge_launch(const SplitMergeArgs& a, cudaStream_t stream) {
    const long long items = (long long)a.listed * a.R;
    if (items == 0) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((items + kSplitThreads / 16 - 1) / (kSplitThreads / 16)));
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_merge_kernel, a);
}

cudaError_t merge_launch(const MergeArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.R * a.H;
    if (rows == 0) return cudaSuccess;
    merge_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
