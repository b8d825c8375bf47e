// prologue.cu -- the pre-attention step of new tokens, fused: QKV bias, YaRN
// rotary embedding of q and k, q to its output and k / v straight into the
// token's page slot.
//
// Source: "GPT-OSS on day 0" (Perplexity), section "Attention: GQA with
// attention sinks": the QKV projections carry a bias and positions are
// encoded with YaRN rotary embeddings (as in DeepSeek-V3).  The frequencies
// (the published YaRN ramp) are computed on the host in double precision and
// passed in; the position of new token i of sequence n is start_pos[n] + i,
// its slot page_table[n][pos / 16], pos % 16.
//
// HBM-bound elementwise work: one CTA per token.  Warp 0 finds the token's
// sequence, position and page and turns position x frequency into a rotation
// (angle taken in double and reduced to [-pi, pi] before a single-precision
// sincos, so that positions of 10^5 and beyond keep full accuracy); then every
// warp takes heads in turn, a lane per rotated pair.
#include "kernels.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) qkv_prologue_kernel(const PrologueArgs a) {
    __shared__ float s_cos[kHeadDim / 2], s_sin[kHeadDim / 2];
    __shared__ int s_page, s_slot;
    const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {
        int lo = 0, hi = a.N - 1;  // sequence holding token t: largest n with cu_seqlens[n] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(&a.cu_seqlens[mid]) <= t) lo = mid;
            else hi = mid - 1;
        }
        const long long pos = (long long)__ldg(&a.start_pos[lo]) + (t - __ldg(&a.cu_seqlens[lo]));
        constexpr double kTwoPi = 6.283185307179586476925286766559;
        double ang = (double)pos * a.inv_freq[lane];
        ang -= kTwoPi * rint(ang / kTwoPi);
        float sv, cv;
        sincosf((float)ang, &sv, &cv);
        s_cos[lane] = cv * a.mscale;
        s_sin[lane] = sv * a.mscale;
        if (lane == 0) {
            int page = -1;
            if (pos < 0 || pos >= (long long)a.max_pages * kPageSize) {
                atomicOr(a.err, kErrBadLength);
            } else {
                page = __ldg(&a.page_table[(long long)lo * a.max_pages + pos / kPageSize]);
                if (page < 0 || page >= a.num_pages) {
                    atomicOr(a.err, kErrBadPage);
                    page = -1;
                }
            }
            s_page = page;
            s_slot = (int)(pos % kPageSize);
        }
    }
    __syncthreads();
    const int heads = a.Hq + 2 * a.Hkv;
    const int e0 = a.interleaved ? 2 * lane : lane;                         // the pair this lane rotates
    const int e1 = a.interleaved ? 2 * lane + 1 : lane + kHeadDim / 2;
    const float c = s_cos[lane], s = s_sin[lane];
    const int page = s_page, slot = s_slot;
    for (int hd = warp; hd < heads; hd += kThreads / 32) {
        const __nv_bfloat16* src = a.qkv + ((long long)t * heads + hd) * kHeadDim;
        float x0 = __bfloat162float(src[e0]), x1 = __bfloat162float(src[e1]);
        if (a.bias) {
            x0 += __bfloat162float(a.bias[hd * kHeadDim + e0]);
            x1 += __bfloat162float(a.bias[hd * kHeadDim + e1]);
        }
        __nv_bfloat16* dst;
        if (hd < a.Hq + a.Hkv) {  // q or k: rotate the pair, scaled by the YaRN temperature factor
            const float y0 = x0 * c - x1 * s, y1 = x1 * c + x0 * s;
            x0 = y0;
            x1 = y1;
        }
        if (hd < a.Hq) {
            dst = a.q_out + ((long long)t * a.Hq + hd) * kHeadDim;
        } else {
            if (page < 0) continue;
            const bool is_k = hd < a.Hq + a.Hkv;
            const int g = hd - a.Hq - (is_k ? 0 : a.Hkv);
            dst = (is_k ? a.k_pages : a.v_pages) + (((long long)page * a.Hkv + g) * kPageSize + slot) * kHeadDim;
        }
        dst[e0] = __float2bfloat16_rn(x0);
        dst[e1] = __float2bfloat16_rn(x1);
    }
}

}  // namespace

cudaError_t qkv_prologue_launch(const PrologueArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    qkv_prologue_kernel<<<a.T, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
