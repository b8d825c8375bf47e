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
// HBM-bound elementwise work: one warp per token.  The lanes find the token's
// sequence, position and page; lane d turns position x frequency of pair d
// into a rotation (angle taken in double and reduced to [-pi, pi] before a
// single-precision sincos, so that positions of 10^5 and beyond keep full
// accuracy) and the lanes share them by shuffles; then four lanes take a head
// (its 32 pairs), each lane eight rotated pairs in two 16-byte pieces (pairs
// (d, d + 32): elements 8l..8l+7 and 8l+32..8l+39; pairs (2d, 2d + 1):
// elements 16l..16l+15), eight heads at a time across the warp, and each lane
// loads several of its heads before it uses any.
#include "args_paged.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarps = 8;  // tokens per CTA

__device__ __forceinline__ float lo_bf16(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// The eight bf16 values of a 16-byte piece, in order, as floats.
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = lo_bf16(w[i]);
        f[2 * i + 1] = hi_bf16(w[i]);
    }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
}

__global__ void __launch_bounds__(kWarps * 32) qkv_prologue_kernel(const PrologueArgs a) {
    const int lane = threadIdx.x & 31;
    // a packing that is not 0 <= cu_seqlens[n] <= cu_seqlens[n+1] <= T is reported (one grid-stride pass)
    for (long long n = (long long)blockIdx.x * blockDim.x + threadIdx.x; n < a.N; n += (long long)gridDim.x * blockDim.x) {
        const int c0 = __ldg(&a.cu_seqlens[n]), c1 = __ldg(&a.cu_seqlens[n + 1]);
        if (c0 < 0 || c1 < c0 || c1 > a.T) atomicOr(a.err, kErrBadLength);
    }
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= a.T) return;
    int lo = 0, hi = a.N - 1;  // sequence holding token t: largest n with cu_seqlens[n] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&a.cu_seqlens[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    // with a corrupted packing the search can land on a sequence that does not hold t: its k / v
    // are not written (q_out still is)
    const bool held = t >= __ldg(&a.cu_seqlens[lo]) && t < __ldg(&a.cu_seqlens[lo + 1]);
    const long long pos = (long long)__ldg(&a.start_pos[lo]) + (t - __ldg(&a.cu_seqlens[lo]));
    int page = -1;
    if (!held || pos < 0 || pos >= (long long)a.max_pages * kPageSize) {
        if (lane == 0) atomicOr(a.err, kErrBadLength);
    } else {
        page = __ldg(&a.page_table[(long long)lo * a.max_pages + pos / kPageSize]);
        if (page < 0 || page >= a.num_pages) {
            if (lane == 0) atomicOr(a.err, kErrBadPage);
            page = -1;
        }
    }
    const int slot = (int)(pos % kPageSize);
    // lane d turns pair d (one double-precision angle per pair and token; double is slow here)
    float cd, sd;
    {
        constexpr double kTwoPi = 6.283185307179586476925286766559, kInvTwoPi = 0.15915494309189533576888376337251;
        double ang = (double)pos * a.inv_freq[lane];
        ang -= kTwoPi * rint(ang * kInvTwoPi);
        sincosf((float)ang, &sd, &cd);
        cd *= a.mscale;
        sd *= a.mscale;
    }
    // this lane's eight pairs: d = 8 (lane % 4) + i, d < 32
    const int l = lane & 3;
    float cs[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cs[i] = __shfl_sync(0xffffffffu, cd, 8 * l + i);
        sn[i] = __shfl_sync(0xffffffffu, sd, 8 * l + i);
    }
    const int heads = a.Hq + 2 * a.Hkv;
    // element offsets of this lane's two 16-byte pieces
    const int o0 = a.interleaved ? 16 * l : 8 * l, o1 = a.interleaved ? 16 * l + 8 : 8 * l + kHeadDim / 2;
    // one head's 16 elements of this lane: bias, rotation (q and k), store
    auto finish = [&](int hd, float (&u)[8], float (&w)[8]) {
        if (a.bias) {
            const uint4* bs = reinterpret_cast<const uint4*>(a.bias + hd * kHeadDim);
            float bu[8], bw[8];
            unpack8(__ldg(bs + o0 / 8), bu);
            unpack8(__ldg(bs + o1 / 8), bw);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                u[i] += bu[i];
                w[i] += bw[i];
            }
        }
        if (hd < a.Hq + a.Hkv) {  // q or k: rotate the pairs, scaled by the YaRN temperature factor
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // pair i = (x, y): halves (u[i], w[i]); interleaved (u or w)[2(i % 4)], [2(i % 4) + 1]
                float& x = a.interleaved ? (i < 4 ? u[2 * i] : w[2 * i - 8]) : u[i];
                float& y = a.interleaved ? (i < 4 ? u[2 * i + 1] : w[2 * i - 7]) : w[i];
                const float rx = x * cs[i] - y * sn[i], ry = y * cs[i] + x * sn[i];
                x = rx;
                y = ry;
            }
        }
        uint4* dst;
        if (hd < a.Hq) {
            dst = reinterpret_cast<uint4*>(a.q_out + ((long long)t * a.Hq + hd) * kHeadDim);
        } else {
            if (page < 0) return;
            const bool is_k = hd < a.Hq + a.Hkv;
            const int g = hd - a.Hq - (is_k ? 0 : a.Hkv);
            dst = reinterpret_cast<uint4*>((is_k ? a.k_pages : a.v_pages) +
                                           (((long long)page * a.Hkv + g) * kPageSize + slot) * kHeadDim);
        }
        dst[o0 / 8] = pack8(u);
        dst[o1 / 8] = pack8(w);
    };
    const uint4* row = reinterpret_cast<const uint4*>(a.qkv + (long long)t * heads * kHeadDim);
    int hd = lane >> 2;
    // this lane's heads are lane / 4 + 8j, taken two per pass with all four 16-byte loads issued
    // before either head is used (one head in flight leaves the warp waiting on DRAM latency)
    for (; hd + 8 < heads; hd += 16) {
        const uint4 x0 = __ldg(row + hd * 8 + o0 / 8), x1 = __ldg(row + hd * 8 + o1 / 8);
        const uint4 y0 = __ldg(row + (hd + 8) * 8 + o0 / 8), y1 = __ldg(row + (hd + 8) * 8 + o1 / 8);
        float u[8], w[8];
        unpack8(x0, u);
        unpack8(x1, w);
        finish(hd, u, w);
        unpack8(y0, u);
        unpack8(y1, w);
        finish(hd + 8, u, w);
    }
    if (hd < heads) {
        float u[8], w[8];
        unpack8(__ldg(row + hd * 8 + o0 / 8), u);
        unpack8(__ldg(row + hd * 8 + o1 / 8), w);
        finish(hd, u, w);
    }
    // this warp's stores are issued: a prefill launched behind this kernel as a programmatic dependent may
    // start its CTAs once every CTA gets here or exits (they wait for this grid to complete before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t qkv_prologue_launch(const PrologueArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    qkv_prologue_kernel<<<(a.T + kWarps - 1) / kWarps, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
