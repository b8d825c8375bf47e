// prefill_mma.cu -- causal varlen prefill with a per-head sink on the legacy
// warp-level tensor path (mma.sync m16n8k16, bf16 -> fp32).
//
// Source of the method: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": the sink-aware kernel template serves prefill as
// well as decode; the online softmax starts from m = sink, d = 1.
//
// This is the FlashAttention-2 style kernel shape that sm_80/sm_90 code uses,
// written for sm_103a: 4 warps x 16 query rows, 64-key tiles double-buffered
// with cp.async, scores and P.V on mma.sync, P kept in registers.  It is the
// baseline the tcgen05 kernel (prefill_tc.cu) is measured against.
#include "args_prefill.h"
#include "ptx.cuh"
#include "tile_order.cuh"

namespace sinkattn {
namespace {

constexpr int kBM = 64, kBN = 64, kPitch = 72;  // 144-byte rows: ldmatrix without bank conflicts
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool pred) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(pred ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows [r0, r0+64) of a [T, H, 64] tensor, head h, into a pitched tile; rows >= rmax are zero-filled.
__device__ __forceinline__ void load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src, long long tok0, int H, int h,
                                          int rvalid) {
#pragma unroll
    for (int i = 0; i < (kBM * 8) / kThreads; ++i) {
        const int c = threadIdx.x + i * kThreads;
        const int r = c >> 3, ch = c & 7;
        const bool ok = r < rvalid;
        const long long tok = tok0 + (ok ? r : 0);
        cp_async16(dst + r * kPitch + ch * 8, src + (tok * H + h) * kHeadDim + ch * 8, ok);
    }
}

__global__ void __launch_bounds__(kThreads) prefill_mma_kernel(const PrefillArgs a) {
    __shared__ __align__(128) __nv_bfloat16 sQ[kBM * kPitch];
    __shared__ __align__(128) __nv_bfloat16 sK[2][kBN * kPitch];
    __shared__ __align__(128) __nv_bfloat16 sV[2][kBN * kPitch];
    extern __shared__ int dyn[];

    TileOrder<kThreads> order;
    order.build(dyn, a.cu_seqlens, a.N, a.T, a.max_seqlen, kBM, a.err);
    const long long lin = blockIdx.x;
    const int idx = (int)(lin / a.Hq), h = (int)(lin % a.Hq);
    if (idx >= order.total) return;
    int seq, qt;
    order.lookup(idx, seq, qt);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const long long s0 = a.cu_seqlens[seq];
    const int L = min(a.cu_seqlens[seq + 1] - a.cu_seqlens[seq], a.max_seqlen);
    const int row0 = qt * kBM;
    const int kvh = h / a.G;
    const int kend = a.causal ? min(L, row0 + kBM) : L;
    const int ntile = (kend + kBN - 1) / kBN;

    load_tile(sQ, a.q, s0 + row0, a.Hq, h, L - row0);
    load_tile(sK[0], a.k, s0, a.Hkv, kvh, kend);
    load_tile(sV[0], a.v, s0, a.Hkv, kvh, kend);
    cp_async_commit();

    const int r_lo = row0 + warp * 16 + gq, r_hi = r_lo + 8;  // this thread's two rows (sequence-relative)
    const float sink2 = __ldg(&a.sinks[h]) * kLog2e;
    float m[2] = {sink2, sink2};
    float d[2] = {tq == 0 ? 1.f : 0.f, tq == 0 ? 1.f : 0.f};  // e^(sink - m) = 1, once per row
    float O[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) O[i][e] = 0.f;
    uint32_t qf[4][4];

    for (int j = 0; j < ntile; ++j) {
        if (j + 1 < ntile) {
            const int kb = (j + 1) * kBN;
            load_tile(sK[(j + 1) & 1], a.k, s0 + kb, a.Hkv, kvh, kend - kb);
            load_tile(sV[(j + 1) & 1], a.v, s0 + kb, a.Hkv, kvh, kend - kb);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int r = warp * 16 + (lane & 15);
                ldmatrix_x4(qf[kk], smem_u32(sQ + r * kPitch + kk * 16 + (lane >> 4) * 8));
            }
        }
        const __nv_bfloat16* Ks = sK[j & 1];
        const __nv_bfloat16* Vs = sV[j & 1];

        float S[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) S[i][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {  // pairs of 8-key n-tiles
                uint32_t b[4];
                const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int col = kk * 16 + ((lane >> 3) & 1) * 8;
                ldmatrix_x4(b, smem_u32(Ks + key * kPitch + col));
                mma_bf16_16816(S[2 * np], qf[kk], b[0], b[1]);
                mma_bf16_16816(S[2 * np + 1], qf[kk], b[2], b[3]);
            }
        }

        // mask + online softmax (base 2)
        const int kb = j * kBN;
        float mx[2] = {kNegInf, kNegInf};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = kb + nt * 8 + 2 * tq + (e & 1);
                const int row = (e < 2) ? r_lo : r_hi;
                const bool vis = key < L && (!a.causal || key <= row);
                S[nt][e] = vis ? S[nt][e] * a.scale_log2 : kNegInf;
                mx[e >> 1] = fmaxf(mx[e >> 1], S[nt][e]);
            }
        float al[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
            mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
            const float mn = fmaxf(m[rr], mx[rr]);
            al[rr] = (mn == kNegInf) ? 1.f : fast_exp2(m[rr] - mn);
            m[rr] = mn;
            d[rr] *= al[rr];
        }
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mn = m[e >> 1];
                p[e] = (mn == kNegInf) ? 0.f : fast_exp2(S[nt][e] - mn);
                d[e >> 1] += p[e];
            }
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p[0], p[1]);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p[2], p[3]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            O[i][0] *= al[0];
            O[i][1] *= al[0];
            O[i][2] *= al[1];
            O[i][3] *= al[1];
        }
        // O += P V ; A = P (rows x keys), B = V (keys x dims) via ldmatrix.trans
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t af[4] = {pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3]};
#pragma unroll
            for (int dp = 0; dp < 4; ++dp) {  // pairs of 8-dim n-tiles
                uint32_t b[4];
                const int key = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int col = dp * 16 + (lane >> 4) * 8;
                ldmatrix_x4_trans(b, smem_u32(Vs + key * kPitch + col));
                mma_bf16_16816(O[2 * dp], af, b[0], b[1]);
                mma_bf16_16816(O[2 * dp + 1], af, b[2], b[3]);
            }
        }
        __syncthreads();
    }

    // finalize: rows r_lo, r_hi
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float dt = d[rr];
        dt += __shfl_xor_sync(0xffffffffu, dt, 1);
        dt += __shfl_xor_sync(0xffffffffu, dt, 2);
        const int row = rr ? r_hi : r_lo;
        if (row >= L) continue;
        const float inv = 1.f / dt;
        const long long tok = s0 + row;
        __nv_bfloat16* orow = a.out + (tok * a.Hq + h) * kHeadDim;
#pragma unroll
        for (int nd = 0; nd < 8; ++nd)
            *reinterpret_cast<__nv_bfloat162*>(orow + nd * 8 + 2 * tq) =
                __floats2bfloat162_rn(O[nd][2 * rr] * inv, O[nd][2 * rr + 1] * inv);
        if (tq == 0 && a.lse) a.lse[tok * a.Hq + h] = (m[rr] + log2f(dt)) * kLn2;
    }
}

}  // namespace

cudaError_t prefill_mma_launch(const PrefillArgs& a, cudaStream_t stream) {
    const int kmax = (a.max_seqlen + kBM - 1) / kBM;
    const long long tiles_ub = (long long)(a.T + kBM - 1) / kBM + a.N;
    const long long grid = tiles_ub * a.Hq;
    if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    const size_t smem = tile_order_smem_ints(a.N, kmax) * sizeof(int);
    const size_t static_smem = sizeof(__nv_bfloat16) * kPitch * (kBM + 4 * kBN);
    if (smem + static_smem > 48 * 1024) {  // above the default limit: opt in (cached per device)
        static thread_local size_t set_to[64] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev >= 64 || set_to[dev] < smem) {
            e = cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (dev < 64) set_to[dev] = smem;
        }
    }
    prefill_mma_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
