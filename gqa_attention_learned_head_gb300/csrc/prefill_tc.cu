// prefill_tc.cu -- causal varlen prefill with a per-head sink on the fifth-
// generation tensor cores (tcgen05 MMA, accumulators in tensor memory).
//
// Source of the method: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": the online softmax starts from m = sink, d = 1, so
// the sink sits in the row normaliser and contributes no value row; the same
// sink-aware kernel serves prefill.
//
// One CTA = one tile of 128 query rows of one head; two CTAs share an SM.
//   warps 0, 3  TMA producers: Q once and K_j tiles into a 3-stage ring
//               (warp 0), V_j tiles into a 2-stage ring (warp 3); 128 keys x 64,
//               128-byte swizzle.
//   warp 1      allocates 256 TMEM columns; issues S_j = Q K_j^T (M=128,
//               N=128, K=64; SMEM x SMEM -> TMEM) as soon as the softmax has
//               read S_{j-1}.
//   warp 2      issues O += P_j V_j (M=128, N=64, K=128; P read from TMEM) as
//               soon as P_j is written.  Two issuers, so that neither chain
//               waits on the other's wake-up; each walks its loop warp-wide and
//               one elected lane issues the products.
//   warps 4-7   softmax: thread r owns query row r (TMEM lane r).  It reads
//               S_j, releases the S columns at once (so S_{j+1} can start),
//               masks the diagonal tile, takes exp2 against a running max that
//               is only moved when it grows by more than 2^8 (rare rescales of
//               O in TMEM), writes P_j as bf16 into TMEM, and at the end writes
//               O / d -- d including the sink term -- and the log-sum-exp.
// TMEM columns: [0,128) S fp32, [128,192) O fp32, [192,256) P bf16 pairs.
// Every wait is bounded; a wait that gives up sets the device error word.
#include "args_prefill.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tile_order.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;

#ifndef SINKATTN_EXP_EMU
#define SINKATTN_EXP_EMU 0  // of every 8 score pairs, this many take exp2 on the FMA pipe (0 measured best)
#endif

constexpr int kKStages = 3, kVStages = 2;  // K runs further ahead: S_{j+1} is issued early

struct __align__(1024) Smem {
    uint8_t q[kTileBytes];
    uint8_t k[kKStages][kTileBytes];
    uint8_t v[kVStages][kTileBytes];
    uint64_t q_full, k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full, s_free, p_full, o_done, mma_done;
    uint64_t v_fixed;  // paged: the last V tile with its rows past the cache end zeroed
    uint32_t tmem_base;
};

// kPaged: K and V come from the page pool through page_table, the new tokens of a sequence sit at
// cache positions start_pos .. start_pos + L - 1 and see the whole cached prefix.
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int* order_ints = reinterpret_cast<int*>(&sm + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Paged: a programmatic dependent of what precedes it on the stream (the append or the prologue that
    // wrote its K / V, whose last CTAs it may overlap): nothing is read before that kernel has completed.
    // It lets no dependent of its own start early, since their waiting CTAs would hold SMs that its later
    // CTAs need.  (The contiguous form follows kernels that do not let it start early: it waits for
    // nothing and launches as a plain kernel, since the wait costs its many short CTAs ~0.3%.)
    if constexpr (kPaged) asm volatile("griddepcontrol.wait;" ::: "memory");

    SeqOrder order;
    order.build_warp0(order_ints, a.cu_seqlens, kPaged ? a.start_pos : nullptr, a.N, a.T, a.max_seqlen, kBM, a.err);
    __syncthreads();
    order.finish_build();
    const int idx = (int)(blockIdx.x / a.Hq), h = (int)(blockIdx.x % a.Hq);
    if (idx >= order.total) return;  // whole CTA: no tile left
    int seq, qt;
    order.lookup_warp(idx, seq, qt);  // every warp on its own
    const int s0 = a.cu_seqlens[seq];
    const int L = min(a.cu_seqlens[seq + 1] - s0, a.max_seqlen);
    const int row0 = qt * kBM;
    const int kvh = h / a.G;
    int start = 0;  // cache position of the sequence's first new token
    if constexpr (kPaged) {
        start = __ldg(&a.start_pos[seq]);
        if (start < 0 || (long long)start + L > (long long)a.max_pages * kPageSize) {
            if (h == 0 && threadIdx.x == 0) atomicOr(a.err, kErrBadLength);
            start = max(0, min(start, a.max_pages * kPageSize - L));
        }
    }
    const int kv_total = start + L;  // cached tokens once the new ones are in
    const int kend = a.causal ? min(kv_total, start + row0 + kBM) : kv_total;
    const int ntile = (kend + kBN - 1) / kBN;
    // paged: the last V tile may end inside a page whose later slots hold anything
    const bool fix_last_v = kPaged && ntile * kBN > kv_total;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);  // released by the S issuer
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);  // released by the PV issuer
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 128);
        mbar_init(&sm.p_full, 128);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.mma_done, 2);
        mbar_init(&sm.v_fixed, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = sm.tmem_base;

    if (warp < 4) {
        // producers: 40 registers (56 for the paged ones, whose whole warp resolves page ids)
        if constexpr (kPaged) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;");
        else asm volatile("setmaxnreg.dec.sync.aligned.u32 40;");
        if (kPaged && (warp == 0 || warp == 3)) {
            // ------------------------------------------------------------ TMA producers over the page pool:
            // warp 0 Q and K_j, warp 3 V_j; lanes 0-7 each copy one 16-token page of a 128-key tile.
            const bool is_k = warp == 0;
            const int stages = is_k ? kKStages : kVStages;
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
            if (lane == 0) {
                tma_prefetch_desc(map);
                if (is_k) {
                    tma_prefetch_desc(&tmap_q);
                    mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
                    tma_load_3d(sm.q, &tmap_q, 0, h, s0 + row0, &sm.q_full);
                }
            }
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < ntile; ++j) {
                const int st = j % stages;
                if (j >= stages) {
                    int got = 0;
                    if (lane == 0) got = mbar_wait(&empty[st], ((j / stages) - 1) & 1);
                    if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
                }
                const int row = page_tile_row(a, seq, kvh, j * (kBN / kPageSize) + (lane & 7), kv_total);
                if (lane == 0) mbar_arrive_expect_tx(&full[st], kTileBytes);
                __syncwarp();
                uint8_t* tile = is_k ? sm.k[st] : sm.v[st];
                if (lane < kBN / kPageSize) tma_load_2d(tile + lane * (kPageSize * 128), map, 0, row, &full[st]);
                issued = j + 1;
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            if (!is_k && ok && fix_last_v) {
                // zero the rows of the last V tile at or past the cache end, then hand it over
                const int j = ntile - 1, st = j % kVStages;
                const bool landed = __all_sync(0xffffffffu, mbar_wait(&sm.v_full[st], (j / kVStages) & 1));
                if (landed) {
                    const int r0 = kv_total - j * kBN;
                    for (int i = r0 * 8 + lane; i < kBN * 8; i += 32)
                        reinterpret_cast<uint4*>(sm.v[st])[i] = make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.v_fixed);
                } else if (lane == 0) {
                    atomicOr(a.err, kErrTimeout);
                }
            }
            // every copy this warp started has landed before the CTA can exit (bounded)
            if (lane == 0) {
                if (is_k) (void)mbar_wait(&sm.q_full, 0);
                for (int j = issued - stages < 0 ? 0 : issued - stages; j < issued; ++j)
                    (void)mbar_wait(&full[j % stages], (j / stages) & 1);
            }
        } else if (!kPaged && warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA producer: Q, then K_j
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            mbar_arrive_expect_tx(&sm.q_full, kTileBytes);
            tma_load_3d(sm.q, &tmap_q, 0, h, s0 + row0, &sm.q_full);
            int issued = 0;
            for (int j = 0; j < ntile; ++j) {
                const int st = j % kKStages;
                if (j >= kKStages && !mbar_wait(&sm.k_empty[st], ((j / kKStages) - 1) & 1)) {
                    atomicOr(a.err, kErrTimeout);
                    break;
                }
                mbar_arrive_expect_tx(&sm.k_full[st], kTileBytes);
                tma_load_3d(sm.k[st], &tmap_k, 0, kvh, s0 + j * kBN, &sm.k_full[st]);
                issued = j + 1;
            }
            // every copy this thread started has landed before the CTA can exit (bounded)
            (void)mbar_wait(&sm.q_full, 0);
            for (int j = issued - kKStages < 0 ? 0 : issued - kKStages; j < issued; ++j)
                (void)mbar_wait(&sm.k_full[j % kKStages], (j / kKStages) & 1);
        } else if (!kPaged && warp == 3 && lane == 0) {
            // ------------------------------------------------------------ TMA producer: V_j
            tma_prefetch_desc(&tmap_v);
            int issued = 0;
            for (int j = 0; j < ntile; ++j) {
                const int st = j % kVStages;
                if (j >= kVStages && !mbar_wait(&sm.v_empty[st], ((j / kVStages) - 1) & 1)) {
                    atomicOr(a.err, kErrTimeout);
                    break;
                }
                mbar_arrive_expect_tx(&sm.v_full[st], kTileBytes);
                tma_load_3d(sm.v[st], &tmap_v, 0, kvh, s0 + j * kBN, &sm.v_full[st]);
                issued = j + 1;
            }
            for (int j = issued - kVStages < 0 ? 0 : issued - kVStages; j < issued; ++j)
                (void)mbar_wait(&sm.v_full[j % kVStages], (j / kVStages) & 1);
        } else if (warp == 1) {
            // ------------------------------------------------------------ S issuer: S_j = Q K_j^T
            // Needs only K_j and the S columns released by the softmax, so S_{j+1} is computed
            // while the softmax still works on tile j.  (The whole warp walks the loop, one elected
            // lane issues.)
            const uint32_t tS = tbase + kColS;
            const uint32_t qaddr = smem_u32(sm.q);
            bool ok = warp_wait(&sm.q_full, 0);
            for (int j = 0; ok && j < ntile; ++j) {
                const int st = j % kKStages;
                ok = warp_wait(&sm.k_full[st], (j / kKStages) & 1) && (j == 0 || warp_wait(&sm.s_free, (j - 1) & 1));
                if (!ok) break;
                tc_fence_after();
                const uint32_t kaddr = smem_u32(sm.k[st]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_ss_warp(tS, sw128_desc(qaddr + kk * 32), sw128_desc(kaddr + kk * 32), kIdescQK, kk > 0);
                tc_commit_warp(&sm.s_full);
                tc_commit_warp(&sm.k_empty[st]);  // K_j read
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);  // every MMA of both issuers has finished before TMEM is released
            (void)warp_wait(&sm.mma_done, 0);
        } else if (warp == 2) {
            // ------------------------------------------------------------ PV issuer: O += P_j V_j
            // (the whole warp walks the loop, one elected lane issues)
            const uint32_t tO = tbase + kColO, tP = tbase + kColP;
            bool ok = true;
            for (int j = 0; ok && j < ntile; ++j) {
                ok = ((fix_last_v && j == ntile - 1) ? warp_wait(&sm.v_fixed, 0)
                                                     : warp_wait(&sm.v_full[j % kVStages], (j / kVStages) & 1)) &&
                     warp_wait(&sm.p_full, j & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t vaddr = smem_u32(sm.v[j % kVStages]);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma_ts_warp(tO, tP + ks * 8, sw128_desc(vaddr + ks * 2048), kIdescPV,
                                   (j > 0 || ks > 0) ? 1u : 0u);
                tc_commit_warp(&sm.v_empty[j % kVStages]);  // V_j read
                tc_commit_warp(&sm.o_done);
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);
            (void)warp_wait(&sm.mma_done, 0);
        }
    } else {
        // 128 x 40 + 128 x 216 = 128 x 56 + 128 x 200 = 256 x 128, the launch's registers
        if constexpr (kPaged) asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
        else asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
        // ---------------------------------------------------------------- softmax warpgroup
        const int r = threadIdx.x - 128;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_off + kColS, tO = tbase + lane_off + kColO, tP = tbase + lane_off + kColP;
        const int qrow = row0 + r;
        const float scale_log2 = a.scale_log2;
        float m = __ldg(&a.sinks[h]) * kLog2e;  // running max, seeded with the sink
        float d = 1.f;                          // e^(sink - m) = 1
        bool ok = true;
        for (int j = 0; j < ntile; ++j) {
            if (!(ok = warp_wait(&sm.s_full, j & 1))) break;
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(&sm.s_free);

            const int kb = j * kBN;
            const bool masked = (kb + kBN > kv_total) || (a.causal && kb + kBN - 1 > start + row0);
            // The row max is taken on the raw scores (scale > 0) with eight independent 3-input max
            // chains; p = exp2(s * scale_log2 - m) is then one FFMA and one MUFU per score.
            float mul = scale_log2;
            if (!(scale_log2 > 0.f)) {  // zero or negative scale: scale first, mask after
#pragma unroll
                for (int c = 0; c < 128; ++c) s[c] *= scale_log2;
                mul = 1.f;
            }
            if (masked) {
                const int lim = (a.causal ? min(kv_total, start + qrow + 1) : kv_total) - kb;  // keys kb + [0, lim)
#pragma unroll
                for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : kNegInf;
            }
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmax3(s[i], s[8 + i], s[16 + i]);
#pragma unroll
            for (int c = 24; c < 120; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmax3(acc[i], s[c + i], s[c + 8 + i]);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaxf(acc[i], s[120 + i]);
            const float mx_raw = fmaxf(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], fmax3(acc[5], acc[6], acc[7])));
            const float mx = mx_raw == kNegInf ? kNegInf : mx_raw * mul;
            const float m_new = fmaxf(m, mx);
            float factor = 1.f;
            bool rescale_o = false;
            if (j == 0 || m_new > m + kRescaleThreshold) {
                factor = (m_new == kNegInf) ? 1.f : fast_exp2(m - m_new);
                rescale_o = (j > 0);
                m = m_new;
                d *= factor;
            }
            const float neg_m = (m == kNegInf) ? 0.f : -m;
            // p = exp2(s * scale_log2 - m) in pairs with packed FMAs; SINKATTN_EXP_EMU of every 8
            // pairs use the FMA-pipe polynomial, the rest the MUFU, so that neither pipe is the limit.
            const float2 mul2 = make_float2(mul, mul), negm2 = make_float2(neg_m, neg_m);
            float2 sums[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float2 xx = ffma2(make_float2(s[2 * c], s[2 * c + 1]), mul2, negm2);
                float2 pp;
                if ((c & 7) < SINKATTN_EXP_EMU) {
                    pp = exp2_fma2(xx);
                } else {
                    pp.x = fast_exp2(xx.x);
                    pp.y = fast_exp2(xx.y);
                }
                sums[c & 3] = fadd2(sums[c & 3], pp);
                pk[c] = pack_bf16(pp.x, pp.y);
            }
            const float2 s01 = fadd2(fadd2(sums[0], sums[1]), fadd2(sums[2], sums[3]));
            const float sum = s01.x + s01.y;
            d += sum;
            if (j > 0) {  // P_{j-1} consumed and O_{j-1} final before P and O are touched
                if (!(ok = warp_wait(&sm.o_done, (j - 1) & 1))) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
                        tmem_st32(tO + c * 32, o);
                    }
                }
            }
            tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.p_full);
        }
        if (ok) ok = warp_wait(&sm.o_done, (ntile - 1) & 1);
        if (ok) {
            tc_fence_after();
            uint32_t o[64];
            tmem_ld32(tO, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
            tmem_ld32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
            tc_wait_ld();
            if (qrow < L) {
                const float inv = d > 0.f ? 1.f / d : 0.f;
                const long long tok = (long long)s0 + qrow;
                uint4* dst = reinterpret_cast<uint4*>(a.out + (tok * a.Hq + h) * kHeadDim);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                    dst[c] = w;
                }
                if (a.lse) a.lse[tok * a.Hq + h] = d > 0.f ? (m + log2f(d)) * kLn2 : kNegInf;
            }
        } else if (lane == 0) {
            atomicOr(a.err, kErrTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

namespace {

template <bool kPaged>
cudaError_t launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   cudaStream_t stream) {
    const long long tiles_ub = (long long)(a.T + kBM - 1) / kBM + a.N;
    const long long grid = tiles_ub * a.Hq;
    if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    const size_t smem = 1024 + sizeof(Smem) + seq_order_smem_ints(a.N) * sizeof(int);
    static thread_local size_t set_to[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || set_to[dev] < smem) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) set_to[dev] = smem;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = kPaged ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<kPaged>, tq, tk, tv, a);
}

}  // namespace

cudaError_t prefill_tc_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream) {
    return launch<false>(a, tq, tk, tv, stream);
}

cudaError_t prefill_paged_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, cudaStream_t stream) {
    return launch<true>(a, tq, tk, tv, stream);
}

}  // namespace sinkattn
