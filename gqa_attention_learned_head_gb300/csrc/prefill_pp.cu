// prefill_pp.cu -- causal varlen prefill with a per-head sink on the tcgen05
// tensor cores, two query heads per CTA whose softmax phases take turns.
//
// Source of the method: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": the online softmax starts from m = sink, d = 1, so
// the sink sits in the row normaliser and contributes no value row.
//
// Why two heads: at head_dim 64 one 128x128 score tile costs the tensor core
// as long (S = Q K^T plus O += P V) as the MUFU needs for its 16384 exp2.  Two
// CTAs per SM that each own one tile drift into lock-step -- both softmaxes
// compete for the MUFU, then both wait for the tensor core.  Here one CTA per
// SM owns the same 128 query rows of two heads h0, h0 + 1 of one KV group, so
// K_j and V_j are loaded once for both, and the two softmax warpgroups hand an
// "exp turn" back and forth through mbarriers, warp by warp on each SM
// sub-partition (whose exp unit warps k and k + 4 of the two groups share): while
// one group exponentiates tile j, the tensor core runs the other's products.
//
//   warp 0      TMA: both Q tiles once, then K_j into a 3-stage ring.
//   warp 3      TMA: V_j into a 3-stage ring.
//   warp 1      allocates all 512 TMEM columns; issues S_w = Q_w K_j^T for
//               w = 0, 1 as soon as warpgroup w has read its previous S.
//   warp 2      issues O_w += P_w V_j as soon as P_w is written.
// The two issuer warps walk their loops warp-wide and one elected lane issues
// each product (operands computed warp-uniformly: the products go out at the
// tensor pipe's rate, which a lone lane in a divergent branch does not reach).
//   warps 4-7   softmax of head h0 (warpgroup 0), thread r owns query row r.
//   warps 8-11  softmax of head h0 + 1 (warpgroup 1).
// TMEM columns: S_w at 128 w, O_w at 256 + 64 w, P_w (bf16 pairs) at 384 + 64 w.
// Every wait is bounded; a wait that gives up sets the device error word and
// the kernel winds down (the other waits then give up too).
#include "args_prefill.h"
#include "ptx.cuh"
#include "tc_tile.cuh"
#include "tile_order.cuh"

namespace sinkattn {
namespace {

using namespace tc;

constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr int kKStages = 3, kVStages = 3;
constexpr uint32_t kProducerRegs = 72, kSoftmaxRegs = 208;  // 128 x 72 + 256 x 208 <= 384 x 168
// Of a row's 64 score pairs, those exponentiated before the exp turn passes to the partner warp (60: measured
// best among 48-64 on the causal and paged prefills, 1.5% over the full 64).
constexpr int kTurnPairs = 60;

#ifndef SINKATTN_PP_EXP_EMU
#define SINKATTN_PP_EXP_EMU 0  // of every 8 score pairs, this many take exp2 on the FMA pipe
#endif

struct __align__(1024) Smem {
    uint8_t q[2][kTileBytes];
    uint8_t k[kKStages][kTileBytes];
    uint8_t v[kVStages][kTileBytes];
    uint64_t q_full, k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
    // turn[w][k]: warp k of warpgroup w may exponentiate; completed by warp k of the other warpgroup (the
    // same SM sub-partition, whose exp unit the two share) when it has finished its exp phase
    uint64_t turn[2][4];
    uint64_t mma_done;
    uint64_t v_fixed;  // paged: the last V tile with its rows past the cache end zeroed
    uint32_t tmem_base;
};

__device__ __forceinline__ float ex2_in_turn(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// kPaged: K and V come from the page pool through page_table, the new tokens of a sequence sit at
// cache positions start_pos .. start_pos + L - 1 and see the whole cached prefix.
template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pp_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
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
    const int npairs = a.Hq >> 1;
    const int idx = (int)(blockIdx.x / npairs), h0 = 2 * (int)(blockIdx.x % npairs);
    if (idx >= order.total) return;  // whole CTA: no tile left
    int seq, qt;
    order.lookup_warp(idx, seq, qt);  // every warp on its own
    const int s0 = a.cu_seqlens[seq];
    const int L = min(a.cu_seqlens[seq + 1] - s0, a.max_seqlen);
    const int row0 = qt * kBM;
    const int kvh = h0 / a.G;  // h0 and h0 + 1 share it: the group size is even
    int start = 0;  // cache position of the sequence's first new token
    if constexpr (kPaged) {
        start = __ldg(&a.start_pos[seq]);
        if (start < 0 || (long long)start + L > (long long)a.max_pages * kPageSize) {
            if (h0 == 0 && threadIdx.x == 0) atomicOr(a.err, kErrBadLength);
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
            mbar_init(&sm.k_empty[i], 1);  // released by the S issuer after both heads' S
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);  // released by the PV issuer after both heads' PV
        }
        for (int w = 0; w < 2; ++w) {
            mbar_init(&sm.s_full[w], 1);
            mbar_init(&sm.s_free[w], 128);
            mbar_init(&sm.p_full[w], 128);
            mbar_init(&sm.o_done[w], 1);
            for (int k = 0; k < 4; ++k) mbar_init(&sm.turn[w][k], 1);
        }
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
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        if (kPaged && (warp == 0 || warp == 3)) {
            // ------------------------------------------------------------ TMA producers over the page pool:
            // warp 0 Q_0, Q_1 and K_j, warp 3 V_j; lanes 0-7 each copy one 16-token page of a 128-key tile.
            const bool is_k = warp == 0;
            const int stages = is_k ? kKStages : kVStages;
            uint64_t* full = is_k ? sm.k_full : sm.v_full;
            uint64_t* empty = is_k ? sm.k_empty : sm.v_empty;
            const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
            if (lane == 0) {
                tma_prefetch_desc(map);
                if (is_k) {
                    tma_prefetch_desc(&tmap_q);
                    mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
                    tma_load_3d(sm.q[0], &tmap_q, 0, h0, s0 + row0, &sm.q_full);
                    tma_load_3d(sm.q[1], &tmap_q, 0, h0 + 1, s0 + row0, &sm.q_full);
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
                    for (int i = (kv_total - j * kBN) * 8 + lane; i < kBN * 8; i += 32)
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
            // ------------------------------------------------------------ TMA producer: Q_0, Q_1, then K_j
            tma_prefetch_desc(&tmap_q);
            tma_prefetch_desc(&tmap_k);
            mbar_arrive_expect_tx(&sm.q_full, 2 * kTileBytes);
            tma_load_3d(sm.q[0], &tmap_q, 0, h0, s0 + row0, &sm.q_full);
            tma_load_3d(sm.q[1], &tmap_q, 0, h0 + 1, s0 + row0, &sm.q_full);
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
            // ------------------------------------------------------------ S issuer: S_w = Q_w K_j^T
            bool ok = warp_wait(&sm.q_full, 0);
            for (int j = 0; ok && j < ntile; ++j) {
                const int st = j % kKStages;
                if (!(ok = warp_wait(&sm.k_full[st], (j / kKStages) & 1))) break;
                const uint32_t kaddr = smem_u32(sm.k[st]);
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (j > 0 && !(ok = warp_wait(&sm.s_free[w], (j - 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t qaddr = smem_u32(sm.q[w]);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_ss_warp(tbase + kColS + 128u * w, sw128_desc(qaddr + kk * 32),
                                       sw128_desc(kaddr + kk * 32), kIdescQK, kk > 0);
                    tc_commit_warp(&sm.s_full[w]);
                }
                if (!ok) break;
                tc_commit_warp(&sm.k_empty[st]);  // K_j read by both products
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);  // every MMA of both issuers has finished before TMEM is released
            (void)warp_wait(&sm.mma_done, 0);
        } else if (warp == 2) {
            // ------------------------------------------------------------ PV issuer: O_w += P_w V_j
            bool ok = true;
            for (int j = 0; ok && j < ntile; ++j) {
                const int st = j % kVStages;
                if (!(ok = (fix_last_v && j == ntile - 1) ? warp_wait(&sm.v_fixed, 0)
                                                           : warp_wait(&sm.v_full[st], (j / kVStages) & 1)))
                    break;
                const uint32_t vaddr = smem_u32(sm.v[st]);
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (!(ok = warp_wait(&sm.p_full[w], j & 1))) break;
                    tc_fence_after();
                    const uint32_t tO = tbase + kColO + 64u * w, tP = tbase + kColP + 64u * w;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc_mma_ts_warp(tO, tP + ks * 8, sw128_desc(vaddr + ks * 2048), kIdescPV,
                                       (j > 0 || ks > 0) ? 1u : 0u);
                    tc_commit_warp(&sm.o_done[w]);
                }
                if (!ok) break;
                tc_commit_warp(&sm.v_empty[st]);  // V_j read by both products
            }
            if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
            tc_commit_warp(&sm.mma_done);
            (void)warp_wait(&sm.mma_done, 0);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // ---------------------------------------------------------------- softmax warpgroups
        const int w = (warp - 4) >> 2;  // warpgroup = which of the two heads
        const int h = h0 + w;
        const int r = threadIdx.x - 128 - 128 * w;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tbase + lane_off + kColS + 128u * w;
        const uint32_t tO = tbase + lane_off + kColO + 64u * w;
        const uint32_t tP = tbase + lane_off + kColP + 64u * w;
        const int qrow = row0 + r;
        const float scale_log2 = a.scale_log2;
        float m = __ldg(&a.sinks[h]) * kLog2e;  // running max, seeded with the sink
        float d = 1.f;                          // e^(sink - m) = 1
        bool ok = true;
        for (int j = 0; j < ntile; ++j) {
            if (!(ok = warp_wait(&sm.s_full[w], j & 1))) break;
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[c * 32]));
            tc_wait_ld();
            tc_fence_before();
            mbar_arrive(&sm.s_free[w]);

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

            // The exp turn, per SM sub-partition: warp k of warpgroup 0 goes first at every tile, warp k
            // of warpgroup 1 (on the same sub-partition) after it.
            if (w == 0 ? j > 0 : true) {
                if (!(ok = warp_wait(&sm.turn[w][warp & 3], (w == 0 ? j - 1 : j) & 1))) break;
            }
            const float2 mul2 = make_float2(mul, mul), negm2 = make_float2(neg_m, neg_m);
            float2 sums[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                              make_float2(0.f, 0.f)};
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float2 xx = ffma2(make_float2(s[2 * c], s[2 * c + 1]), mul2, negm2);
                float2 pp;
                if ((c & 7) < SINKATTN_PP_EXP_EMU) {
                    pp = exp2_fma2(xx);
                } else {
                    pp.x = ex2_in_turn(xx.x);
                    pp.y = ex2_in_turn(xx.y);
                }
                sums[c & 3] = fadd2(sums[c & 3], pp);
                pk[c] = pack_bf16(pp.x, pp.y);
                if (c == kTurnPairs - 1) {
                    // Hand the turn to the partner warp once this many pairs are summed, so its first exps
                    // overlap this warp's last few and the hand-off's latency: the partial sum is >= 0
                    // always, but the test makes the arrival wait for those exp2.
                    const float2 part = fadd2(fadd2(sums[0], sums[1]), fadd2(sums[2], sums[3]));
                    __syncwarp();
                    if (lane == 0 && !(part.x + part.y < 0.f)) mbar_arrive(&sm.turn[w ^ 1][warp & 3]);
                }
            }
            const float2 s01 = fadd2(fadd2(sums[0], sums[1]), fadd2(sums[2], sums[3]));
            d += s01.x + s01.y;
            if (j > 0) {  // P_{j-1} consumed and O_{j-1} final before P and O are touched
                if (!(ok = warp_wait(&sm.o_done[w], (j - 1) & 1))) break;
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
            mbar_arrive(&sm.p_full[w]);
        }
        if (ok) ok = warp_wait(&sm.o_done[w], (ntile - 1) & 1);
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
                    uint4 v;
                    v.x = pack_bf16(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                    v.y = pack_bf16(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                    v.z = pack_bf16(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                    v.w = pack_bf16(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                    dst[c] = v;
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
cudaError_t launch_pp(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      cudaStream_t stream) {
    if (a.G % 2 != 0) return cudaErrorInvalidValue;  // heads are taken in pairs of one KV group
    const long long tiles_ub = (long long)(a.T + kBM - 1) / kBM + a.N;
    const long long grid = tiles_ub * (a.Hq / 2);
    if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    const size_t smem = 1024 + sizeof(Smem) + seq_order_smem_ints(a.N) * sizeof(int);
    static thread_local size_t set_to[64] = {};
    static thread_local int regs_ok[64] = {};  // 0 unknown, 1 checked
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !regs_ok[dev]) {
        // The register split (setmaxnreg) must fit in what the block is launched with.
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, prefill_pp_kernel<kPaged>)) != cudaSuccess) return e;
        if ((long long)fa.numRegs * kThreads < 128ll * kProducerRegs + 256ll * kSoftmaxRegs)
            return cudaErrorInvalidConfiguration;
        if (dev < 64) regs_ok[dev] = 1;
    }
    if (dev >= 64 || set_to[dev] < smem) {
        e = cudaFuncSetAttribute(prefill_pp_kernel<kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
    return cudaLaunchKernelEx(&cfg, prefill_pp_kernel<kPaged>, tq, tk, tv, a);
}

}  // namespace

cudaError_t prefill_pp_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, cudaStream_t stream) {
    return launch_pp<false>(a, tq, tk, tv, stream);
}

cudaError_t prefill_pp_paged_launch(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, cudaStream_t stream) {
    return launch_pp<true>(a, tq, tk, tv, stream);
}

}  // namespace sinkattn
