// verify.cu -- attention of drafted tokens over the paged cache (verification
// in speculative decoding), with a per-head learned sink.
//
// Source: "Accelerating Sonar through speculation" (Perplexity), sections
// "Speculative decoding" (the target model runs over the drafted tokens and
// produces logits for every one of them, so up to n + 1 tokens come out of one
// step) and "Inference with speculative decoding" (verification batches over
// the paged KV cache); the attention itself is the sink attention of "GPT-OSS
// on day 0", section "Kernels for GPT-OSS / Sink Attention".  Query token i of
// request b is the cache token at position kv_len - q_len + i (its K and V are
// already in the pages) and sees cache tokens 0 .. that position -- or, for a
// tree of drafts (section "EAGLE": the target checks the drafted tree with a
// custom attention mask), every token before the draft and the drafted tokens
// on its own path, given as a bit mask per token.
//
// GB300 design: the decode's work split (split_kv.cuh: contiguous per-CTA
// shares of (request, KV head, page) units, pieces, merge in the same launch),
// but the R = q_len x G query rows of a (request, KV head) go through ONE pass
// over its pages, so the draft costs the cache bytes once:
//  * consumer warp w < W owns rows 16w .. 16w+15 (row r = i * G + head within
//    the group); all consumer warps read every page of the share from one CTA ring
//    of 3W + 1 stages, which a producer warp (warp W) fills by TMA (K and V
//    slices of one (page, KV head), 128-byte swizzle) as soon as every consumer
//    has released a stage.  The producer is a warp of its own so that its
//    waits -- for the slowest consumer, for page ids, for a TMA issue slot --
//    never hold up the products;
//  * per warp and page: S[16 rows x 16 tokens] = Q K^T and O[16 x 64] += P V
//    with mma.m16n8k16 (rows on M, so P goes from the accumulators straight
//    into the next product), online softmax in registers, each row masked at
//    its own causal limit;
//  * no combine between warps (they own different rows); a piece that is not
//    a whole segment writes fp32 partials per row and the CTA completing the
//    segment merges them by log-sum-exp.
// Every wait is bounded; a wait that gives up sets the device error word.
#include <climits>

#include "args_verify.h"
#include "ptx.cuh"
#include "split_kv.cuh"

namespace sinkattn {
namespace {

constexpr int kSliceBytes = kPageSize * kHeadDim * 2;  // 2048: one (page, KV head) of K or V
constexpr int kStageBytes = 2 * kSliceBytes;
constexpr int kMinPages = 32;  // automatic mode: never cut shares finer than this
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
// The library's choice between the two kernels: the tcgen05 kernel from this many query rows per
// (request, KV head) on (measured faster at 8, 16, 32 and 64 rows).
constexpr int kTcMinRows = 1;

// Shared memory: ring | full / empty barriers | bad-page flags | misc | pend | queue | prefix[B+1].
struct Layout {
    size_t ring, full, empty, bad, misc, pend, queue, prefix, total;
    __host__ __device__ Layout(int stages, int B) {
        ring = 0;
        full = size_t(stages) * kStageBytes;
        empty = full + size_t(stages) * 8;
        bad = empty + size_t(stages) * 8;
        misc = bad + size_t(stages) * 4;  // [0..8] scan scratch, [12] merge queue count, [13] pend count
        pend = misc + 16 * 4;
        queue = pend + 2 * 4;
        prefix = queue + 2 * 4;
        total = prefix + size_t(B + 1) * 4 + 1024 /* alignment slack */;
    }
};

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Keeps the bf16 halves of x whose token (lo: t, hi: t + 1) lies below `valid`.
__device__ __forceinline__ uint32_t keep_tokens(uint32_t x, int t, int valid) {
    return x & ((t < valid ? 0x0000FFFFu : 0u) | (t + 1 < valid ? 0xFFFF0000u : 0u));
}

// Log-sum-exp merge of one query row of one segment from its partials (base-2 lse), by the 4
// lanes of a quad: lane l owns head-dims 16l..16l+15.  Pieces are taken 4 at a time with all
// loads issued together and combined online; a quad per row keeps many rows in flight at once.
__device__ __forceinline__ void merge_row(const VerifyArgs& a, int b, int g, int r, long long slot0, int pieces,
                                          int hl) {
    constexpr int kChunk = 4;
    const int R = a.R;
    const float* lp = a.part_lse + slot0 * R + r;
    const float* op = a.part_o + (slot0 * R + r) * kHeadDim + 16 * hl;
    float M = kNegInf, sum = 0.f;
    float o[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = 0.f;
    for (int c0 = 0; c0 < pieces; c0 += kChunk) {
        float l[kChunk];
        float4 v[kChunk][4];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const bool in = c0 + i < pieces;
            const float4* src = reinterpret_cast<const float4*>(op + (long long)(c0 + i) * R * kHeadDim);
            l[i] = in ? __ldcg(lp + (long long)(c0 + i) * R) : kNegInf;
#pragma unroll
            for (int k = 0; k < 4; ++k) v[i][k] = in ? __ldcg(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mc = M;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) Mc = fmaxf(Mc, l[i]);
        if (Mc == kNegInf) continue;
        const float rs = M == kNegInf ? 0.f : exp2f(M - Mc);
        sum *= rs;
#pragma unroll
        for (int k = 0; k < 16; ++k) o[k] *= rs;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const float w = l[i] == kNegInf ? 0.f : exp2f(l[i] - Mc);
            sum += w;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                o[4 * k + 0] += w * v[i][k].x;
                o[4 * k + 1] += w * v[i][k].y;
                o[4 * k + 2] += w * v[i][k].z;
                o[4 * k + 3] += w * v[i][k].w;
            }
        }
        M = Mc;
    }
    const int i = r / a.G, h = g * a.G + r % a.G;
    const long long row = ((long long)b * a.QL + i) * a.Hq + h;
    uint4* dst = reinterpret_cast<uint4*>(a.out + row * kHeadDim + 16 * hl);
    if (M == kNegInf) {  // no live key and no finite sink in any piece
        dst[0] = dst[1] = make_uint4(0u, 0u, 0u, 0u);
        if (hl == 0 && a.lse) a.lse[row] = kNegInf;
        return;
    }
    const float inv = 1.f / sum;
#pragma unroll
    for (int k = 0; k < 2; ++k)
        dst[k] = make_uint4(pack_bf16(o[8 * k + 0] * inv, o[8 * k + 1] * inv), pack_bf16(o[8 * k + 2] * inv, o[8 * k + 3] * inv),
                            pack_bf16(o[8 * k + 4] * inv, o[8 * k + 5] * inv), pack_bf16(o[8 * k + 6] * inv, o[8 * k + 7] * inv));
    if (hl == 0 && a.lse) a.lse[row] = (M + log2f(sum)) * kLn2;
}

// Resident CTAs per SM the launch bounds ask for: a register cap of 128 (one consumer warp) or
// 136 (two or four), which the consumers need without spilling.
template <int W>
constexpr int min_blocks() { return W == 1 ? 8 : W == 2 ? 5 : 3; }

template <int W>  // W consumer warps = W groups of 16 query rows, plus one producer warp
__global__ void __launch_bounds__((W + 1) * 32, min_blocks<W>())
    verify_split_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const VerifyArgs a) {
    constexpr int S = 3 * W + 1;  // ring stages: slack for consumers that drift apart
    const Layout L(S, a.B);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = sm + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(sm + L.empty);
    int* bad = reinterpret_cast<int*>(sm + L.bad);
    int* misc = reinterpret_cast<int*>(sm + L.misc);
    int* pend = reinterpret_cast<int*>(sm + L.pend);    // segments of this share's partial pieces
    int* queue = reinterpret_cast<int*>(sm + L.queue);  // segments this CTA completes and merges
    int* prefix = reinterpret_cast<int*>(sm + L.prefix);  // [B + 1] exclusive prefix of pages per request

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, Hkv = a.Hkv, G = a.G, QL = a.QL, R = a.R, cap = a.max_pages * kPageSize;

    // ---- 1. pages per request -> exclusive prefix sum (every CTA, in shared memory)
    int running = 0;
    for (int base = 0; base < B; base += (W + 1) * 32) {
        const int b = base + tid;
        int n = 0;
        if (b < B) {
            const int Lb = a.kv_lens[b];
            if ((Lb < 0 || Lb > cap) && blockIdx.x == 0) atomicOr(a.err, kErrBadLength);
            n = (clamp_len(Lb, cap) + kPageSize - 1) / kPageSize;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) misc[warp] = incl;
        __syncthreads();
        int woff = 0, tot = 0;
#pragma unroll
        for (int w = 0; w <= W; ++w) {
            const int v = misc[w];
            woff += (w < warp) ? v : 0;
            tot += v;
        }
        if (b < B) prefix[b] = running + woff + incl - n;
        running += tot;
        __syncthreads();
    }
    if (tid == 0) {
        prefix[B] = running;
        misc[12] = 0;
    }
    __syncthreads();

    // ---- 2. requests with no cached token: every row's mass on the sink (out = 0, lse = sink)
    {
        const long long rows = (long long)B * QL * a.Hq;
        for (long long r = (long long)blockIdx.x * blockDim.x + tid; r < rows; r += (long long)gridDim.x * blockDim.x) {
            const int b = (int)(r / ((long long)QL * a.Hq));
            if (prefix[b + 1] != prefix[b]) continue;
            uint4* dst = reinterpret_cast<uint4*>(a.out + r * kHeadDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
            if (a.lse) a.lse[r] = __ldg(&a.sinks[r % a.Hq]);
        }
    }

    const long long U = (long long)running * Hkv;
    if (U == 0) return;
    const long long C = effective_shares(a.workers, a.fixed_workers, a.min_pages_per_worker, U);
    const long long cta = blockIdx.x;
    if (cta >= C) return;
    const long long x0 = cta * U / C, x1 = (cta + 1) * U / C;
    const int total = (int)(x1 - x0);

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);  // every consumer warp releases every page
        }
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    __syncthreads();

    // ---- 3. producer (warp W): walks the share's pages; lanes resolve 32 page ids at a time
    SegPiece pp;
    piece_first(pp, prefix, B, Hkv, x0, x1);
    int pt = 0, win_base = -64, win_row = -1, issued = 0;
    auto issue_next = [&]() {  // warp-uniform; the stage of page `issued` is free
        if (pt >= pp.len()) {
            piece_next(pp, prefix, B, Hkv, x1);
            pt = 0;
            win_base = -64;
        }
        if (pt - win_base >= 32) {
            win_base = pt;
            int row = -1;
            if (pt + lane < pp.len()) {
                const int pid = __ldg(&a.page_table[(long long)pp.b * a.max_pages + pp.page0() + pt + lane]);
                if (pid >= 0 && pid < a.num_pages) row = (pid * Hkv + pp.g) * kPageSize;
            }
            win_row = row;
        }
        const int row = __shfl_sync(0xffffffffu, win_row, pt - win_base);
        if (lane == 0) {
            const int s = issued % S;
            uint8_t* dst = ring + s * kStageBytes;
            if (row >= 0) {
                bad[s] = 0;
                mbar_arrive_expect_tx(&full[s], kStageBytes);
                tma_load_2d(dst, &tmap_k, 0, row, &full[s]);
                tma_load_2d(dst + kSliceBytes, &tmap_v, 0, row, &full[s]);
            } else {
                bad[s] = 1;
                atomicOr(a.err, kErrBadPage);
                mbar_arrive(&full[s]);
            }
        }
        ++pt;
        ++issued;
    };
    if (warp == W) {
        bool ok = true;
        while (ok && issued < total) {
            if (issued >= S) {  // the stage's previous page must be released by every consumer
                int got = 0;
                if (lane == 0) got = mbar_wait(&empty[issued % S], ((issued / S) - 1) & 1);
                ok = __shfl_sync(0xffffffffu, got, 0) != 0;
                if (!ok) break;
            }
            issue_next();
        }
        if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
        // every copy it started has landed before the CTA can exit (bounded)
        for (int j = issued > S ? issued - S : 0; j < issued; ++j) (void)mbar_wait(&full[j % S], (j / S) & 1);
    }

    // ---- 4. consumers (warps 0 .. W-1): piece by piece, page by page
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
    int consumed = 0;
    bool failed = false;
    int pend_n = 0;  // partial pieces of this share (at most its first and its last), thread 0 only
    SegPiece cp;
    piece_first(cp, prefix, B, Hkv, x0, x1);
    for (; warp < W && cp.ps < x1; piece_next(cp, prefix, B, Hkv, x1)) {
        const int kv_len = clamp_len(__ldg(&a.kv_lens[cp.b]), cap);
        const int pos0 = kv_len - QL;  // cache position of drafted token 0 (negative for a short cache)
        // This lane's two query rows (mma rows gq and gq + 8 of the warp's 16): keys [0, lim) visible;
        // with a draft tree, a drafted key j (position pos0 + j) only if bit j of the row's mask is set.
        const bool tree = a.tree_mask != nullptr;
        int rr[2], lim[2];
        float sink2[2];
        unsigned long long bits[2] = {0ull, 0ull};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            rr[e] = 16 * warp + gq + 8 * e;
            const bool live = rr[e] < R;
            lim[e] = !live ? 0 : tree ? kv_len : pos0 + rr[e] / G + 1;
            sink2[e] = live ? __ldg(&a.sinks[cp.g * G + rr[e] % G]) * kLog2e : kNegInf;
            if (tree && live) bits[e] = __ldg(&a.tree_mask[(long long)cp.b * QL + rr[e] / G]);
        }
        // smallest limit over the warp's live rows (for a tree: the draft's start): pages below it
        // need no mask
        const int first_masked = tree ? max(pos0, 0) : INT_MAX;
        int lim_lo = min(rr[0] < R ? min(lim[0], first_masked) : INT_MAX, rr[1] < R ? min(lim[1], first_masked) : INT_MAX);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) lim_lo = min(lim_lo, __shfl_xor_sync(0xffffffffu, lim_lo, o));
        // A fragments of Q (rows gq, gq + 8; dims 2tq, 2tq+1 and +8 within each 16-dim step)
        uint32_t qa[4][4];
        {
            const __nv_bfloat16* qr[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = rr[e] < R ? rr[e] : 0;
                qr[e] = a.q + (((long long)cp.b * QL + r / G) * a.Hq + cp.g * G + r % G) * kHeadDim;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                qa[kk][0] = rr[0] < R ? ld_u32(qr[0] + kk * 16 + 2 * tq) : 0u;
                qa[kk][1] = rr[1] < R ? ld_u32(qr[1] + kk * 16 + 2 * tq) : 0u;
                qa[kk][2] = rr[0] < R ? ld_u32(qr[0] + kk * 16 + 8 + 2 * tq) : 0u;
                qa[kk][3] = rr[1] < R ? ld_u32(qr[1] + kk * 16 + 8 + 2 * tq) : 0u;
            }
        }
        const bool seeded = cp.page0() == 0;  // this piece holds token 0: it carries the sink
        const int seg = cp.b * Hkv + cp.g;
        const bool whole = seeded && (cp.pe == cp.seg_start + cp.n);
        float m[2], d[2], O[8][4];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            m[e] = seeded ? sink2[e] : kNegInf;
            d[e] = (seeded && tq == 0) ? 1.f : 0.f;  // the sink's own e^(sink-m)=1, once per row
        }
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) O[n][e] = 0.f;

        const int npg = cp.len();
        for (int t = 0; t < npg; ++t) {
            const int s = consumed % S;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (consumed / S) & 1))) {
                failed = true;
                if (lane == 0) atomicOr(a.err, kErrTimeout);
                break;
            }
            const int page = cp.page0() + t;
            const int valid = bad[s] ? 0 : min(kPageSize, kv_len - page * kPageSize);
            const uint32_t kb = smem_u32(ring + s * kStageBytes), vb = kb + kSliceBytes;

            // S = Q K^T : 16 rows x 16 tokens (two n-tiles of 8 tokens); K rows give B fragments
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int tok = ((lane >> 4) << 3) + (lane & 7);
                const int chunk = 2 * kk + ((lane >> 3) & 1);
                uint32_t kf[4];
                ldmatrix_x4(kf, kb + tok * 128 + ((chunk ^ (tok & 7)) << 4));
                mma_bf16_16816(acc[0], qa[kk], kf[0], kf[1]);
                mma_bf16_16816(acc[1], qa[kk], kf[2], kf[3]);
            }

            // online softmax (base 2): element e of n-tile j is row rr[e >> 1], token 8j + 2tq + (e & 1).
            // Only the pages holding the draft or the cache end need the per-row limits.
            float sc[2][4];
            if (valid == kPageSize && (page + 1) * kPageSize <= lim_lo) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[j][e] = acc[j][e] * a.scale_log2;
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int slot_tok = 8 * j + 2 * tq + (e & 1);
                        const int tok = page * kPageSize + slot_tok;
                        const bool live = slot_tok < valid && tok < lim[e >> 1] &&
                                          (tok < pos0 || !tree || ((bits[e >> 1] >> (tok - pos0)) & 1ull));
                        sc[j][e] = live ? acc[j][e] * a.scale_log2 : kNegInf;
                    }
            }
            float mx[2];
            mx[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mx[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) {
                mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
                mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
            }
            float al[2], p[2][4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float mn = fmaxf(m[e], mx[e]);
                const bool dead = mn == kNegInf;
                al[e] = dead ? 1.f : fast_exp2(m[e] - mn);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    p[j][2 * e] = dead ? 0.f : fast_exp2(sc[j][2 * e] - mn);
                    p[j][2 * e + 1] = dead ? 0.f : fast_exp2(sc[j][2 * e + 1] - mn);
                }
                d[e] = d[e] * al[e] + ((p[0][2 * e] + p[0][2 * e + 1]) + (p[1][2 * e] + p[1][2 * e + 1]));
                m[e] = mn;
            }
            if (!__all_sync(0xffffffffu, al[0] == 1.f && al[1] == 1.f)) {  // some row's max moved
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    O[n][0] *= al[0];
                    O[n][1] *= al[0];
                    O[n][2] *= al[1];
                    O[n][3] *= al[1];
                }
            }
            // P as the A operand: the accumulator layout is the A layout (no shuffle)
            uint32_t pa[4];
            pa[0] = pack_bf16(p[0][0], p[0][1]);  // row gq,     tokens 2tq, 2tq+1
            pa[1] = pack_bf16(p[0][2], p[0][3]);  // row gq + 8, tokens 2tq, 2tq+1
            pa[2] = pack_bf16(p[1][0], p[1][1]);  // row gq,     tokens 8+2tq, 9+2tq
            pa[3] = pack_bf16(p[1][2], p[1][3]);  // row gq + 8, tokens 8+2tq, 9+2tq

            // O += P V : 8 n-tiles of 8 head-dims; V rows give B fragments through the transposing
            // load.  Slots at or past the cache end (or of a skipped page) may hold anything; their
            // value halves are zeroed in registers so that a 0 weight times garbage cannot make NaN.
#pragma unroll
            for (int nn = 0; nn < 4; ++nn) {
                const int tok = ((lane >> 3) & 1) * 8 + (lane & 7);
                const int chunk = 2 * nn + (lane >> 4);
                uint32_t vf[4];
                ldmatrix_x4_trans(vf, vb + tok * 128 + ((chunk ^ (tok & 7)) << 4));
                if (valid < kPageSize) {
                    vf[0] = keep_tokens(vf[0], 2 * tq, valid);
                    vf[1] = keep_tokens(vf[1], 8 + 2 * tq, valid);
                    vf[2] = keep_tokens(vf[2], 2 * tq, valid);
                    vf[3] = keep_tokens(vf[3], 8 + 2 * tq, valid);
                }
                mma_bf16_16816(O[2 * nn], pa, vf[0], vf[1]);
                mma_bf16_16816(O[2 * nn + 1], pa, vf[2], vf[3]);
            }

            // release the stage to the producer
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++consumed;
        }
        if (failed) break;

        // ---- end of the piece: normaliser over the quad, then this warp's rows
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int o = 1; o < 4; o <<= 1) d[e] += __shfl_xor_sync(0xffffffffu, d[e], o);
        const long long slot = cta + seg;  // partial slot of this piece
        if (!whole && tid == 0) pend[pend_n++] = seg;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int r = rr[e];
            if (r >= R) continue;
            const float inv = d[e] > 0.f ? 1.f / d[e] : 0.f;
            if (whole) {
                __nv_bfloat16* dst =
                    a.out + (((long long)cp.b * QL + r / G) * a.Hq + cp.g * G + r % G) * kHeadDim + 2 * tq;
#pragma unroll
                for (int n = 0; n < 8; ++n)
                    *reinterpret_cast<uint32_t*>(dst + 8 * n) = pack_bf16(O[n][2 * e] * inv, O[n][2 * e + 1] * inv);
            } else {
                float* dst = a.part_o + (slot * R + r) * kHeadDim + 2 * tq;
#pragma unroll
                for (int n = 0; n < 8; ++n)
                    *reinterpret_cast<float2*>(dst + 8 * n) = make_float2(O[n][2 * e] * inv, O[n][2 * e + 1] * inv);
            }
            if (tq == 0) {
                const float l2 = d[e] > 0.f ? m[e] + log2f(d[e]) : kNegInf;
                if (whole) {
                    if (a.lse) a.lse[((long long)cp.b * QL + r / G) * a.Hq + cp.g * G + r % G] = l2 * kLn2;
                } else {
                    a.part_lse[slot * R + r] = l2;
                }
            }
        }
    }

    if (tid == 0) misc[13] = pend_n;

    // ---- 5. count this share's partial pieces (at most two); merge the segments it completes
    __syncthreads();  // every partial of this CTA is written (CTA scope) ...
    if (tid < 2 && tid < misc[13]) {  // ... and the release CAS publishes them device-wide
        const int seg = pend[tid];
        const int b = seg / Hkv, g = seg - b * Hkv;
        const int n = prefix[b + 1] - prefix[b];
        long long c_first;
        int pieces;
        segment_pieces((long long)prefix[b] * Hkv + (long long)g * n, n, C, U, c_first, pieces);
        if (arrive_last(&a.counters[seg], a.epoch, pieces)) queue[atomicAdd(&misc[12], 1)] = seg;
    }
    __syncthreads();
    const int nq = misc[12];
    // (segment, row) items over quads of lanes: 8 per warp and pass
    for (int item = warp * 8 + (lane >> 2); item < nq * R; item += (W + 1) * 8) {
        const int seg = queue[item / R], r = item % R;
        const int b = seg / Hkv, g = seg - b * Hkv;
        const int n = prefix[b + 1] - prefix[b];
        long long c_first;
        int pieces;
        segment_pieces((long long)prefix[b] * Hkv + (long long)g * n, n, C, U, c_first, pieces);
        merge_row(a, b, g, r, c_first + seg, pieces, lane & 3);
    }
}

template <int W>
cudaError_t ensure_smem_attr(size_t smem) {
    static thread_local size_t set_to[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && set_to[dev] >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(verify_split_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && dev < 64) set_to[dev] = smem;
    return e;
}

template <int W>
cudaError_t occupancy(size_t smem, int* per_sm) {
    cudaError_t e = ensure_smem_attr<W>(smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, verify_split_kernel<W>, (W + 1) * 32, smem);
}

// Consumer warps for R query rows: groups of 16 rows, rounded up to a power of two.
int warps_for(int R) {
    const int n = (R + 15) / 16;
    return n <= 1 ? 1 : n <= 2 ? 2 : 4;
}

// Resident CTAs for (device, warps, shared memory), remembered so that repeated calls skip the query.
cudaError_t resident(int W, size_t smem, long long* ctas) {
    struct Entry {
        int dev, W;
        size_t smem;
        long long ctas;
    };
    static thread_local Entry cache[8] = {};
    static thread_local int next = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    for (const Entry& c : cache)
        if (c.ctas > 0 && c.dev == dev && c.W == W && c.smem == smem) {
            *ctas = c.ctas;
            return cudaSuccess;
        }
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    switch (W) {
        case 1: e = occupancy<1>(smem, &per_sm); break;
        case 2: e = occupancy<2>(smem, &per_sm); break;
        default: e = occupancy<4>(smem, &per_sm); break;
    }
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cache[next] = Entry{dev, W, smem, (long long)sms * per_sm};
    next = (next + 1) % 8;
    *ctas = (long long)sms * per_sm;
    return cudaSuccess;
}

}  // namespace

cudaError_t verify_plan(int B, int QL, int Hq, int Hkv, int num_workers, int use_tc, VerifyPlan* plan) {
    const int G = Hq / Hkv, R = QL * G;
    // mma.sync kernel: one share per resident CTA (or num_workers shares)
    const int W = warps_for(R);
    const int S = 3 * W + 1;
    const size_t smem = Layout(S, B).total;
    long long res = 0;
    cudaError_t e = resident(W, smem, &res);
    if (e != cudaSuccess) return e;
    const long long shares = num_workers > 0 ? num_workers : res;
    plan->grid = (int)shares;
    plan->warps = W;
    plan->stages = S;
    plan->smem = smem;
    // tcgen05 kernel: one share of the (request, KV head, 128-key tile) units per resident slot
    // (num_workers > 0: that many shares)
    int per_sm = 0, sms = 0, dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = verify_tc_occupancy(&per_sm)) != cudaSuccess) return e;
    const long long segs = (long long)B * Hkv;
    plan->tc_grid = num_workers > 0 ? num_workers : (long long)sms * (per_sm > 0 ? per_sm : 1);
    plan->tc = use_tc >= 0 ? use_tc != 0 : R >= kTcMinRows;
    // workspace for either kernel: partials (o, lse) per slot and row, then a counter per segment
    plan->slots = (size_t)shares + (size_t)segs;
    const size_t tc_slots = (size_t)plan->tc_grid + (size_t)segs;  // partial slot = share + segment
    if (tc_slots > plan->slots) plan->slots = tc_slots;
    size_t bytes = plan->slots * R * kHeadDim * 4;  // partial o
    bytes += plan->slots * R * 4;                   // partial lse (base 2)
    plan->counters_offset = (bytes + 255) & ~size_t(255);
    plan->ws_bytes = plan->counters_offset + (size_t)segs * sizeof(unsigned long long);
    return cudaSuccess;
}

cudaError_t verify_launch(const VerifyArgs& args, const VerifyPlan& plan, const CUtensorMap& tk, const CUtensorMap& tv,
                          cudaStream_t stream) {
    if (args.B == 0) return cudaSuccess;
    VerifyArgs a = args;
    a.min_pages_per_worker = kMinPages;
    switch (plan.warps) {
        case 1: verify_split_kernel<1><<<plan.grid, 64, plan.smem, stream>>>(tk, tv, a); break;
        case 2: verify_split_kernel<2><<<plan.grid, 96, plan.smem, stream>>>(tk, tv, a); break;
        default: verify_split_kernel<4><<<plan.grid, 160, plan.smem, stream>>>(tk, tv, a); break;
    }
    return cudaGetLastError();
}

}  // namespace sinkattn
