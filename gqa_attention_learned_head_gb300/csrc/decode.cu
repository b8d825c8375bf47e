// decode.cu -- paged split-KV decode with a per-head learned sink.
//
// Source of the method: "GPT-OSS on day 0" (Perplexity), section "Kernels for
// GPT-OSS / Sink Attention": attention is parallelised over independent heads
// and along the KV length; the softmax runs online with a running max m and
// scale d, and seeding m from the head's sink makes the sink count in the
// normaliser -- in the first block along the sequence only.  Pages come from a
// per-request page table ("Accelerating Sonar through speculation", section
// "Inference with speculative decoding": KV pages allocated per request, page
// metadata copied to the GPU).
//
// GB300 design (not the pages' FlashInfer template):
//  * Work = the flattened list of (request b, KV head g, page) units.  Every
//    CTA recomputes the per-request page prefix sum from kv_lens in shared
//    memory, so the split needs no host-side knowledge of the lengths (no
//    host sync; graph-capturable).  Worker warp w takes the contiguous share
//    [w*U/W, (w+1)*U/W) of the U units: the load is balanced to one page.
//  * A share that covers a whole (b, g) segment writes the final output;
//    otherwise each piece writes an fp32 partial (o_c, lse_c) and
//    merge_pieces_kernel combines them.  Only the piece holding page 0 is
//    seeded with the sink, so the sink is counted exactly once.
//  * Each warp streams its pages through a private ring of kStages shared-
//    memory stages.  One stage = the K and V slices of one (page, KV head):
//    2 x 2 KiB, loaded by two TMA tensor copies with 128-byte swizzle (so the
//    ldmatrix reads below are bank-conflict free) and tracked by one mbarrier.
//  * All G <= 8 query heads of the group share one pass over K/V.  Scores are
//    computed transposed, S^T[16 tokens x 8 heads] = K * Q^T, with
//    mma.m16n8k16 (no padding: M = a page, N = the group); the row max per
//    head is a 3-step shuffle; P^T is re-laid out for the next MMA with
//    movmatrix; O^T[64 x 8] += V^T * P^T.  Everything stays in registers.
#include "kernels.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarps = 4;             // worker warps per CTA
constexpr int kStages = 4;            // ring depth per warp
constexpr int kSliceBytes = kPageSize * kHeadDim * 2;  // 2048: one (page, KV head) of K or V
constexpr int kStageBytes = 2 * kSliceBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

__host__ __device__ constexpr size_t split_smem_fixed() {
    return 1024 /* alignment slack */ + size_t(kWarps) * kStages * (kStageBytes + 8 + 4) + kWarps * 4;
}

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// Position of unit x in the flattened (request, KV head, page) order.
struct Cursor {
    int b, g, page, n;  // request, KV head, page within the request, pages of the request
};

__device__ __forceinline__ Cursor locate(const int* prefix, int B, int Hkv, long long x) {
    int lo = 0, hi = B - 1;  // smallest b with prefix[b+1]*Hkv > x
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if ((long long)prefix[mid + 1] * Hkv > x) hi = mid;
        else lo = mid + 1;
    }
    Cursor c;
    c.b = lo;
    c.n = prefix[lo + 1] - prefix[lo];
    long long off = x - (long long)prefix[lo] * Hkv;
    c.g = (int)(off / c.n);
    c.page = (int)(off - (long long)c.g * c.n);
    return c;
}

__device__ __forceinline__ void advance(Cursor& c, const int* prefix, int B, int Hkv) {
    if (++c.page < c.n) return;
    c.page = 0;
    if (++c.g < Hkv) return;
    c.g = 0;
    do { ++c.b; } while (c.b < B && prefix[c.b + 1] == prefix[c.b]);
    if (c.b < B) c.n = prefix[c.b + 1] - prefix[c.b];
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Worker count actually used for U units (identical in every CTA).
__device__ __forceinline__ long long effective_workers(const DecodeArgs& a, long long U) {
    long long w = a.workers;
    if (!a.fixed_workers) {
        long long want = (U + a.min_pages_per_worker - 1) / a.min_pages_per_worker;
        if (want < w) w = want;
    }
    if (w > U) w = U;
    return w < 1 ? 1 : w;
}

template <int NT>  // NT = ceil(G / 8) groups of 8 query heads
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                   const __grid_constant__ CUtensorMap tmap_v,
                                                                   const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + kWarps * kStages * kStageBytes);
    int* bad = reinterpret_cast<int*>(bars + kWarps * kStages);
    int* wtot = bad + kWarps * kStages;
    int* prefix = wtot + kWarps;  // [B + 1] exclusive prefix of pages per request

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.B, Hkv = a.Hkv, G = a.G, cap = a.max_pages * kPageSize;

    // ---- 1. pages per request -> exclusive prefix sum (every CTA, in shared memory)
    int running = 0;
    for (int base = 0; base < B; base += kWarps * 32) {
        int b = base + tid, n = 0;
        if (b < B) {
            int L = a.kv_lens[b];
            if ((L < 0 || L > cap) && blockIdx.x == 0) atomicOr(a.err, kErrBadLength);
            n = (clamp_len(L, cap) + kPageSize - 1) / kPageSize;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        int woff = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            int v = wtot[w];
            woff += (w < warp) ? v : 0;
            tot += v;
        }
        if (b < B) prefix[b] = running + woff + incl - n;
        running += tot;
        __syncthreads();
    }
    if (tid == 0) prefix[B] = running;
    __syncthreads();

    const long long U = (long long)running * Hkv;
    if (U == 0) return;
    const long long W = effective_workers(a, U);
    const long long w = (long long)blockIdx.x * kWarps + warp;
    if (w >= W) return;
    const long long x0 = w * U / W, x1 = (w + 1) * U / W;
    const int npg = (int)(x1 - x0);

    uint8_t* my_ring = ring + warp * kStages * kStageBytes;
    uint64_t* my_bars = bars + warp * kStages;
    int* my_bad = bad + warp * kStages;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&my_bars[s], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
    __syncwarp();

    // ---- 2. producer: lane l resolves unit (x0 + base + l) to a pool row, 32 units at a time
    int win_base = -64, win_row = -1;
    auto issue = [&](int j) {  // warp-uniform; stage j % kStages must be free
        if (j - win_base >= 32) {
            win_base = j;
            int jj = j + lane, row = -1;
            if (jj < npg) {
                Cursor c = locate(prefix, B, Hkv, x0 + jj);
                int pid = __ldg(&a.page_table[(long long)c.b * a.max_pages + c.page]);
                if (pid >= 0 && pid < a.num_pages) row = (pid * Hkv + c.g) * kPageSize;
            }
            win_row = row;
        }
        int row = __shfl_sync(0xffffffffu, win_row, j - win_base);
        if (lane == 0) {
            int s = j % kStages;
            uint8_t* dst = my_ring + s * kStageBytes;
            if (row >= 0) {
                my_bad[s] = 0;
                mbar_arrive_expect_tx(&my_bars[s], kStageBytes);
                tma_load_2d(dst, &tmap_k, 0, row, &my_bars[s]);
                tma_load_2d(dst + kSliceBytes, &tmap_v, 0, row, &my_bars[s]);
            } else {
                my_bad[s] = 1;
                atomicOr(a.err, kErrBadPage);
                mbar_arrive(&my_bars[s]);
            }
        }
    };
    for (int j = 0; j < kStages && j < npg; ++j) issue(j);

    // ---- 3. consumer
    const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
    Cursor cc = locate(prefix, B, Hkv, x0);
    uint32_t qf[NT][4][2];
    float O[4][NT][4];
    float m[NT][2], d[NT][2];
    int kv_len = 0;
    bool piece_open = false, piece_first = false;
    int stopped_at = -1;  // consumer position of a wait that gave up
    int issued = min(kStages, npg);

    for (int i = 0; i < npg; ++i) {
        if (!piece_open) {
            piece_open = true;
            piece_first = (cc.page == 0);
            kv_len = clamp_len(__ldg(&a.kv_lens[cc.b]), cap);
            const __nv_bfloat16* qb = a.q + ((long long)cc.b * a.Hq + (long long)cc.g * G) * kHeadDim;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hl = nt * 8 + gq;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    qf[nt][kk][0] = hl < G ? ld_u32(qb + hl * kHeadDim + kk * 16 + 2 * tq) : 0u;
                    qf[nt][kk][1] = hl < G ? ld_u32(qb + hl * kHeadDim + kk * 16 + 8 + 2 * tq) : 0u;
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int h = nt * 8 + 2 * tq + e;
                    m[nt][e] = (piece_first && h < G) ? __ldg(&a.sinks[cc.g * G + h]) * kLog2e : kNegInf;
                    d[nt][e] = (piece_first && lane < 4) ? 1.f : 0.f;  // the sink's own e^(sink-m)=1, once per head
                }
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) O[mt][nt][e] = 0.f;
            }
        }

        const int s = i % kStages;
        const bool ok = mbar_wait(&my_bars[s], (i / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
            stopped_at = i;
            break;
        }
        const int valid = my_bad[s] ? 0 : min(kPageSize, kv_len - cc.page * kPageSize);
        uint8_t* st = my_ring + s * kStageBytes;
        if (valid < kPageSize) {
            // Rows past the cache end (or a skipped page) may hold anything; zero the
            // value rows so that 0-weight * garbage cannot produce NaN.
            uint4* vz = reinterpret_cast<uint4*>(st + kSliceBytes);
            for (int c = valid * 8 + lane; c < kPageSize * 8; c += 32) vz[c] = make_uint4(0, 0, 0, 0);
            __syncwarp();
        }
        const uint32_t kb = smem_u32(st), vb = kb + kSliceBytes;

        // S^T = K Q^T : 16 tokens x 8 heads per n-tile
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int row = ((lane >> 3) & 1) * 8 + (lane & 7);
            const int chunk = 2 * kk + (lane >> 4);
            uint32_t af[4];
            ldmatrix_x4(af, kb + row * 128 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], af, qf[nt][kk][0], qf[nt][kk][1]);
        }

        // online softmax (base 2); this thread holds tokens gq, gq+8 and heads 2tq, 2tq+1
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float sc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = gq + (e >= 2 ? 8 : 0);
                sc[e] = tok < valid ? acc[nt][e] * a.scale_log2 : kNegInf;
            }
            float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
            const bool dead0 = (mn0 == kNegInf), dead1 = (mn1 == kNegInf);
            const float al0 = dead0 ? 1.f : fast_exp2(m[nt][0] - mn0);
            const float al1 = dead1 ? 1.f : fast_exp2(m[nt][1] - mn1);
            const float p0 = dead0 ? 0.f : fast_exp2(sc[0] - mn0);
            const float p2 = dead0 ? 0.f : fast_exp2(sc[2] - mn0);
            const float p1 = dead1 ? 0.f : fast_exp2(sc[1] - mn1);
            const float p3 = dead1 ? 0.f : fast_exp2(sc[3] - mn1);
            d[nt][0] = d[nt][0] * al0 + (p0 + p2);
            d[nt][1] = d[nt][1] * al1 + (p1 + p3);
            m[nt][0] = mn0;
            m[nt][1] = mn1;
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                O[mt][nt][0] *= al0;
                O[mt][nt][1] *= al1;
                O[mt][nt][2] *= al0;
                O[mt][nt][3] *= al1;
            }
            pb[nt][0] = movmatrix_trans(pack_bf16(p0, p1));  // tokens 0..7  -> B rows k = 2tq, 2tq+1
            pb[nt][1] = movmatrix_trans(pack_bf16(p2, p3));  // tokens 8..15
        }

        // O^T += V^T P^T : 4 tiles of 16 head-dims
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int j = lane >> 3;
            const int row = (j >> 1) * 8 + (lane & 7);
            const int chunk = 2 * mt + (j & 1);
            uint32_t af[4];
            ldmatrix_x4_trans(af, vb + row * 128 + ((chunk ^ (row & 7)) << 4));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(O[mt][nt], af, pb[nt][0], pb[nt][1]);
        }

        // release the stage and refill it
        fence_proxy_async_smem();
        __syncwarp();
        if (issued < npg) issue(issued++);

        // end of a piece: normalise and write
        const bool seg_last = (cc.page == cc.n - 1);
        if (seg_last || i == npg - 1) {
            const int seg = cc.b * Hkv + cc.g;
            const bool whole = piece_first && seg_last;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float inv[2], lse2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float dt = d[nt][e];
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) dt += __shfl_xor_sync(0xffffffffu, dt, o);
                    inv[e] = dt > 0.f ? 1.f / dt : 0.f;
                    lse2[e] = dt > 0.f ? (m[nt][e] + log2f(dt)) * kLn2 : kNegInf;
                }
#pragma unroll
                for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = nt * 8 + 2 * tq + (e & 1);
                        const int dim = mt * 16 + gq + (e >= 2 ? 8 : 0);
                        if (h >= G) continue;
                        const float v = O[mt][nt][e] * inv[e & 1];
                        if (whole)
                            a.out[((long long)cc.b * a.Hq + cc.g * G + h) * kHeadDim + dim] = __float2bfloat16_rn(v);
                        else
                            a.part_o[((w + seg) * G + h) * kHeadDim + dim] = v;
                    }
                if (lane < 4) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = nt * 8 + 2 * tq + e;
                        if (h >= G) continue;
                        if (whole) {
                            if (a.lse) a.lse[(long long)cc.b * a.Hq + cc.g * G + h] = lse2[e];
                        } else {
                            a.part_lse[(w + seg) * G + h] = lse2[e];
                        }
                    }
                }
            }
            if (piece_first && lane == 0) {
                // pieces of this segment: owners of its first and last unit are consecutive workers
                const long long seg_end = (long long)prefix[cc.b] * Hkv + (long long)(cc.g + 1) * cc.n;
                const long long w_last = (seg_end * W - 1) / U;
                a.seg_meta[seg] = make_int2((int)(w + seg), (int)(w_last - w + 1));
            }
            piece_open = false;
        }
        advance(cc, prefix, B, Hkv);
    }

    if (stopped_at >= 0) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        // let copies already in flight land (bounded) before the CTA's shared memory is released
        for (int j = stopped_at; j < issued; ++j) (void)mbar_wait(&my_bars[j % kStages], (j / kStages) & 1);
    }
}

// Combines the pieces of every split (request, KV head) segment; also writes the
// rows of empty requests (all mass on the sink: out = 0, lse = sink).
__global__ void __launch_bounds__(128) merge_pieces_kernel(const DecodeArgs a) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= (long long)a.B * a.Hq) return;
    const int b = (int)(row / a.Hq), h = (int)(row - (long long)b * a.Hq);
    const int g = h / a.G, hl = h - g * a.G;
    const int L = clamp_len(__ldg(&a.kv_lens[b]), a.max_pages * kPageSize);
    __nv_bfloat162* out2 = reinterpret_cast<__nv_bfloat162*>(a.out + row * kHeadDim) + lane;
    if (L == 0) {
        *out2 = __floats2bfloat162_rn(0.f, 0.f);
        if (lane == 0 && a.lse) a.lse[row] = __ldg(&a.sinks[h]);
        return;
    }
    const int2 meta = a.seg_meta[(long long)b * a.Hkv + g];
    if (meta.y <= 1) return;
    const float* lp = a.part_lse + (long long)meta.x * a.G + hl;
    const float* op = a.part_o + ((long long)meta.x * a.G + hl) * kHeadDim + 2 * lane;
    float M = kNegInf;
    for (int c = 0; c < meta.y; ++c) M = fmaxf(M, lp[(long long)c * a.G]);
    float sum = 0.f, ox = 0.f, oy = 0.f;
    for (int c = 0; c < meta.y; ++c) {
        const float wgt = __expf(lp[(long long)c * a.G] - M);
        sum += wgt;
        const float2 v = *reinterpret_cast<const float2*>(op + (long long)c * a.G * kHeadDim);
        ox += wgt * v.x;
        oy += wgt * v.y;
    }
    const float inv = 1.f / sum;
    *out2 = __floats2bfloat162_rn(ox * inv, oy * inv);
    if (lane == 0 && a.lse) a.lse[row] = M + logf(sum);
}

template <int NT>
cudaError_t launch_split(const DecodeArgs& args, const DecodePlan& plan, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t stream) {
    decode_split_kernel<NT><<<plan.grid, kWarps * 32, plan.smem, stream>>>(tk, tv, args);
    return cudaGetLastError();
}

template <int NT>
cudaError_t ensure_smem_attr(size_t smem) {
    static thread_local size_t set_to[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && set_to[dev] >= smem) return cudaSuccess;
    e = cudaFuncSetAttribute(decode_split_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && dev < 64) set_to[dev] = smem;
    return e;
}

}  // namespace

cudaError_t decode_plan(int B, int Hq, int Hkv, int num_workers, DecodePlan* plan) {
    const int G = Hq / Hkv;
    const size_t smem = split_smem_fixed() + size_t(B + 1) * 4;
    cudaError_t e = G <= 8 ? ensure_smem_attr<1>(smem) : ensure_smem_attr<2>(smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = G <= 8 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<1>, kWarps * 32, smem)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<2>, kWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long workers = num_workers > 0 ? num_workers : (long long)sms * per_sm * kWarps;
    plan->workers = (int)workers;
    plan->grid = (int)((workers + kWarps - 1) / kWarps);
    plan->smem = smem;
    plan->slots = (size_t)workers + (size_t)B * Hkv;
    size_t bytes = plan->slots * G * kHeadDim * 4;   // partial o
    bytes += plan->slots * G * 4;                    // partial lse
    bytes = (bytes + 255) & ~size_t(255);
    bytes += (size_t)B * Hkv * sizeof(int2);         // segment table
    plan->ws_bytes = bytes;
    return cudaSuccess;
}

cudaError_t decode_launch(const DecodeArgs& args, const DecodePlan& plan, const CUtensorMap& tk,
                          const CUtensorMap& tv, cudaStream_t stream) {
    if (args.B == 0) return cudaSuccess;
    cudaError_t e = args.G <= 8 ? launch_split<1>(args, plan, tk, tv, stream) : launch_split<2>(args, plan, tk, tv, stream);
    if (e != cudaSuccess) return e;
    const long long rows = (long long)args.B * args.Hq;
    merge_pieces_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(args);
    return cudaGetLastError();
}

}  // namespace sinkattn
