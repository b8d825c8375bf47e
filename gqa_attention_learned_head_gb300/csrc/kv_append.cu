// kv_append.cu -- writes the K and V of new tokens into their requests' pages.
//
// Source: "Accelerating Sonar through speculation" (Perplexity), section
// "Inference with speculative decoding": before a batch runs, slots for the
// next tokens are allocated in the per-request KV pages; the model then writes
// the new tokens' keys and values there and attends over the pages.  New token
// i of sequence n goes to cache position start_pos[n] + i: page
// page_table[n][pos / 16], slot pos % 16.
//
// HBM-bound scatter: one warp per new token; its lanes move the token's
// Hkv x 64 bf16 keys and values in 16-byte pieces (a (page, KV head, slot) row
// of 128 B is contiguous in the pool).  Page ids outside the pool and
// positions past the page-table row are skipped and flagged.
#include "args_paged.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) kv_append_kernel(const AppendArgs a) {
    const int lane = threadIdx.x & 31;
    // a packing that is not 0 <= cu_seqlens[n] <= cu_seqlens[n+1] <= T is reported (one grid-stride pass)
    for (long long n = (long long)blockIdx.x * blockDim.x + threadIdx.x; n < a.N; n += (long long)gridDim.x * blockDim.x) {
        const int c0 = __ldg(&a.cu_seqlens[n]), c1 = __ldg(&a.cu_seqlens[n + 1]);
        if (c0 < 0 || c1 < c0 || c1 > a.T) atomicOr(a.err, kErrBadLength);
    }
    const long long t = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (t >= a.T) return;
    // sequence holding token t: largest n with cu_seqlens[n] <= t (all lanes, same addresses)
    int lo = 0, hi = a.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&a.cu_seqlens[mid]) <= t) lo = mid;
        else hi = mid - 1;
    }
    const int n = lo;
    // with a corrupted packing the search can land on a sequence that does not hold t: skip it
    if (t < __ldg(&a.cu_seqlens[n]) || t >= __ldg(&a.cu_seqlens[n + 1])) {
        if (lane == 0) atomicOr(a.err, kErrBadLength);
        return;
    }
    const long long pos = (long long)__ldg(&a.start_pos[n]) + (t - __ldg(&a.cu_seqlens[n]));
    if (pos < 0 || pos >= (long long)a.max_pages * kPageSize) {
        if (lane == 0) atomicOr(a.err, kErrBadLength);
        return;
    }
    const int page = __ldg(&a.page_table[(long long)n * a.max_pages + pos / kPageSize]);
    if (page < 0 || page >= a.num_pages) {
        if (lane == 0) atomicOr(a.err, kErrBadPage);
        return;
    }
    const int slot = (int)(pos % kPageSize);
    const int chunks = a.Hkv * (kHeadDim / 8);  // 16-byte pieces of one token's K (or V)
    const uint4* ks = reinterpret_cast<const uint4*>(a.k + t * a.Hkv * kHeadDim);
    const uint4* vs = reinterpret_cast<const uint4*>(a.v + t * a.Hkv * kHeadDim);
    for (int c = lane; c < chunks; c += 32) {
        const int g = c >> 3, part = c & 7;
        const long long row = ((long long)page * a.Hkv + g) * kPageSize + slot;
        const uint4 kx = __ldg(ks + c), vx = __ldg(vs + c);
        reinterpret_cast<uint4*>(a.k_pages + row * kHeadDim)[part] = kx;
        reinterpret_cast<uint4*>(a.v_pages + row * kHeadDim)[part] = vx;
    }
    // this warp's stores are issued: a prefill launched behind this kernel as a programmatic dependent may
    // start its CTAs once every CTA gets here or exits (they wait for this grid to complete before reading)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace

cudaError_t kv_append_launch(const AppendArgs& a, cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const long long blocks = (a.T + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    kv_append_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
