// decode_noalloc.cu -- sinkattn_decode_noalloc: the paged split-KV decode for
// callers that cannot allocate device memory.
//
// sinkattn_decode needs a caller-provided workspace for its split-KV partial
// results.  Some callers have no way to provide one: a framework that has
// already reserved the whole device for its own memory pool (a cudaMalloc then
// fails even though the pool has room), a plugin interface that hands the
// operator only its input and output buffers, or a latency-critical serving
// loop that must not call cudaMalloc / cudaFree because those calls can
// synchronise the device and stall every other stream.  This entry point runs
// the same decode kernels with a fixed scratch area that belongs to the
// library: a file-scope __device__ array, which the CUDA driver places in
// device memory when the library's code is loaded onto a device, and which
// every such device keeps until the process exits.
//
// Properties a caller must know:
//   * Size limit: SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB).  A problem
//     whose workspace (sinkattn_decode_workspace_size) is larger is rejected
//     with SINKATTN_ERR_WORKSPACE before anything is launched.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); later calls reuse it.
//     Make that first call before any stream capture begins.
//   * All calls share the one array and it keeps whatever the last call left
//     in it.  Nothing in it has to start at zero: each call writes every
//     scratch value before reading it.  Calls whose kernels may run at the
//     same time on the GPU (different streams, no ordering between them) race
//     on the array and give wrong results; order them on one stream or with
//     events.
//   * No cudaMalloc, cudaFree or allocating library routine is called.
#include <sinkattn.h>

#include "call_range.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr int kMaxDevices = 64;

// The scratch area itself; host code must never use this symbol as an address.
static __device__ __align__(256) unsigned char g_decode_scratch[SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once per device).
sinkattn_status_t scratch_address(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SINKATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return SINKATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return SINKATTN_OK;
}

}  // namespace

extern "C" sinkattn_status_t sinkattn_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                                     const int32_t* page_table, const int32_t* kv_lens,
                                                     const float* sinks, float scale, void* out, float* lse,
                                                     const sinkattn_decode_dims_t* dims, void* stream) {
    sinkattn::CallRange range("sinkattn_decode_noalloc");
    const size_t need = sinkattn_decode_workspace_size(dims);
    if (need == 0)  // invalid sizes: let the regular entry point report which check failed
        return sinkattn_decode(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, out, lse, dims, nullptr, 0,
                               stream);
    if (need > SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES) return SINKATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    const sinkattn_status_t st = scratch_address(&scratch);
    if (st != SINKATTN_OK) return st;
    return sinkattn_decode(q, k_pages, v_pages, page_table, kv_lens, sinks, scale, out, lse, dims, scratch,
                           SINKATTN_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
