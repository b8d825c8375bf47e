// api.cu -- the C ABI of libsinkattn (declared in include/sinkattn.h):
// host-side validation, TMA descriptor encoding, launch, and the per-device
// error word that kernels report into instead of trapping.
#include <sinkattn.h>


#include <cmath>
#include <cstring>
#include <mutex>

#include "call_range.h"
#include "kernels.h"

namespace sinkattn {
namespace {

// One word per device (each device holds its own copy of a __device__ variable).
__device__ unsigned g_error_word = 0;
// Where sinkattn_get_error's exchange leaves the word it took (read back by the host).
__device__ unsigned g_error_taken = 0;

// Takes the error word and clears it in one atomic step, ordered on the caller's stream: a bit
// that a kernel on another stream sets afterwards stays in the word for the next read.
__global__ void take_error_kernel(unsigned* err, unsigned* taken) { *taken = atomicExch(err, 0u); }

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    unsigned* err = nullptr;    // device address of g_error_word
    unsigned* taken = nullptr;  // device address of g_error_taken
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

sinkattn_status_t device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SINKATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return SINKATTN_ERR_CUDA;
        s.err = static_cast<unsigned*>(p);
        if (cudaGetSymbolAddress(&p, g_error_taken) != cudaSuccess) return SINKATTN_ERR_CUDA;
        s.taken = static_cast<unsigned*>(p);
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return SINKATTN_ERR_CUDA;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        s.ready = true;
    }
    *out = &s;
    return SINKATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A bf16, 128-byte-swizzled tensor map of `rank` dimensions (the innermost one 64 elements of
// 128 B), encoded once per distinct (base, dims, strides, box) in each host thread: a serving loop
// calling with the same buffers every step skips the encoder after its first call.
bool encode_cached(CUtensorMap* map, int rank, const void* base, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box) {
    struct Entry {
        const void* base;
        int rank;
        cuuint64_t dims[3], strides[2];
        cuuint32_t box[3];
        CUtensorMap map;
    };
    constexpr int kEntries = 16;
    static thread_local Entry cache[kEntries];
    static thread_local int used = 0, next = 0;
    auto same = [&](const Entry& e) {
        if (e.base != base || e.rank != rank) return false;
        for (int i = 0; i < rank; ++i)
            if (e.dims[i] != dims[i] || e.box[i] != box[i]) return false;
        for (int i = 0; i < rank - 1; ++i)
            if (e.strides[i] != strides[i]) return false;
        return true;
    };
    for (int i = 0; i < used; ++i)
        if (same(cache[i])) {
            *map = cache[i].map;
            return true;
        }
    const cuuint32_t estride[3] = {1, 1, 1};
    if (g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
                 estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    Entry& e = cache[next];
    e.base = base;
    e.rank = rank;
    for (int i = 0; i < rank; ++i) {
        e.dims[i] = dims[i];
        e.box[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) e.strides[i] = strides[i];
    e.map = *map;
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return true;
}

// 3-D map over q [tokens, H, 64] whose box is 64 x box_heads heads x box_tokens tokens (the rows of
// one query-head group of several consecutive tokens).
bool encode_token_groups(CUtensorMap* map, const void* base, long long tokens, int H, unsigned box_heads,
                         unsigned box_tokens) {
    const cuuint64_t dims[3] = {64, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {128, (cuuint64_t)H * 128};
    const cuuint32_t box[3] = {64, box_heads, box_tokens};
    return encode_cached(map, 3, base, dims, strides, box);
}

// 2-D map over rows of 64 elements (128 B), box = box_rows x 64.
bool encode_rows(CUtensorMap* map, const void* base, unsigned long long rows, unsigned long long row_stride_bytes,
                 unsigned box_rows) {
    const cuuint64_t dims[2] = {64, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {64, box_rows};
    return encode_cached(map, 2, base, dims, strides, box);
}

// 3-D map over [T, H, 64] (token-major), box = box_rows tokens x 1 head x 64.
bool encode_thd(CUtensorMap* map, const void* base, int T, int H, unsigned box_rows) {
    const cuuint64_t dims[3] = {64, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {128, (cuuint64_t)H * 128};
    const cuuint32_t box[3] = {64, 1, box_rows};
    return encode_cached(map, 3, base, dims, strides, box);
}

sinkattn_status_t check_decode_dims(const sinkattn_decode_dims_t* d) {
    if (!d) return SINKATTN_ERR_INVALID_ARG;
    if (d->batch < 0 || d->batch > 32768 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->num_pages < 0 ||
        d->max_pages < 1 || d->num_workers < 0 || d->num_workers > (1 << 22))
        return SINKATTN_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads) return SINKATTN_ERR_INVALID_ARG;
    if (d->head_dim != kHeadDim || d->page_size != kPageSize) return SINKATTN_ERR_UNSUPPORTED;
    if (d->num_q_heads / d->num_kv_heads > 16) return SINKATTN_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit: pages * Hkv * 16 rows must fit; so must the token cap.
    if ((long long)d->num_pages * d->num_kv_heads * kPageSize >= (1ll << 31)) return SINKATTN_ERR_UNSUPPORTED;
    if ((long long)d->max_pages * kPageSize >= (1ll << 31)) return SINKATTN_ERR_UNSUPPORTED;
    return SINKATTN_OK;
}

sinkattn_status_t check_verify_dims(const sinkattn_verify_dims_t* d) {
    if (!d) return SINKATTN_ERR_INVALID_ARG;
    const sinkattn_decode_dims_t dd = {d->batch,     d->num_q_heads, d->num_kv_heads, d->head_dim,  d->page_size,
                                       d->num_pages, d->max_pages,   d->num_workers};
    const sinkattn_status_t st = check_decode_dims(&dd);
    if (st != SINKATTN_OK) return st;
    if (d->q_len < 1) return SINKATTN_ERR_INVALID_ARG;
    if (d->q_len > 16 || d->q_len * (d->num_q_heads / d->num_kv_heads) > kVerifyMaxRows) return SINKATTN_ERR_UNSUPPORTED;
    return SINKATTN_OK;
}

sinkattn_status_t check_paged_dims(const sinkattn_paged_dims_t* d, bool need_q_heads) {
    if (!d) return SINKATTN_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->total_tokens < 0 || d->max_seqlen < 0 || d->num_kv_heads <= 0 || d->num_pages < 0 ||
        d->max_pages < 1)
        return SINKATTN_ERR_INVALID_ARG;
    if (need_q_heads && (d->num_q_heads <= 0 || d->num_q_heads % d->num_kv_heads)) return SINKATTN_ERR_INVALID_ARG;
    if (need_q_heads && d->share_sms != 0 && d->share_sms != 1) return SINKATTN_ERR_INVALID_ARG;
    if (d->head_dim != kHeadDim || d->page_size != kPageSize) return SINKATTN_ERR_UNSUPPORTED;
    if (d->num_seqs > 16384 || d->max_seqlen > (1 << 20)) return SINKATTN_ERR_UNSUPPORTED;
    if ((long long)d->num_pages * d->num_kv_heads * kPageSize >= (1ll << 31)) return SINKATTN_ERR_UNSUPPORTED;
    if ((long long)d->max_pages * kPageSize >= (1ll << 31)) return SINKATTN_ERR_UNSUPPORTED;
    return SINKATTN_OK;
}

}  // namespace
}  // namespace sinkattn

using namespace sinkattn;

extern "C" {

int32_t sinkattn_version(void) { return 10000; }

const char* sinkattn_status_string(sinkattn_status_t s) {
    switch (s) {
        case SINKATTN_OK: return "ok";
        case SINKATTN_ERR_INVALID_ARG: return "invalid argument";
        case SINKATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case SINKATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case SINKATTN_ERR_BAD_PAGE: return "page id out of range";
        case SINKATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
        case SINKATTN_ERR_CUDA: return "CUDA runtime error";
        case SINKATTN_ERR_BAD_LENGTH: return "sequence length out of range";
    }
    return "unknown status";
}

size_t sinkattn_decode_workspace_size(const sinkattn_decode_dims_t* dims) {
    if (check_decode_dims(dims) != SINKATTN_OK) return 0;
    DecodePlan plan;
    if (decode_plan(dims->batch, dims->num_q_heads, dims->num_kv_heads, dims->num_workers, &plan) != cudaSuccess)
        return 0;
    return plan.ws_bytes;
}

sinkattn_status_t sinkattn_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                  const int32_t* kv_lens, const float* sinks, float scale, void* out, float* lse,
                                  const sinkattn_decode_dims_t* dims, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    CallRange range("sinkattn_decode");
    sinkattn_status_t st = check_decode_dims(dims);
    if (st != SINKATTN_OK) return st;
    if (dims->batch == 0) return SINKATTN_OK;
    if (!q || !page_table || !kv_lens || !sinks || !out) return SINKATTN_ERR_INVALID_ARG;
    if (dims->num_pages > 0 && (!k_pages || !v_pages)) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(page_table, 4) || !aligned(kv_lens, 4) || !aligned(sinks, 4) || (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return SINKATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    DecodePlan plan;
    if (decode_plan(dims->batch, dims->num_q_heads, dims->num_kv_heads, dims->num_workers, &plan) != cudaSuccess)
        return SINKATTN_ERR_CUDA;
    if (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)) return SINKATTN_ERR_WORKSPACE;

    const int Hkv = dims->num_kv_heads, G = dims->num_q_heads / Hkv;
    // With an empty pool every page id is out of range, so no copy is ever issued
    // and the (zeroed) maps are never read.
    CUtensorMap tk, tv;
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    const unsigned long long rows = (unsigned long long)dims->num_pages * Hkv * kPageSize;
    if (rows > 0 &&
        (!encode_rows(&tk, k_pages, rows, 128, kPageSize) || !encode_rows(&tv, v_pages, rows, 128, kPageSize)))
        return SINKATTN_ERR_INVALID_ARG;

    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.page_table = page_table;
    a.kv_lens = kv_lens;
    a.sinks = sinks;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = a.part_o + plan.slots * G * kHeadDim;
    a.merge_list = reinterpret_cast<int2*>(ws + plan.merge_list_offset);
    a.err = ds->err;
    a.B = dims->batch;
    a.Hq = dims->num_q_heads;
    a.Hkv = Hkv;
    a.G = G;
    a.num_pages = dims->num_pages;
    a.max_pages = dims->max_pages;
    a.workers = plan.workers;
    a.min_pages_per_worker = plan.min_pages;
    a.fixed_workers = dims->num_workers > 0 ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    // One share (a fixed single worker, or an automatic split whose largest possible work,
    // every request at max_pages, stays under the minimum share) cuts no segment.
    const long long max_units = (long long)dims->batch * Hkv * dims->max_pages;
    const bool may_split = plan.workers > 1 && (a.fixed_workers || max_units > plan.min_pages);
    return decode_launch(a, plan, tk, tv, may_split, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SINKATTN_OK
               : SINKATTN_ERR_CUDA;
}

size_t sinkattn_verify_workspace_size(const sinkattn_verify_dims_t* dims) {
    if (check_verify_dims(dims) != SINKATTN_OK) return 0;
    VerifyPlan plan;
    if (verify_plan(dims->batch, dims->q_len, dims->num_q_heads, dims->num_kv_heads, dims->num_workers, &plan) !=
        cudaSuccess)
        return 0;
    return plan.ws_bytes;
}

namespace sinkattn {
namespace {
sinkattn_status_t verify_common(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                const int32_t* kv_lens, const uint64_t* tree_mask, const float* sinks, float scale,
                                void* out, float* lse, const sinkattn_verify_dims_t* dims, void* workspace,
                                size_t workspace_bytes, void* stream);
}  // namespace
}  // namespace sinkattn

sinkattn_status_t sinkattn_verify(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                  const int32_t* kv_lens, const float* sinks, float scale, void* out, float* lse,
                                  const sinkattn_verify_dims_t* dims, void* workspace, size_t workspace_bytes,
                                  void* stream) {
    CallRange range("sinkattn_verify");
    return verify_common(q, k_pages, v_pages, page_table, kv_lens, nullptr, sinks, scale, out, lse, dims, workspace,
                         workspace_bytes, stream);
}

sinkattn_status_t sinkattn_verify_tree(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* page_table, const int32_t* kv_lens, const uint64_t* tree_mask,
                                       const float* sinks, float scale, void* out, float* lse,
                                       const sinkattn_verify_dims_t* dims, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    CallRange range("sinkattn_verify_tree");
    if (!tree_mask) return SINKATTN_ERR_INVALID_ARG;
    if (dims && dims->q_len > 64) return SINKATTN_ERR_UNSUPPORTED;
    return verify_common(q, k_pages, v_pages, page_table, kv_lens, tree_mask, sinks, scale, out, lse, dims, workspace,
                         workspace_bytes, stream);
}

namespace sinkattn {
namespace {
sinkattn_status_t verify_common(const void* q, const void* k_pages, const void* v_pages, const int32_t* page_table,
                                const int32_t* kv_lens, const uint64_t* tree_mask, const float* sinks, float scale,
                                void* out, float* lse, const sinkattn_verify_dims_t* dims, void* workspace,
                                size_t workspace_bytes, void* stream) {
    sinkattn_status_t st = check_verify_dims(dims);
    if (st != SINKATTN_OK) return st;
    if (dims->batch == 0) return SINKATTN_OK;
    if (!q || !page_table || !kv_lens || !sinks || !out) return SINKATTN_ERR_INVALID_ARG;
    if (dims->num_pages > 0 && (!k_pages || !v_pages)) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(page_table, 4) || !aligned(kv_lens, 4) || !aligned(sinks, 4) || (lse && !aligned(lse, 4)) ||
        (tree_mask && !aligned(tree_mask, 8)))
        return SINKATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return SINKATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    VerifyPlan plan;
    if (verify_plan(dims->batch, dims->q_len, dims->num_q_heads, dims->num_kv_heads, dims->num_workers, &plan) !=
        cudaSuccess)
        return SINKATTN_ERR_CUDA;
    if (!workspace || workspace_bytes < plan.ws_bytes || !aligned(workspace, 256)) return SINKATTN_ERR_WORKSPACE;

    const int Hkv = dims->num_kv_heads, G = dims->num_q_heads / Hkv;
    CUtensorMap tk, tv;
    const unsigned long long rows = (unsigned long long)dims->num_pages * Hkv * kPageSize;
    if (rows > 0 &&
        (!encode_rows(&tk, k_pages, rows, 128, kPageSize) || !encode_rows(&tv, v_pages, rows, 128, kPageSize)))
        return SINKATTN_ERR_INVALID_ARG;

    VerifyArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.page_table = page_table;
    a.kv_lens = kv_lens;
    a.sinks = sinks;
    a.tree_mask = reinterpret_cast<const unsigned long long*>(tree_mask);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = a.part_o + plan.slots * (size_t)dims->q_len * G * kHeadDim;
    a.merge_list = reinterpret_cast<int2*>(ws + plan.merge_list_offset);
    a.err = ds->err;
    a.B = dims->batch;
    a.QL = dims->q_len;
    a.Hq = dims->num_q_heads;
    a.Hkv = Hkv;
    a.G = G;
    a.R = dims->q_len * G;
    a.num_pages = dims->num_pages;
    a.max_pages = dims->max_pages;
    a.fixed_workers = dims->num_workers > 0 ? 1 : 0;
    a.tc_grid = plan.tc_grid;
    a.scale_log2 = scale * 1.4426950408889634f;
    // An empty pool has no page to copy (and no memory for a tensor map to describe): every
    // cached token is absent, so every row is the sink's alone.
    if (rows == 0)
        return verify_empty_pool_launch(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINKATTN_OK
                                                                                           : SINKATTN_ERR_CUDA;
    CUtensorMap tq;
    if (!encode_token_groups(&tq, q, (long long)dims->batch * dims->q_len, dims->num_q_heads, (unsigned)G,
                             (unsigned)dims->q_len))
        return SINKATTN_ERR_INVALID_ARG;
    // one share (a fixed single worker, or an automatic split whose largest possible work stays
    // under the minimum share) cuts no segment
    const long long max_tiles = (long long)dims->batch * Hkv * (((long long)dims->max_pages * kPageSize + 127) / 128);
    const bool may_split = plan.tc_grid > 1 && (a.fixed_workers || max_tiles > kVerifyMinTiles);
    const cudaError_t e = verify_tc_launch(a, tq, tk, tv, may_split, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}
}  // namespace
}  // namespace sinkattn

sinkattn_status_t sinkattn_kv_append(const void* k, const void* v, const int32_t* cu_seqlens, const int32_t* start_pos,
                                     const int32_t* page_table, void* k_pages, void* v_pages,
                                     const sinkattn_paged_dims_t* dims, void* stream) {
    CallRange range("sinkattn_kv_append");
    sinkattn_status_t st = check_paged_dims(dims, false);
    if (st != SINKATTN_OK) return st;
    if (dims->num_seqs == 0 || dims->total_tokens == 0) return SINKATTN_OK;
    if (!k || !v || !cu_seqlens || !start_pos || !page_table || !k_pages || !v_pages) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        !aligned(cu_seqlens, 4) || !aligned(start_pos, 4) || !aligned(page_table, 4))
        return SINKATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    AppendArgs a;
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.cu_seqlens = cu_seqlens;
    a.start_pos = start_pos;
    a.page_table = page_table;
    a.k_pages = static_cast<__nv_bfloat16*>(k_pages);
    a.v_pages = static_cast<__nv_bfloat16*>(v_pages);
    a.err = ds->err;
    a.N = dims->num_seqs;
    a.T = dims->total_tokens;
    a.Hkv = dims->num_kv_heads;
    a.num_pages = dims->num_pages;
    a.max_pages = dims->max_pages;
    return kv_append_launch(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                                         const int32_t* page_table, const int32_t* cu_seqlens, const int32_t* start_pos,
                                         const float* sinks, float scale, void* out, float* lse,
                                         const sinkattn_paged_dims_t* dims, void* stream) {
    CallRange range("sinkattn_prefill_paged");
    sinkattn_status_t st = check_paged_dims(dims, true);
    if (st != SINKATTN_OK) return st;
    const sinkattn_paged_dims_t& d = *dims;
    if (d.num_seqs == 0 || d.total_tokens == 0 || d.max_seqlen == 0) return SINKATTN_OK;
    if (!q || !page_table || !cu_seqlens || !start_pos || !sinks || !out) return SINKATTN_ERR_INVALID_ARG;
    if (d.num_pages > 0 && (!k_pages || !v_pages)) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(page_table, 4) || !aligned(cu_seqlens, 4) || !aligned(start_pos, 4) || !aligned(sinks, 4) ||
        (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return SINKATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    CUtensorMap tq, tk, tv;
    std::memset(&tk, 0, sizeof tk);
    std::memset(&tv, 0, sizeof tv);
    if (!encode_thd(&tq, q, d.total_tokens, d.num_q_heads, 128)) return SINKATTN_ERR_INVALID_ARG;
    // With an empty pool every page reads as out of range (zero-filled copies from a map over one
    // row would still need a pool), so an empty pool is only accepted without cached tokens.
    const unsigned long long rows = (unsigned long long)d.num_pages * d.num_kv_heads * kPageSize;
    if (rows == 0) return SINKATTN_ERR_INVALID_ARG;
    if (!encode_rows(&tk, k_pages, rows, 128, kPageSize) || !encode_rows(&tv, v_pages, rows, 128, kPageSize))
        return SINKATTN_ERR_INVALID_ARG;
    PrefillArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k_pages);
    a.v = static_cast<const __nv_bfloat16*>(v_pages);
    a.cu_seqlens = cu_seqlens;
    a.sinks = sinks;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.err = ds->err;
    a.N = d.num_seqs;
    a.T = d.total_tokens;
    a.max_seqlen = d.max_seqlen;
    a.Hq = d.num_q_heads;
    a.Hkv = d.num_kv_heads;
    a.G = d.num_q_heads / d.num_kv_heads;
    a.causal = 1;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.page_table = page_table;
    a.start_pos = start_pos;
    a.num_pages = d.num_pages;
    a.max_pages = d.max_pages;
    // the two-head kernel for an even query-head group (unless the caller shares the SMs)
    const bool two_head = a.G % 2 == 0 && !d.share_sms;
    const cudaError_t e = two_head ? prefill_pp_paged_launch(a, tq, tk, tv, static_cast<cudaStream_t>(stream))
                                   : prefill_paged_launch(a, tq, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_qkv_prologue(const void* qkv, const void* bias, const int32_t* cu_seqlens,
                                        const int32_t* start_pos, const int32_t* page_table, const sinkattn_rope_t* rope,
                                        void* q_out, void* k_pages, void* v_pages, const sinkattn_paged_dims_t* dims,
                                        void* stream) {
    CallRange range("sinkattn_qkv_prologue");
    sinkattn_status_t st = check_paged_dims(dims, true);
    if (st != SINKATTN_OK) return st;
    if (!rope) return SINKATTN_ERR_INVALID_ARG;
    const sinkattn_rope_t& r = *rope;
    if (!(r.theta > 1.f) || !(r.factor >= 1.f) || r.original_max_position <= 0 || !(r.beta_slow > 0.f) ||
        !(r.beta_fast > r.beta_slow) || !(r.attn_factor >= 0.f))
        return SINKATTN_ERR_INVALID_ARG;
    const sinkattn_paged_dims_t& d = *dims;
    if (d.num_seqs == 0 || d.total_tokens == 0) return SINKATTN_OK;
    if (!qkv || !cu_seqlens || !start_pos || !page_table || !q_out || !k_pages || !v_pages)
        return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(qkv, 16) || (bias && !aligned(bias, 16)) || !aligned(q_out, 16) || !aligned(k_pages, 16) ||
        !aligned(v_pages, 16) || !aligned(cu_seqlens, 4) || !aligned(start_pos, 4) || !aligned(page_table, 4))
        return SINKATTN_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    PrologueArgs a;
    a.qkv = static_cast<const __nv_bfloat16*>(qkv);
    a.bias = static_cast<const __nv_bfloat16*>(bias);
    a.cu_seqlens = cu_seqlens;
    a.start_pos = start_pos;
    a.page_table = page_table;
    a.q_out = static_cast<__nv_bfloat16*>(q_out);
    a.k_pages = static_cast<__nv_bfloat16*>(k_pages);
    a.v_pages = static_cast<__nv_bfloat16*>(v_pages);
    a.err = ds->err;
    a.N = d.num_seqs;
    a.T = d.total_tokens;
    a.Hq = d.num_q_heads;
    a.Hkv = d.num_kv_heads;
    a.num_pages = d.num_pages;
    a.max_pages = d.max_pages;
    a.interleaved = r.interleaved ? 1 : 0;
    // YaRN: pairs that turn often over the original context keep their frequency, slow ones are
    // stretched by the factor, with a linear ramp in the number of turns between.
    const double s = r.factor, pi = 3.14159265358979323846;
    for (int i = 0; i < kHeadDim / 2; ++i) {
        const double th = std::pow((double)r.theta, -2.0 * i / kHeadDim);
        const double turns = (double)r.original_max_position * th / (2.0 * pi);
        double gamma = (turns - r.beta_slow) / ((double)r.beta_fast - r.beta_slow);
        gamma = gamma < 0.0 ? 0.0 : (gamma > 1.0 ? 1.0 : gamma);
        a.inv_freq[i] = (1.0 - gamma) * th / s + gamma * th;
    }
    a.mscale = r.attn_factor > 0.f ? r.attn_factor : (s > 1.0 ? (float)(0.1 * std::log(s) + 1.0) : 1.f);
    return qkv_prologue_launch(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_prefill(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                                   const float* sinks, float scale, int32_t causal, void* out, float* lse,
                                   const sinkattn_prefill_dims_t* dims, void* stream) {
    CallRange range("sinkattn_prefill");
    if (!dims) return SINKATTN_ERR_INVALID_ARG;
    const sinkattn_prefill_dims_t& d = *dims;
    if (d.num_seqs < 0 || d.total_tokens < 0 || d.max_seqlen < 0 || d.num_q_heads <= 0 || d.num_kv_heads <= 0 ||
        d.num_q_heads % d.num_kv_heads)
        return SINKATTN_ERR_INVALID_ARG;
    if (d.head_dim != kHeadDim) return SINKATTN_ERR_UNSUPPORTED;
    if (d.share_sms != 0 && d.share_sms != 1) return SINKATTN_ERR_INVALID_ARG;
    if (d.num_seqs > 16384 || d.max_seqlen > (1 << 20)) return SINKATTN_ERR_UNSUPPORTED;
    if (d.num_seqs == 0 || d.total_tokens == 0 || d.max_seqlen == 0) return SINKATTN_OK;
    if (!q || !k || !v || !cu_seqlens || !sinks || !out) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(cu_seqlens, 4) ||
        !aligned(sinks, 4) || (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    if (!(scale == scale)) return SINKATTN_ERR_INVALID_ARG;
    sinkattn_status_t st;
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != SINKATTN_OK) return st;
    PrefillArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.cu_seqlens = cu_seqlens;
    a.sinks = sinks;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.err = ds->err;
    a.N = d.num_seqs;
    a.T = d.total_tokens;
    a.max_seqlen = d.max_seqlen;
    a.Hq = d.num_q_heads;
    a.Hkv = d.num_kv_heads;
    a.G = d.num_q_heads / d.num_kv_heads;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.page_table = nullptr;
    a.start_pos = nullptr;
    a.num_pages = a.max_pages = 0;
    CUtensorMap tq, tk, tv;
    if (!encode_thd(&tq, q, d.total_tokens, d.num_q_heads, 128) ||
        !encode_thd(&tk, k, d.total_tokens, d.num_kv_heads, 128) ||
        !encode_thd(&tv, v, d.total_tokens, d.num_kv_heads, 128))
        return SINKATTN_ERR_INVALID_ARG;
    // the two-head kernel for an even query-head group (unless the caller shares the SMs), else
    // the one-head kernel
    const cudaError_t e = (a.G % 2 == 0 && !d.share_sms)
                              ? prefill_pp_launch(a, tq, tk, tv, static_cast<cudaStream_t>(stream))
                              : prefill_tc_launch(a, tq, tk, tv, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_merge(const float* partial_o, const float* partial_lse, const float* sinks, void* out,
                                 float* lse, const sinkattn_merge_dims_t* dims, void* stream) {
    CallRange range("sinkattn_merge");
    if (!dims) return SINKATTN_ERR_INVALID_ARG;
    if (dims->num_splits < 0 || dims->num_rows < 0 || dims->num_heads <= 0) return SINKATTN_ERR_INVALID_ARG;
    if (dims->head_dim != kHeadDim) return SINKATTN_ERR_UNSUPPORTED;
    if (dims->num_rows == 0) return SINKATTN_OK;
    if (!out || (dims->num_splits > 0 && (!partial_o || !partial_lse))) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(partial_o, 8) || !aligned(partial_lse, 4) || (sinks && !aligned(sinks, 4)) ||
        (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    MergeArgs a;
    a.part_o = partial_o;
    a.part_lse = partial_lse;
    a.sinks = sinks;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.S = dims->num_splits;
    a.R = dims->num_rows;
    a.H = dims->num_heads;
    return merge_launch(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINKATTN_OK : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_selftest_wait_timeout(void* stream) {
    DeviceState* ds = nullptr;
    sinkattn_status_t st = device_state(&ds);
    if (st != SINKATTN_OK) return st;
    return wait_timeout_selftest_launch(ds->err, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SINKATTN_OK
                                                                                                  : SINKATTN_ERR_CUDA;
}

sinkattn_status_t sinkattn_get_error(void* stream) {
    CallRange range("sinkattn_get_error");
    DeviceState* ds = nullptr;
    sinkattn_status_t st = device_state(&ds);
    if (st != SINKATTN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one reader at a time per process: the exchange's destination word is shared
    static std::mutex take_mu;
    std::lock_guard<std::mutex> lock(take_mu);
    unsigned word = 0;
    take_error_kernel<<<1, 1, 0, s>>>(ds->err, ds->taken);
    if (cudaGetLastError() != cudaSuccess) return SINKATTN_ERR_CUDA;
    if (cudaMemcpyAsync(&word, ds->taken, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SINKATTN_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SINKATTN_ERR_CUDA;
    for (int code = 1; code < 32; ++code)
        if (word & (1u << code)) return static_cast<sinkattn_status_t>(code);
    return SINKATTN_OK;
}

}  // extern "C"
