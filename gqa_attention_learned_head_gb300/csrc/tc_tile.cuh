// tc_tile.cuh -- pieces shared by the tcgen05 attention kernels (the prefills and the
// verification): the two instruction descriptors of a 128-row attention tile, the shared-memory
// descriptor of a 128-byte-swizzled operand, 32-column tensor-memory loads and stores, and the
// bounded warp-wide mbarrier wait.
#pragma once

#include "ptx.cuh"

namespace sinkattn {
namespace tc {

constexpr int kBM = 128, kBN = 128;         // query rows, keys per tile
constexpr uint32_t kTileBytes = 128 * 128;  // 128 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O / d may grow by up to 2^8 before a rescale

// Cubic for 2^f on [-1/2, 1/2], minimax in relative error (max 7.5e-5); derived by exp2_poly.py.
constexpr float kExp2C0 = 0.9999280571937561f;
constexpr float kExp2C1 = 0.6932609677314758f;
constexpr float kExp2C2 = 0.2426111251115799f;
constexpr float kExp2C3 = 0.0551716685295105f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer in the low bits

// exp2 of two values without the MUFU: 2^x = 2^round(x) * p(x - round(x)).  Arguments below -125
// (including -inf) are clamped there, giving ~2e-38 instead of 0, which no sum can notice.
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
    x.x = fmaxf(x.x, -125.f);
    x.y = fmaxf(x.y, -125.f);
    const float2 t = fadd2(x, make_float2(kRoundMagic, kRoundMagic));
    const float2 r = fadd2(t, make_float2(-kRoundMagic, -kRoundMagic));
    const float2 f = ffma2(r, make_float2(-1.f, -1.f), x);
    float2 p = ffma2(f, make_float2(kExp2C3, kExp2C3), make_float2(kExp2C2, kExp2C2));
    p = ffma2(p, f, make_float2(kExp2C1, kExp2C1));
    p = ffma2(p, f, make_float2(kExp2C0, kExp2C0));
    return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                       __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

// Instruction descriptors, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28; bit 16 = B is MN-major.
constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPV =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((64u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory matrix descriptor for a 128-byte-swizzled tile whose 8-row groups are 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)       // start address
           | ((uint64_t)(1024u >> 4) << 16)          // leading-dimension byte offset (unused by these shapes)
           | ((uint64_t)(1024u >> 4) << 32)          // stride-dimension byte offset: next 8-row group
           | (1ull << 46)                            // descriptor version
           | (2ull << 61);                           // 128-byte swizzle
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Paged cache: TMA row of page pg of request / sequence `seq` and KV head kvh in the 2-D map over the
// page pool (rows of 64 elements, a (page, KV head) slice = 16 rows).  A page past the cache end
// (kv_len tokens) or past the page-table row, and a page id outside the pool, give a row past the
// pool's end, which the copy fills with zeros; an id outside the pool is also reported.
template <class Args>
__device__ __forceinline__ int page_tile_row(const Args& a, int seq, int kvh, int pg, int kv_len) {
    const int oob = a.num_pages * a.Hkv * kPageSize;
    if (pg >= a.max_pages || pg * kPageSize >= kv_len) return oob;
    const int pid = __ldg(&a.page_table[(long long)seq * a.max_pages + pg]);
    if (pid < 0 || pid >= a.num_pages) {
        atomicOr(a.err, kErrBadPage);
        return oob;
    }
    return (pid * a.Hkv + kvh) * kPageSize;
}

// Every lane waits (bounded); true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

}  // namespace tc
}  // namespace sinkattn
