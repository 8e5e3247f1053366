// Blackwell (sm_100 family, built for sm_103a) tensor-core helpers: TMA tile
// loads, tensor memory (TMEM) allocation / load / store, tcgen05.mma with
// shared-memory matrix descriptors, and commit-to-mbarrier.  Inline PTX.
//
// Shared-memory operand layout used throughout: a tile of R rows x 64 bf16
// (128 bytes per row) in the 128-byte swizzle pattern that TMA produces with
// CU_TENSOR_MAP_SWIZZLE_128B: row r starts at byte r * 128 and its 16-byte
// chunk j is stored at chunk position j ^ (r % 8).  A 128-column operand is two
// such sub-tiles back to back.  Sub-tiles start on 1024-byte boundaries.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace path {
namespace tc {

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 3-D tiled load (x innermost) completing on `bar` with transaction bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 3-D tiled store of a shared-memory box to global memory (bulk-group
// completion: commit with bulk_commit, wait with bulk_wait_read/bulk_wait).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            map),
        "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// All committed bulk stores have finished reading their shared-memory source.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// All committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Brings a 3-D box into L2 ahead of a later tiled load.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// All committed bulk stores but the N most recent groups are complete.
template <int N>
__device__ __forceinline__ void bulk_wait_all_but() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Brings `bytes` (a multiple of 16) at the 16-byte aligned global address
// `p` into L2, without waiting.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (MMA/TMA).
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ shared memory

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Async-proxy global writes (completed bulk stores) -> later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Four consecutive fp32 atomic adds in one vector reduction (16-byte aligned).
__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a),
                 "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Named barrier over n threads.  bar.sync is a warp-aligned instruction: every
// lane of the warp must execute it together, so the warp is reconverged first
// (lanes may leave a bounded wait loop at different iterations).
__device__ __forceinline__ void named_bar(int id, int n) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also ANDs `ok` across its threads, so that a wait that
// gave up in one thread makes the whole group leave together.
__device__ __forceinline__ bool group_all(int id, int n, bool ok) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

#define PATH_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                   "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])

// 32 consecutive columns of this thread's lane (warp lane quadrant
// 32 * (warp % 4)); the wait is part of the same asm statement so the
// outputs are complete when the statement ends.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : PATH_R8(0), PATH_R8(8), PATH_R8(16), PATH_R8(24)
        : "r"(addr)
        : "memory");
}

// 64 consecutive columns of this thread's lane, one load and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t addr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(addr)
        : "memory");
}

// 128 consecutive columns of this thread's lane, one load and one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t addr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(addr)
        : "memory");
}

#define PATH_W8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                   "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(addr),
        PATH_W8(0), PATH_W8(8), PATH_W8(16), PATH_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ MMA

// Shared-memory matrix descriptor (sm_100 format): start address, leading and
// stride byte offsets (16-byte units), version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16 with bf16 A/B and f32 accumulation.
// a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Byte offset of 16-byte chunk j (0..15) of row r in a 128-column bf16
// operand made of two [R][64] swizzled sub-tiles.
__device__ __forceinline__ uint32_t swz_off(int r, int j, int R) {
    return (uint32_t)((j >> 3) * R * 128 + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// D[128 x 128] (+)= A[128 x 128] * B over K = 128 in eight K = 16 steps.
// A: K-major two-sub-tile operand at a_base.  B: K-major (rows = N) when
// !b_mn, else MN-major with rows = K (each row 128 N-values as two
// sub-tiles).
__device__ __forceinline__ void gemm_128x128x128(uint32_t d_tmem, uint32_t a_base,
                                                 uint32_t b_base, bool b_mn, bool accumulate) {
    const uint32_t idesc = idesc_bf16(128, 128, false, b_mn);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_addr = a_base + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t ad = sdesc(a_addr, 16, 1024);
        uint64_t bd;
        if (!b_mn)
            bd = sdesc(b_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        else
            bd = sdesc(b_base + kk * 2048, 16384, 1024);
        mma_bf16(d_tmem, ad, bd, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Low / high 32-bit words of an SW128 descriptor for a tile at `saddr`:
// K-major (leading offset unused) or MN-major (leading offset = 16 KB, the
// distance between the two 64-column sub-tiles of a 128-row tile).  The high
// word holds the 1024-byte stride, the version and the swizzle mode.  A
// shared address is below 2^18, so adding (byte offset >> 4) to the low word
// never carries out of the 14-bit start-address field.
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, bool mn_major) {
    return ((saddr >> 4) & 0x3FFFu) | ((mn_major ? (16384u >> 4) : 1u) << 16);
}
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);

__device__ __forceinline__ void mma_bf16_lohi(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 ad, {%1, %5};\n\t"
        "mov.b64 bd, {%2, %5};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
        : "memory");
}

// gemm_128x128x128 with precomputed descriptor low words; A_MN / B_MN select
// MN-major operands (rows = K; each row holds 128 M or N values as two
// 64-column sub-tiles 16 KB apart), else K-major.
template <bool B_MN, bool A_MN>
__device__ __forceinline__ void gemm128_lo2(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                            bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16(128, 128, A_MN, B_MN);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2);
        const uint32_t aoff = A_MN ? (uint32_t)(kk * 128) : koff;
        const uint32_t boff = B_MN ? (uint32_t)(kk * 128) : koff;
        mma_bf16_lohi(d_tmem, a_lo + aoff, b_lo + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// gemm_128x128x128 with precomputed descriptor low words (a_lo K-major;
// b_lo K-major or MN-major per B_MN).
template <bool B_MN>
__device__ __forceinline__ void gemm128_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                           bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16(128, 128, false, B_MN);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2);
        const uint32_t boff = B_MN ? (uint32_t)(kk * 128) : aoff;
        mma_bf16_lohi(d_tmem, a_lo + aoff, b_lo + boff, idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// D (+)= A * B with A read from tensor memory at column a_tmem (lane field 0):
// row i of A in lane i, 16-bit elements packed two per 32-bit column (even k
// in the low half), K = 16 per instruction = 8 columns.  B as in mma_bf16_lohi.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 bd, {%2, %5};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kDescHi)
        : "memory");
}

// gemm128_lo with the 128 x 128 bf16 A operand in tensor memory (64 columns
// from a_tmem, packed as in mma_bf16_ta).
template <bool B_MN>
__device__ __forceinline__ void gemm128_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                           bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16(128, 128, false, B_MN);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t boff = B_MN ? (uint32_t)(kk * 128) : (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2);
        mma_bf16_ta(d_tmem, a_tmem + (uint32_t)(kk * 8), b_lo + boff, idesc,
                    (accumulate || kk > 0) ? 1u : 0u);
    }
}

}  // namespace tc
}  // namespace path
