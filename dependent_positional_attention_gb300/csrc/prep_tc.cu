// PaTH prefill prep on tensor cores (bf16 inputs, head_dim 128, chunk 128).
//
// UT transform of each chunk's transitions (PaTH Attention summary, section
// "3. 효율적인 학습 및 추론", UT transform and boundary-adjusted rows).  For a
// chunk with rows Q, K, W (128 x 128 bf16) and coefficients beta:
//   G  = W W^T,  T = (I + strict_lower(diag(beta) G))^{-1} diag(beta)
//   Wt = T W                                   (compact chunk product factor)
//   Y  = (M_gt * K W^T) T^T
//   Qh = Q - (M_le * Q W^T) Wt                 (boundary-adjusted queries)
//   Kh = K - Y W                               (boundary-adjusted keys)
//   Sd = Q K^T - (M_le * Q W^T) Y^T            (within-chunk logits)
//   Pm = I - W^T Wt                            (chunk product H_first...H_last,
//                                               as the d x d matrix applied to
//                                               carried query rows: q <- q Pm)
// with M_le[r][s] = s <= r and M_gt[r][s] = s > r.  Nine 128 x 128 x 128
// contractions run as tcgen05 MMAs (bf16 operands, fp32 accumulation in
// TMEM); T is solved in fp32 on the CUDA cores by forward substitution, two
// threads per column.  Persistent CTAs, one chunk at a time.
//
// Phases per chunk (one thread issues TMA and MMAs; waits are bounded):
//   P1 TMA Q,K,W; MMA G->cols 0, QW->128, KW->256, QK->384
//   P2 G -> fp32 smem
//   P3 solve T (fp32 smem)
//   P4 T -> bf16 tile, -(M_le*QW) -> bf16 tile, (M_gt*KW) -> bf16 tile
//   P5 MMA Wt = T W -> cols 0, Y = (M_gt*KW) T^T -> cols 256
//   P6 Wt -> bf16 tile, Y -> bf16 tile
//   P7 MMA -(M_le*QW) Wt -> cols 128, Y W -> cols 0, += -(M_le*QW) Y^T -> cols 384,
//      W^T Wt -> cols 256   (the chunk's V is loaded meanwhile)
//   P8 Qh, Kh, Pm -> workspace
//   P9 causal softmax of the within-chunk logits (cols 384) -> P bf16 tile;
//      MMA P V -> cols 256
//   P10 the chunk's own attention output (normalised, bf16) and its log-sum-exp
//      -> workspace; the scan starts every query tile from them

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kTile = kC * kC * 2;  // bf16 128 x 128 operand tile
constexpr int kThreadsP = 256;
constexpr int kGs = kC + 1;  // fp32 G row stride (conflict-free row writes and row reads)
constexpr int kOffQ = 0, kOffK = kTile, kOffW = 2 * kTile;
constexpr int kOffR1 = 3 * kTile;            // G fp32, then T bf16 | -(M_le*QW) bf16
constexpr int kR1Bytes = 65 * 1024;          // >= 128 * 129 * 4
constexpr int kOffR2 = kOffR1 + kR1Bytes;    // T fp32, then KWm/Y bf16 | Wt bf16
constexpr int kOffBar = kOffR2 + 64 * 1024;
constexpr int kSmemP = kOffBar + 640 + 1024;
static_assert(kC * kGs * 4 <= kR1Bytes, "G staging does not fit");
static_assert(kSmemP <= 232448, "shared memory budget exceeded");
constexpr uint32_t kColA = 0, kColB = 128, kColC = 256, kColD = 384;

struct PBars {
    uint64_t tma, mma, vbar;
    uint32_t tmem_base;
    int ok;
    float beta[kC];
};
static_assert(sizeof(PBars) <= 640, "barrier block too large");

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

// 32 TMEM columns of row r (as floats), scaled per column by mask(s) into a
// swizzled bf16 tile at 16-byte chunks 4*cc .. 4*cc+3.
template <class F>
__device__ __forceinline__ void tile_store32(uint32_t tile, int r, int cc, const uint32_t (&v)[32],
                                             F f) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int s0 = cc * 32 + q * 8 + 2 * e;
            w[e] = pack2(f(s0, __uint_as_float(v[q * 8 + 2 * e])),
                         f(s0 + 1, __uint_as_float(v[q * 8 + 2 * e + 1])));
        }
        sts128(tile + tc::swz_off(r, cc * 4 + q, kC), w[0], w[1], w[2], w[3]);
    }
}

// 8 bf16 values of row r, 16-byte chunk j of a swizzled tile, as floats.
__device__ __forceinline__ void tile_load8(uint32_t tile, int r, int j, float (&f)[8]) {
    const uint4 u = lds128(tile + tc::swz_off(r, j, kC));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
        f[2 * e] = x.x;
        f[2 * e + 1] = x.y;
    }
}

// Linv = (I + A)^{-1} for A[i][k] = beta_i G[i][k] (k < i), by blocks:
// invert the eight 16 x 16 diagonal blocks by forward substitution, then
// merge sibling blocks (sizes 16, 32, 64) with X21 = -Inv(B2) A21 Inv(B1).
// G: fp32 [128][kGs] (symmetric, only k < i used).  Tf: fp32 [128][128]
// receives Linv, zero above the diagonal.  The intermediate A21 Inv(B1) of a
// merge is parked in the upper-right block of the pair (zero afterwards).
// 256 threads; each merge step gives every active thread one 4 x 4 tile.
__device__ __forceinline__ void unit_lower_inverse(const float *G, float *Tf, const float *beta,
                                                   int tid) {
    for (int e = tid; e < kC * kC / 4; e += kThreadsP)
        reinterpret_cast<float4 *>(Tf)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    if (tid < kC) {
        const int o = (tid >> 4) * 16, c = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float s = (i == c) ? 1.f : 0.f;
            const float bi = beta[o + i];
#pragma unroll
            for (int k = 0; k < i; ++k) s = fmaf(-bi * G[(o + i) * kGs + o + k], x[k], s);
            x[i] = (i < c) ? 0.f : s;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[(o + i) * kC + o + c] = x[i];
    }
    __syncthreads();
    for (int s = 16; s < kC; s *= 2) {
        const int tiles_per_pair = (s / 4) * (s / 4);
        const int ntiles = (kC / (2 * s)) * tiles_per_pair;
        const bool active = tid < ntiles;
        const int pair = tid / tiles_per_pair, t = tid % tiles_per_pair;
        const int i0 = (t / (s / 4)) * 4, j0 = (t % (s / 4)) * 4;
        const int r1 = pair * 2 * s, r2 = r1 + s;
        // P = A21 Inv(B1)  ->  Tf[r1 + i][r2 + j]
        if (active) {
            float acc[4][4] = {};
            for (int k = 0; k < s; ++k) {
                const float4 bv = *reinterpret_cast<const float4 *>(Tf + (r1 + k) * kC + r1 + j0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float av = G[(r2 + i0 + u) * kGs + r1 + k];
                    acc[u][0] = fmaf(av, bv.x, acc[u][0]);
                    acc[u][1] = fmaf(av, bv.y, acc[u][1]);
                    acc[u][2] = fmaf(av, bv.z, acc[u][2]);
                    acc[u][3] = fmaf(av, bv.w, acc[u][3]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float bi = beta[r2 + i0 + u];
                *reinterpret_cast<float4 *>(Tf + (r1 + i0 + u) * kC + r2 + j0) =
                    make_float4(bi * acc[u][0], bi * acc[u][1], bi * acc[u][2], bi * acc[u][3]);
            }
        }
        __syncthreads();
        // X21 = -Inv(B2) P  ->  Tf[r2 + i][r1 + j]
        if (active) {
            float acc[4][4] = {};
            for (int k = 0; k < s; ++k) {
                const float4 pv = *reinterpret_cast<const float4 *>(Tf + (r1 + k) * kC + r2 + j0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float av = Tf[(r2 + i0 + u) * kC + r2 + k];
                    acc[u][0] = fmaf(av, pv.x, acc[u][0]);
                    acc[u][1] = fmaf(av, pv.y, acc[u][1]);
                    acc[u][2] = fmaf(av, pv.z, acc[u][2]);
                    acc[u][3] = fmaf(av, pv.w, acc[u][3]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4 *>(Tf + (r2 + i0 + u) * kC + r1 + j0) =
                    make_float4(-acc[u][0], -acc[u][1], -acc[u][2], -acc[u][3]);
        }
        __syncthreads();
        if (active)
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4 *>(Tf + (r1 + i0 + u) * kC + r2 + j0) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kThreadsP, 1)
    prep_tc_kernel(const __grid_constant__ PrepTcMaps maps, PrepTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    PBars &bars = *reinterpret_cast<PBars *>(smem + kOffBar);
    const uint32_t sQ = smem_u32(smem + kOffQ), sK = smem_u32(smem + kOffK);
    const uint32_t sW = smem_u32(smem + kOffW);
    const uint32_t sR1 = smem_u32(smem + kOffR1), sR2 = smem_u32(smem + kOffR2);
    float *Gf = reinterpret_cast<float *>(smem + kOffR1);
    float *Tf = reinterpret_cast<float *>(smem + kOffR2);
    float *bsm = bars.beta;
    const uint32_t sT = sR1, sQm = sR1 + kTile;   // after the solve
    const uint32_t sY = sR2, sWt = sR2 + kTile;   // KWm, then Y | Wt
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;               // TMEM lane / tile row of this thread
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int total = a.N * a.BH;

    if (tid == 0) {
        mbar_init(&bars.tma, 1);
        mbar_init(&bars.mma, 1);
        mbar_init(&bars.vbar, 1);
        bars.ok = 1;
        fence_mbar_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&bars.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    uint32_t ph_tma = 0, ph_mma = 0, ph_v = 0;
    const float sl2 = a.scale * 1.4426950408889634f;

    // thread 0 waits for the MMAs committed so far; result shared by the block
    auto mma_sync = [&]() {
        if (tid == 0) {
            tc::mma_commit(&bars.mma);
            if (!mbar_wait(&bars.mma, ph_mma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
        }
        ph_mma ^= 1;
        __syncthreads();
        tc::fence_after_sync();
        return bars.ok != 0;
    };

    for (int job = blockIdx.x; job < total; job += gridDim.x) {
        const int bh = job / a.N, chunk = job % a.N;
        const int c0 = chunk * kC;
        const int n = min(kC, a.L - c0);
        // ---------------------------------------------------------------- P1
        if (tid == 0) {
            mbar_arrive_expect_tx(&bars.tma, 3 * kTile);
            tc::tma_load_3d(smem + kOffQ, &maps.q, 0, c0, bh, &bars.tma);
            tc::tma_load_3d(smem + kOffQ + kTile / 2, &maps.q, 64, c0, bh, &bars.tma);
            tc::tma_load_3d(smem + kOffK, &maps.k, 0, c0, bh, &bars.tma);
            tc::tma_load_3d(smem + kOffK + kTile / 2, &maps.k, 64, c0, bh, &bars.tma);
            tc::tma_load_3d(smem + kOffW, &maps.w, 0, c0, bh, &bars.tma);
            tc::tma_load_3d(smem + kOffW + kTile / 2, &maps.w, 64, c0, bh, &bars.tma);
            if (!mbar_wait(&bars.tma, ph_tma, a.err, nullptr, kWaitLimitNs)) {
                bars.ok = 0;
            } else {
                tc::fence_after_sync();
                tc::gemm_128x128x128(tmem + kColA, sW, sW, false, false);  // G
                tc::gemm_128x128x128(tmem + kColB, sQ, sW, false, false);  // Q W^T
                tc::gemm_128x128x128(tmem + kColC, sK, sW, false, false);  // K W^T
                tc::gemm_128x128x128(tmem + kColD, sQ, sK, false, false);  // Q K^T
            }
        }
        ph_tma ^= 1;
        if (!mma_sync()) break;
        // ---------------------------------------------------------------- P2
        if (tid < kC) bsm[tid] = (tid < n) ? a.beta[(size_t)bh * a.L + c0 + tid] : 0.f;
        {
            uint32_t v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = half * 64 + cc * 32;
                tc::tmem_ld32(tmem + lane_off + kColA + col, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) Gf[r * kGs + col + i] = __uint_as_float(v[i]);
            }
        }
        __syncthreads();
        // ---------------------------------------------------------------- P3
        // Linv = (I + strict_lower(diag(beta) G))^{-1} into Tf (fp32, unit lower
        // triangular); T = Linv diag(beta) is formed when converting to bf16.
        unit_lower_inverse(Gf, Tf, bsm, tid);
        // ---------------------------------------------------------------- P4
        if (warp < 4) {
            // T fp32 -> bf16 tile (row i, column c), one column per thread
            const int c = tid;
            const float bc = bsm[c];
            for (int i = 0; i < kC; ++i) {
                const float t = (i >= c) ? Tf[i * kC + c] * bc : 0.f;
                const __nv_bfloat16 h = __float2bfloat16_rn(t);
                const uint32_t addr = sT + tc::swz_off(i, c >> 3, kC) + (c & 7) * 2;
                asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                             "h"(*reinterpret_cast<const unsigned short *>(&h))
                             : "memory");
            }
        } else {
            // -(M_le * Q W^T) -> bf16 tile
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + kColB + cc * 32, v);
                tile_store32(sQm, r, cc, v, [&](int s, float x) { return s <= r ? -x : 0.f; });
            }
        }
        __syncthreads();
        {
            // (M_gt * K W^T) -> bf16 tile in the first half of R2 (T fp32 done)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                const int c32 = half * 2 + cc;
                tc::tmem_ld32(tmem + lane_off + kColC + c32 * 32, v);
                tile_store32(sY, r, c32, v, [&](int s, float x) { return s > r ? x : 0.f; });
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------------------------------------------------------- P5
        if (tid == 0) {
            tc::gemm_128x128x128(tmem + kColA, sT, sW, true, false);   // Wt = T W
            tc::gemm_128x128x128(tmem + kColC, sY, sT, false, false);  // Y = KWm T^T
        }
        if (!mma_sync()) break;
        if (tid == 0) {
            // the chunk's values, for its own attention block, into the free T tile
            mbar_arrive_expect_tx(&bars.vbar, kTile);
            tc::tma_load_3d(smem + kOffR1, &maps.v, 0, c0, bh, &bars.vbar);
            tc::tma_load_3d(smem + kOffR1 + kTile / 2, &maps.v, 64, c0, bh, &bars.vbar);
        }
        // ---------------------------------------------------------------- P6
        {
            const uint32_t src = (half == 0) ? kColA : kColC;
            const uint32_t dst = (half == 0) ? sWt : sY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + src + cc * 32, v);
                tile_store32(dst, r, cc, v, [](int, float x) { return x; });
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------------------------------------------------------- P7
        if (tid == 0) {
            tc::gemm_128x128x128(tmem + kColB, sQm, sWt, true, false);  // -(M_le*QW) Wt
            tc::gemm_128x128x128(tmem + kColA, sY, sW, true, false);    // Y W
            tc::gemm_128x128x128(tmem + kColD, sQm, sY, false, true);   // QK^T - (M_le*QW) Y^T
            tc::gemm128_lo2<true, true>(tmem + kColC, tc::desc_lo(sW, true),
                                        tc::desc_lo(sWt, true), false);  // W^T Wt
        }
        if (!mma_sync()) break;
        // ---------------------------------------------------------------- P8
        {
            const size_t row = (size_t)bh * a.Lp + c0 + r;
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(half == 0 ? a.Qh : a.Kh) + row * kC;
            const uint32_t src_tile = half == 0 ? sQ : sK;
            const uint32_t col = half == 0 ? kColB : kColA;
            const float sign = half == 0 ? 1.f : -1.f;  // Qh = Q + (-M QW) Wt, Kh = K - Y W
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + col + cc * 32, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
                    tile_load8(src_tile, r, cc * 4 + q, x);
                    uint4 u;
                    u.x = pack2(x[0] + sign * __uint_as_float(v[q * 8 + 0]),
                                x[1] + sign * __uint_as_float(v[q * 8 + 1]));
                    u.y = pack2(x[2] + sign * __uint_as_float(v[q * 8 + 2]),
                                x[3] + sign * __uint_as_float(v[q * 8 + 3]));
                    u.z = pack2(x[4] + sign * __uint_as_float(v[q * 8 + 4]),
                                x[5] + sign * __uint_as_float(v[q * 8 + 5]));
                    u.w = pack2(x[6] + sign * __uint_as_float(v[q * 8 + 6]),
                                x[7] + sign * __uint_as_float(v[q * 8 + 7]));
                    *reinterpret_cast<uint4 *>(dst + cc * 32 + q * 8) = u;
                }
            }
            // Pm = I - W^T Wt, row r (input dimension), columns half*64 ..
            __nv_bfloat16 *pm = static_cast<__nv_bfloat16 *>(a.Pm) + row * kC;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                const int col = half * 64 + cc * 32;
                tc::tmem_ld32(tmem + lane_off + kColC + col, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        x[e] = ((col + q * 8 + e) == r ? 1.f : 0.f) - __uint_as_float(v[q * 8 + e]);
                    uint4 u;
                    u.x = pack2(x[0], x[1]);
                    u.y = pack2(x[2], x[3]);
                    u.z = pack2(x[4], x[5]);
                    u.w = pack2(x[6], x[7]);
                    *reinterpret_cast<uint4 *>(pm + col + q * 8) = u;
                }
            }
        }
        // ---------------------------------------------------------------- P9
        // causal softmax of the within-chunk logits, rows r, columns half*64..
        float m_row, l_row;
        {
            // per-row partial max / sum of the two column halves, in the R2
            // region (its Y / Wt tiles were last read by the P7 MMAs)
            float(*red)[2][kC] = reinterpret_cast<float(*)[2][kC]>(smem + kOffR2);
            const float *F = a.F ? a.F + (size_t)bh * a.Lp + c0 : nullptr;
            const float fi = F ? F[r] * 1.4426950408889634f : 0.f;
            uint32_t v[64];
            tc::tmem_ld64(tmem + lane_off + kColD + half * 64, v);
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int j = half * 64 + i;
                float x = __uint_as_float(v[i]) * sl2;
                if (F) x += fi - F[j] * 1.4426950408889634f;
                x = (j <= r) ? x : -INFINITY;
                v[i] = __float_as_uint(x);
                mx = fmaxf(mx, x);
            }
            red[0][half][r] = mx;
            __syncthreads();
            m_row = fmaxf(red[0][0][r], red[0][1][r]);  // finite: column r is unmasked
            float sum = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x = __uint_as_float(v[q * 8 + e]);
                    float y;
                    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x - m_row));
                    p[e] = (x == -INFINITY) ? 0.f : y;
                    sum += p[e];
                }
                sts128(sQm + tc::swz_off(r, half * 8 + q, kC), pack2(p[0], p[1]), pack2(p[2], p[3]),
                       pack2(p[4], p[5]), pack2(p[6], p[7]));
            }
            red[1][half][r] = sum;
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            l_row = red[1][0][r] + red[1][1][r];
        }
        if (tid == 0) {
            if (!mbar_wait(&bars.vbar, ph_v, a.err, nullptr, kWaitLimitNs)) {
                bars.ok = 0;
            } else {
                tc::gemm_128x128x128(tmem + kColC, sQm, sT, true, false);  // P V
            }
        }
        ph_v ^= 1;
        if (!mma_sync()) break;
        // ---------------------------------------------------------------- P10
        {
            const size_t row = (size_t)bh * a.Lp + c0 + r;
            __nv_bfloat16 *od = a.OD + row * kC + half * 64;
            const float inv = 1.f / l_row;
            uint32_t v[64];
            tc::tmem_ld64(tmem + lane_off + kColC + half * 64, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint4 u;
                u.x = pack2(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv);
                u.y = pack2(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv);
                u.z = pack2(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv);
                u.w = pack2(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv);
                *reinterpret_cast<uint4 *>(od + q * 8) = u;
            }
            if (half == 0) a.LSD[row] = (m_row + log2f(l_row)) * 0.6931471805599453f;
        }
        tc::fence_before_sync();
        __syncthreads();  // Q, K tiles and TMEM free before the next chunk's loads
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_prep_tc(const PrepTcMaps &maps, const PrepTcArgs &a, int num_sms,
                           cudaStream_t st) {
    const int total = a.N * a.BH;
    const int grid = total < num_sms ? total : num_sms;
    cudaError_t e =
        cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
    if (e != cudaSuccess) return e;
    prep_tc_kernel<<<grid, kThreadsP, kSmemP, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace path
