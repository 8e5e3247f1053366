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
//                                               carried query rows: q <- q Pm;
//                                               stored transposed for the
//                                               forward scan)
// with M_le[r][s] = s <= r and M_gt[r][s] = s > r.  Eleven 128 x 128 x 128
// contractions run as tcgen05 MMAs (bf16 operands, fp32 accumulation in
// TMEM).  T is solved blockwise in fp32: the 16 x 16 diagonal blocks by
// forward substitution on the CUDA cores, their merges (T21 = -T22 G21 T11)
// as TF32 mma.sync products with a hi/lo split (about fp32 accuracy).
// Persistent CTAs, one chunk at a time.
//
// Phases per chunk (one thread issues TMA and MMAs; waits are bounded):
//   P1 MMA G -> cols 0 alone, as soon as the chunk's W lands (its TMA load,
//      and Q's and K's, were issued during the previous chunk's P10); the
//      next chunk's boxes are prefetched into L2
//   P3 (start) MMA QW -> 128, KW -> 256, QK -> 384, issued by a thread the
//      diagonal-block solve leaves idle
//   P2 G -> fp32 smem (swizzled)
//   P3 solve T (fp32 smem)
//   P4 T -> bf16 tile, -(M_le*QW) -> bf16 tile, (M_gt*KW) -> bf16 tile
//   P5 MMA Wt = T W -> cols 0, Y = (M_gt*KW) T^T -> cols 256
//   P6 Wt -> bf16 tile, Y -> bf16 tile
//   P7 MMA -(M_le*QW) Wt -> cols 128, Y W -> cols 0, += -(M_le*QW) Y^T -> cols 384,
//      W^T Wt -> cols 256   (the chunk's V is loaded meanwhile)
//   P8 Qh, Kh, Pm over their dead operand tiles, stored by TMA
//   P9 causal softmax of the within-chunk logits (cols 384) -> P bf16 tile;
//      MMA P V -> cols 256
//   P10 the chunk's own attention output (normalised, bf16, stored by TMA) and
//      its log-sum-exp -> workspace; the scan starts every query tile from them

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "ut_solve_tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kTile = kC * kC * 2;  // bf16 128 x 128 operand tile
constexpr int kThreadsP = 256;
constexpr int kOffQ = 0, kOffK = kTile, kOffW = 2 * kTile;
constexpr int kOffR1 = 3 * kTile;            // G fp32, then T bf16 | -(M_le*QW) bf16
constexpr int kR1Bytes = 64 * 1024;
constexpr int kOffR2 = kOffR1 + kR1Bytes;    // T fp32, then KWm/Y bf16 | Wt bf16
constexpr int kOffBar = kOffR2 + 64 * 1024;
constexpr int kBarBytes = 1152;
constexpr int kSmemP = kOffBar + kBarBytes + 1024;
static_assert(kC * kC * 4 <= kR1Bytes, "G staging does not fit");
static_assert(kSmemP <= 232448, "shared memory budget exceeded");
constexpr uint32_t kColA = 0, kColB = 128, kColC = 256, kColD = 384;

struct PBars {
    uint64_t tma, tma2, mma, mma2, vbar;
    uint32_t tmem_base;
    int ok;
    alignas(16) float beta[kC];
    float fsm[kC];  // PaTH-FoX: the chunk's prefix sums relative to its first, log2 units
};
static_assert(sizeof(PBars) <= kBarBytes, "barrier block too large");

using tc::lds128;
using tc::pack2;
using tc::sts128;

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

using utc::sw;
using utc::sw_f;
using utc::ut_solve;

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
    const int total = a.nloc * a.BH;

    if (tid == 0) {
        mbar_init(&bars.tma, 1);
        mbar_init(&bars.tma2, 1);
        mbar_init(&bars.mma, 1);
        mbar_init(&bars.mma2, 1);
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
    uint32_t ph_tma = 0, ph_mma = 0, ph_mma2 = 0, ph_v = 0;
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

    // W, Q and K of a chunk: issued for the first chunk here, and for each
    // following chunk as soon as the current one's output stores have read
    // the tiles (during P9), so that the loads overlap P9-P10.  Inputs and
    // outputs are addressed by local row (local chunk i at row 128 i).
    auto issue_loads = [&](int job) {
        const int bh = job / a.nloc, c0 = (job % a.nloc) * kC;
        tc::bulk_wait_read();
        mbar_arrive_expect_tx(&bars.tma, kTile);
        tc::tma_load_3d(smem + kOffW, &maps.w, 0, c0, bh, &bars.tma);
        tc::tma_load_3d(smem + kOffW + kTile / 2, &maps.w, 64, c0, bh, &bars.tma);
        mbar_arrive_expect_tx(&bars.tma2, 2 * kTile);
        tc::tma_load_3d(smem + kOffQ, &maps.q, 0, c0, bh, &bars.tma2);
        tc::tma_load_3d(smem + kOffQ + kTile / 2, &maps.q, 64, c0, bh, &bars.tma2);
        tc::tma_load_3d(smem + kOffK, &maps.k, 0, c0, bh, &bars.tma2);
        tc::tma_load_3d(smem + kOffK + kTile / 2, &maps.k, 64, c0, bh, &bars.tma2);
    };
    if (tid == 0 && blockIdx.x < total) issue_loads(blockIdx.x);
    for (int job = blockIdx.x; job < total; job += gridDim.x) {
        const int bh = job / a.nloc, li = job % a.nloc;
        const int chunk = a.cm.global_of_local(li);
        const int c0 = chunk * kC;  // first row of the chunk in the whole sequence
        const int r0 = li * kC;     // its first row in the local inputs and outputs
        const int n = min(kC, a.L - c0);
        // beta of the chunk, read ahead of its use in P2
        const float beta_r = (tid < kC && tid < n) ? a.beta[(size_t)bh * a.Lin + r0 + tid] : 0.f;
        // PaTH-FoX: the chunk's prefix sums, relative to its first (the bias
        // F_i - F_j is unchanged), read ahead of their use in P9
        const float f_r = (a.F && tid < kC)
                              ? (a.F[(size_t)bh * a.Lp + c0 + tid] - a.F[(size_t)bh * a.Lp + c0]) *
                                    1.4426950408889634f
                              : 0.f;
        // ---------------------------------------------------------------- P1
        // W first: G = W W^T alone lets the solve for T start while the
        // other three products run
        if (tid == 0) {
            const int next = job + gridDim.x;
            if (next < total) {
                const int nbh = next / a.nloc, nc0 = (next % a.nloc) * kC;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    tc::tma_prefetch_3d(&maps.q, 64 * x, nc0, nbh);
                    tc::tma_prefetch_3d(&maps.k, 64 * x, nc0, nbh);
                    tc::tma_prefetch_3d(&maps.w, 64 * x, nc0, nbh);
                    tc::tma_prefetch_3d(&maps.v, 64 * x, nc0, nbh);
                }
            }
            if (!mbar_wait(&bars.tma, ph_tma, a.err, nullptr, kWaitLimitNs)) {
                bars.ok = 0;
            } else {
                tc::fence_after_sync();
                tc::gemm_128x128x128(tmem + kColA, sW, sW, false, false);  // G
                tc::mma_commit(&bars.mma);
                if (!mbar_wait(&bars.mma, ph_mma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
            }
            // the previous chunk's OD (and V copy) stores read R1, which P2
            // overwrites with G
            tc::bulk_wait_read();
        }
        // Q W^T, K W^T, Q K^T are issued at the start of P3 by a thread that
        // the diagonal-block solve leaves idle, so that this thread is not held
        // on the MMA queue before it can release the block into the solve
        const uint32_t ph_q = ph_tma;
        ph_tma ^= 1;
        ph_mma ^= 1;
        __syncthreads();
        tc::fence_after_sync();
        if (!bars.ok) break;
        // ---------------------------------------------------------------- P2
        if (tid < kC) {
            bsm[tid] = beta_r;
            bars.fsm[tid] = f_r;
        }
        {
            uint32_t v[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = half * 64 + cc * 32;
                tc::tmem_ld32(tmem + lane_off + kColA + col, v);
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    *reinterpret_cast<float4 *>(Gf + sw(r, col + 4 * g)) =
                        make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                    __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
            }
        }
        __syncthreads();
        // ---------------------------------------------------------------- P3
        if (tid == 128) {
            if (!mbar_wait(&bars.tma2, ph_q, a.err, nullptr, kWaitLimitNs)) {
                bars.ok = 0;
            } else {
                tc::fence_after_sync();
                tc::gemm_128x128x128(tmem + kColB, sQ, sW, false, false);  // Q W^T
                tc::gemm_128x128x128(tmem + kColC, sK, sW, false, false);  // K W^T
                tc::gemm_128x128x128(tmem + kColD, sQ, sK, false, false);  // Q K^T
                tc::mma_commit(&bars.mma2);
            }
        }
        // T = (I + strict_lower(diag(beta) G))^{-1} diag(beta) into Tf (fp32)
        ut_solve(Gf, Tf, bsm, tid);
        // Q W^T, K W^T, Q K^T
        if (tid == 0 && bars.ok && !mbar_wait(&bars.mma2, ph_mma2, a.err, nullptr, kWaitLimitNs))
            bars.ok = 0;
        ph_mma2 ^= 1;
        __syncthreads();
        tc::fence_after_sync();
        if (!bars.ok) break;
        // ---------------------------------------------------------------- P4
        if (warp < 4) {
            // T fp32 -> bf16 tile, one row per thread.  Stored group pairs
            // (2n, 2n+1) hold the logical pair n ^ (sw_f >> 1), swapped when
            // sw_f is odd; visiting them in an order rotated by the row makes
            // the eight lanes of a load phase read different banks.
            const int f = sw_f(r);
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                const int n = (j + r) & 15;
                const float4 y0 = *reinterpret_cast<const float4 *>(Tf + r * kC + n * 8);
                const float4 y1 = *reinterpret_cast<const float4 *>(Tf + r * kC + n * 8 + 4);
                const float4 x0 = (f & 1) ? y1 : y0, x1 = (f & 1) ? y0 : y1;
                sts128(sT + tc::swz_off(r, n ^ (f >> 1), kC), pack2(x0.x, x0.y), pack2(x0.z, x0.w),
                       pack2(x1.x, x1.y), pack2(x1.z, x1.w));
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
            tc::tma_load_3d(smem + kOffR1, &maps.v, 0, r0, bh, &bars.vbar);
            tc::tma_load_3d(smem + kOffR1 + kTile / 2, &maps.v, 64, r0, bh, &bars.vbar);
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
            // W^T Wt, or its transpose Wt^T W when the chunk product is wanted
            // as Pm^T (rows = output dimension), the K-major layout the scan's
            // fused carried-query/logit product reads
            if (a.pm_transposed)
                tc::gemm128_lo2<true, true>(tmem + kColC, tc::desc_lo(sWt, true),
                                            tc::desc_lo(sW, true), false);
            else
                tc::gemm128_lo2<true, true>(tmem + kColC, tc::desc_lo(sW, true),
                                            tc::desc_lo(sWt, true), false);
        }
        if (!mma_sync()) break;
        // ---------------------------------------------------------------- P8
        // Qh (rows of threads 0-127) over the Q tile and Kh (threads 128-255)
        // over the K tile, in place; Pm over the W tile (its last readers, the
        // P7 MMAs, are complete); then one thread stores the three tiles.
        {
            const uint32_t tile = half == 0 ? sQ : sK;
            const uint32_t col = half == 0 ? kColB : kColA;
            const float sign = half == 0 ? 1.f : -1.f;  // Qh = Q + (-M QW) Wt, Kh = K - Y W
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + col + cc * 32, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
                    tile_load8(tile, r, cc * 4 + q, x);
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] += sign * __uint_as_float(v[q * 8 + e]);
                    sts128(tile + tc::swz_off(r, cc * 4 + q, kC), pack2(x[0], x[1]),
                           pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
                }
            }
            // Pm = I - W^T Wt, row r (input dimension), columns half*64 ..
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                const int col0 = half * 64 + cc * 32;
                tc::tmem_ld32(tmem + lane_off + kColC + col0, v);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        x[e] = ((col0 + q * 8 + e) == r ? 1.f : 0.f) - __uint_as_float(v[q * 8 + e]);
                    sts128(sW + tc::swz_off(r, half * 8 + cc * 4 + q, kC), pack2(x[0], x[1]),
                           pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
                }
            }
        }
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                tc::tma_store_3d(&maps.qh, smem + kOffQ + x * (kTile / 2), 64 * x, r0, bh);
                tc::tma_store_3d(&maps.kh, smem + kOffK + x * (kTile / 2), 64 * x, r0, bh);
                tc::tma_store_3d(&maps.pm, smem + kOffW + x * (kTile / 2), 64 * x, r0, bh);
            }
            tc::bulk_commit();
        }
        // ---------------------------------------------------------------- P9
        // causal softmax of the within-chunk logits, rows r, columns half*64..
        float m_row, l_row;
        {
            // per-row partial max / sum of the two column halves, in the R2
            // region (its Y / Wt tiles were last read by the P7 MMAs)
            float(*red)[2][kC] = reinterpret_cast<float(*)[2][kC]>(smem + kOffR2);
            const bool fox = a.F != nullptr;
            const float fi = fox ? bars.fsm[r] : 0.f;
            uint32_t v[64];
            tc::tmem_ld64(tmem + lane_off + kColD + half * 64, v);
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int j = half * 64 + i;
                float x = __uint_as_float(v[i]) * sl2;
                if (fox) x += fi - bars.fsm[j];
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
                // the next chunk's W, Q, K: the P8 stores have long been issued
                if (job + (int)gridDim.x < total) issue_loads(job + gridDim.x);
                if (a.copy_v) {
                    // sharded prefill: the chunk's V tile for the exchange with
                    // the other ranks (read by TMA while the MMA reads it too)
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        tc::tma_store_3d(&maps.vx, smem + kOffR1 + x * (kTile / 2), 64 * x, r0, bh);
                    tc::bulk_commit();
                }
            }
        }
        ph_v ^= 1;
        if (!mma_sync()) break;
        // ---------------------------------------------------------------- P10
        // the chunk's own attention output, normalised, over the P tile (the
        // PV MMA is complete), then stored by one thread
        {
            const float inv = 1.f / l_row;
            uint32_t v[64];
            tc::tmem_ld64(tmem + lane_off + kColC + half * 64, v);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                sts128(sQm + tc::swz_off(r, half * 8 + q, kC),
                       pack2(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv),
                       pack2(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv),
                       pack2(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv),
                       pack2(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv));
            if (half == 0)
                a.LSD[(size_t)bh * a.Lq + r0 + r] = (m_row + log2f(l_row)) * 0.6931471805599453f;
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();  // TMEM free, P tile rewritten, before the next chunk
        if (tid == 0) {
#pragma unroll
            for (int x = 0; x < 2; ++x)
                tc::tma_store_3d(&maps.od, smem + kOffR1 + kTile + x * (kTile / 2), 64 * x, r0, bh);
            tc::bulk_commit();
        }
    }
    if (tid == 0) tc::bulk_wait();  // no store may outlive the CTA's shared memory
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
    const int total = a.nloc * a.BH;
    const int grid = total < num_sms ? total : num_sms;
    cudaError_t e =
        cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
    if (e != cudaSuccess) return e;
    prep_tc_kernel<<<grid, kThreadsP, kSmemP, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace path
