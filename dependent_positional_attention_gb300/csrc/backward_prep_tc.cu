// Backward prep on tensor cores (bf16, head_dim 128, chunk 128; PaTH and
// PaTH-FoX): the chunk's own causal block and the gradient through the
// boundary adjustment and the UT transform, as a sequence of batched
// 128 x 128 x 128 contractions over all chunks (bf16 operands, fp32
// accumulation in TMEM) plus small CUDA-core steps: the per-row D, the UT
// solve, the chunk's own softmax block, fp32 -> bf16 conversions and dbeta.  The formulas are
// those of bwd_prep_kernel (backward_simt.cu); here
//   T = Ti diag(beta),  Ti = (I + strict_lower(diag(beta) G))^{-1},
// so that the solve dX = (I + Lo)^{-T} dT becomes the product Ti^T dT.
// Intermediate tiles live in the workspace as [BH][Lp][128] arrays.

#include "common.cuh"
#include "kernels.h"
#include "simt_gemm.cuh"
#include "tc.cuh"
#include "ut_solve_tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kTile = kC * kC * 2;
constexpr int kStages = 3;      // (A, B) tile pairs in flight
constexpr int kThreadsG = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue

struct GBars {
    uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_word;
};
constexpr int kSmemG = (int)sizeof(GBars) + 1023 + kStages * 2 * kTile;
static_assert(kSmemG <= 232448, "shared memory budget exceeded");

// D = alpha * sum_p (+/-) op(A_p) op(B_p) (+ E), masked, for every chunk.
// Persistent and warp-specialised: a three-stage TMA ring of operand pairs,
// one MMA thread accumulating into two TMEM buffers (128 columns each) so
// that the epilogue of one chunk overlaps the products of the next, and eight
// epilogue warps (two per TMEM lane quadrant, thread = chunk row, one half of
// the columns each).  Staging the rows through shared memory for contiguous
// global stores was tried and was slower: it left room for only two stages.
__global__ void __launch_bounds__(kThreadsG, 1)
    chunk_gemm_tc_kernel(const __grid_constant__ ChunkGemmMaps maps, ChunkGemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    GBars &bars = *reinterpret_cast<GBars *>(smem_raw);
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(GBars) + 1023) &
        ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int jobs = a.N * a.BH;
    volatile int *abort_word = &bars.abort_word;
    const uint64_t lim = kWaitLimitNs;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_empty[b], 8);
        }
        mbar_init(&bars.drain, 1);
        bars.abort_word = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bars.tmem_base, 256);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int par[kStages];
            for (int i = 0; i < kStages; ++i) par[i] = -1;
            bool ok = true;
            for (int job = blockIdx.x; job < jobs && ok; job += gridDim.x) {
                const int c0 = (job % a.N) * kC, bh = job / a.N;
                for (int p = 0; p < a.np; ++p) {
                    if (!mbar_wait(&bars.empty[s], ph ^ 1, a.err, abort_word, lim)) {
                        ok = false;
                        break;
                    }
                    const ChunkGemmProd &pr = a.prod[p];
                    uint8_t *dst = tiles + s * 2 * kTile;
                    mbar_arrive_expect_tx(&bars.full[s], 2 * kTile);
                    tc::tma_load_3d(dst, &maps.m[pr.a], 0, c0, bh, &bars.full[s]);
                    tc::tma_load_3d(dst + kTile / 2, &maps.m[pr.a], 64, c0, bh, &bars.full[s]);
                    tc::tma_load_3d(dst + kTile, &maps.m[pr.b], 0, c0, bh, &bars.full[s]);
                    tc::tma_load_3d(dst + kTile + kTile / 2, &maps.m[pr.b], 64, c0, bh,
                                    &bars.full[s]);
                    par[s] = (int)ph;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            if (!ok)  // let the copies in flight land before the CTA's memory goes away
                for (int i = 0; i < kStages; ++i)
                    if (par[i] >= 0) mbar_wait(&bars.full[i], (uint32_t)par[i], nullptr, nullptr, lim);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int s = 0, it = 0;
            uint32_t ph = 0, ae_ph[2] = {0, 0};
            bool ok = true, issued = false;
            for (int job = blockIdx.x; job < jobs && ok; job += gridDim.x, ++it) {
                const int buf = it & 1;
                if (!mbar_wait(&bars.acc_empty[buf], ae_ph[buf] ^ 1, a.err, abort_word, lim)) {
                    ok = false;
                    break;
                }
                ae_ph[buf] ^= 1;
                tc::fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(buf * 128);
                for (int p = 0; p < a.np; ++p) {
                    if (!mbar_wait(&bars.full[s], ph, a.err, abort_word, lim)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const ChunkGemmProd &pr = a.prod[p];
                    // A: op = X (K-major) or X^T (MN-major).  B: op = X is
                    // MN-major (rows of X along K), X^T is K-major.
                    const bool a_mn = pr.at, b_mn = !pr.bt;
                    const uint32_t idesc =
                        tc::idesc_bf16(128, 128, a_mn, b_mn) | (pr.neg ? (1u << 13) : 0u);
                    const uint32_t sA = smem_u32(tiles + s * 2 * kTile), sB = sA + kTile;
                    const uint32_t a_lo = tc::desc_lo(sA, a_mn), b_lo = tc::desc_lo(sB, b_mn);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2);
                        tc::mma_bf16_lohi(d, a_lo + (a_mn ? (uint32_t)(kk * 128) : koff),
                                          b_lo + (b_mn ? (uint32_t)(kk * 128) : koff), idesc,
                                          (p > 0 || kk > 0) ? 1u : 0u);
                    }
                    issued = true;
                    tc::mma_commit(&bars.empty[s]);  // frees the stage once read
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&bars.acc_full[buf]);
            }
            if (!ok && issued) {  // every issued MMA completes before TMEM is freed
                tc::mma_commit(&bars.drain);
                mbar_wait(&bars.drain, 0, nullptr, nullptr, lim);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3, hcol = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint32_t af_ph[2] = {0, 0};
        int it = 0;
        for (int job = blockIdx.x; job < jobs; job += gridDim.x, ++it) {
            const int buf = it & 1;
            bool ok = mbar_wait(&bars.acc_full[buf], af_ph[buf], a.err, abort_word, lim);
            af_ph[buf] ^= 1;
            if (!__all_sync(0xffffffffu, ok)) break;
            tc::fence_after_sync();
            const int chunk = job % a.N, bh = job / a.N;
            const int c0 = chunk * kC;
            const int n = min(kC, a.L - c0);
            const size_t ws_row = ((size_t)bh * a.Lp + c0 + r) * kC;
            const size_t io_row = ((size_t)bh * a.L + c0 + r) * kC;
            const bool live = r < n;
            const float rs = (a.rowscale && live) ? a.rowscale[(size_t)bh * a.L + c0 + r] : 0.f;
#pragma unroll 1
            for (int cc = 2 * hcol; cc < 2 * hcol + 2; ++cc) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + lane_off + (uint32_t)(buf * 128 + cc * 32), v);
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = cc * 32 + e;
                    float y = a.alpha * __uint_as_float(v[e]);
                    if (a.E) y += a.E[ws_row + j];
                    const bool keep = live && (a.mask == 0 || (a.mask == 1 && j <= r) ||
                                               (a.mask == 2 && j > r) || (a.mask == 3 && j < r));
                    x[e] = keep ? y : 0.f;
                }
                if (a.out_f32) {
                    float4 *dst = reinterpret_cast<float4 *>(a.out_f32 + ws_row + cc * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        dst[k4] = make_float4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
                }
                if (a.out_bf16 && (!a.out_final || live)) {
                    const float sc = a.rowscale ? rs : 1.f;
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        a.out_bf16 + (a.out_final ? io_row : ws_row) + cc * 32);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        dst[k4] = make_uint4(tc::pack2(sc * x[8 * k4], sc * x[8 * k4 + 1]),
                                             tc::pack2(sc * x[8 * k4 + 2], sc * x[8 * k4 + 3]),
                                             tc::pack2(sc * x[8 * k4 + 4], sc * x[8 * k4 + 5]),
                                             tc::pack2(sc * x[8 * k4 + 6], sc * x[8 * k4 + 7]));
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.acc_empty[buf]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

// Ti = (I + strict_lower(diag(beta) G))^{-1} by the tensor-core prep's blocked
// solve in inverse mode, written as bf16 Ti and T = Ti diag(beta).  One block
// of 256 threads per chunk.
// 16 bytes global -> shared without registers (cp.async, L2 only); the
// group below completes in issue order.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Ti = (I + strict_lower(diag(beta) G))^{-1} and T = Ti diag(beta) (bf16) of
// every chunk.  Persistent: each CTA solves its chunks one after another
// while the next chunk's G streams into the second of two shared buffers.
__global__ void __launch_bounds__(utc::kThr) bwd_solve_kernel(const float *G, const float *beta,
                                                               __nv_bfloat16 *T, __nv_bfloat16 *Ti,
                                                               int BH, int L, int Lp, int N) {
    extern __shared__ uint8_t smem_raw[];
    float *Gbuf = reinterpret_cast<float *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
    float *Tf = Gbuf + 2 * kC * kC;
    float *bsm = Tf + kC * kC;  // two beta rows
    const int tid = threadIdx.x;
    const int total = N * BH;
    // G of job -> buffer b, in the solve's swizzled layout; beta alongside
    auto fetch = [&](int job, int b) {
        const int chunk = job % N, bh = job / N;
        const int c0 = chunk * kC, n = min(kC, L - c0);
        const float *src = G + ((size_t)bh * Lp + c0) * kC;
        float *dst = Gbuf + b * kC * kC;
        for (int e = tid; e < kC * kC / 4; e += utc::kThr) {
            const int r = e / (kC / 4), c = (e % (kC / 4)) * 4;
            cp_async16(dst + utc::sw(r, c), src + (size_t)e * 4);
        }
        if (tid < kC) bsm[b * kC + tid] = tid < n ? beta[(size_t)bh * L + c0 + tid] : 0.f;
        cp_async_commit();
    };
    int k = 0;
    if (blockIdx.x < total) fetch(blockIdx.x, 0);
    for (int job = blockIdx.x; job < total; job += gridDim.x, ++k) {
        const int b = k & 1;
        const int next = job + gridDim.x;
        // the next chunk's G streams in while this one is solved
        if (next < total) {
            fetch(next, b ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        float *Gs = Gbuf + b * kC * kC;
        const float *bs = bsm + b * kC;
        utc::ut_solve<true>(Gs, Tf, bs, tid);
        __syncthreads();
        // Ti and T rows, eight columns a store
        const int chunk = job % N, bh = job / N;
        const size_t base = ((size_t)bh * Lp + chunk * kC) * kC;
        for (int e = tid; e < kC * kC / 8; e += utc::kThr) {
            const int r = e / (kC / 8), c = (e % (kC / 8)) * 8;
            const float4 t0 = *reinterpret_cast<const float4 *>(Tf + utc::sw(r, c));
            const float4 t1 = *reinterpret_cast<const float4 *>(Tf + utc::sw(r, c + 4));
            const float t[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
            uint32_t wi[4], wt[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                wi[q] = tc::pack2(t[2 * q], t[2 * q + 1]);
                wt[q] = tc::pack2(t[2 * q] * bs[c + 2 * q], t[2 * q + 1] * bs[c + 2 * q + 1]);
            }
            *reinterpret_cast<uint4 *>(Ti + base + (size_t)e * 8) = make_uint4(wi[0], wi[1], wi[2], wi[3]);
            *reinterpret_cast<uint4 *>(T + base + (size_t)e * 8) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
        }
        // every thread is done with this buffer before the fetch after next
        // (issued at the start of the next job) reuses it
        __syncthreads();
    }
    cp_async_wait<0>();
}

// D = dout . out - dlse for every row of the padded layout [BH][Lp] (0 on the
// padding), one warp per row.
__global__ void bwd_rowdot_kernel(const __nv_bfloat16 *out, const __nv_bfloat16 *dout,
                                  const float *dlse, float *Dg, int BH, int L, int Lp) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= (size_t)BH * Lp) return;
    const int bh = (int)(row / Lp), i = (int)(row % Lp);
    float s = 0.f;
    if (i < L) {
        const size_t off = ((size_t)bh * L + i) * kC + 4 * lane;
        const uint2 x = *reinterpret_cast<const uint2 *>(out + off);
        const uint2 y = *reinterpret_cast<const uint2 *>(dout + off);
        const float2 x0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
        const float2 x1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
        const float2 y0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&y.x));
        const float2 y1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&y.y));
        s = x0.x * y0.x + x0.y * y0.y + x1.x * y1.x + x1.y * y1.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) Dg[row] = (i < L) ? s - (dlse ? dlse[(size_t)bh * L + i] : 0.f) : 0.f;
}

// The chunk's own block: P = exp(scale Sd + F_i - F_j - lse) (j <= i; the
// FoX term only for PaTH-FoX), dSd = scale P (dP - D), as bf16 tiles; for
// PaTH-FoX also dF_i += sum_j dlogit_ij and dF_j -= sum_i dlogit_ij.  One
// block per chunk; dlogit staged in shared memory for the sums.
__global__ void __launch_bounds__(kThreads) bwd_diag_kernel(BwdDiagArgs a) {
    extern __shared__ float dls[];  // [C][C + 1] dlogit (PaTH-FoX only)
    __shared__ float rD[kC], rL[kC], rF[kC];
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int c0 = chunk * kC, n = min(kC, a.L - c0);
    const size_t base = ((size_t)bh * a.Lp + c0) * kC;
    const float *F = a.F ? a.F + (size_t)bh * a.Lp + c0 : nullptr;
    for (int r = threadIdx.x; r < kC; r += kThreads) {
        rD[r] = a.Dg[(size_t)bh * a.Lp + c0 + r];
        rL[r] = r < n ? a.lse[(size_t)bh * a.L + c0 + r] : 0.f;
        rF[r] = F ? F[r] - F[0] : 0.f;  // chunk-relative prefix
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kC * kC; e += kThreads) {
        const int r = e / kC, j = e - r * kC;
        float p = 0.f;
        if (r < n && j <= r) p = expf(a.scale * a.Sd[base + e] + rF[r] - rF[j] - rL[r]);
        const float dl = p * (a.dP[base + e] - rD[r]);
        a.P[base + e] = __float2bfloat16_rn(p);
        a.dSd[base + e] = __float2bfloat16_rn(a.scale * dl);
        if (F) dls[r * (kC + 1) + j] = dl;
    }
    if (!F) return;
    __syncthreads();
    for (int r = threadIdx.x; r < n; r += kThreads) {
        float sr = 0.f, sc = 0.f;
        for (int j = 0; j < kC; ++j) sr += dls[r * (kC + 1) + j];
        for (int i = 0; i < kC; ++i) sc += dls[i * (kC + 1) + r];
        atomicAdd(a.dF + (size_t)bh * a.Lp + c0 + r, sr - sc);
    }
}

__global__ void bwd_cvt_kernel(const float *x, __nv_bfloat16 *y, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = reinterpret_cast<const float4 *>(x)[i];
        reinterpret_cast<uint2 *>(y)[i] = make_uint2(tc::pack2(v.x, v.y), tc::pack2(v.z, v.w));
    }
}

// dbeta_s = dX_ss + sum_{t<s} dLo_st G_st, one warp per row (dLo is zero for
// t >= s, so the whole row is summed).
__global__ void bwd_dbeta_kernel(const float *dX, const float *dLo, const float *G, float *dbeta,
                                 int L, int Lp, int N, int BH) {
    const size_t row = (size_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;  // over BH * Lp
    const int lane = threadIdx.x & 31;
    if (row >= (size_t)BH * Lp) return;
    const int bh = (int)(row / Lp), i = (int)(row % Lp);
    if (i >= L) return;
    const size_t base = row * kC;
    const float4 x = reinterpret_cast<const float4 *>(dLo + base)[lane];
    const float4 g = reinterpret_cast<const float4 *>(G + base)[lane];
    float v = x.x * g.x + x.y * g.y + x.z * g.z + x.w * g.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) dbeta[(size_t)bh * L + i] = v + dX[base + i % kC];
}

}  // namespace

cudaError_t launch_chunk_gemm_tc(const ChunkGemmMaps &maps, const ChunkGemmArgs &a,
                                 int num_sms, cudaStream_t st) {
    // set on every call: function attributes are per device
    cudaError_t e = cudaFuncSetAttribute(chunk_gemm_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemG);
    if (e != cudaSuccess) return e;
    const int jobs = a.N * a.BH;
    chunk_gemm_tc_kernel<<<jobs < num_sms ? jobs : num_sms, kThreadsG, kSmemG, st>>>(maps, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_solve(const float *G, const float *beta, __nv_bfloat16 *T,
                             __nv_bfloat16 *Ti, int BH, int L, int Lp, int N, cudaStream_t st) {
    const size_t sm = sizeof(float) * (3 * kC * kC + 2 * kC) + 16;
    cudaError_t e =
        cudaFuncSetAttribute(bwd_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long total = (long long)N * BH;
    const int grid = (int)(total < sms ? total : sms);
    if (grid <= 0) return cudaSuccess;
    bwd_solve_kernel<<<grid, utc::kThr, sm, st>>>(G, beta, T, Ti, BH, L, Lp, N);
    return cudaGetLastError();
}

cudaError_t launch_bwd_rowdot(const __nv_bfloat16 *out, const __nv_bfloat16 *dout,
                              const float *dlse, float *Dg, int BH, int L, int Lp,
                              cudaStream_t st) {
    const size_t rows = (size_t)BH * Lp;
    bwd_rowdot_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(out, dout, dlse, Dg, BH, L, Lp);
    return cudaGetLastError();
}

cudaError_t launch_bwd_diag(const BwdDiagArgs &a, cudaStream_t st) {
    const size_t sm = a.F ? sizeof(float) * kC * (kC + 1) : 0;
    cudaError_t e =
        cudaFuncSetAttribute(bwd_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    bwd_diag_kernel<<<dim3(a.N, a.BH), kThreads, sm, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_cvt(const float *x, __nv_bfloat16 *y, size_t n, cudaStream_t st) {
    const size_t n4 = n / 4;
    const int blocks = (int)((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096);
    bwd_cvt_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(x, y, n4);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dbeta(const float *dX, const float *dLo, const float *G, float *dbeta,
                             int BH, int L, int Lp, int N, cudaStream_t st) {
    const size_t rows = (size_t)BH * Lp;
    bwd_dbeta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(dX, dLo, G, dbeta, L, Lp, N, BH);
    return cudaGetLastError();
}

}  // namespace path
