// PaTH prefill, SIMT path (fp32 arithmetic on CUDA cores).
//
// Used for PATH_F32 inputs, where tensor-core rounding would exceed the
// fp32 tolerance.  Same algorithm as the tensor-core path (PaTH Attention
// summary, section "3. 효율적인 학습 및 추론"):
//   1. per chunk of C tokens, the UT transform of the chunk's transitions:
//        T = (I + strict_lower(diag(beta) W W^T))^{-1} diag(beta), so that
//        H_first ... H_last = I - W^T T^T W;
//      from it the boundary-adjusted rows
//        Qh = Q - (M_le * Q W^T) (T W),   Kh = K - (M_gt * K W^T) (T^T W),
//      the compact product factor Wt = T W, and the within-chunk logits
//        Sd = Q K^T - (M_le * Q W^T) T (M_gt * K W^T)^T
//      (M_le[r][s] = s <= r, M_gt[r][s] = s > r);
//   2. per query chunk b, a scan over key chunks c = b, b-1, ..., 0 with an
//      online softmax; after chunk c the carried query rows take the chunk
//      product: Qt <- Qt - (Qt W_c^T) Wt_c.
// The prep kernel is also instantiated for bf16 inputs/outputs.

#include "common.cuh"
#include "kernels.h"
#include "simt_gemm.cuh"

namespace path {
namespace {

// ------------------------------------------------------------------ prep

template <class T, class TO>
__global__ void __launch_bounds__(kThreads) prep_simt_kernel(PrepSimtArgs a) {
    extern __shared__ float smem[];
    float *sA = smem, *sB = smem + kTK * kTS;
    float *big = smem + 2 * kTK * kTS;  // [C][C+1] x 2 for the triangular solve

    const int C = a.C, d = a.d, L = a.L;
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int c0 = chunk * C;
    const int n = min(C, L - c0);  // valid rows in this chunk
    const size_t in_base = (size_t)bh * L * d + (size_t)c0 * d;
    const T *q = static_cast<const T *>(a.q) + in_base;
    const T *k = static_cast<const T *>(a.k) + in_base;
    const T *w = static_cast<const T *>(a.w) + in_base;
    const float *beta = a.beta + (size_t)bh * L + c0;
    const size_t ws_rows = (size_t)bh * a.Lp + c0;
    TO *Qh = static_cast<TO *>(a.Qh) + ws_rows * d;
    TO *Kh = static_cast<TO *>(a.Kh) + ws_rows * d;
    TO *Wt = static_cast<TO *>(a.Wt) + ws_rows * d;
    const bool queries = !a.keys_only;
    const size_t cc = (size_t)C * C;
    const size_t chunk_id = (size_t)bh * a.N + chunk;
    float *Sd = a.Sd + chunk_id * cc;
    float *G = a.scratch + chunk_id * 5 * cc;  // G, later T
    float *QW = G + cc, *KW = G + 2 * cc, *Z = G + 3 * cc, *Y = G + 4 * cc;

    auto W_ = [&](int r, int m) { return r < n ? to_f32(w[(size_t)r * d + m]) : 0.f; };
    auto Q_ = [&](int r, int m) { return r < n ? to_f32(q[(size_t)r * d + m]) : 0.f; };
    auto K_ = [&](int r, int m) { return r < n ? to_f32(k[(size_t)r * d + m]) : 0.f; };
    float acc[8][8];

    // S1: G = W W^T, QW = Q W^T, KW = K W^T, Sd = Q K^T.
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, W_, [&](int m, int s) { return W_(s, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { G[r * C + c] = v; });
    if (queries) {
        zero(acc);
        block_gemm<true, true>(acc, C, C, d, Q_, [&](int m, int s) { return W_(s, m); }, sA, sB);
        for_owned(acc, C, C, [&](int r, int c, float v) { QW[r * C + c] = v; });
        zero(acc);
        block_gemm<true, true>(acc, C, C, d, Q_, [&](int m, int s) { return K_(s, m); }, sA, sB);
        for_owned(acc, C, C, [&](int r, int c, float v) { Sd[r * C + c] = v; });
    }
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, K_, [&](int m, int s) { return W_(s, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { KW[r * C + c] = v; });
    __syncthreads();

    // S2: T = (I + strict_lower(diag(beta) G))^{-1} diag(beta), in place of G.
    ut_solve(G, beta, n, C, G, big);
    const float *Tm = G;

    // S3: Wt = T W, Z = (M_le * QW) T, Y = (M_gt * KW) T^T.
    zero(acc);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return Tm[r * C + s]; }, W_, sA, sB);
    for_owned(acc, C, d, [&](int r, int m, float v) { Wt[(size_t)r * d + m] = from_f32<TO>(v); });
    if (queries) {
        zero(acc);
        block_gemm<true, false>(
            acc, C, C, C, [&](int r, int s) { return s <= r ? QW[r * C + s] : 0.f; },
            [&](int s, int t) { return Tm[s * C + t]; }, sA, sB);
        for_owned(acc, C, C, [&](int r, int c, float v) { Z[r * C + c] = v; });
    }
    zero(acc);
    block_gemm<true, true>(
        acc, C, C, C, [&](int r, int s) { return s > r ? KW[r * C + s] : 0.f; },
        [&](int s, int t) { return Tm[t * C + s]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { Y[r * C + c] = v; });
    __syncthreads();

    // S4: Qh = Q - Z W, Kh = K - Y W, Sd -= (M_le * QW) Y^T.
    zero(acc);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return Y[r * C + s]; }, W_, sA, sB);
    for_owned(acc, C, d, [&](int r, int m, float v) {
        Kh[(size_t)r * d + m] = from_f32<TO>(K_(r, m) - v);
    });
    if (!queries) return;
    zero(acc);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return Z[r * C + s]; }, W_, sA, sB);
    for_owned(acc, C, d, [&](int r, int m, float v) {
        Qh[(size_t)r * d + m] = from_f32<TO>(Q_(r, m) - v);
    });
    zero(acc);
    block_gemm<true, true>(
        acc, C, C, C, [&](int r, int s) { return s <= r ? QW[r * C + s] : 0.f; },
        [&](int s, int j) { return Y[j * C + s]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { Sd[r * C + c] -= v; });
}

// ------------------------------------------------------------------ FoX prefix

// F[bh][i] = sum_{s<=i} log_f[bh][s] (fp64 sums, stored fp32); padded
// positions repeat the last value.  One block of kPrefixThreads per head,
// over tiles of kPrefixThreads * 16 positions: each thread sums its 16
// consecutive values, a block-wide exclusive scan of those sums (warp
// shuffles, then the warp totals) gives each thread its offset, and a second
// pass over the values held in registers writes the prefixes.  (One warp per
// head with a serial fp64 chain per lane took tens of microseconds at
// B8 H12 L4096, on the path of every PaTH-FoX call.)
constexpr int kPrefixThreads = 256;
__global__ void __launch_bounds__(kPrefixThreads)
    fox_prefix_kernel(const float *log_f, float *F, int L, int Lp, int BH) {
    constexpr int kPer = 16, kWarps = kPrefixThreads / 32;
    __shared__ double wtot[kWarps];
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (bh >= BH) return;
    const float *lf = log_f + (size_t)bh * L;
    float *out = F + (size_t)bh * Lp;
    double base = 0.0;
    for (int t0 = 0; t0 < Lp; t0 += kPrefixThreads * kPer) {
        const int i0 = t0 + tid * kPer;
        float x[kPer];
        double part = 0.0;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            x[e] = (i0 + e < L) ? lf[i0 + e] : 0.f;
            part += (double)x[e];
        }
        // exclusive scan of the threads' sums: within the warp, then over warps
        double incl = part;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        double before = 0.0, total = 0.0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const double t = wtot[w];
            if (w < warp) before += t;
            total += t;
        }
        __syncthreads();  // wtot is rewritten by the next tile
        double run = base + before + (incl - part);
        if (i0 < Lp) {
            float y[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                run += (double)x[e];
                y[e] = (float)run;
            }
            if (i0 + kPer <= Lp && (reinterpret_cast<uintptr_t>(out + i0) & 15) == 0) {
#pragma unroll
                for (int e = 0; e < kPer; e += 4)
                    *reinterpret_cast<float4 *>(out + i0 + e) =
                        make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < kPer; ++e)
                    if (i0 + e < Lp) out[i0 + e] = y[e];
            }
        }
        base += total;
    }
}

// ------------------------------------------------------------------ scan

// TIO: element type of w, v and out (float, or bf16 for bf16 inputs whose head
// dimension the tensor-core route does not take); Qh, Kh, Wt, Sd are fp32.
template <class TIO>
__global__ void __launch_bounds__(kThreads) flash_simt_kernel(FlashSimtArgs a) {
    extern __shared__ float smem[];
    const int C = a.C, d = a.d, L = a.L;
    float *sA = smem, *sB = smem + kTK * kTS;
    float *Qt = smem + 2 * kTK * kTS;  // [C][d]
    float *S = Qt + C * d;             // [C][C] logits, then probabilities
    float *X = S + C * C;              // [C][C]
    float *rowm = X + C * C, *rowl = rowm + C, *rowa = rowl + C;

    const int b = blockIdx.x, bh = blockIdx.y;
    const int nq = min(C, L - b * C);
    const float *Qh = static_cast<const float *>(a.Qh) + ((size_t)bh * a.Lp + (size_t)b * C) * d;
    const float *Kh = static_cast<const float *>(a.Kh) + (size_t)bh * a.Lp * d;
    const float *Wt = static_cast<const float *>(a.Wt) + (size_t)bh * a.Lp * d;
    const TIO *W = static_cast<const TIO *>(a.w) + (size_t)bh * L * d;
    const TIO *V = static_cast<const TIO *>(a.v) + (size_t)bh * L * d;
    const float *Sd = a.Sd + ((size_t)bh * a.N + b) * C * C;
    const float *F = a.F ? a.F + (size_t)bh * a.Lp : nullptr;

    for (int e = threadIdx.x; e < C * d; e += kThreads) Qt[e] = Qh[e];
    for (int r = threadIdx.x; r < C; r += kThreads) { rowm[r] = -INFINITY; rowl[r] = 0.f; }
    float o[8][8];
    zero(o);
    float acc[8][8];
    __syncthreads();

    for (int c = b; c >= 0; --c) {
        const int k0 = c * C;
        if (c == b) {
            for (int e = threadIdx.x; e < C * C; e += kThreads) S[e] = Sd[e];
        } else {
            zero(acc);
            block_gemm<false, true>(
                acc, C, C, d, [&](int r, int m) { return Qt[r * d + m]; },
                [&](int m, int j) { return Kh[(size_t)(k0 + j) * d + m]; }, sA, sB);
            for_owned(acc, C, C, [&](int r, int j, float v) { S[r * C + j] = v; });
            if (c >= 1) {
                zero(acc);
                block_gemm<false, true>(
                    acc, C, C, d, [&](int r, int m) { return Qt[r * d + m]; },
                    [&](int m, int s) { return to_f32(W[(size_t)(k0 + s) * d + m]); }, sA, sB);
                for_owned(acc, C, C, [&](int r, int s, float v) { X[r * C + s] = v; });
            }
        }
        __syncthreads();
        // online softmax, one thread per query row
        for (int r = threadIdx.x; r < C; r += kThreads) {
            float *srow = S + r * C;
            const int jmax = (c == b) ? r : C - 1;  // causal within the diagonal chunk
            const float fi = F ? F[b * C + r] : 0.f;
            float mx = -INFINITY;
            for (int j = 0; j < C; ++j) {
                float l = -INFINITY;
                if (r < nq && j <= jmax) {
                    l = a.scale * srow[j];
                    if (F) l += fi - F[k0 + j];
                }
                srow[j] = l;
                mx = fmaxf(mx, l);
            }
            const float mold = rowm[r];
            const float mnew = fmaxf(mold, mx);
            const float alpha = (mnew == -INFINITY) ? 1.f : expf(mold - mnew);
            float sum = 0.f;
            for (int j = 0; j < C; ++j) {
                float p = (srow[j] == -INFINITY) ? 0.f : expf(srow[j] - mnew);
                srow[j] = p;
                sum += p;
            }
            rowl[r] = rowl[r] * alpha + sum;
            rowm[r] = mnew;
            rowa[r] = alpha;
        }
        __syncthreads();
        {
            const int ty = threadIdx.x >> 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int r = ty + 16 * i;
                float al = r < C ? rowa[r] : 1.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) o[i][j] *= al;
            }
        }
        block_gemm<true, false>(
            o, C, d, C, [&](int r, int j) { return S[r * C + j]; },
            [&](int j, int m) { return (k0 + j < L) ? to_f32(V[(size_t)(k0 + j) * d + m]) : 0.f; }, sA,
            sB);
        if (c >= 1 && c < b) {
            zero(acc);
            block_gemm<true, false>(
                acc, C, d, C, [&](int r, int s) { return X[r * C + s]; },
                [&](int s, int m) { return Wt[(size_t)(k0 + s) * d + m]; }, sA, sB);
            for_owned(acc, C, d, [&](int r, int m, float v) { Qt[r * d + m] -= v; });
        }
        __syncthreads();
    }
    TIO *out = static_cast<TIO *>(a.out) + ((size_t)bh * L + (size_t)b * C) * d;
    for_owned(o, nq, d,
              [&](int r, int m, float v) { out[(size_t)r * d + m] = from_f32<TIO>(v / rowl[r]); });
    if (a.lse)
        for (int r = threadIdx.x; r < nq; r += kThreads)
            a.lse[(size_t)bh * L + (size_t)b * C + r] = rowm[r] + logf(rowl[r]);
}

}  // namespace

size_t prep_simt_smem(int C) {
    return sizeof(float) * (2 * kTK * kTS + 2 * C * (C + 1));
}
size_t flash_simt_smem(int C, int d) {
    return sizeof(float) * (2 * kTK * kTS + C * d + 2 * C * C + 3 * C);
}

cudaError_t launch_prep_simt(const PrepSimtArgs &a, bool bf16_in, bool bf16_out,
                             cudaStream_t st) {
    dim3 grid(a.N, a.BH);
    size_t sm = prep_simt_smem(a.C);
    void (*kern)(PrepSimtArgs);
    if (bf16_in)
        kern = bf16_out ? prep_simt_kernel<__nv_bfloat16, __nv_bfloat16>
                        : prep_simt_kernel<__nv_bfloat16, float>;
    else
        kern = prep_simt_kernel<float, float>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    kern<<<grid, kThreads, sm, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fox_prefix(const float *log_f, float *F, int L, int Lp, int BH,
                              cudaStream_t st) {
    if (BH <= 0) return cudaSuccess;
    fox_prefix_kernel<<<BH, kPrefixThreads, 0, st>>>(log_f, F, L, Lp, BH);
    return cudaGetLastError();
}

cudaError_t launch_flash_simt(const FlashSimtArgs &a, bool bf16_io, cudaStream_t st) {
    dim3 grid(a.N, a.BH);
    size_t sm = flash_simt_smem(a.C, a.d);
    void (*kern)(FlashSimtArgs) =
        bf16_io ? flash_simt_kernel<__nv_bfloat16> : flash_simt_kernel<float>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    kern<<<grid, kThreads, sm, st>>>(a);
    return cudaGetLastError();
}

}  // namespace path
