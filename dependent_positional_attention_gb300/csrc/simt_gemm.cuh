// Block-level SIMT GEMM helper (fp32 FMA), 256 threads, tiles up to 128x128.
#pragma once

#include "common.cuh"

namespace path {

constexpr int kThreads = 256;
constexpr int kTK = 16;       // k-depth of one smem stage
constexpr int kTS = 132;      // smem row stride of a stage (floats)

// out[r][c] (+)= sum_k A(r, k) B(k, c) for r < M <= 128, c < N <= 128.
// Thread (ty, tx) = (tid / 16, tid % 16) owns rows ty + 16 a and columns
// tx + 16 b.  AK / BK: the source is contiguous along k (selects the
// global-load mapping only).  Callers pass functors returning 0 outside the
// valid region.
template <bool AK, bool BK, class FA, class FB>
__device__ __forceinline__ void block_gemm(float (&acc)[8][8], int M, int N, int K, FA fa, FB fb, float *sA,
                           float *sB) {
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    for (int k0 = 0; k0 < K; k0 += kTK) {
        for (int e = tid; e < kTK * 128; e += kThreads) {
            int kk, r;
            if (AK) { kk = e % kTK; r = e / kTK; } else { r = e % 128; kk = e / 128; }
            sA[kk * kTS + r] = (r < M && k0 + kk < K) ? fa(r, k0 + kk) : 0.f;
            int c;
            if (BK) { kk = e % kTK; c = e / kTK; } else { c = e % 128; kk = e / 128; }
            sB[kk * kTS + c] = (c < N && k0 + kk < K) ? fb(k0 + kk, c) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kTK; ++kk) {
            float a[8], b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = sA[kk * kTS + ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = sB[kk * kTS + tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
}

__device__ __forceinline__ void zero(float (&acc)[8][8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
}

// Calls f(r, c, value) for every owned element with r < M, c < N.
template <class F>
__device__ __forceinline__ void for_owned(const float (&acc)[8][8], int M, int N, F f) {
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int r = ty + 16 * i, c = tx + 16 * j;
            if (r < M && c < N) f(r, c, acc[i][j]);
        }
}

// T = (I + strict_lower(diag(beta) G))^{-1} diag(beta) of one chunk, one
// column per thread by forward substitution:
//   T[i][c] = beta_i ([i == c] - sum_{c <= k < i} G[i][k] T[k][c]).
// G and T are row-major [C][C] (they may alias); rows >= n have beta = 0.
// big: 2 C (C + 1) floats of shared memory.  Ends with __syncthreads().
__device__ __forceinline__ void ut_solve(const float *G, const float *beta, int n, int C,
                                         float *T, float *big) {
    float *Gs = big, *Ts = big + C * (C + 1);
    for (int e = threadIdx.x; e < C * C; e += kThreads) Gs[(e / C) * (C + 1) + e % C] = G[e];
    __syncthreads();
    if (threadIdx.x < C) {
        const int c = threadIdx.x;
        for (int i = 0; i < C; ++i) {
            float t = 0.f;
            if (i >= c) {
                float s = (i == c) ? 1.f : 0.f;
                for (int kk = c; kk < i; ++kk) s -= Gs[i * (C + 1) + kk] * Ts[kk * (C + 1) + c];
                t = (i < n ? beta[i] : 0.f) * s;
            }
            Ts[i * (C + 1) + c] = t;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * C; e += kThreads) T[e] = Ts[(e / C) * (C + 1) + e % C];
    __syncthreads();
}

}  // namespace path
