// Blocked solve of the chunk's UT transform in fp32 shared memory, for 256
// threads and a 128-row chunk (PaTH Attention summary, section "3. 효율적인
// 학습 및 추론", UT transform): the 16 x 16 diagonal blocks by forward
// substitution on the CUDA cores, their merges as 3 x TF32 mma.sync products
// (about fp32 accuracy).  Used by the tensor-core prep (T) and by the
// tensor-core backward (Ti = T diag(beta)^-1 without the division).
#pragma once

#include "common.cuh"

namespace path {
namespace utc {

constexpr int kN = 128;    // chunk rows
constexpr int kThr = 256;  // threads that run the solve: warps 0-7 of the calling block

// Barrier over the solving threads only (named barrier 1), so that a block may
// hold further warps that do other work meanwhile.  bar.sync is warp-aligned:
// the warp is reconverged first.
__device__ __forceinline__ void solve_sync() {
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kThr) : "memory");
}

// fp32 128 x 128 matrices in shared memory (G, then T): row stride 128 floats,
// the 16-byte groups of row r permuted by group ^ sw_f(r).  sw_f takes eight
// different values on eight consecutive rows (from a multiple of 8) and four
// different values of sw_f >> 1 on four consecutive rows (from a multiple of
// 4), so that a warp touches every bank once both when it reads an m16n8k8
// A fragment (8 rows x 4 columns) and a B fragment (4 rows x 8 columns), and
// when one lane per row writes one group.
__device__ __forceinline__ int sw_f(int r) { return ((r & 3) << 1) | ((r >> 2) & 1); }
__device__ __forceinline__ int sw(int r, int c) {
    return r * kN + (((c >> 2) ^ sw_f(r)) << 2) + (c & 3);
}

// x = hi + lo + e with hi, lo tf32 values (fp32 bit patterns whose low 13
// mantissa bits are clear) and |e| < 2^-20 |x|: hi*hi + hi*lo + lo*hi carries
// a product to about fp32 accuracy ("3xTF32").  Truncation by a bit mask
// keeps the split on the integer pipes.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi)) & 0xffffe000u;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc[n] + acc2[n] += X[rows ra .. ra+15][k] * Y[k][cols cb + 8n .. +7] for k in
// [k_lo, k_hi), X and Y fp32 in the sw layout (X's column and Y's row offsets
// included in xc, yr); three tf32 MMAs per 16 x 8 x 8 step, the two small
// cross terms accumulated apart from the main one.
template <int NT>
__device__ __forceinline__ void mma3_rows(float (&acc)[NT][4], float (&acc2)[NT][4], const float *X,
                                          int ra, int xc, const float *Y, int yr, int cb, int k_lo,
                                          int k_hi, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int k0 = k_lo; k0 < k_hi; k0 += 8) {
        uint32_t ah[4], al[4];
        split_tf32(X[sw(ra + g, xc + k0 + t)], ah[0], al[0]);
        split_tf32(X[sw(ra + g + 8, xc + k0 + t)], ah[1], al[1]);
        split_tf32(X[sw(ra + g, xc + k0 + t + 4)], ah[2], al[2]);
        split_tf32(X[sw(ra + g + 8, xc + k0 + t + 4)], ah[3], al[3]);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            uint32_t bh[2], bl[2];
            split_tf32(Y[sw(yr + k0 + t, cb + 8 * n + g)], bh[0], bl[0]);
            split_tf32(Y[sw(yr + k0 + t + 4, cb + 8 * n + g)], bh[1], bl[1]);
            mma_tf32(acc2[n], al, bh);
            mma_tf32(acc2[n], ah, bl);
            mma_tf32(acc[n], ah, bh);
        }
    }
}

// Writes sign * (acc + acc2) (m16n8 accumulator fragments) to
// Z[rows ra ..][cols cb + 8n ..].
template <int NT>
__device__ __forceinline__ void store_frag(float *Z, int ra, int cb, const float (&acc)[NT][4],
                                           const float (&acc2)[NT][4], float sign, int lane,
                                           const float *rs = nullptr) {
    const int g = lane >> 2, t = lane & 3;
    const float s0 = rs ? sign * rs[g] : sign, s1 = rs ? sign * rs[g + 8] : sign;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        *reinterpret_cast<float2 *>(Z + sw(ra + g, cb + 8 * n + 2 * t)) =
            make_float2(s0 * (acc[n][0] + acc2[n][0]), s0 * (acc[n][1] + acc2[n][1]));
        *reinterpret_cast<float2 *>(Z + sw(ra + g + 8, cb + 8 * n + 2 * t)) =
            make_float2(s1 * (acc[n][2] + acc2[n][2]), s1 * (acc[n][3] + acc2[n][3]));
    }
}

// One merge level of the blocked solve for T.  For each pair of sibling
// diagonal blocks of size S starting at r1 and r2 = r1 + S,
//   T21 = -T22 G21 T11
// (from T = L^{-1} diag(beta), L = I + strict_lower(diag(beta) G): the
// lower-left block of L^{-1} is -L22^{-1} diag(beta_2) G21 L11^{-1}).
// Phase A forms P = G21 T11 and parks it in G's upper-right block of the
// pair, which the solve never reads otherwise (G is symmetric and only its
// lower blocks are used); phase B forms -T22 P into T.  Warp w takes one
// 16-row stripe and half of the columns of one pair; the k range skips the
// steps where T11 (upper triangle, phase A) or T22 (phase B) is zero.  The
// two warps that share a scheduler (w and w + 4) take the left and right
// column halves and mirrored stripes, so that both phases give them equal
// work.
template <int S, bool kInv>
__device__ __forceinline__ void ut_merge(float *G, float *Tf, const float *beta, int warp,
                                         int lane) {
    constexpr int M = S / 16;    // 16-row stripes per block
    constexpr int NT = S / 16;   // 8-column tiles per warp
    static_assert((kN / (2 * S)) * 2 * M == kThr / 32, "one stripe per warp");
    const int sched = warp & 3, h = warp >> 2;
    const int pair = sched / M, u = sched % M;
    const int r1 = pair * 2 * S, r2 = r1 + S;
    const int i0 = (h ? M - 1 - u : u) * 16, j0 = h * NT * 8;
    float acc[NT][4], acc2[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = acc2[n][e] = 0.f;
    // P[i][j] = sum_k G21[i][k] T11[k][j]; T11[k][j] = 0 for k < j
    mma3_rows<NT>(acc, acc2, G, r2 + i0, r1, Tf, r1, r1 + j0, j0, S, lane);
    // inverse mode: P = diag(beta_2) G21 Ti11, so that Ti21 = -Ti22 P
    store_frag<NT>(G, r1 + i0, r2 + j0, acc, acc2, 1.f, lane, kInv ? beta + r2 + i0 : nullptr);
    solve_sync();
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = acc2[n][e] = 0.f;
    // T21[i][j] = -sum_k T22[i][k] P[k][j]; T22[i][k] = 0 for k > i
    mma3_rows<NT>(acc, acc2, Tf, r2 + i0, r2, G, r1, r2 + j0, 0, i0 + 16, lane);
    store_frag<NT>(Tf, r2 + i0, r1 + j0, acc, acc2, -1.f, lane);
    solve_sync();
}

// T = (I + strict_lower(diag(beta) G))^{-1} diag(beta) into Tf (fp32, sw
// layout, zero above the diagonal); with kInv, Ti = (I + strict_lower(diag(beta)
// G))^{-1} instead (no column scaling; the merges scale the rows of their
// intermediate product by beta).  G: fp32 in the sw layout (symmetric; its
// upper blocks are overwritten).  The eight 16 x 16 diagonal blocks are
// solved by forward substitution (one column per thread, scaled by beta of
// that column), then merged at sizes 16, 32 and 64 on the tensor cores.
template <bool kInv = false>
__device__ __forceinline__ void ut_solve(float *G, float *Tf, const float *beta, int tid) {
    // zero the blocks above the 16 x 16 diagonal; nothing else writes them
    for (int e = tid; e < kN * kN / 4; e += kThr) {
        const int row = e >> 5, lgrp = (e & 31) ^ sw_f(row);
        if ((lgrp >> 2) > (row >> 4))
            reinterpret_cast<float4 *>(Tf)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < kN) {
        // column c of the diagonal block at o: x = (I + strict_lower(diag(beta) G))^{-1} e_c,
        // right-looking: s[i] accumulates sum_{k<i} G[i][k] x[k] and x[k] = [k == c] - beta_k s[k].
        // G[i][k] is read as G[k][i] (symmetry), one 16-byte group at a time.
        const int o = (tid >> 4) * 16, c = tid & 15;
        float bt[16], s_[16], x[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 b4 = *reinterpret_cast<const float4 *>(beta + o + 4 * q);
            bt[4 * q] = b4.x; bt[4 * q + 1] = b4.y; bt[4 * q + 2] = b4.z; bt[4 * q + 3] = b4.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) s_[i] = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            x[k] = (k < c) ? 0.f : fmaf(-bt[k], s_[k], (k == c) ? 1.f : 0.f);
#pragma unroll
            for (int q = (k + 1) >> 2; q < 4; ++q) {
                const float4 g4 = *reinterpret_cast<const float4 *>(G + sw(o + k, o + 4 * q));
                const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e > k) s_[4 * q + e] = fmaf(gv[e], x[k], s_[4 * q + e]);
            }
        }
        const float bc = kInv ? 1.f : beta[o + c];
#pragma unroll
        for (int i = 0; i < 16; ++i) Tf[sw(o + i, o + c)] = x[i] * bc;
    }
    solve_sync();
    const int warp = tid >> 5, lane = tid & 31;
    ut_merge<16, kInv>(G, Tf, beta, warp, lane);
    ut_merge<32, kInv>(G, Tf, beta, warp, lane);
    ut_merge<64, kInv>(G, Tf, beta, warp, lane);
}

}  // namespace utc
}  // namespace path
