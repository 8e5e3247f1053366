// PaTH prefill backward on CUDA cores (fp32 arithmetic).
//
// Gradients of sum(dout * out) + sum(dlse * lse) with respect to q, k, v, w,
// beta and (PaTH-FoX) log f, by reverse-mode differentiation of the blockwise
// forward of prefill_simt.cu (PaTH Attention summary, section "3. 효율적인
// 학습 및 추론").  Notation of that file: per chunk the UT transform T, the
// boundary-adjusted rows Qh = Q - a T W and Kh = K - b T^T W with
// a = M_le * Q W^T and b = M_gt * K W^T, Wt = T W, the within-chunk logits
// Sd = Q K^T - a T b^T, and the chunk product A_c = I - W_c^T Wt_c that the
// carried query rows take after key chunk c: Qt_{c-1} = Qt_c A_c.
//
//   bwd_scan_kernel (one block per query chunk b, key chunks c < b):
//     (R) the forward's right-to-left chain Qt_{b-1} = Qh_b, Qt_{c-1} = Qt_c A_c,
//         every Qt_c stored;
//     (L) c = 0 .. b-1: probabilities from the saved lse, dP = dout V_c^T,
//         dlogit = P * (dP - D + dlse) with D = dout . out; then
//           dV_c  += P^T dout                     (atomic, over query chunks)
//           dKh_c += scale dlogit^T Qt_c          (atomic)
//           dA_c  += Qt_c^T G_{c-1}               (atomic)
//           G_c    = scale dlogit Kh_c + G_{c-1} A_c^T,  G_{-1} = 0,
//         and dQh_b = G_{b-1}.
//         The pages remark that the backward pays for atomic accumulation;
//         these three sums are where it does.
//   bwd_prep_kernel (one block per chunk): the chunk's own causal block
//     (its logits Sd recomputed, dSd = scale dlogit, dV's diagonal part),
//     then from dQh, dKh, dSd and dA back through the boundary adjustment,
//     Wt = T W and the UT transform to dq, dk, dw, dbeta (the derivation is
//     written out step by step below).  It recomputes everything it needs
//     from the inputs, so it serves the CUDA-core and the tensor-core scans.
//   fox_suffix_kernel: with the FoX bias F_i - F_j (F the inclusive prefix of
//     log f), dF_i = sum_j dlogit_ij - sum_i' dlogit_i'i and
//     dlog f_s = sum_{i >= s} dF_i.

#include "common.cuh"
#include "kernels.h"
#include "simt_gemm.cuh"

namespace path {
namespace {

template <class TIO>
__global__ void __launch_bounds__(kThreads) bwd_scan_kernel(BwdArgs a) {
    extern __shared__ float smem[];
    const int C = a.C, d = a.d, L = a.L;
    float *sA = smem, *sB = smem + kTK * kTS;
    float *Gs = smem + 2 * kTK * kTS;  // [C][d]: carried query rows (R), then G (L)
    float *S = Gs + C * d;             // [C][C]
    float *X = S + C * C;              // [C][C]
    float *rD = X + C * C, *rL = rD + C, *rF = rL + C, *rR = rF + C;

    const int b = a.N - 1 - blockIdx.x;  // longest rows first
    const int bh = blockIdx.y;
    const int nq = min(C, L - b * C);
    const size_t head = (size_t)bh * a.Lp * d;
    const float *Kh = a.Kh + head, *Wt = a.Wt + head;
    const TIO *W = static_cast<const TIO *>(a.w) + (size_t)bh * L * d;
    const TIO *V = static_cast<const TIO *>(a.v) + (size_t)bh * L * d;
    const TIO *dO = static_cast<const TIO *>(a.dout) + ((size_t)bh * L + (size_t)b * C) * d;
    const TIO *O = static_cast<const TIO *>(a.out) + ((size_t)bh * L + (size_t)b * C) * d;
    const float *F = a.F ? a.F + (size_t)bh * a.Lp : nullptr;
    float *Qts = a.Qts + ((size_t)bh * a.N * (a.N - 1) / 2 + (size_t)b * (b - 1) / 2) * C * d;
    float *dKh = a.dKh + head, *dV = a.dV + head;
    float *dA = a.dA + (size_t)bh * a.N * d * d;
    float *dF = a.dF ? a.dF + (size_t)bh * a.Lp : nullptr;

    auto dO_ = [&](int r, int m) { return r < nq ? to_f32(dO[(size_t)r * d + m]) : 0.f; };

    // row constants: D - dlse (so that dlogit = P (dP - rD)), lse, F_i
    for (int r = threadIdx.x; r < C; r += kThreads) {
        float D = 0.f, l = 0.f, f = 0.f;
        if (r < nq) {
            for (int m = 0; m < d; ++m) D = fmaf(to_f32(dO[(size_t)r * d + m]), to_f32(O[(size_t)r * d + m]), D);
            const size_t row = (size_t)bh * L + (size_t)b * C + r;
            if (a.dlse) D -= a.dlse[row];
            l = a.lse[row];
            f = F ? F[b * C + r] : 0.f;
        }
        rD[r] = D; rL[r] = l; rF[r] = f; rR[r] = 0.f;
    }
    float acc[8][8];

    // (R) carried query rows for c = b-1 .. 0
    if (b >= 1) {
        const float *Qh = a.Qh + head + (size_t)b * C * d;
        for (int e = threadIdx.x; e < C * d; e += kThreads) Gs[e] = Qh[e];
        __syncthreads();
        for (int c = b - 1; c >= 0; --c) {
            float *dst = Qts + (size_t)c * C * d;
            for (int e = threadIdx.x; e < C * d; e += kThreads) dst[e] = Gs[e];
            if (c >= 1) {
                const int k0 = c * C;
                zero(acc);
                block_gemm<true, true>(
                    acc, C, C, d, [&](int r, int m) { return Gs[r * d + m]; },
                    [&](int m, int s) { return to_f32(W[(size_t)(k0 + s) * d + m]); }, sA, sB);
                for_owned(acc, C, C, [&](int r, int s, float v) { X[r * C + s] = v; });
                __syncthreads();
                zero(acc);
                block_gemm<true, false>(
                    acc, C, d, C, [&](int r, int s) { return X[r * C + s]; },
                    [&](int s, int m) { return Wt[(size_t)(k0 + s) * d + m]; }, sA, sB);
                for_owned(acc, C, d, [&](int r, int m, float v) { Gs[r * d + m] -= v; });
            }
            __syncthreads();
        }
    }

    // (L) c = 0 .. b-1
    for (int e = threadIdx.x; e < C * d; e += kThreads) Gs[e] = 0.f;
    __syncthreads();
    for (int c = 0; c < b; ++c) {
        const int k0 = c * C;
        const float *Qt = Qts + (size_t)c * C * d;
        zero(acc);
        block_gemm<true, true>(
            acc, C, C, d, [&](int r, int m) { return Qt[(size_t)r * d + m]; },
            [&](int m, int j) { return Kh[(size_t)(k0 + j) * d + m]; }, sA, sB);
        for_owned(acc, C, C, [&](int r, int j, float v) { S[r * C + j] = v; });
        zero(acc);
        block_gemm<true, true>(
            acc, C, C, d, dO_,
            [&](int m, int j) { return (k0 + j < L) ? to_f32(V[(size_t)(k0 + j) * d + m]) : 0.f; },
            sA, sB);
        for_owned(acc, C, C, [&](int r, int j, float v) { X[r * C + j] = v; });
        __syncthreads();
        for (int e = threadIdx.x; e < C * C; e += kThreads) {
            const int r = e / C, j = e - r * C;
            const bool valid = r < nq;  // key chunk c < b is full
            float p = 0.f;
            if (valid) {
                float l = a.scale * S[e] + (F ? rF[r] - F[k0 + j] : 0.f);
                p = expf(l - rL[r]);
            }
            S[e] = p;
            X[e] = p * (X[e] - rD[r]);
        }
        __syncthreads();
        if (dF) {
            for (int r = threadIdx.x; r < C; r += kThreads) {
                float s = 0.f;
                for (int j = 0; j < C; ++j) s += X[r * C + j];
                rR[r] += s;
            }
            for (int j = threadIdx.x; j < C; j += kThreads) {
                float s = 0.f;
                for (int r = 0; r < C; ++r) s += X[r * C + j];
                if (k0 + j < L) atomicAdd(dF + k0 + j, -s);
            }
        }
        // dV_c += P^T dout
        zero(acc);
        block_gemm<false, false>(
            acc, C, d, C, [&](int j, int r) { return S[r * C + j]; }, dO_, sA, sB);
        for_owned(acc, C, d, [&](int j, int m, float v) {
            if (k0 + j < L) atomicAdd(dV + (size_t)(k0 + j) * d + m, v);
        });
        // dKh_c += scale dlogit^T Qt_c
        zero(acc);
        block_gemm<false, false>(
            acc, C, d, C, [&](int j, int r) { return X[r * C + j]; },
            [&](int r, int m) { return Qt[(size_t)r * d + m]; }, sA, sB);
        for_owned(acc, C, d, [&](int j, int m, float v) {
            if (k0 + j < L) atomicAdd(dKh + (size_t)(k0 + j) * d + m, a.scale * v);
        });
        if (c >= 1) {
            // dA_c += Qt_c^T G_{c-1}
            zero(acc);
            block_gemm<false, false>(
                acc, d, d, C, [&](int m, int r) { return Qt[(size_t)r * d + m]; },
                [&](int r, int n) { return Gs[r * d + n]; }, sA, sB);
            float *dAc = dA + (size_t)c * d * d;
            for_owned(acc, d, d, [&](int m, int n, float v) { atomicAdd(dAc + m * d + n, v); });
            // E = G_{c-1} Wt_c^T into S (P is no longer needed)
            zero(acc);
            block_gemm<true, true>(
                acc, C, C, d, [&](int r, int m) { return Gs[r * d + m]; },
                [&](int m, int s) { return Wt[(size_t)(k0 + s) * d + m]; }, sA, sB);
            for_owned(acc, C, C, [&](int r, int s, float v) { S[r * C + s] = v; });
            __syncthreads();
        }
        // G_c = G_{c-1} + [scale dlogit | -E] [Kh_c ; W_c]
        zero(acc);
        block_gemm<true, false>(
            acc, C, d, c >= 1 ? 2 * C : C,
            [&](int r, int kk) { return kk < C ? a.scale * X[r * C + kk] : -S[r * C + kk - C]; },
            [&](int kk, int m) {
                return kk < C ? Kh[(size_t)(k0 + kk) * d + m]
                              : to_f32(W[(size_t)(k0 + kk - C) * d + m]);
            },
            sA, sB);
        for_owned(acc, C, d, [&](int r, int m, float v) { Gs[r * d + m] += v; });
        __syncthreads();
    }
    __syncthreads();
    float *dQh = a.dQh + head + (size_t)b * C * d;
    for (int e = threadIdx.x; e < C * d; e += kThreads) dQh[e] = Gs[e];
    if (dF)
        for (int r = threadIdx.x; r < nq; r += kThreads) atomicAdd(dF + b * C + r, rR[r]);
}

// One chunk's own causal block and the gradient through its prep.  The block:
//   Sd = Q K^T - a Y^T, P = exp(scale Sd + F_i - F_j - lse_i) (j <= i),
//   dlogit = P (dout V^T - D + dlse), dSd = scale dlogit, dV += P^T dout.
// Then, with dQh, dKh from the scan and dA (the chunk product's gradient):
//   dWt  = -W dA                     dW  = -Wt dA^T + ...
//   da   = -(dSd b T^T + dQh Wt^T)   (a = M_le * Q W^T)
//   db   = -(dSd^T a + dKh W^T) T    (b = M_gt * K W^T)
//   dT   = -a^T (dSd b + dQh W^T) - (W dKh^T) b + dWt W^T
//   T = (I + Lo)^{-1} diag(beta), Lo = strict_lower(diag(beta) G), G = W W^T:
//     dX = (I + Lo)^{-T} dT,  dLo = strict_lower(-dX T^T),
//     dbeta_s = dX_ss + sum_{t<s} dLo_st G_st,  dG_st = beta_s dLo_st (t < s)
//   dq = dQh + dSd K + (M_le * da) W
//   dk = dKh + dSd^T Q + (M_gt * db) W
//   dw = -Wt dA^T - Z^T dQh - Y^T dKh + T^T dWt + (M_le * da)^T Q
//        + (M_gt * db)^T K + (dG + dG^T) W,    Z = a T, Y = b T^T.
template <class TIO>
__global__ void __launch_bounds__(kThreads) bwd_prep_kernel(BwdArgs a) {
    extern __shared__ float smem[];
    float *sA = smem, *sB = smem + kTK * kTS;
    float *big = smem + 2 * kTK * kTS;  // 2 [C][C+1] for the two triangular solves

    const int C = a.C, d = a.d, L = a.L;
    const int chunk = blockIdx.x, bh = blockIdx.y;
    const int c0 = chunk * C;
    const int n = min(C, L - c0);
    const size_t in_base = (size_t)bh * L * d + (size_t)c0 * d;
    const TIO *q = static_cast<const TIO *>(a.q) + in_base;
    const TIO *k = static_cast<const TIO *>(a.k) + in_base;
    const TIO *w = static_cast<const TIO *>(a.w) + in_base;
    const float *beta = a.beta + (size_t)bh * L + c0;
    const size_t ws_rows = ((size_t)bh * a.Lp + c0) * d;
    const float *dQh = a.dQh + ws_rows, *dKh = a.dKh + ws_rows, *dVa = a.dV + ws_rows;
    const size_t chunk_id = (size_t)bh * a.N + chunk;
    const float *dA = a.dA + chunk_id * d * d;
    const size_t cc = (size_t)C * C;
    float *G = a.scratch + chunk_id * kBwdPrepCC * cc;
    float *Tm = G + cc, *QW = G + 2 * cc, *KW = G + 3 * cc, *Z = G + 4 * cc, *Y = G + 5 * cc;
    float *R = G + 6 * cc, *dam = G + 7 * cc, *dbm = G + 8 * cc, *dT = G + 9 * cc;
    float *dSd = G + 10 * cc;
    float *dWt = a.scratch + (size_t)a.BH * a.N * kBwdPrepCC * cc + chunk_id * 2 * C * d;
    float *Wt = dWt + C * d;
    const size_t io_rows = (size_t)bh * L + c0;
    const TIO *v = static_cast<const TIO *>(a.v) + in_base;
    const TIO *dO = static_cast<const TIO *>(a.dout) + in_base;
    const TIO *O = static_cast<const TIO *>(a.out) + in_base;
    const float *F = a.F ? a.F + (size_t)bh * a.Lp + c0 : nullptr;
    float *dF = a.dF ? a.dF + (size_t)bh * a.Lp + c0 : nullptr;

    auto W_ = [&](int r, int m) { return r < n ? to_f32(w[(size_t)r * d + m]) : 0.f; };
    auto Q_ = [&](int r, int m) { return r < n ? to_f32(q[(size_t)r * d + m]) : 0.f; };
    auto K_ = [&](int r, int m) { return r < n ? to_f32(k[(size_t)r * d + m]) : 0.f; };
    auto am = [&](int r, int s) { return s <= r ? QW[r * C + s] : 0.f; };
    auto bm = [&](int r, int s) { return s > r ? KW[r * C + s] : 0.f; };
    float acc[8][8];

    // recompute G, Q W^T, K W^T, T, Z = a T, Y = b T^T (as the forward prep)
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, W_, [&](int m, int s) { return W_(s, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { G[r * C + c] = v; });
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, Q_, [&](int m, int s) { return W_(s, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { QW[r * C + c] = v; });
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, K_, [&](int m, int s) { return W_(s, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { KW[r * C + c] = v; });
    __syncthreads();
    ut_solve(G, beta, n, C, Tm, big);
    zero(acc);
    block_gemm<true, false>(acc, C, C, C, am, [&](int s, int t) { return Tm[s * C + t]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { Z[r * C + c] = v; });
    zero(acc);
    block_gemm<true, true>(acc, C, C, C, bm, [&](int s, int t) { return Tm[t * C + s]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int c, float v) { Y[r * C + c] = v; });
    // Wt = T W
    zero(acc);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return Tm[r * C + s]; }, W_, sA, sB);
    for_owned(acc, C, d, [&](int r, int m, float v) { Wt[r * d + m] = v; });

    // The chunk's own block.  Row constants in the (idle) solve area.
    float *rD = big, *rL = big + C, *rF = big + 2 * C;
    for (int r = threadIdx.x; r < C; r += kThreads) {
        float D = 0.f, l = 0.f, f = 0.f;
        if (r < n) {
            for (int m = 0; m < d; ++m)
                D = fmaf(to_f32(dO[(size_t)r * d + m]), to_f32(O[(size_t)r * d + m]), D);
            if (a.dlse) D -= a.dlse[io_rows + r];
            l = a.lse[io_rows + r];
            f = F ? F[r] : 0.f;
        }
        rD[r] = D; rL[r] = l; rF[r] = f;
    }
    auto dO_ = [&](int r, int m) { return r < n ? to_f32(dO[(size_t)r * d + m]) : 0.f; };
    // Sd = Q K^T - a Y^T into R; dP = dout V^T into dam
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, Q_, [&](int m, int j) { return K_(j, m); }, sA, sB);
    block_gemm<true, true>(acc, C, C, C, [&](int r, int s) { return -am(r, s); },
                           [&](int s, int j) { return Y[j * C + s]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int j, float v) { R[r * C + j] = v; });
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, dO_,
                           [&](int m, int j) { return j < n ? to_f32(v[(size_t)j * d + m]) : 0.f; },
                           sA, sB);
    for_owned(acc, C, C, [&](int r, int j, float x) { dam[r * C + j] = x; });
    __syncthreads();
    for (int e = threadIdx.x; e < C * C; e += kThreads) {
        const int r = e / C, j = e - r * C;
        float p = 0.f;
        if (r < n && j <= r) p = expf(a.scale * R[e] + (F ? rF[r] - F[j] : 0.f) - rL[r]);
        const float dl = p * (dam[e] - rD[r]);
        R[e] = p;
        dam[e] = dl;
        dSd[e] = a.scale * dl;
    }
    __syncthreads();
    if (dF) {
        // FoX: dF_i += sum_j dlogit_ij, dF_j -= sum_i dlogit_ij
        for (int r = threadIdx.x; r < n; r += kThreads) {
            float srow = 0.f, scol = 0.f;
            for (int j = 0; j < C; ++j) srow += dam[r * C + j];
            for (int i = 0; i < C; ++i) scol += dam[i * C + r];
            atomicAdd(dF + r, srow - scol);
        }
    }
    // dv = dV (scan) + P^T dout
    zero(acc);
    block_gemm<false, false>(acc, C, d, C, [&](int j, int r) { return R[r * C + j]; }, dO_, sA, sB);
    TIO *dv = static_cast<TIO *>(a.dv) + in_base;
    for_owned(acc, n, d, [&](int r, int m, float x) {
        dv[(size_t)r * d + m] = from_f32<TIO>(x + dVa[(size_t)r * d + m]);
    });
    __syncthreads();

    // dWt = -W dA
    zero(acc);
    block_gemm<true, false>(acc, C, d, d, W_, [&](int m, int nn) { return dA[m * d + nn]; }, sA, sB);
    for_owned(acc, C, d, [&](int r, int m, float v) { dWt[r * d + m] = -v; });
    // R = dSd b
    zero(acc);
    block_gemm<true, false>(acc, C, C, C, [&](int r, int s) { return dSd[r * C + s]; }, bm, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { R[r * C + t] = v; });
    __syncthreads();
    // da = -(R T^T + dQh Wt^T)
    zero(acc);
    block_gemm<true, true>(acc, C, C, C, [&](int r, int s) { return R[r * C + s]; },
                           [&](int s, int t) { return Tm[t * C + s]; }, sA, sB);
    block_gemm<true, true>(acc, C, C, d, [&](int r, int m) { return dQh[(size_t)r * d + m]; },
                           [&](int m, int t) { return Wt[(size_t)t * d + m]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { dam[r * C + t] = -v; });
    // db = -(dSd^T a + dKh W^T) T  (the bracket first, into dbm)
    zero(acc);
    block_gemm<false, false>(acc, C, C, C, [&](int r, int s) { return dSd[s * C + r]; }, am, sA, sB);
    block_gemm<true, true>(acc, C, C, d, [&](int r, int m) { return dKh[(size_t)r * d + m]; },
                           [&](int m, int t) { return W_(t, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { dbm[r * C + t] = v; });
    __syncthreads();
    zero(acc);
    block_gemm<true, false>(acc, C, C, C, [&](int r, int s) { return dbm[r * C + s]; },
                            [&](int s, int t) { return Tm[s * C + t]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { dbm[r * C + t] = -v; });
    // R += dQh W^T  (R = dSd b + dQh W^T)
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, [&](int r, int m) { return dQh[(size_t)r * d + m]; },
                           [&](int m, int t) { return W_(t, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { R[r * C + t] += v; });
    // dT = -(a^T R + (W dKh^T) b - dWt W^T); W dKh^T goes to dT first
    zero(acc);
    block_gemm<true, true>(acc, C, C, d, W_, [&](int m, int t) { return dKh[(size_t)t * d + m]; },
                           sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { dT[r * C + t] = v; });
    __syncthreads();
    zero(acc);
    block_gemm<false, false>(acc, C, C, C, [&](int r, int s) { return am(s, r); },
                             [&](int s, int t) { return R[s * C + t]; }, sA, sB);
    block_gemm<true, false>(acc, C, C, C, [&](int r, int s) { return dT[r * C + s]; }, bm, sA, sB);
    block_gemm<true, true>(acc, C, C, d, [&](int r, int m) { return -dWt[r * d + m]; },
                           [&](int m, int t) { return W_(t, m); }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { dT[r * C + t] = -v; });
    __syncthreads();

    // dX = (I + Lo)^{-T} dT in place: X_i = dT_i - sum_{k > i} beta_k G[k][i] X_k,
    // one column per thread, rows from the last to the first.
    {
        float *Gs = big, *Xs = big + C * (C + 1);
        for (int e = threadIdx.x; e < C * C; e += kThreads) {
            const int r = e / C, c = e - r * C;
            Gs[r * (C + 1) + c] = (r < n ? beta[r] : 0.f) * G[e];
            Xs[r * (C + 1) + c] = dT[e];
        }
        __syncthreads();
        if (threadIdx.x < C) {
            const int c = threadIdx.x;
            for (int i = C - 1; i >= 0; --i) {
                float s = Xs[i * (C + 1) + c];
                for (int kk = i + 1; kk < C; ++kk) s -= Gs[kk * (C + 1) + i] * Xs[kk * (C + 1) + c];
                Xs[i * (C + 1) + c] = s;
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < C * C; e += kThreads)
            dT[e] = Xs[(e / C) * (C + 1) + e % C];
        __syncthreads();
    }
    const float *dX = dT;
    // dLo = strict_lower(-dX T^T) into R
    zero(acc);
    block_gemm<true, true>(acc, C, C, C, [&](int r, int s) { return dX[r * C + s]; },
                           [&](int s, int t) { return Tm[t * C + s]; }, sA, sB);
    for_owned(acc, C, C, [&](int r, int t, float v) { R[r * C + t] = t < r ? -v : 0.f; });
    __syncthreads();
    float *dbeta = a.dbeta + (size_t)bh * L + c0;
    for (int s = threadIdx.x; s < n; s += kThreads) {
        float v = dX[s * C + s];
        for (int t = 0; t < s; ++t) v = fmaf(R[s * C + t], G[s * C + t], v);
        dbeta[s] = v;
    }
    auto dG = [&](int x, int y) { return (x < n ? beta[x] : 0.f) * R[x * C + y]; };

    // dw
    zero(acc);
    block_gemm<true, false>(acc, C, d, d, [&](int r, int m) { return -Wt[(size_t)r * d + m]; },
                            [&](int m, int nn) { return dA[nn * d + m]; }, sA, sB);
    block_gemm<false, false>(acc, C, d, C, [&](int r, int s) { return -Z[s * C + r]; },
                             [&](int s, int m) { return dQh[(size_t)s * d + m]; }, sA, sB);
    block_gemm<false, false>(acc, C, d, C, [&](int r, int s) { return -Y[s * C + r]; },
                             [&](int s, int m) { return dKh[(size_t)s * d + m]; }, sA, sB);
    block_gemm<false, false>(acc, C, d, C, [&](int r, int s) { return Tm[s * C + r]; },
                             [&](int s, int m) { return dWt[s * d + m]; }, sA, sB);
    block_gemm<false, false>(acc, C, d, C,
                             [&](int r, int s) { return r <= s ? dam[s * C + r] : 0.f; }, Q_, sA, sB);
    block_gemm<false, false>(acc, C, d, C,
                             [&](int r, int s) { return r > s ? dbm[s * C + r] : 0.f; }, K_, sA, sB);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return dG(r, s) + dG(s, r); }, W_,
                            sA, sB);
    TIO *dw = static_cast<TIO *>(a.dw) + in_base;
    for_owned(acc, n, d, [&](int r, int m, float v) { dw[(size_t)r * d + m] = from_f32<TIO>(v); });
    // dq
    zero(acc);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return dSd[r * C + s]; }, K_, sA, sB);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return s <= r ? dam[r * C + s] : 0.f; },
                            W_, sA, sB);
    TIO *dq = static_cast<TIO *>(a.dq) + in_base;
    for_owned(acc, n, d, [&](int r, int m, float v) {
        dq[(size_t)r * d + m] = from_f32<TIO>(v + dQh[(size_t)r * d + m]);
    });
    // dk
    zero(acc);
    block_gemm<false, false>(acc, C, d, C, [&](int r, int s) { return dSd[s * C + r]; }, Q_, sA, sB);
    block_gemm<true, false>(acc, C, d, C, [&](int r, int s) { return s > r ? dbm[r * C + s] : 0.f; },
                            W_, sA, sB);
    TIO *dk = static_cast<TIO *>(a.dk) + in_base;
    for_owned(acc, n, d, [&](int r, int m, float v) {
        dk[(size_t)r * d + m] = from_f32<TIO>(v + dKh[(size_t)r * d + m]);
    });
}

// dlog f_s = sum_{i >= s} dF_i (fp64 running sum from the right), one warp per head.
__global__ void fox_suffix_kernel(const float *dF, float *dlog_f, int L, int Lp, int BH) {
    const int bh = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (bh >= BH) return;
    const float *src = dF + (size_t)bh * Lp;
    float *out = dlog_f + (size_t)bh * L;
    const int seg = (L + 31) / 32;
    const int s0 = lane * seg, s1 = min(L, s0 + seg);
    double tot = 0.0;
    for (int i = s0; i < s1; ++i) tot += (double)src[i];
    // exclusive sum over the lanes to the right
    double incl = tot;
    for (int o = 1; o < 32; o <<= 1) {
        double v = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += v;
    }
    double run = incl - tot;
    for (int i = s1 - 1; i >= s0; --i) {
        run += (double)src[i];
        out[i] = (float)run;
    }
}

}  // namespace

size_t bwd_scan_smem(int C, int d) {
    return sizeof(float) * (2 * kTK * kTS + C * d + 2 * C * C + 4 * C);
}
size_t bwd_prep_smem(int C) {
    return sizeof(float) * (2 * kTK * kTS + 2 * C * (C + 1));
}

cudaError_t launch_bwd(const BwdArgs &a, bool bf16_io, cudaStream_t st) {
    dim3 grid(a.N, a.BH);
    const size_t sm = bwd_scan_smem(a.C, a.d);
    void (*kern)(BwdArgs) = bf16_io ? bwd_scan_kernel<__nv_bfloat16> : bwd_scan_kernel<float>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    kern<<<grid, kThreads, sm, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_bwd_prep(a, bf16_io, st);
}

cudaError_t launch_bwd_prep(const BwdArgs &a, bool bf16_io, cudaStream_t st) {
    dim3 grid(a.N, a.BH);
    {
        const size_t sm = bwd_prep_smem(a.C);
        void (*kern)(BwdArgs) = bf16_io ? bwd_prep_kernel<__nv_bfloat16> : bwd_prep_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        kern<<<grid, kThreads, sm, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (a.dF) return launch_fox_suffix(a.dF, a.dlog_f, a.L, a.Lp, a.BH, st);
    return cudaSuccess;
}

cudaError_t launch_fox_suffix(const float *dF, float *dlog_f, int L, int Lp, int BH,
                              cudaStream_t st) {
    const int warps = 4;
    fox_suffix_kernel<<<(BH + warps - 1) / warps, 32 * warps, 0, st>>>(dF, dlog_f, L, Lp, BH);
    return cudaGetLastError();
}

}  // namespace path
