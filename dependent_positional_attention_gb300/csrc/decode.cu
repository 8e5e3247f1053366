// PaTH decode step and key-cache build.
//
// Decode (PaTH Attention summary, section "3. 효율적인 학습 및 추론",
// inference bullet): the new token's transition H_t = I - beta_t w_t w_t^T is
// applied in place to every cached key, so the cache never stores w, and the
// attention itself reads the cache like ordinary flash-decoding.
//
// decode_split_kernel: grid (splits, B*H); each CTA streams a contiguous
// range of keys once.  A key of D bf16 is read by D/8 lanes with one 16-byte
// load each; per key the lanes reduce a = w_t.k_j and b = q_t.k_j with
// shuffles, write k_j - beta a w_t back (16-byte store) and form the logit
// scale * (b - beta a (q_t.w_t)) — the logit of the updated key, without
// re-reading it.  An online softmax (base 2) accumulates sum p v_j.  The
// CTA's 16 key groups merge in shared memory into one (m, l, o[D]) partial.
// decode_combine_kernel: one CTA per (b,h) merges the partials with the new
// token's own term (k_t enters untransformed) and appends k_t, v_t.
//
// Key-cache build: kc_j = H_{L-1} ... H_{j+1} k_j.  With chunk products
// P_c = H_{c,first} ... H_{c,last} = I - Wt_c^T W_c (Wt_c = T_c W_c) and
// boundary-adjusted keys Kh_c, kc_j = (Kh_j^T P_{c+1} ... P_{N-1})^T.
// The right-to-left product M_c = P_{c+1} ... P_{N-1} (d x d) is built in
// three phases so that the sequential part is short: per super-chunk of G
// chunks its product; per head the chain over super-chunks; per
// super-chunk the sweep that writes the keys.

#include "common.cuh"
#include "kernels.h"
#include "simt_gemm.cuh"

namespace path {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 x = __bfloat1622float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

template <int LPK>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = LPK / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kDecThreads = 256;
// Keys in flight per thread and loop iteration: 8 (88% of measured HBM copy
// bandwidth on GB300 at a 64K-token cache, against 76% with 4).  The split
// kernel is held to 128 registers (two CTAs per SM): left free, the PaTH-FoX
// instance took 147 and ran one CTA per SM at 60% of the bandwidth; held,
// it runs at 88% (it ran at 84% with 4 keys in flight).
template <bool FOX>
__host__ __device__ constexpr int dec_unroll() { return 8; }

// F_t = F_{t-1} + log f_t of the new token (PaTH-FoX), F_{-1} = 0.
__device__ __forceinline__ float fox_prefix_now(const DecodeArgs &a, int bh) {
    const float *fc = a.f_cache + (size_t)bh * a.cap;
    return (a.cache_len > 0 ? fc[a.cache_len - 1] : 0.f) + a.log_f_t[bh];
}

template <int D, bool FOX>
__global__ void __launch_bounds__(kDecThreads, 2) decode_split_kernel(DecodeArgs a) {
    constexpr int UNROLL = dec_unroll<FOX>();
    constexpr int LPK = D / 8;                      // lanes per key
    constexpr int KPW = 32 / LPK;                   // keys per warp per load
    constexpr int GROUPS = (kDecThreads / 32) * KPW;  // key groups per CTA
    __shared__ float sm_m[GROUPS], sm_l[GROUPS];
    __shared__ float sm_o[GROUPS][D + 4];

    const int bh = blockIdx.y, split = blockIdx.x;
    const int j0 = split * a.keys_per_split;
    const int j1 = min(a.cache_len, j0 + a.keys_per_split);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = warp * KPW + lane / LPK;
    const int sub = lane % LPK;

    const __nv_bfloat16 *qt = static_cast<const __nv_bfloat16 *>(a.q_t) + (size_t)bh * D + sub * 8;
    const __nv_bfloat16 *wt = static_cast<const __nv_bfloat16 *>(a.w_t) + (size_t)bh * D + sub * 8;
    float q[8], w[8];
    unpack8(*reinterpret_cast<const uint4 *>(qt), q);
    unpack8(*reinterpret_cast<const uint4 *>(wt), w);
    const float beta = a.beta_t[bh];
    float qw = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) qw = fmaf(q[i], w[i], qw);
    qw = group_sum<LPK>(qw);
    const float sl2 = a.scale * kLog2e;
    // PaTH-FoX: key j's logit gains sum_{s=j+1}^{t} log f_s = F_t - F_j
    const float *fc = FOX ? a.f_cache + (size_t)bh * a.cap : nullptr;
    const float Ft = FOX ? fox_prefix_now(a, bh) : 0.f;

    __nv_bfloat16 *kc = static_cast<__nv_bfloat16 *>(a.k_cache) + (size_t)bh * a.cap * D + sub * 8;
    const __nv_bfloat16 *vc =
        static_cast<const __nv_bfloat16 *>(a.v_cache) + (size_t)bh * a.cap * D + sub * 8;

    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;

    for (int base = j0; base < j1; base += GROUPS * UNROLL) {
        uint4 kr[UNROLL], vr[UNROLL];
        float fj[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int j = base + g + u * GROUPS;
            if (j < j1) {
                kr[u] = *reinterpret_cast<const uint4 *>(kc + (size_t)j * D);
                vr[u] = ld_stream(vc + (size_t)j * D);
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        if (FOX) {
            // lane u of the key group loads the prefix of the group's key u;
            // the group's lanes then take all UNROLL of them by shuffles
            const int jl = base + g + sub * GROUPS;
            const float fl = (sub < UNROLL && jl < j1) ? fc[jl] : 0.f;
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) fj[u] = __shfl_sync(0xffffffffu, fl, lane - sub + u);
        }
        float s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int j = base + g + u * GROUPS;
            float k[8];
            unpack8(kr[u], k);
            float pa = 0.f, pb = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pa = fmaf(w[i], k[i], pa);
                pb = fmaf(q[i], k[i], pb);
            }
            pa = group_sum<LPK>(pa);
            pb = group_sum<LPK>(pb);
            const float ba = beta * pa;
#pragma unroll
            for (int i = 0; i < 8; ++i) k[i] = fmaf(-ba, w[i], k[i]);
            if (j < j1) st_stream(kc + (size_t)j * D, pack8(k));
            float sj = sl2 * fmaf(-ba, qw, pb);
            if (FOX) sj = fmaf(Ft - fj[u], kLog2e, sj);  // difference first: no cancellation
            s[u] = (j < j1) ? sj : -INFINITY;
        }
        float mnew = m;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) mnew = fmaxf(mnew, s[u]);
        // mref keeps exp2 finite while no valid key has been seen (then every
        // term is exp2(-inf) = 0 and the state stays empty).
        const float mref = (mnew == -INFINITY) ? 0.f : mnew;
        const float alpha = exp2f(m - mref);
        l *= alpha;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] *= alpha;
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const float p = exp2f(s[u] - mref);
            l += p;
            float v[8];
            unpack8(vr[u], v);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = fmaf(p, v[i], o[i]);
        }
        m = mnew;
    }
    if (sub == 0) {
        sm_m[g] = m;
        sm_l[g] = l;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sm_o[g][sub * 8 + i] = o[i];
    __syncthreads();
    float *part = a.partials + ((size_t)bh * a.max_splits + split) * (D + 2);
    for (int dim = threadIdx.x; dim < D; dim += kDecThreads) {
        float M = -INFINITY;
#pragma unroll
        for (int gg = 0; gg < GROUPS; ++gg) M = fmaxf(M, sm_m[gg]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int gg = 0; gg < GROUPS; ++gg) {
            const float f = (sm_m[gg] == -INFINITY) ? 0.f : exp2f(sm_m[gg] - M);
            Ls = fmaf(sm_l[gg], f, Ls);
            Os = fmaf(sm_o[gg][dim], f, Os);
        }
        part[2 + dim] = Os;
        if (dim == 0) {
            part[0] = M;
            part[1] = Ls;
        }
    }
}

template <int D, bool FOX>
__global__ void __launch_bounds__(D) decode_combine_kernel(DecodeArgs a, int nsplit) {
    __shared__ float red[D / 32];
    const int bh = blockIdx.x, dim = threadIdx.x;
    const __nv_bfloat16 *qt = static_cast<const __nv_bfloat16 *>(a.q_t) + (size_t)bh * D;
    const __nv_bfloat16 *kt = static_cast<const __nv_bfloat16 *>(a.k_t) + (size_t)bh * D;
    const __nv_bfloat16 *vt = static_cast<const __nv_bfloat16 *>(a.v_t) + (size_t)bh * D;
    float x = __bfloat162float(qt[dim]) * __bfloat162float(kt[dim]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((dim & 31) == 0) red[dim >> 5] = x;
    __syncthreads();
    float self = 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) self += red[i];
    self *= a.scale * kLog2e;  // the new key enters untransformed (empty product)

    const float *part = a.partials + (size_t)bh * a.max_splits * (D + 2);
    float M = self;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part[s * (D + 2)]);
    float Ls = exp2f(self - M);
    float Os = Ls * __bfloat162float(vt[dim]);
    for (int s = 0; s < nsplit; ++s) {
        const float *p = part + s * (D + 2);
        const float f = (p[0] == -INFINITY) ? 0.f : exp2f(p[0] - M);
        Ls = fmaf(p[1], f, Ls);
        Os = fmaf(p[2 + dim], f, Os);
    }
    static_cast<__nv_bfloat16 *>(a.out)[(size_t)bh * D + dim] = __float2bfloat16_rn(Os / Ls);
    const size_t slot = ((size_t)bh * a.cap + a.cache_len) * D + dim;
    static_cast<__nv_bfloat16 *>(a.k_cache)[slot] = kt[dim];
    static_cast<__nv_bfloat16 *>(a.v_cache)[slot] = vt[dim];
    if (FOX && dim == 0) a.f_cache[(size_t)bh * a.cap + a.cache_len] = fox_prefix_now(a, bh);
}

// ------------------------------------------------------------ key-cache build

// M (smem, d x d) <- P_c M = M - Wt_c^T (W_c M); Y is a C x d smem scratch.
__device__ void apply_chunk_product(float *M, float *Y, const __nv_bfloat16 *Wc, const float *Wtc,
                                    int n, int C, int d, float *sA, float *sB) {
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    block_gemm<true, false>(
        acc, C, d, d,
        [&](int r, int s) { return r < n ? __bfloat162float(Wc[(size_t)r * d + s]) : 0.f; },
        [&](int s, int m) { return M[s * d + m]; }, sA, sB);
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int r = ty + 16 * i, c = tx + 16 * j;
            if (r < C && c < d) Y[r * d + c] = acc[i][j];
            acc[i][j] = 0.f;
        }
    __syncthreads();
    block_gemm<false, false>(
        acc, d, d, C, [&](int m1, int r) { return Wtc[(size_t)r * d + m1]; },
        [&](int r, int m2) { return Y[r * d + m2]; }, sA, sB);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int r = ty + 16 * i, c = tx + 16 * j;
            if (r < d && c < d) M[r * d + c] -= acc[i][j];
        }
    __syncthreads();
}

__device__ void set_identity(float *M, int d) {
    for (int e = threadIdx.x; e < d * d; e += kThreads) M[e] = (e / d == e % d) ? 1.f : 0.f;
    __syncthreads();
}

// Phase 1: Pi[s] = P_first ... P_last over the chunks of super-chunk s.
__global__ void __launch_bounds__(kThreads) kc_product_kernel(KcacheArgs a) {
    extern __shared__ float smem[];
    float *sA = smem, *sB = sA + kTK * kTS, *M = sB + kTK * kTS, *Y = M + a.d * a.d;
    const int s = blockIdx.x, h = blockIdx.y, d = a.d, C = a.C;
    const int c_first = s * a.G, c_last = min(a.N, c_first + a.G) - 1;
    set_identity(M, d);
    for (int c = c_last; c >= c_first; --c) {
        const int n = min(C, a.L - c * C);
        const __nv_bfloat16 *Wc = a.w + ((size_t)h * a.L + (size_t)c * C) * d;
        const float *Wtc = a.Wt + ((size_t)h * a.Lp + (size_t)c * C) * d;
        apply_chunk_product(M, Y, Wc, Wtc, n, C, d, sA, sB);
    }
    float *out = a.Pi + ((size_t)h * a.S + s) * d * d;
    for (int e = threadIdx.x; e < d * d; e += kThreads) out[e] = M[e];
}

// Phase 2: per head, Mout[s] = Pi[s+1] ... Pi[S-1] (identity for the last).
__global__ void __launch_bounds__(kThreads) kc_chain_kernel(KcacheArgs a) {
    extern __shared__ float smem[];
    float *sA = smem, *sB = sA + kTK * kTS, *M = sB + kTK * kTS, *Y = M + a.d * a.d;
    const int h = blockIdx.x, d = a.d;
    set_identity(M, d);
    for (int s = a.S - 1; s >= 0; --s) {
        float *mo = a.Mout + ((size_t)h * a.S + s) * d * d;
        for (int e = threadIdx.x; e < d * d; e += kThreads) mo[e] = M[e];
        if (s == 0) break;
        const float *Pi = a.Pi + ((size_t)h * a.S + s) * d * d;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
        block_gemm<true, false>(
            acc, d, d, d, [&](int r, int k) { return Pi[(size_t)r * d + k]; },
            [&](int k, int m) { return M[k * d + m]; }, sA, sB);
        const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int r = ty + 16 * i, c = tx + 16 * j;
                if (r < d && c < d) Y[r * d + c] = acc[i][j];
            }
        __syncthreads();
        for (int e = threadIdx.x; e < d * d; e += kThreads) M[e] = Y[e];
        __syncthreads();
    }
}

// Phase 3: sweep each super-chunk right to left writing kc rows = Kh_c M_c.
__global__ void __launch_bounds__(kThreads) kc_apply_kernel(KcacheArgs a) {
    extern __shared__ float smem[];
    float *sA = smem, *sB = sA + kTK * kTS, *M = sB + kTK * kTS, *Y = M + a.d * a.d;
    const int s = blockIdx.x, h = blockIdx.y, d = a.d, C = a.C;
    const int c_first = s * a.G, c_last = min(a.N, c_first + a.G) - 1;
    const float *mo = a.Mout + ((size_t)h * a.S + s) * d * d;
    for (int e = threadIdx.x; e < d * d; e += kThreads) M[e] = mo[e];
    __syncthreads();
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    for (int c = c_last; c >= c_first; --c) {
        const int n = min(C, a.L - c * C);
        const float *Khc = a.Kh + ((size_t)h * a.Lp + (size_t)c * C) * d;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
        block_gemm<true, false>(
            acc, C, d, d, [&](int r, int k) { return Khc[(size_t)r * d + k]; },
            [&](int k, int m) { return M[k * d + m]; }, sA, sB);
        __nv_bfloat16 *dst = a.k_cache + ((size_t)(a.h0 + h) * a.cap + (size_t)c * C) * d;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int r = ty + 16 * i, m = tx + 16 * j;
                if (r < n && m < d) dst[(size_t)r * d + m] = __float2bfloat16_rn(acc[i][j]);
            }
        if (c > c_first) {
            const __nv_bfloat16 *Wc = a.w + ((size_t)h * a.L + (size_t)c * C) * d;
            const float *Wtc = a.Wt + ((size_t)h * a.Lp + (size_t)c * C) * d;
            apply_chunk_product(M, Y, Wc, Wtc, n, C, d, sA, sB);
        }
    }
}

}  // namespace

int decode_keys_per_split() { return 1024; }

template <int D, bool FOX>
void launch_decode_t(const DecodeArgs &a, int nsplit, cudaStream_t st) {
    if (nsplit > 0) decode_split_kernel<D, FOX><<<dim3(nsplit, a.BH), kDecThreads, 0, st>>>(a);
    decode_combine_kernel<D, FOX><<<a.BH, D, 0, st>>>(a, nsplit);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
    const int nsplit = (a.cache_len + a.keys_per_split - 1) / a.keys_per_split;
    const bool fox = a.f_cache != nullptr;
    if (a.d == 128) {
        if (fox) launch_decode_t<128, true>(a, nsplit, st);
        else launch_decode_t<128, false>(a, nsplit, st);
    } else {
        if (fox) launch_decode_t<64, true>(a, nsplit, st);
        else launch_decode_t<64, false>(a, nsplit, st);
    }
    return cudaGetLastError();
}

size_t kcache_smem(int d, int C) {
    return sizeof(float) * (2 * kTK * kTS + d * d + (size_t)(C > d ? C : d) * d);
}

cudaError_t launch_kcache_sweep(const KcacheArgs &a, cudaStream_t st) {
    const size_t sm = kcache_smem(a.d, a.C);
    cudaFuncSetAttribute(kc_product_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    cudaFuncSetAttribute(kc_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    cudaFuncSetAttribute(kc_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    kc_product_kernel<<<dim3(a.S, a.HB), kThreads, sm, st>>>(a);
    kc_chain_kernel<<<a.HB, kThreads, sm, st>>>(a);
    kc_apply_kernel<<<dim3(a.S, a.HB), kThreads, sm, st>>>(a);
    return cudaGetLastError();
}

}  // namespace path
