// PaTH prefill backward scan on tensor cores (bf16, head_dim 128, chunk 128).
//
// The off-diagonal part of the backward of the blockwise forward (PaTH
// Attention summary, section "3. 효율적인 학습 및 추론"); the chunk's own
// block and the gradient through the UT transform follow in
// bwd_prep_kernel.  Per query chunk b, with the tensor-core prep's bf16 Qh,
// Kh and chunk products Pm_c (the carried rows take Qt <- Qt Pm_c after key
// chunk c):
//   (R) Qt_{b-1} = Qh_b, Qt_{c-1} = Qt_c Pm_c: the forward's right-to-left
//       chain, recomputed exactly as the forward scan forms it (bf16 rows,
//       fp32 product, re-rounded per chunk), every Qt_c stored by TMA;
//   (L) c = 0 .. b-1, with D = dout . out - dlse per row (bwd_rowdot_kernel):
//         S  = Qt_c Kh_c^T,  dP = dout V_c^T,  P = 2^(S scale log2e - lse log2e)
//         dl = scale P (dP - D)                     (bf16 tile)
//         dA_c += Qt_c^T G  (c >= 1),  G <- G Pm_c^T + dl Kh_c  (G = 0 before c = 0)
//       and dQh_b = G.  dA's sum over query chunks is a vector fp32
//       reduction into HBM (the pages remark that the backward pays for
//       atomic accumulation; this is where it does).
// Six 128 x 128 x 128 MMAs per (b, c) pair: S, dP, dA, G Pm^T, dl Kh and the
// chain product of (R).
//
// bwd_kv_tc_kernel, one key chunk c per job: for every later query chunk b it
// reloads the stored Qt_c (of that b) and dout_b, recomputes S, dP, P and dl
// as above, and accumulates dV_c = sum_b P^T dout_b and dKh_c = sum_b dl^T
// Qt_c in TMEM, written once at the end (four MMAs per pair, no reductions).
//
// One thread issues TMA and MMAs; 256 threads run the epilogues (thread =
// TMEM lane / tile row, half of the columns).  Persistent CTAs, jobs in
// decreasing order of work.  Every wait is bounded; on timeout a kernel sets
// the device error flag and stops.
//
// Query-side shared memory: seven 32 KB bf16 tiles (dout_b, Qt, Kh_c, V_c,
// Pm_c, dl, G).  TMEM columns: [0,128) S, [128,256) dP, [256,384) G,
// [384,512) the chain product U then dA.  The loads of step c are issued as
// soon as step c-1's MMAs are done, and step c's S and dP MMAs at the end of
// step c-1's epilogue.
//
// PaTH-FoX (kFox): the logit gains F_i - F_j (F the inclusive prefix of log f),
// split as in the forward scan into a per-row term and a chunk-relative column
// term; dF gets exact row sums of dlogit on the query side and column sums on
// the key side.

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kTile = kC * kC * 2;
constexpr int kThreadsB = 256;
constexpr uint32_t kColS = 0, kColDP = 128, kColG = 256, kColU = 384;
constexpr float kLog2e = 1.4426950408889634f;
enum { kDO = 0, kQt, kKh, kVP, kPm, kDL, kGs, kSlots };  // kVP: V (the key side's P slot)

struct BBars {
    uint64_t tma, mma;
    uint32_t tmem_base;
    int ok;
    float rD[kC];    // dout . out - dlse
    float rL[kC];    // lse * log2e (PaTH-FoX: less the row's bias term)
    float fcol[kC];  // PaTH-FoX: (F_j - F_ref) * log2e of the current key chunk
};
constexpr int kSmemB = (int)sizeof(BBars) + 1023 + kSlots * kTile;
static_assert(kSmemB <= 232448, "shared memory budget exceeded");

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool kFox>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_scan_tc_kernel(const __grid_constant__ BwdTcMaps maps, BwdTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    BBars &bars = *reinterpret_cast<BBars *>(smem_raw);
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(BBars) + 1023) &
        ~static_cast<uintptr_t>(1023));
    const uint32_t s0 = smem_u32(tiles);
    auto slot = [&](int s) { return s0 + (uint32_t)(s * kTile); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int T = (a.N - 1) * a.BH;
    const float sl2 = a.scale * kLog2e;

    if (tid == 0) {
        mbar_init(&bars.tma, 1);
        mbar_init(&bars.mma, 1);
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
    uint32_t ph_tma = 0, ph_mma = 0;

    // Thread 0 waits for the MMAs issued so far; the result is shared by the block.
    auto mma_sync = [&]() {
        if (tid == 0) {
            tc::mma_commit(&bars.mma);
            if (!mbar_wait(&bars.mma, ph_mma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
        }
        ph_mma ^= 1;
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        return bars.ok != 0;
    };
    // Thread 0 waits for the TMA loads issued against `bytes`; shared result.
    auto tma_sync = [&]() {
        if (tid == 0) {
            if (!mbar_wait(&bars.tma, ph_tma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
            tc::fence_after_sync();
        }
        ph_tma ^= 1;
        __syncthreads();
        return bars.ok != 0;
    };
    auto load_tile = [&](int s, const CUtensorMap *map, int y, int z) {
        tc::tma_load_3d(tiles + s * kTile, map, 0, y, z, &bars.tma);
        tc::tma_load_3d(tiles + s * kTile + kTile / 2, map, 64, y, z, &bars.tma);
    };
    // 64 fp32 TMEM values (this thread's row, columns half*64 ..) -> bf16 tile row
    auto store_row = [&](uint32_t tile, const uint32_t (&v)[64]) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            tc::sts128(tile + tc::swz_off(r, half * 8 + q, kC),
                       tc::pack2(__uint_as_float(v[q * 8 + 0]), __uint_as_float(v[q * 8 + 1])),
                       tc::pack2(__uint_as_float(v[q * 8 + 2]), __uint_as_float(v[q * 8 + 3])),
                       tc::pack2(__uint_as_float(v[q * 8 + 4]), __uint_as_float(v[q * 8 + 5])),
                       tc::pack2(__uint_as_float(v[q * 8 + 6]), __uint_as_float(v[q * 8 + 7])));
    };
    // 64 fp32 TMEM values added into 64 consecutive floats of global memory
    auto red_row = [&](float *dst, const uint32_t (&v)[64]) {
#pragma unroll
        for (int q = 0; q < 16; ++q)
            tc::red_add_v4(dst + 4 * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
    };

    for (int job = blockIdx.x; job < T && bars.ok; job += gridDim.x) {
        const int b = a.N - 1 - job / a.BH, bh = job % a.BH;  // b >= 1
        const int nq = min(kC, a.L - b * kC);
        const int pair0 = b * (b - 1) / 2;  // first (b, c) pair of this chunk in the head
        const size_t head_rows = (size_t)bh * a.Lp;

        // row constants (D from bwd_rowdot_kernel)
        if (half == 0) {
            bars.rD[r] = a.Dg[head_rows + (size_t)b * kC + r];
            bars.rL[r] = r < nq ? a.lse[(size_t)bh * a.L + (size_t)b * kC + r] * kLog2e : 0.f;
        }
        // PaTH-FoX: the row's prefix (log2 units) and its dF row sum
        const float fi2 = kFox ? a.F[head_rows + (size_t)b * kC + r] * kLog2e : 0.f;
        float frow = 0.f;
        // (R) dout_b and Qh_b, then the chain
        if (tid == 0) {
            mbar_arrive_expect_tx(&bars.tma, 2 * kTile);
            load_tile(kDO, &maps.dout, b * kC, bh);
            load_tile(kQt, &maps.qh, b * kC, bh);
        }
        if (!tma_sync()) break;
        bool ok = true;
        for (int c = b - 1; c >= 0; --c) {
            if (tid == 0) {
                tc::tma_store_3d(&maps.qts, tiles + kQt * kTile, 0, (pair0 + c) * kC, bh);
                tc::tma_store_3d(&maps.qts, tiles + kQt * kTile + kTile / 2, 64, (pair0 + c) * kC, bh);
                tc::bulk_commit();
            }
            if (c == 0) break;
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars.tma, kTile);
                load_tile(kPm, &maps.pm, c * kC, bh);
            }
            if (!(ok = tma_sync())) break;
            if (tid == 0)
                tc::gemm128_lo<true>(tmem + kColU, tc::desc_lo(slot(kQt), false),
                                     tc::desc_lo(slot(kPm), true), false);
            if (tid == 0) tc::bulk_wait_read();  // the store of Qt_c has read the tile
            if (!(ok = mma_sync())) break;
            {
                uint32_t v[64];
                tc::tmem_ld64(tmem + lane_off + kColU + half * 64, v);
                store_row(slot(kQt), v);
            }
            tc::fence_proxy_async();
            __syncthreads();
        }
        if (!ok) break;
        if (tid == 0) {
            tc::bulk_wait();  // every Qt_c is in HBM before it is loaded back
            tc::fence_proxy_async_global();
        }
        __syncthreads();

        // (L)
        // the loads of step c are issued as soon as step c-1's MMAs are done,
        // so that they overlap its epilogue
        auto issue_loads = [&](int c) {
            const int k0 = c * kC;
            // Qt_0 is still in its tile from the end of (R)
            mbar_arrive_expect_tx(&bars.tma, (c > 0 ? 4 : 2) * kTile);
            if (c > 0) load_tile(kQt, &maps.qts, (pair0 + c) * kC, bh);
            load_tile(kKh, &maps.kh, k0, bh);
            load_tile(kVP, &maps.v, k0, bh);
            if (c > 0) load_tile(kPm, &maps.pm, k0, bh);
            if (c + 1 < b) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    tc::tma_prefetch_3d(&maps.qts, 64 * x, (pair0 + c + 1) * kC, bh);
                    tc::tma_prefetch_3d(&maps.kh, 64 * x, k0 + kC, bh);
                    tc::tma_prefetch_3d(&maps.v, 64 * x, k0 + kC, bh);
                    tc::tma_prefetch_3d(&maps.pm, 64 * x, k0 + kC, bh);
                }
            }
        };
        // S and dP of step c: issued by thread 0 once the step's tiles have
        // landed, for c > 0 at the end of step c-1's epilogue (their TMEM
        // columns are free once step c-1's first epilogue has read them)
        auto issue_s_dp = [&]() {
            if (!mbar_wait(&bars.tma, ph_tma, a.err, nullptr, kWaitLimitNs)) {
                bars.ok = 0;
                return;
            }
            tc::fence_after_sync();
            tc::gemm128_lo<false>(tmem + kColS, tc::desc_lo(slot(kQt), false),
                                  tc::desc_lo(slot(kKh), false), false);  // S = Qt Kh^T
            tc::gemm128_lo<false>(tmem + kColDP, tc::desc_lo(slot(kDO), false),
                                  tc::desc_lo(slot(kVP), false), false);  // dP = dout V^T
        };
        if (tid == 0) {
            issue_loads(0);
            issue_s_dp();
        }
        for (int c = 0; c < b; ++c) {
            ph_tma ^= 1;  // the wait on step c's tiles was done in issue_s_dp
            if (kFox && half == 0)
                bars.fcol[r] = (a.F[head_rows + (size_t)c * kC + r] - a.F[head_rows + (size_t)c * kC]) *
                               kLog2e;
            if (!(ok = mma_sync())) break;
            // dl (scaled) as a bf16 tile
            {
                uint32_t sv[64], pv[64];
                tc::tmem_ld64(tmem + lane_off + kColS + half * 64, sv);
                tc::tmem_ld64(tmem + lane_off + kColDP + half * 64, pv);
                // FoX: logit (log2) = S scale log2e - fcol[j] + (fi2 - fref2) with
                // fref2 = F_ref log2e; folded into the row offset below
                const float lr = bars.rL[r] -
                                 (kFox ? fi2 - a.F[head_rows + (size_t)c * kC] * kLog2e : 0.f);
                const float dr = bars.rD[r];
                const bool live = r < nq;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float p[8], g[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x = __uint_as_float(sv[q * 8 + e]);
                        const float fb = kFox ? bars.fcol[half * 64 + q * 8 + e] : 0.f;
                        p[e] = live ? ex2(fmaf(x, sl2, -lr - fb)) : 0.f;
                        const float gu = p[e] * (__uint_as_float(pv[q * 8 + e]) - dr);
                        if (kFox) frow += gu;
                        g[e] = a.scale * gu;
                    }
                    const uint32_t off = tc::swz_off(r, half * 8 + q, kC);
                    tc::sts128(slot(kDL) + off, tc::pack2(g[0], g[1]), tc::pack2(g[2], g[3]),
                               tc::pack2(g[4], g[5]), tc::pack2(g[6], g[7]));
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                if (c > 0) {
                    // dA = Qt^T G, then G <- G Pm^T
                    tc::gemm128_lo2<true, true>(tmem + kColU, tc::desc_lo(slot(kQt), true),
                                                tc::desc_lo(slot(kGs), true), false);
                    tc::gemm128_lo<false>(tmem + kColG, tc::desc_lo(slot(kGs), false),
                                          tc::desc_lo(slot(kPm), false), false);
                }
                // G += dl Kh
                tc::gemm128_lo<true>(tmem + kColG, tc::desc_lo(slot(kDL), false),
                                     tc::desc_lo(slot(kKh), true), c > 0);
            }
            if (!(ok = mma_sync())) break;
            if (tid == 0 && c + 1 < b) issue_loads(c + 1);  // every reader of the tiles is done
            {
                uint32_t v[64];
                if (c > 0) {
                    tc::tmem_ld64(tmem + lane_off + kColU + half * 64, v);
                    red_row(a.dA + (((size_t)bh * a.N + c) * kC + r) * kC + half * 64, v);
                }
                tc::tmem_ld64(tmem + lane_off + kColG + half * 64, v);
                store_row(slot(kGs), v);
            }
            if (tid == 0 && c + 1 < b) issue_s_dp();
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
        }
        if (!ok) break;
        if (kFox && r < nq) atomicAdd(a.dF + head_rows + (size_t)b * kC + r, frow);
        // dQh_b = G (fp32)
        {
            uint32_t v[64];
            tc::tmem_ld64(tmem + lane_off + kColG + half * 64, v);
            float4 *dst = reinterpret_cast<float4 *>(a.dQh + (head_rows + (size_t)b * kC + r) * kC +
                                                     half * 64);
#pragma unroll
            for (int q = 0; q < 16; ++q)
                dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (tid == 0) tc::bulk_wait();  // no store may outlive the CTA's shared memory
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Key side: dV_c and dKh_c of key chunk c from every later query chunk.
// Shared memory: six 32 KB tiles (Kh_c, V_c resident; Qt_c of b, dout_b, P,
// dl per step).  TMEM columns: [0,128) S, [128,256) dP, [256,384) dV,
// [384,512) dKh.
enum { kvKh = 0, kvV, kvQt, kvDO, kvP, kvDL, kvSlots };
constexpr int kSmemKV = (int)sizeof(BBars) + 1023 + kvSlots * kTile;
static_assert(kSmemKV <= 232448, "shared memory budget exceeded");
constexpr uint32_t kColDV = 256, kColDK = 384;

template <bool kFox>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_kv_tc_kernel(const __grid_constant__ BwdTcMaps maps, BwdTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    BBars &bars = *reinterpret_cast<BBars *>(smem_raw);
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(BBars) + 1023) &
        ~static_cast<uintptr_t>(1023));
    const uint32_t s0 = smem_u32(tiles);
    auto slot = [&](int s) { return s0 + (uint32_t)(s * kTile); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int T = (a.N - 1) * a.BH;
    const float sl2 = a.scale * kLog2e;

    if (tid == 0) {
        mbar_init(&bars.tma, 1);
        mbar_init(&bars.mma, 1);
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
    uint32_t ph_tma = 0, ph_mma = 0;
    auto mma_sync = [&]() {
        if (tid == 0) {
            tc::mma_commit(&bars.mma);
            if (!mbar_wait(&bars.mma, ph_mma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
        }
        ph_mma ^= 1;
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        return bars.ok != 0;
    };
    auto tma_sync = [&]() {
        if (tid == 0) {
            if (!mbar_wait(&bars.tma, ph_tma, a.err, nullptr, kWaitLimitNs)) bars.ok = 0;
            tc::fence_after_sync();
        }
        ph_tma ^= 1;
        __syncthreads();
        return bars.ok != 0;
    };
    auto load_tile = [&](int s, const CUtensorMap *map, int y, int z) {
        tc::tma_load_3d(tiles + s * kTile, map, 0, y, z, &bars.tma);
        tc::tma_load_3d(tiles + s * kTile + kTile / 2, map, 64, y, z, &bars.tma);
    };

    for (int job = blockIdx.x; job < T && bars.ok; job += gridDim.x) {
        const int c = job / a.BH, bh = job % a.BH;  // c <= N - 2, heaviest first
        const int k0 = c * kC;
        const size_t head_rows = (size_t)bh * a.Lp;
        bool ok = true;
        // PaTH-FoX: the key chunk's relative prefixes (fixed for the job) and
        // this thread's column sum of dlogit (column tid % 128, rows of its half)
        const float fref2 = kFox ? a.F[head_rows + k0] * kLog2e : 0.f;
        if (kFox && half == 0) bars.fcol[r] = a.F[head_rows + k0 + r] * kLog2e - fref2;
        float fcolsum = 0.f;
        for (int b = c + 1; b < a.N; ++b) {
            const int nq = min(kC, a.L - b * kC);
            if (half == 0) {
                const size_t row = head_rows + (size_t)b * kC + r;
                bars.rD[r] = a.Dg[row];
                float l = r < nq ? a.lse[(size_t)bh * a.L + (size_t)b * kC + r] * kLog2e : 0.f;
                if (kFox) l -= a.F[row] * kLog2e - fref2;
                bars.rL[r] = l;
            }
            if (tid == 0) {
                mbar_arrive_expect_tx(&bars.tma, (b == c + 1 ? 4 : 2) * kTile);
                if (b == c + 1) {
                    load_tile(kvKh, &maps.kh, k0, bh);
                    load_tile(kvV, &maps.v, k0, bh);
                }
                load_tile(kvQt, &maps.qts, (b * (b - 1) / 2 + c) * kC, bh);
                load_tile(kvDO, &maps.dout, b * kC, bh);
                if (b + 1 < a.N) {
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        tc::tma_prefetch_3d(&maps.qts, 64 * x, ((b + 1) * b / 2 + c) * kC, bh);
                        tc::tma_prefetch_3d(&maps.dout, 64 * x, (b + 1) * kC, bh);
                    }
                }
            }
            if (!(ok = tma_sync())) break;
            if (tid == 0) {
                tc::gemm128_lo<false>(tmem + kColS, tc::desc_lo(slot(kvQt), false),
                                      tc::desc_lo(slot(kvKh), false), false);  // S = Qt Kh^T
                tc::gemm128_lo<false>(tmem + kColDP, tc::desc_lo(slot(kvDO), false),
                                      tc::desc_lo(slot(kvV), false), false);   // dP = dout V^T
            }
            if (!(ok = mma_sync())) break;
            {
                uint32_t sv[64], pv[64];
                tc::tmem_ld64(tmem + lane_off + kColS + half * 64, sv);
                tc::tmem_ld64(tmem + lane_off + kColDP + half * 64, pv);
                const float lr = bars.rL[r], dr = bars.rD[r];
                const bool live = r < nq;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float p[8], g[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x = __uint_as_float(sv[q * 8 + e]);
                        const float fb = kFox ? bars.fcol[half * 64 + q * 8 + e] : 0.f;
                        p[e] = live ? ex2(fmaf(x, sl2, -lr - fb)) : 0.f;
                        g[e] = a.scale * p[e] * (__uint_as_float(pv[q * 8 + e]) - dr);
                    }
                    const uint32_t off = tc::swz_off(r, half * 8 + q, kC);
                    tc::sts128(slot(kvP) + off, tc::pack2(p[0], p[1]), tc::pack2(p[2], p[3]),
                               tc::pack2(p[4], p[5]), tc::pack2(p[6], p[7]));
                    tc::sts128(slot(kvDL) + off, tc::pack2(g[0], g[1]), tc::pack2(g[2], g[3]),
                               tc::pack2(g[4], g[5]), tc::pack2(g[6], g[7]));
                }
            }
            tc::fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                // dV += P^T dout, dKh += dl^T Qt
                tc::gemm128_lo2<true, true>(tmem + kColDV, tc::desc_lo(slot(kvP), true),
                                            tc::desc_lo(slot(kvDO), true), b > c + 1);
                tc::gemm128_lo2<true, true>(tmem + kColDK, tc::desc_lo(slot(kvDL), true),
                                            tc::desc_lo(slot(kvQt), true), b > c + 1);
            }
            if (!(ok = mma_sync())) break;
            if (kFox) {
                // column tid % 128 of scale * dlogit, rows of this thread's half
                const int j = tid & (kC - 1), r0 = (tid >> 7) * 64;
                const uint8_t *dl = tiles + kvDL * kTile;
                float cs = 0.f;
#pragma unroll 8
                for (int rr = r0; rr < r0 + 64; ++rr) {
                    const uint32_t off = tc::swz_off(rr, j >> 3, kC) + (uint32_t)((j & 7) * 2);
                    cs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(dl + off));
                }
                fcolsum += cs;
            }
        }
        if (!ok) break;
        if (kFox) atomicAdd(a.dF + head_rows + k0 + (tid & (kC - 1)), -fcolsum / a.scale);
        {
            uint32_t v[64];
            const size_t krow = (head_rows + k0 + r) * kC + half * 64;
#pragma unroll 1
            for (int w = 0; w < 2; ++w) {
                tc::tmem_ld64(tmem + lane_off + (w ? kColDK : kColDV) + half * 64, v);
                float4 *dst = reinterpret_cast<float4 *>((w ? a.dKh : a.dV) + krow);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                         __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_bwd_kv_tc(const BwdTcMaps &maps, const BwdTcArgs &a, int num_sms,
                             cudaStream_t st) {
    const int total = (a.N - 1) * a.BH;
    if (total <= 0) return cudaSuccess;
    const int grid = total < num_sms ? total : num_sms;
    void (*kern)(const BwdTcMaps, BwdTcArgs) =
        a.F ? bwd_kv_tc_kernel<true> : bwd_kv_tc_kernel<false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemKV);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsB, kSmemKV, st>>>(maps, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_scan_tc(const BwdTcMaps &maps, const BwdTcArgs &a, int num_sms,
                               cudaStream_t st) {
    const int total = (a.N - 1) * a.BH;
    if (total <= 0) return cudaSuccess;
    const int grid = total < num_sms ? total : num_sms;
    void (*kern)(const BwdTcMaps, BwdTcArgs) =
        a.F ? bwd_scan_tc_kernel<true> : bwd_scan_tc_kernel<false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemB);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsB, kSmemB, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace path
