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
// Roles.  Warp 8 issues every TMA copy and MMA: a tcgen05.mma stalls its
// issuing thread for about as long as the product runs, so no warp that does
// CUDA-core work issues one.  Warps 0-7 (the "compute" warps) stage G, solve
// for T and run every epilogue; they wait on the MMA commits (one mbarrier per
// product group) and hand each operand tile to warp 8 through an mbarrier
// that every compute warp (or each half) arrives on.  Per chunk:
//   G (early: issued for the next chunk while this one finishes)
//   P2 G -> fp32 smem (region Ra)             | QW -> B, KW -> C, QK -> D
//   P3 solve T (fp32, region Rb)              |   (run during the solve)
//   P4 T -> bf16, -(M_le*QW) -> bf16  (rdy4a) | Wt = T W -> A
//      (M_gt*KW) -> bf16              (rdy4b) | Y = KWm T^T -> C
//   P6 Wt -> bf16 (half 0, rdy6a),            | -(M_le*QW) Wt -> B       (b1)
//      Y -> bf16 (half 1, rdy6b)              | Y W -> A (b2), W^T Wt -> C (b3),
//                                             | += -(M_le*QW) Y^T -> D   (b4);
//                                             | V over the T tile
//   P8 Qh (half 0, after b1), Kh (half 1,     | Qh, Kh, Pm stored by TMA
//      after b2), Pm (after b3)       (rdy8)  |
//   P9 causal softmax of Sd -> P      (rdy9)  | P V -> C; then the next chunk's
//                                             | W, Q, K over the stored tiles
//   P10 own-chunk output and LSE      (rdy10) | output stored; next G
// The two 64 KB staging regions swap roles every chunk: Ra holds G (fp32),
// then the T / -(M_le*QW) / V / P / output tiles, Rb holds T (fp32), then the
// KWm / Y / Wt tiles and the softmax scratch.  So the next chunk's G staging
// never waits for this chunk's output store, only its solve does.

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "ut_solve_tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kTile = kC * kC * 2;  // bf16 128 x 128 operand tile
constexpr int kCompute = 256;       // warps 0-7
// warps 8-11: one warpgroup, so that registers can be moved to the compute
// warps (setmaxnreg works per warpgroup); warp 8 issues, 9-11 idle
constexpr int kThreadsP = kCompute + 128;
// launched at 65536 / 384 = 168 registers a thread; 2 x 128 x 224 + 128 x 56
// = 64512 = 384 x 168, so the increase never waits on registers that are not
// released
constexpr int kRegCompute = 224, kRegIssuer = 56;
static_assert(2 * 128 * kRegCompute + 128 * kRegIssuer <= kThreadsP * 168, "register split");
constexpr int kOffQ = 0, kOffK = kTile, kOffW = 2 * kTile;
constexpr int kOffR1 = 3 * kTile;   // the two staging regions (Ra / Rb by chunk parity)
constexpr int kRBytes = 64 * 1024;
constexpr int kOffR2 = kOffR1 + kRBytes;
constexpr int kOffBar = kOffR2 + kRBytes;
constexpr int kBarBytes = 1280;
constexpr int kSmemP = kOffBar + kBarBytes + 1024;
static_assert(kC * kC * 4 <= kRBytes, "G staging does not fit");
static_assert(kSmemP <= 232448, "shared memory budget exceeded");
static_assert(utc::kThr == kCompute, "the solve runs on the compute warps");
constexpr uint32_t kColA = 0, kColB = 128, kColC = 256, kColD = 384;
// named barrier 1 (all compute warps) is also the solve's
constexpr int kBarAll = 1;

struct PBars {
    // TMA arrivals
    uint64_t tma_w, tma_qk, vbar;
    // MMA completions (warp 8 commits, compute warps wait)
    uint64_t g_done, qkw_done, wt_done, y_done, b1, b2, b3, b4, pv_done, drain;
    // tiles written by the compute warps (warp 8 waits)
    uint64_t rdy4a, rdy4b, rdy6a, rdy6b, rdy8, rdy9, rdy10;
    // warp 8 -> compute warps: the finished chunk's Ra region has been read by
    // its output stores
    uint64_t xfree;
    uint32_t tmem_base;
    int abort_word;
    alignas(16) float beta[kC];
    float fsm[kC];  // PaTH-FoX: the chunk's prefix sums relative to its first, log2 units
};
static_assert(sizeof(PBars) <= kBarBytes, "barrier block too large");

using tc::group_all;
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

// Hands tiles this warp wrote (generic proxy) and TMEM it read to the MMA /
// TMA issuer: every lane orders its own accesses, then one lane arrives.
__device__ __forceinline__ void warp_release(uint64_t *bar, int lane) {
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// A shared address the compiler cannot hoist out of a loop: the issuer forms
// each MMA's descriptors at the product, instead of keeping dozens of
// loop-invariant 64-bit descriptors live (and spilled).
__device__ __forceinline__ uint32_t opaque(uint32_t x) {
    uint32_t y;
    asm volatile("mov.b32 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D (+)= A B over one 128 x 128 x 128 product, as gemm_128x128x128, with
// operand bases formed at the call.
__device__ __forceinline__ void gemm(uint32_t d, uint32_t a_base, uint32_t b_base, bool b_mn,
                                     bool accumulate) {
    tc::gemm_128x128x128(d, opaque(a_base), opaque(b_base), b_mn, accumulate);
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
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = a.nloc * a.BH;
    volatile int *abort_word = &bars.abort_word;
    constexpr uint64_t lim = kWaitLimitNs;
    // a scan launched behind this grid may take each SM this grid leaves;
    // it waits on the per-head counters (a.ready) before reading any output
    launch_dependents();

    if (tid == 0) {
        uint64_t *one[] = {&bars.tma_w, &bars.tma_qk, &bars.vbar, &bars.g_done, &bars.qkw_done,
                           &bars.wt_done, &bars.y_done, &bars.b1, &bars.b2, &bars.b3, &bars.b4,
                           &bars.pv_done, &bars.drain};
        for (uint64_t *p : one) mbar_init(p, 1);
        // compute -> issuer: one arrival per compute warp (or per warp of a half)
        mbar_init(&bars.rdy4a, 8);
        mbar_init(&bars.rdy4b, 8);
        mbar_init(&bars.rdy6a, 4);
        mbar_init(&bars.rdy6b, 4);
        mbar_init(&bars.rdy8, 8);
        mbar_init(&bars.rdy9, 8);
        mbar_init(&bars.rdy10, 8);
        mbar_init(&bars.xfree, 1);
        bars.abort_word = 0;
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

    if (warp >= 8) {
        // ============================================================ issuer
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegIssuer) : "memory");
        if (warp == 8 && lane == 0) {
            bool ok = true;
            // outstanding loads (parity of the phase still to land, or -1),
            // waited for before the CTA exits after an abort
            int pend_w = -1, pend_qk = -1, pend_v = -1;
            // the head of the previous chunk, counted in a.ready once its
            // stores are complete (checked a chunk later, when they long are)
            int done_bh = -1;
            auto publish = [&](int bh) {
                tc::fence_proxy_async_global();
                counter_release_add(a.ready + bh, 1);
            };
            auto wait = [&](uint64_t *bar, uint32_t ph) {
                ok = ok && mbar_wait(bar, ph, a.err, abort_word, lim);
                if (ok) tc::fence_after_sync();
                return ok;
            };
            // W, Q and K of a chunk (inputs and outputs are addressed by
            // local row: local chunk i at row 128 i)
            auto issue_loads = [&](int job, int it) {
                const int bh = job / a.nloc, c0 = (job % a.nloc) * kC;
                mbar_arrive_expect_tx(&bars.tma_w, kTile);
                tc::tma_load_3d(smem + kOffW, &maps.w, 0, c0, bh, &bars.tma_w);
                tc::tma_load_3d(smem + kOffW + kTile / 2, &maps.w, 64, c0, bh, &bars.tma_w);
                mbar_arrive_expect_tx(&bars.tma_qk, 2 * kTile);
                tc::tma_load_3d(smem + kOffQ, &maps.q, 0, c0, bh, &bars.tma_qk);
                tc::tma_load_3d(smem + kOffQ + kTile / 2, &maps.q, 64, c0, bh, &bars.tma_qk);
                tc::tma_load_3d(smem + kOffK, &maps.k, 0, c0, bh, &bars.tma_qk);
                tc::tma_load_3d(smem + kOffK + kTile / 2, &maps.k, 64, c0, bh, &bars.tma_qk);
                pend_w = pend_qk = it & 1;
            };
            issue_loads(blockIdx.x, 0);
            if (wait(&bars.tma_w, 0)) {
                pend_w = -1;
                gemm(tmem + kColA, sW, sW, false, false);  // G
                tc::mma_commit(&bars.g_done);
            }
            int it = 0;
            for (int job = blockIdx.x; job < total && ok; job += gridDim.x, ++it) {
                const uint32_t ph = it & 1;
                const int bh = job / a.nloc, r0 = (job % a.nloc) * kC;
                const int next = job + gridDim.x;
                const uint32_t sRa = smem_u32(smem + (ph ? kOffR2 : kOffR1));
                const uint32_t sRb = smem_u32(smem + (ph ? kOffR1 : kOffR2));
                const uint32_t sT = sRa, sQm = sRa + kTile;   // T | -(M_le*QW); V | P, output
                const uint32_t sY = sRb, sWt = sRb + kTile;   // KWm, then Y | Wt
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
                // QW -> B, KW -> C, QK -> D: B, C, D were last read by the
                // previous chunk's epilogues (rdy10, waited below)
                if (!wait(&bars.tma_qk, ph)) break;
                pend_qk = -1;
                gemm(tmem + kColB, sQ, sW, false, false);  // Q W^T
                gemm(tmem + kColC, sK, sW, false, false);  // K W^T
                gemm(tmem + kColD, sQ, sK, false, false);  // Q K^T
                tc::mma_commit(&bars.qkw_done);
                // Wt = T W -> A (G in A was read in P2)
                if (!wait(&bars.rdy4a, ph)) break;
                gemm(tmem + kColA, sT, sW, true, false);
                tc::mma_commit(&bars.wt_done);
                // Y = KWm T^T -> C (KW in C was read in P4)
                if (!wait(&bars.rdy4b, ph)) break;
                gemm(tmem + kColC, sY, sT, false, false);
                tc::mma_commit(&bars.y_done);
                // -(M_le*QW) Wt -> B
                if (!wait(&bars.rdy6a, ph)) break;
                gemm(tmem + kColB, sQm, sWt, true, false);
                tc::mma_commit(&bars.b1);
                // Y W -> A, W^T Wt -> C, QK^T - (M_le*QW) Y^T -> D
                if (!wait(&bars.rdy6b, ph)) break;
                gemm(tmem + kColA, sY, sW, true, false);
                tc::mma_commit(&bars.b2);
                // W^T Wt, or its transpose Wt^T W when the chunk product is
                // wanted as Pm^T (rows = output dimension), the K-major layout
                // the scan's fused carried-query/logit product reads
                if (a.pm_transposed)
                    tc::gemm128_lo2<true, true>(tmem + kColC, tc::desc_lo(opaque(sWt), true),
                                                tc::desc_lo(opaque(sW), true), false);
                else
                    tc::gemm128_lo2<true, true>(tmem + kColC, tc::desc_lo(opaque(sW), true),
                                                tc::desc_lo(opaque(sWt), true), false);
                tc::mma_commit(&bars.b3);
                gemm(tmem + kColD, sQm, sY, false, true);
                tc::mma_commit(&bars.b4);
                // the chunk's values, for its own attention block, over the T tile
                // (free once Y = KWm T^T is complete; loaded after b1-b4 so that
                // this wait does not hold them up)
                if (!wait(&bars.y_done, ph)) break;
                mbar_arrive_expect_tx(&bars.vbar, kTile);
                tc::tma_load_3d(smem + (ph ? kOffR2 : kOffR1), &maps.v, 0, r0, bh, &bars.vbar);
                tc::tma_load_3d(smem + (ph ? kOffR2 : kOffR1) + kTile / 2, &maps.v, 64, r0, bh,
                                &bars.vbar);
                pend_v = ph;
                // Qh, Kh, Pm -> global; then the next chunk's W, Q, K over them
                if (!wait(&bars.rdy8, ph)) break;
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    tc::tma_store_3d(&maps.qh, smem + kOffQ + x * (kTile / 2), 64 * x, r0, bh);
                    tc::tma_store_3d(&maps.kh, smem + kOffK + x * (kTile / 2), 64 * x, r0, bh);
                    tc::tma_store_3d(&maps.pm, smem + kOffW + x * (kTile / 2), 64 * x, r0, bh);
                }
                tc::bulk_commit();
                if (!wait(&bars.vbar, ph)) break;
                pend_v = -1;
                if (a.copy_v) {
                    // sharded prefill: the chunk's V tile for the exchange
                    // with the other ranks
#pragma unroll
                    for (int x = 0; x < 2; ++x)
                        tc::tma_store_3d(&maps.vx, smem + (ph ? kOffR2 : kOffR1) + x * (kTile / 2),
                                         64 * x, r0, bh);
                    tc::bulk_commit();
                }
                // P V -> C (Pm in C was read in P8), ahead of the wait for the
                // stores above to read their tiles, which takes a while
                if (!wait(&bars.rdy9, ph)) break;
                gemm(tmem + kColC, sQm, sT, true, false);
                tc::mma_commit(&bars.pv_done);
                // the next chunk's W, Q, K over the stored tiles, then its G -> A
                // (Kh's YW in A was read in P8)
                if (next < total) {
                    tc::bulk_wait_read();
                    issue_loads(next, it + 1);
                    if (!wait(&bars.tma_w, ph ^ 1)) break;
                    pend_w = -1;
                    gemm(tmem + kColA, sW, sW, false, false);
                    tc::mma_commit(&bars.g_done);
                }
                // the chunk's own attention output -> global; Ra is free once read
                if (!wait(&bars.rdy10, ph)) break;
#pragma unroll
                for (int x = 0; x < 2; ++x)
                    tc::tma_store_3d(&maps.od, smem + (ph ? kOffR2 : kOffR1) + kTile + x * (kTile / 2),
                                     64 * x, r0, bh);
                tc::bulk_commit();
                tc::bulk_wait_read();
                mbar_arrive(&bars.xfree);
                if (a.ready) {
                    // every group but this chunk's (Qh/Kh/Pm, V copy, OD) is
                    // complete: the previous chunk is in global memory
                    if (done_bh >= 0) {
                        if (a.copy_v)
                            tc::bulk_wait_all_but<3>();
                        else
                            tc::bulk_wait_all_but<2>();
                        publish(done_bh);
                    }
                    done_bh = bh;
                }
            }
            if (!ok) {
                // let every copy this thread issued land before the CTA exits
                if (pend_w >= 0) mbar_wait(&bars.tma_w, pend_w, a.err, nullptr, lim);
                if (pend_qk >= 0) mbar_wait(&bars.tma_qk, pend_qk, a.err, nullptr, lim);
                if (pend_v >= 0) mbar_wait(&bars.vbar, pend_v, a.err, nullptr, lim);
            }
            // every MMA this thread issued has completed before TMEM is
            // released, and no store outlives the CTA's shared memory
            tc::mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, a.err, nullptr, lim);
            tc::bulk_wait();
            if (a.ready && ok && done_bh >= 0) publish(done_bh);
        }
        __syncwarp();
    } else {
        // ============================================================ compute
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegCompute) : "memory");
        const int quad = warp & 3, half = warp >> 2;
        const int r = quad * 32 + lane;  // TMEM lane / tile row of this thread
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const float sl2 = a.scale * 1.4426950408889634f;
        float *bsm = bars.beta;
        bool ok = true;
        auto wait = [&](uint64_t *bar, uint32_t ph) {
            ok = ok && mbar_wait(bar, ph, a.err, abort_word, lim);
            __syncwarp();
            tc::fence_after_sync();
        };
        int it = 0;
        for (int job = blockIdx.x; job < total; job += gridDim.x, ++it) {
            const uint32_t ph = it & 1;
            const int bh = job / a.nloc, li = job % a.nloc;
            const int chunk = a.cm.global_of_local(li);
            const int c0 = chunk * kC;  // first row of the chunk in the whole sequence
            const int r0 = li * kC;     // its first row in the local inputs and outputs
            const int n = min(kC, a.L - c0);
            uint8_t *Ra = smem + (ph ? kOffR2 : kOffR1), *Rb = smem + (ph ? kOffR1 : kOffR2);
            float *Gf = reinterpret_cast<float *>(Ra);
            float *Tf = reinterpret_cast<float *>(Rb);
            const uint32_t sT = smem_u32(Ra), sQm = sT + kTile;
            const uint32_t sY = smem_u32(Rb), sWt = sY + kTile;
            // beta of the chunk and (PaTH-FoX) its prefix sums relative to its
            // first (the bias F_i - F_j is unchanged), read ahead of their use
            const float beta_r = (tid < kC && tid < n) ? a.beta[(size_t)bh * a.Lin + r0 + tid] : 0.f;
            const float f_r = (a.F && tid < kC)
                                  ? (a.F[(size_t)bh * a.Lp + c0 + tid] - a.F[(size_t)bh * a.Lp + c0]) *
                                        1.4426950408889634f
                                  : 0.f;
            // ------------------------------------------------------------ P2
            wait(&bars.g_done, ph);
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
            // Rb held the previous chunk's V and output tiles until their stores read them
            if (it > 0) wait(&bars.xfree, ph ^ 1);
            if (!group_all(kBarAll, kCompute, ok)) break;
            // ------------------------------------------------------------ P3
            // T = (I + strict_lower(diag(beta) G))^{-1} diag(beta) into Tf (fp32)
            ut_solve(Gf, Tf, bsm, tid);
            // ------------------------------------------------------------ P4
            // T fp32 -> bf16 tile and -(M_le * Q W^T) -> bf16 tile, half a row
            // each.  Stored group pairs (2p, 2p+1) hold the logical pair
            // p ^ (sw_f >> 1), swapped when sw_f is odd; visiting them in an
            // order rotated by the row, and taking the pair's two halves in an
            // order set by bit 2 of the row, spreads a warp's loads over all
            // banks.
            wait(&bars.qkw_done, ph);
            {
                const int f = sw_f(r), hsel = (r >> 2) & 1;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int p = half * 8 + ((i + r) & 7);
                    const float *src = Tf + r * kC + p * 8;
                    float4 y0, y1;
                    if (hsel) {
                        y1 = *reinterpret_cast<const float4 *>(src + 4);
                        y0 = *reinterpret_cast<const float4 *>(src);
                    } else {
                        y0 = *reinterpret_cast<const float4 *>(src);
                        y1 = *reinterpret_cast<const float4 *>(src + 4);
                    }
                    const float4 x0 = (f & 1) ? y1 : y0, x1 = (f & 1) ? y0 : y1;
                    sts128(sT + tc::swz_off(r, p ^ (f >> 1), kC), pack2(x0.x, x0.y),
                           pack2(x0.z, x0.w), pack2(x1.x, x1.y), pack2(x1.z, x1.w));
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t v[32];
                    const int c32 = half * 2 + cc;
                    tc::tmem_ld32(tmem + lane_off + kColB + c32 * 32, v);
                    tile_store32(sQm, r, c32, v, [&](int s, float x) { return s <= r ? -x : 0.f; });
                }
            }
            warp_release(&bars.rdy4a, lane);
            // every read of T fp32 is done before (M_gt * K W^T) goes over it
            if (!group_all(kBarAll, kCompute, ok)) break;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[32];
                const int c32 = half * 2 + cc;
                tc::tmem_ld32(tmem + lane_off + kColC + c32 * 32, v);
                tile_store32(sY, r, c32, v, [&](int s, float x) { return s > r ? x : 0.f; });
            }
            warp_release(&bars.rdy4b, lane);
            // ------------------------------------------------------------ P6
            // Wt (half 0) and Y (half 1) -> bf16 tiles, each as soon as its
            // product completes
            {
                wait(half == 0 ? &bars.wt_done : &bars.y_done, ph);
                const uint32_t src = half == 0 ? kColA : kColC;
                const uint32_t dst = half == 0 ? sWt : sY;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t v[32];
                    tc::tmem_ld32(tmem + lane_off + src + cc * 32, v);
                    tile_store32(dst, r, cc, v, [](int, float x) { return x; });
                }
                warp_release(half == 0 ? &bars.rdy6a : &bars.rdy6b, lane);
            }
            // ------------------------------------------------------------ P8
            // Qh (half 0, after b1) over the Q tile and Kh (half 1, after b2)
            // over the K tile, in place; then Pm (after b3) over the W tile
            {
                wait(half == 0 ? &bars.b1 : &bars.b2, ph);
                wait(&bars.tma_qk, ph);  // the Q and K tiles as the TMA wrote them
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
                wait(&bars.b3, ph);
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
                warp_release(&bars.rdy8, lane);
            }
            // ------------------------------------------------------------ P9
            // causal softmax of the within-chunk logits, rows r, columns
            // half*64 ..; per-row partial max / sum of the two column halves
            // in Rb (its Y / Wt tiles were last read by the b1-b4 products)
            float m_row, l_row;
            {
                float(*red)[2][kC] = reinterpret_cast<float(*)[2][kC]>(Rb);
                const bool fox = a.F != nullptr;
                const float fi = fox ? bars.fsm[r] : 0.f;
                // columns half*64 + 8g .. +7 are above the diagonal for every
                // row of this warp when 64 half + 8 g > 32 quad + 31
                const int ngrp = min(8, max(0, (32 * quad + 32 - 64 * half + 7) / 8));
                wait(&bars.b4, ph);
                uint32_t v[64];
                tc::tmem_ld64(tmem + lane_off + kColD + half * 64, v);
                // eight interleaved partial maxima (exact in any order), so that
                // no chain of 64 dependent max operations sits in the phase
                float mp[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int j = half * 64 + i;
                    float x = __uint_as_float(v[i]) * sl2;
                    if (fox) x += fi - bars.fsm[j];
                    x = (j <= r) ? x : -INFINITY;
                    v[i] = __float_as_uint(x);
                    mp[i & 7] = fmaxf(mp[i & 7], x);
                }
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 8; ++i) mx = fmaxf(mx, mp[i]);
                red[0][half][r] = mx;
                tc::named_bar(kBarAll, kCompute);
                m_row = fmaxf(red[0][0][r], red[0][1][r]);  // finite: column r is unmasked
                float sum = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float p[8];
                    if (q < ngrp) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float x = __uint_as_float(v[q * 8 + e]);
                            float y;
                            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x - m_row));
                            p[e] = (x == -INFINITY) ? 0.f : y;
                            sum += p[e];
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) p[e] = 0.f;
                    }
                    sts128(sQm + tc::swz_off(r, half * 8 + q, kC), pack2(p[0], p[1]),
                           pack2(p[2], p[3]), pack2(p[4], p[5]), pack2(p[6], p[7]));
                }
                red[1][half][r] = sum;
                warp_release(&bars.rdy9, lane);
                tc::named_bar(kBarAll, kCompute);
                l_row = red[1][0][r] + red[1][1][r];
            }
            // ------------------------------------------------------------ P10
            // the chunk's own attention output, normalised, over the P tile
            // (the P V product is complete)
            {
                wait(&bars.pv_done, ph);
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
                warp_release(&bars.rdy10, lane);
            }
            if (!group_all(kBarAll, kCompute, ok)) break;
        }
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
    const int total = a.nloc * a.BH;
    const int grid = total < num_sms ? total : num_sms;
    cudaError_t e =
        cudaFuncSetAttribute(prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
    if (e != cudaSuccess) return e;
    prep_tc_kernel<<<grid, kThreadsP, kSmemP, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace path
