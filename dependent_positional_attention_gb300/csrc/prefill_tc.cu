// PaTH prefill scan on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Blockwise algorithm of the PaTH Attention summary (section "3. 효율적인
// 학습 및 추론", FlashAttention-style algorithm): per query chunk b (128 rows)
// the key chunks are visited right to left.  The prep kernel has already
// attended each chunk to itself (normalised output OD and log-sum-exp LSD);
// the online softmax starts from that state, and for every earlier chunk c
// the carried query rows Qt (which start as the boundary-adjusted rows Qh_b)
// give
//     S_c = Qt Kh_c^T            (logits against boundary-adjusted keys)
//     Qt <- Qt Pm_c              (chunk product, Pm_c = I - W_c^T T_c W_c)
//     O  += softmax-weights(S_c) V_c           (online softmax)
// Each contraction is a 128 x 128 x 128 bf16 MMA with fp32 accumulation in
// tensor memory.  The carried rows (after the first step) and the softmax
// weights P are written back to tensor memory as bf16 and read from there as
// the A operand, so that shared memory only carries the B operands: at
// M = N = 128 an MMA with both operands in shared memory would take all of
// its bandwidth.  Applying the whole chunk product as one d x d
// matrix takes one MMA per chunk instead of two (Qt W^T, then X Wt) and
// re-rounds the carried rows once per chunk rather than rounding a
// correction term of their own size.
//
// One CTA per SM (persistent), tiles ordered by decreasing work.  Warp roles:
//   warps 0-3   carried-query warpgroup: Qt Pm_c (TMEM, fp32) -> bf16 (TMEM)
//   warps 4-7   softmax warpgroup: logits, online softmax with lazy rescale
//               of O, P -> bf16 (TMEM), epilogue (out, lse)
//   warp 8      TMA producer: Qh_b, then a 6-slot ring of Pm_c, Kh_c, V
//   warp 9      MMA issuer (one thread) and TMEM owner; warps 10-11 idle
// Registers are rebalanced at start (setmaxnreg): the producer/MMA group
// drops to 120 per thread, the two compute groups rise to 192 (the launch's
// 168 x 384 budget is redistributed exactly: 120*128 + 2*192*128 = 64512).
// MMA issue order per step c: U_c = Qt Pm_c (the critical chain), S_c,
// PV_{c+1}; the PV of a chunk runs one step late so the softmax has a full
// step of slack.  Chunk-0 tiles need no scan: the softmax group copies the
// prep's result.  TMEM columns: [0,128) U, [128,192) Qt (bf16 pairs),
// [192,256) P (bf16 pairs), [256,384) S, [384,512) O.
// Every wait is bounded; on timeout the kernel sets the device error flag,
// drains its outstanding copies and MMAs, frees TMEM and exits.

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace path {
namespace {

constexpr int kD = 128, kC = 128;
constexpr int kSlots = 6;
constexpr int kTileBytes = kC * kD * 2;  // 32 KB bf16 tile
constexpr int kThreadsTC = 384;  // 3 warpgroups
constexpr uint32_t kColU = 0, kColQt = 128, kColP = 192, kColS = 256, kColO = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffQb = 0;
constexpr int kOffRing = kOffQb + kTileBytes;
constexpr int kOffBar = kOffRing + kSlots * kTileBytes;

struct Bars {
    uint64_t full[kSlots], empty[kSlots];
    uint64_t qb_tma_full, qb_empty, u_done, qb_free, qb_conv_full;
    uint64_t s_full, s_empty, p_full, o_done, drain;
    uint32_t tmem_base;
    int abort_word;
    float fsm[kC];  // FoX prefix of the current key chunk (log2 units)
};
// barriers/misc after the ring, plus slack to align the dynamic base to 1024
constexpr int kSmemBytes = kOffBar + (int)((sizeof(Bars) + 127) / 128 * 128) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");

// Warpgroup barrier.  bar.sync is a warp-aligned instruction: every lane of
// the warp must execute it together, so the warp is reconverged first (lanes
// may leave a bounded wait loop at different iterations).
__device__ __forceinline__ void named_bar(int id, int n) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over a warpgroup that also ANDs `ok` across its threads, so that a
// wait that gave up in one thread makes the whole group leave together.
__device__ __forceinline__ bool group_all(int id, int n, bool ok) {
    uint32_t r;
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// 2^x on the MUFU unit (inputs here are <= 0 after the max subtraction;
// results below 2^-126 flush to zero, which a softmax weight can ignore).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

struct Tile {
    int b, bh;
};

__device__ __forceinline__ Tile tile_of(int t, int BH, int N) {
    Tile x;
    x.b = N - 1 - t / BH;
    x.bh = t % BH;
    return x;
}

template <bool kFox>
__global__ void __launch_bounds__(kThreadsTC, 1)
    flash_tc_kernel(const __grid_constant__ FlashTcMaps maps, FlashTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars &bars = *reinterpret_cast<Bars *>(smem + kOffBar);
    const uint32_t sQb = smem_u32(smem + kOffQb);
    const uint32_t sRing = smem_u32(smem + kOffRing);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.N * a.BH;
    volatile int *abort_word = &bars.abort_word;
    const uint64_t lim = kWaitLimitNs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
        }
        mbar_init(&bars.qb_tma_full, 1);
        mbar_init(&bars.qb_empty, 2);  // MMA commit + carried-query group
        mbar_init(&bars.u_done, 1);
        mbar_init(&bars.qb_free, 1);
        mbar_init(&bars.qb_conv_full, 1);
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.s_empty, 1);
        mbar_init(&bars.p_full, 1);
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.drain, 1);
        bars.abort_word = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tc::tmem_alloc(&bars.tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    if (warp >= 8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 120;" ::: "memory");
      if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::prefetch_tmap(&maps.qh);
            tc::prefetch_tmap(&maps.kh);
            tc::prefetch_tmap(&maps.pm);
            tc::prefetch_tmap(&maps.v);
            int slot = 0;
            uint32_t ph = 0, qe_ph = 0;
            int last_par[kSlots];
            for (int i = 0; i < kSlots; ++i) last_par[i] = -1;
            int q_last_par = -1;
            uint32_t q_loads = 0;
            bool ok = true;
            auto load = [&](const CUtensorMap *m, int y, int z) -> bool {
                if (!mbar_wait(&bars.empty[slot], ph ^ 1, a.err, abort_word, lim)) return false;
                uint8_t *dst = smem + kOffRing + slot * kTileBytes;
                mbar_arrive_expect_tx(&bars.full[slot], kTileBytes);
                tc::tma_load_3d(dst, m, 0, y, z, &bars.full[slot]);
                tc::tma_load_3d(dst + kTileBytes / 2, m, 64, y, z, &bars.full[slot]);
                last_par[slot] = (int)ph;
                if (++slot == kSlots) {
                    slot = 0;
                    ph ^= 1;
                }
                return true;
            };
            for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
                const Tile tl = tile_of(t, a.BH, a.N);
                const int b = tl.b, bh = tl.bh;
                if (b == 0) continue;
                ok = mbar_wait(&bars.qb_empty, qe_ph ^ 1, a.err, abort_word, lim);
                qe_ph ^= 1;
                if (!ok) break;
                mbar_arrive_expect_tx(&bars.qb_tma_full, kTileBytes);
                tc::tma_load_3d(smem + kOffQb, &maps.qh, 0, b * kC, bh, &bars.qb_tma_full);
                tc::tma_load_3d(smem + kOffQb + kTileBytes / 2, &maps.qh, 64, b * kC, bh,
                                &bars.qb_tma_full);
                q_last_par = (int)(q_loads++ & 1);
                for (int c = b - 1; c >= 0 && ok; --c) {
                    if (c >= 1) ok = ok && load(&maps.pm, c * kC, bh);
                    ok = ok && load(&maps.kh, c * kC, bh);
                    if (c < b - 1) ok = ok && load(&maps.v, (c + 1) * kC, bh);
                }
                ok = ok && load(&maps.v, 0, bh);
            }
            if (*abort_word) {
                // let every copy this thread issued land before the CTA exits
                for (int s = 0; s < kSlots; ++s)
                    if (last_par[s] >= 0) mbar_wait(&bars.full[s], last_par[s], a.err, nullptr, lim);
                if (q_last_par >= 0) mbar_wait(&bars.qb_tma_full, q_last_par, a.err, nullptr, lim);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int slot = 0;
            uint32_t ph = 0, qt_ph = 0, qc_ph = 0, se_ph = 0, pf_ph = 0;
            const uint32_t qb_lo = tc::desc_lo(sQb, false);
            bool ok = true;
            auto take = [&](uint32_t &addr) -> bool {
                if (!mbar_wait(&bars.full[slot], ph, a.err, abort_word, lim)) return false;
                addr = sRing + slot * kTileBytes;
                return true;
            };
            auto release = [&]() {
                tc::mma_commit(&bars.empty[slot]);
                if (++slot == kSlots) {
                    slot = 0;
                    ph ^= 1;
                }
            };
            // O already holds the chunk's own attention block (written by the
            // softmax group), so every PV accumulates
            auto pv = [&]() -> bool {
                uint32_t vaddr;
                if (!take(vaddr)) return false;
                if (!mbar_wait(&bars.p_full, pf_ph, a.err, abort_word, lim)) return false;
                pf_ph ^= 1;
                tc::fence_after_sync();
                tc::gemm128_ta<true>(tmem + kColO, tmem + kColP, tc::desc_lo(vaddr, true), true);
                release();
                tc::mma_commit(&bars.o_done);
                return true;
            };
            for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
                const int b = tile_of(t, a.BH, a.N).b;
                if (b == 0) continue;
                for (int c = b - 1; c >= 0 && ok; --c) {
                    if (c == b - 1) {
                        ok = mbar_wait(&bars.qb_tma_full, qt_ph, a.err, abort_word, lim);
                        qt_ph ^= 1;
                    } else {
                        ok = mbar_wait(&bars.qb_conv_full, qc_ph, a.err, abort_word, lim);
                        qc_ph ^= 1;
                    }
                    if (!ok) break;
                    tc::fence_after_sync();
                    // the first step reads Qh_b from shared memory, later steps
                    // the carried rows from tensor memory
                    const bool first = (c == b - 1);
                    uint32_t addr;
                    if (c >= 1) {
                        // carried rows through the chunk product: U = Qt Pm_c
                        if (!(ok = take(addr))) break;
                        if (first)
                            tc::gemm128_lo<true>(tmem + kColU, qb_lo, tc::desc_lo(addr, true), false);
                        else
                            tc::gemm128_ta<true>(tmem + kColU, tmem + kColQt, tc::desc_lo(addr, true),
                                                 false);
                        release();
                        tc::mma_commit(&bars.u_done);
                    }
                    if (!(ok = take(addr))) break;
                    if (!(ok = mbar_wait(&bars.s_empty, se_ph ^ 1, a.err, abort_word, lim))) break;
                    se_ph ^= 1;
                    tc::fence_after_sync();
                    if (first)
                        tc::gemm128_lo<false>(tmem + kColS, qb_lo, tc::desc_lo(addr, false), false);
                    else
                        tc::gemm128_ta<false>(tmem + kColS, tmem + kColQt, tc::desc_lo(addr, false),
                                              false);
                    release();
                    tc::mma_commit(&bars.s_full);
                    // Qh_b's tile is free after the first step; the carried rows
                    // may be overwritten once U_c and S_c (their readers) complete
                    if (first) tc::mma_commit(&bars.qb_empty);
                    if (c >= 1) tc::mma_commit(&bars.qb_free);
                    if (c < b - 1) ok = pv();
                }
                ok = ok && pv();
            }
            // every MMA issued so far has completed before TMEM is released
            tc::mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, a.err, nullptr, lim);
        }
        __syncwarp();
      }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
      if (warp < 4) {
        // ------------------------------------------------------------ carried query
        const int quad = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t ud_ph = 0, qf_ph = 0, qt_ph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
            const int b = tile_of(t, a.BH, a.N).b;
            if (b == 0) continue;
            ok = group_all(1, 128, mbar_wait(&bars.qb_tma_full, qt_ph, a.err, abort_word, lim));
            if (!ok) break;
            qt_ph ^= 1;
            // second arrival on qb_empty (the first is the MMA commit after the
            // last S of this tile): the next Qh load waits for this group too,
            // so the Qh barrier never runs a phase ahead of it.
            named_bar(1, 128);
            if (threadIdx.x == 0) mbar_arrive(&bars.qb_empty);
            for (int c = b - 1; c >= 1; --c) {
                ok = group_all(1, 128, mbar_wait(&bars.u_done, ud_ph, a.err, abort_word, lim));
                if (!ok) break;
                ud_ph ^= 1;
                tc::fence_after_sync();
                uint32_t pk[64];
                {
                    uint32_t v[128];
                    tc::tmem_ld128(lane_addr + kColU, v);
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        pk[j] = pack_bf16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                }
                ok = group_all(1, 128, mbar_wait(&bars.qb_free, qf_ph, a.err, abort_word, lim));
                if (!ok) break;
                qf_ph ^= 1;
                tc::fence_after_sync();
                tc::tmem_st32(lane_addr + kColQt, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                tc::tmem_st32(lane_addr + kColQt + 32,
                              *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
                tc::tmem_wait_st();
                tc::fence_before_sync();
                named_bar(1, 128);
                if (threadIdx.x == 0) mbar_arrive(&bars.qb_conv_full);
            }
        }
      } else {
        // ------------------------------------------------------------ softmax
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
        const float sl2 = a.scale * kLog2e;
        constexpr bool fox = kFox;
        uint32_t sf_ph = 0, od_ph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T && ok; t += gridDim.x) {
            const Tile tl = tile_of(t, a.BH, a.N);
            const int b = tl.b, bh = tl.bh;
            const float *Frow = fox ? a.F + (size_t)bh * a.Lp : nullptr;
            const float fi = fox ? Frow[b * kC + r] * kLog2e : 0.f;
            const int row = b * kC + r;
            const __nv_bfloat16 *odrow = a.OD + ((size_t)bh * a.Lp + row) * kD;
            const float lsd = a.LSD[(size_t)bh * a.Lp + row];
            if (b == 0) {
                // the chunk attends only to itself: the prep's result is final
                if (row < a.L) {
                    __nv_bfloat16 *orow = a.out + ((size_t)bh * a.L + row) * kD;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        reinterpret_cast<uint4 *>(orow)[j] = reinterpret_cast<const uint4 *>(odrow)[j];
                    if (a.lse) a.lse[(size_t)bh * a.L + row] = lsd;
                }
                continue;
            }
            // start from the chunk's own block: O = OD (weights summing to 1
            // against the reference m = LSD in log2 units), l = 1
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 u = reinterpret_cast<const uint4 *>(odrow)[cc * 4 + q];
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
                        o[q * 8 + 2 * e] = __float_as_uint(f.x);
                        o[q * 8 + 2 * e + 1] = __float_as_uint(f.y);
                    }
                }
                tc::tmem_st32(lane_addr + kColO + cc * 32, o);
            }
            tc::tmem_wait_st();
            float m = lsd * kLog2e, l = 1.f;
            for (int c = b - 1; c >= 0; --c) {
                // FoX: the bias fi - F_j splits into a row term (fi - F_ref) and
                // a column term F_j - F_ref, F_ref the chunk's first prefix
                float dlt = 0.f;
                if (fox) {
                    const float fref = Frow[c * kC];
                    bars.fsm[r] = (Frow[c * kC + r] - fref) * kLog2e;
                    dlt = fi - fref * kLog2e;
                }
                ok = group_all(2, 128, mbar_wait(&bars.s_full, sf_ph, a.err, abort_word, lim));
                if (!ok) break;
                sf_ph ^= 1;
                tc::fence_after_sync();
                // one load of the logit row, then S is released to the next MMA
                uint32_t v[128];
                tc::tmem_ld128(lane_addr + kColS, v);
                tc::fence_before_sync();
                named_bar(2, 128);  // also publishes this chunk's FoX prefix
                if (threadIdx.x == 128) mbar_arrive(&bars.s_empty);
                float mx = -INFINITY;
                if (kFox) {
#pragma unroll
                    for (int j = 0; j < kC; ++j) {
                        const float t = fmaf(__uint_as_float(v[j]), sl2, -bars.fsm[j]);
                        v[j] = __float_as_uint(t);
                        mx = fmaxf(mx, t);
                    }
                    mx += dlt;
                } else {
                    // max of the scaled logits from the raw extreme (min if scale < 0)
                    if (sl2 >= 0.f) {
#pragma unroll
                        for (int j = 0; j < kC; ++j) mx = fmaxf(mx, __uint_as_float(v[j]));
                    } else {
                        mx = INFINITY;
#pragma unroll
                        for (int j = 0; j < kC; ++j) mx = fminf(mx, __uint_as_float(v[j]));
                    }
                    mx *= sl2;
                }
                // lazy rescale: keep the reference max unless it grows by > 2^8.
                // The decision is made per warp (the O rescale uses warp-aligned
                // TMEM loads/stores); a lane that did not need it rescales by its
                // exact factor, which is <= 1.
                const bool rescale = __any_sync(0xffffffffu, mx - m > kRescaleThreshold);
                const float mnew = rescale ? fmaxf(m, mx) : m;
                const float alpha = rescale ? exp2f(m - mnew) : 1.f;
                // probabilities, packed to bf16 pairs (the logits die as they go)
                // FoX rows already hold the scaled logits less the row term
                const float xs = kFox ? 1.f : sl2;
                const float off = kFox ? dlt - mnew : -mnew;
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[kC / 2];
#pragma unroll
                for (int j4 = 0; j4 < kC / 4; ++j4) {
                    float p[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        p[e] = kFox ? ex2(__uint_as_float(v[4 * j4 + e]) + off)
                                    : ex2(fmaf(__uint_as_float(v[4 * j4 + e]), xs, off));
                    sum0 += p[0] + p[1];
                    sum1 += p[2] + p[3];
                    pk[2 * j4] = pack_bf16(p[0], p[1]);
                    pk[2 * j4 + 1] = pack_bf16(p[2], p[3]);
                }
                // previous PV done: P buffer free and O stable (the first step
                // follows the previous tile's epilogue, which waited already)
                if (c < b - 1) {
                    ok = group_all(2, 128, mbar_wait(&bars.o_done, od_ph, a.err, abort_word, lim));
                    if (!ok) break;
                    od_ph ^= 1;
                    tc::fence_after_sync();
                }
                if (rescale) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t o[32];
                        tc::tmem_ld32(lane_addr + kColO + cc * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::tmem_st32(lane_addr + kColO + cc * 32, o);
                    }
                    tc::tmem_wait_st();
                }
                tc::tmem_st32(lane_addr + kColP, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                tc::tmem_st32(lane_addr + kColP + 32,
                              *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
                tc::tmem_wait_st();
                l = l * alpha + (sum0 + sum1);
                m = mnew;
                tc::fence_before_sync();
                named_bar(2, 128);
                if (threadIdx.x == 128) mbar_arrive(&bars.p_full);
            }
            if (!ok) break;
            // epilogue: out = O / l, lse = ln(2) * (m + log2 l)
            ok = group_all(2, 128, mbar_wait(&bars.o_done, od_ph, a.err, abort_word, lim));
            if (!ok) break;
            od_ph ^= 1;
            tc::fence_after_sync();
            const float inv = 1.f / l;
            __nv_bfloat16 *orow = a.out + ((size_t)bh * a.L + row) * kD;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t v[64];
                __syncwarp();  // the ragged-row branch below diverges; the load is warp-aligned
                tc::tmem_ld64(lane_addr + kColO + cc * 64, v);
                if (row < a.L) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint4 u;
                        u.x = pack_bf16(__uint_as_float(v[q * 8 + 0]) * inv,
                                        __uint_as_float(v[q * 8 + 1]) * inv);
                        u.y = pack_bf16(__uint_as_float(v[q * 8 + 2]) * inv,
                                        __uint_as_float(v[q * 8 + 3]) * inv);
                        u.z = pack_bf16(__uint_as_float(v[q * 8 + 4]) * inv,
                                        __uint_as_float(v[q * 8 + 5]) * inv);
                        u.w = pack_bf16(__uint_as_float(v[q * 8 + 6]) * inv,
                                        __uint_as_float(v[q * 8 + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + cc * 64 + q * 8) = u;
                    }
                }
            }
            if (a.lse && row < a.L) a.lse[(size_t)bh * a.L + row] = (m + log2f(l)) * kLn2;
            tc::fence_before_sync();
        }
    }

    }
    tc::fence_before_sync();
    __syncwarp();
    __syncthreads();
    if (warp == 9) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_flash_tc(const FlashTcMaps &maps, const FlashTcArgs &a, int num_sms,
                            cudaStream_t st) {
    const int T = a.N * a.BH;
    const int grid = T < num_sms ? T : num_sms;
    void (*kern)(const FlashTcMaps, FlashTcArgs) =
        a.F ? flash_tc_kernel<true> : flash_tc_kernel<false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreadsTC, kSmemBytes, st>>>(maps, a);
    return cudaGetLastError();
}

}  // namespace path
