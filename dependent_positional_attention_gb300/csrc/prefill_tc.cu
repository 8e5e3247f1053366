// PaTH prefill scan on 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Blockwise algorithm of the PaTH Attention summary (section "3. 효율적인
// 학습 및 추론", FlashAttention-style algorithm): per query chunk b (128 rows)
// the key chunks are visited right to left.  The prep kernel has already
// attended each chunk to itself (normalised output OD and log-sum-exp LSD);
// the online softmax starts from that state, and for every earlier chunk c
// the carried query rows Qt (which start as the boundary-adjusted rows Qh_b)
// give
//     [U_c | S_c] = Qt [Pm_c | Kh_c^T]   (carried rows through the chunk
//                                          product, and the logits)
//     Qt <- U_c
//     O  += softmax-weights(S_c) V_c      (online softmax)
// Pm_c = I - W_c^T T_c W_c is the chunk's whole transition as one d x d
// matrix; the prep stores it transposed, so that Pm_c^T and Kh_c stack into
// one 256-row K-major operand and U_c and S_c come from ONE 128 x 256 x 128
// MMA (eight tcgen05.mma of N = 256): half the instructions of two N = 128
// products, which matters because the issuing thread shares its schedulers
// with the softmax and carried-query warps (a 128 x 128 x 16 instruction
// then issues in about 84 cycles instead of 64, while an N = 256 one still
// runs at its 128).  P V is a 128 x 128 x 128 MMA.  fp32 accumulation in
// tensor memory throughout.  The carried rows (after the first step) and the
// softmax weights P are written back to tensor memory as bf16 and read from
// there as the A operand, so that shared memory only carries B operands.
//
// One CTA per SM (persistent), tiles ordered by decreasing work.  Warp roles:
//   warps 0-7   row group: warp w owns TMEM lanes 32 (w & 3) .. + 31 (query
//               rows) and column half w >> 2.  Per step it converts its half
//               of U_c (fp32) into the next carried rows Qt (bf16, TMEM),
//               then runs the online softmax over its half of the logits
//               (row maxima exchanged with the other half's warp, lazy
//               rescale of its half of O, P -> bf16 in TMEM); epilogue (out,
//               lse) per half.  Two warps per scheduler share the work that
//               a carried-query and a softmax warpgroup used to split by role.
//   warp 8      TMA producer: Qh_b, then two rings: [Pm_c^T | Kh_c] pairs
//               (64 KB slots) and V_c (32 KB slots)
//   warp 9      MMA issuer of the [U|S] products (one thread), TMEM owner
//   warp 11     MMA issuer of the P V products (one thread); warp 10 idle
// The two product streams touch disjoint tensor memory (U, S, Qt against P,
// O) and each thread's commits track only its own MMAs, so the carried-query
// chain never waits behind the issue of a P V product.
// Registers are rebalanced at start (setmaxnreg): the producer/MMA group
// drops to 120 per thread, the row group rises to 192 (the launch's
// 168 x 384 budget is redistributed exactly: 120*128 + 2*192*128 = 64512);
// PaTH-FoX uses 136 / 184 (136*128 + 2*184*128 = 64512), the split at which
// that instance compiles without spills.
// Per step c the products are [U|S]_c and PV_{c+1} (one step late, so the
// softmax has a full step of slack).  The first step of a tile reads Qh_b
// from shared memory; the last (c = 0) needs no U and computes S_0 alone.
// Chunk-0 tiles need no scan: the row group copies the prep's result.
// TMEM columns: [0,128) U, [128,256) S, [256,320) Qt (bf16 pairs),
// [320,384) P (bf16 pairs), [384,512) O.
// Every wait is bounded; on timeout the kernel sets the device error flag,
// drains its outstanding copies and MMAs, frees TMEM and exits.

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace path {
namespace {

constexpr int kC = 128;
constexpr int kThreadsTC = 384;  // 3 warpgroups
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Query tiles reach the roles through a ring of tile indices that the
// producer fills: after the CTA's first tile, in the order of a device
// counter (a dynamic queue over the tiles of one head group after another,
// each group's in decreasing order of work; each CTA claims its next tile
// when it starts the current one), or round-robin when there is no counter.  Readers: the two MMA issuers and the row group.
constexpr int kTileRing = 4, kTileReaders = 3;

// Layout for head dimension D (128, or 64).  Rows of 64 bf16 are one
// 128-byte swizzled sub-tile; a D-wide operand has D / 64 of them.  Dynamic
// shared memory (offsets from a 1024-aligned base): Qh_b, the pair slots and
// the V slots.  A pair slot holds the (D + 128)-row K-major operand
// [Pm^T ; Kh] sub-tile by sub-tile: [Pm^T k0-63 | Kh k0-63 | Pm^T k64-127 |
// Kh k64-127], so that its rows are 8-row groups 1024 bytes apart within a
// sub-tile.  Tensor memory: [U | S] contiguous for the fused product, then Qt
// (bf16 pairs), P (bf16 pairs), O.
template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int kSub = D / 64;
    static constexpr int kTileBytes = kC * D * 2;          // Qh_b or V: 128 rows
    static constexpr int kPairSub = (D + kC) * 128;        // one sub-tile of a pair
    static constexpr int kPairBytes = kSub * kPairSub;
    static constexpr int kPairSlots = D == 64 ? 4 : 2, kVSlots = D == 64 ? 4 : 2;
    static constexpr uint32_t kColU = 0, kColS = D, kColQt = D + kC, kColP = kColQt + D / 2,
                              kColO = kColP + kC / 2;
    static constexpr int kOffQb = 0;
    static constexpr int kOffPair = kOffQb + kTileBytes;
    static constexpr int kOffV = kOffPair + kPairSlots * kPairBytes;
    static constexpr int kOffBar = kOffV + kVSlots * kTileBytes;
    static_assert(kColO + D <= 512, "tensor memory budget exceeded");
};

template <int D>
struct Bars {
    uint64_t pair_full[Cfg<D>::kPairSlots], pair_empty[Cfg<D>::kPairSlots];
    uint64_t v_full[Cfg<D>::kVSlots], v_empty[Cfg<D>::kVSlots];
    uint64_t qb_tma_full, qb_empty, s_full, qb_conv_full;
    uint64_t s_empty, p_full, o_done, drain, drain_pv;
    uint64_t tile_full[kTileRing], tile_empty[kTileRing];
    int tile_ring[kTileRing];  // query tile index, -1 once the queue is empty
    uint32_t tmem_base;
    int abort_word;
    alignas(16) float fsm[kC];  // FoX prefix of the current key chunk (log2 units)
    float xm[2][kC];            // per-row maxima (then partial sums) of the two column halves
};
// barriers/misc after the rings, plus slack to align the dynamic base to 1024
template <int D>
constexpr int smem_bytes() {
    return Cfg<D>::kOffBar + (int)((sizeof(Bars<D>) + 127) / 128 * 128) + 1024;
}
static_assert(smem_bytes<128>() <= 232448 && smem_bytes<64>() <= 232448,
              "shared memory budget exceeded");

using tc::group_all;
using tc::named_bar;

// Next query tile from the ring (slot ts, phase parity ph), for a reader
// role: -1 when the queue is exhausted, -2 when a wait gave up.  A group
// reader (n threads behind named barrier id) reads the slot together and
// releases it once every thread has read it; a single-thread reader passes
// id = 0.
template <int D>
__device__ __forceinline__ int next_tile(Bars<D> &bars, int &ts, uint32_t &ph, int id, int n,
                                         bool first_thread, uint32_t *err,
                                         volatile int *abort_word) {
    bool ok = mbar_wait(&bars.tile_full[ts], ph, err, abort_word, kWaitLimitNs);
    if (id) ok = group_all(id, n, ok);
    if (!ok) return -2;
    const int t = *reinterpret_cast<volatile int *>(&bars.tile_ring[ts]);
    if (id) named_bar(id, n);
    if (first_thread) mbar_arrive(&bars.tile_empty[ts]);
    if (++ts == kTileRing) {
        ts = 0;
        ph ^= 1;
    }
    return t;
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

// Query tile t: local chunk i (tiles in decreasing order of work: local
// chunks run in increasing global order), head bh, global chunk b.
struct Tile {
    int i, b, bh;
};

__device__ __forceinline__ Tile tile_of(int t, const FlashTcArgs &a) {
    Tile x;
    // heads in groups of tile_group (the last group may be smaller); within a
    // group, tiles in decreasing order of work, the group's heads interleaved
    const int g = a.tile_group;
    const int grp = t / (g * a.nloc), rem = t - grp * g * a.nloc;
    const int gs = min(g, a.BH - grp * g);
    x.i = a.nloc - 1 - rem / gs;
    x.bh = grp * g + rem % gs;
    x.b = a.cm.global_of_local(x.i);
    return x;
}

// Fused carried-query / logit product for step c: D[0,256) = A [Pm_c^T ; Kh_c]^T
// over K = 128 (eight N = 256 instructions).  A is the carried rows in TMEM
// (a_tmem) or, on a tile's first step, Qh_b in shared memory (a_lo).
template <int D, bool kAFromSmem>
__device__ __forceinline__ void gemm_us(uint32_t d_tmem, uint32_t a, uint32_t pair_lo) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, D + kC, false, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t boff = (uint32_t)((kk >> 2) * (Cfg<D>::kPairSub / 16) + (kk & 3) * 2);
        if (kAFromSmem)
            tc::mma_bf16_lohi(d_tmem, a + (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                              pair_lo + boff, idesc, kk > 0 ? 1u : 0u);
        else
            tc::mma_bf16_ta(d_tmem, a + (uint32_t)(kk * 8), pair_lo + boff, idesc,
                            kk > 0 ? 1u : 0u);
    }
}

// Logits alone (the last step, c = 0, has no chunk product to apply): N = 128
// over the Kh half of a pair slot, whose sub-tiles are 32 KB apart.
template <int D, bool kAFromSmem>
__device__ __forceinline__ void gemm_s(uint32_t d_tmem, uint32_t a, uint32_t kh_lo) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, 128, false, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t boff = (uint32_t)((kk >> 2) * (Cfg<D>::kPairSub / 16) + (kk & 3) * 2);
        if (kAFromSmem)
            tc::mma_bf16_lohi(d_tmem, a + (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                              kh_lo + boff, idesc, kk > 0 ? 1u : 0u);
        else
            tc::mma_bf16_ta(d_tmem, a + (uint32_t)(kk * 8), kh_lo + boff, idesc,
                            kk > 0 ? 1u : 0u);
    }
}

// O (+)= P V over the 128 keys of a chunk: N = D, the V tile MN-major.
template <int D>
__device__ __forceinline__ void gemm_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                        bool accumulate) {
    constexpr uint32_t idesc = tc::idesc_bf16(128, D, false, true);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        tc::mma_bf16_ta(d_tmem, p_tmem + (uint32_t)(kk * 8), v_lo + (uint32_t)(kk * 128), idesc,
                        (accumulate || kk > 0) ? 1u : 0u);
}

template <bool kFox, int D>
__global__ void __launch_bounds__(kThreadsTC, 1)
    flash_tc_kernel(const __grid_constant__ FlashTcMaps maps, FlashTcArgs a) {
    using K = Cfg<D>;
    constexpr int kTileBytes = K::kTileBytes, kPairBytes = K::kPairBytes;
    constexpr int kPairSlots = K::kPairSlots, kVSlots = K::kVSlots;
    constexpr int kOffQb = K::kOffQb, kOffPair = K::kOffPair, kOffV = K::kOffV;
    constexpr uint32_t kColU = K::kColU, kColS = K::kColS, kColQt = K::kColQt, kColP = K::kColP,
                       kColO = K::kColO;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Bars<D> &bars = *reinterpret_cast<Bars<D> *>(smem + K::kOffBar);
    const uint32_t sQb = smem_u32(smem + kOffQb);
    const uint32_t sPair = smem_u32(smem + kOffPair);
    const uint32_t sV = smem_u32(smem + kOffV);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.nloc * a.BH;
    volatile int *abort_word = &bars.abort_word;
    const uint64_t lim = kWaitLimitNs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairSlots; ++s) {
            mbar_init(&bars.pair_full[s], 1);
            mbar_init(&bars.pair_empty[s], 1);
        }
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        mbar_init(&bars.qb_tma_full, 1);
        mbar_init(&bars.qb_empty, 1);  // the MMA commit of the tile's first product
        mbar_init(&bars.s_full, 1);
        // one arrival per warp of the row group
        mbar_init(&bars.qb_conv_full, 8);
        mbar_init(&bars.s_empty, 8);
        mbar_init(&bars.p_full, 8);
        mbar_init(&bars.o_done, 1);
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.drain_pv, 1);
        for (int s = 0; s < kTileRing; ++s) {
            mbar_init(&bars.tile_full[s], 1);
            mbar_init(&bars.tile_empty[s], kTileReaders);
        }
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
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFox ? 136 : 120) : "memory");
      if (warp == 8) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::prefetch_tmap(&maps.qh);
            tc::prefetch_tmap(&maps.kh);
            tc::prefetch_tmap(&maps.pm);
            tc::prefetch_tmap(&maps.v);
            int ps = 0, vs = 0;
            uint32_t pph = 0, vph = 0, qe_ph = 0;
            int pair_par[kPairSlots], v_par[kVSlots];
            for (int i = 0; i < kPairSlots; ++i) pair_par[i] = -1;
            for (int i = 0; i < kVSlots; ++i) v_par[i] = -1;
            int q_last_par = -1;
            uint32_t q_loads = 0;
            bool ok = true;
            // key side of chunk c of head bh, wherever it lives (ChunkMap):
            // [Pm_c^T | Kh_c] into a pair slot (Kh_c alone for c = 0)
            auto load_pair = [&](int c, int bh) -> bool {
                int owner, idx;
                a.cm.home_of_global(c, owner, idx);
                const int y = idx * kC, z = owner * a.zs + bh;
                if (!mbar_wait(&bars.pair_empty[ps], pph ^ 1, a.err, abort_word, lim)) return false;
                uint8_t *dst = smem + kOffPair + ps * kPairBytes;
                uint64_t *full = &bars.pair_full[ps];
                // per sub-tile: Pm^T's D rows (box of D rows), then Kh's 128
                mbar_arrive_expect_tx(full, c >= 1 ? kPairBytes : kTileBytes);
#pragma unroll
                for (int sub = 0; sub < K::kSub; ++sub) {
                    uint8_t *ds = dst + sub * K::kPairSub;
                    if (c >= 1) tc::tma_load_3d(ds, &maps.pm, 64 * sub, y, z, full);
                    tc::tma_load_3d(ds + D * 128, &maps.kh, 64 * sub, y, z, full);
                }
                // PaTH-FoX: the row group reads the chunk's prefixes about a
                // step before the product runs; bring them to L2 with the pair
                if (kFox) tc::bulk_prefetch_l2(a.F + (size_t)bh * a.Lp + (size_t)c * kC, kC * 4);
                pair_par[ps] = (int)pph;
                if (++ps == kPairSlots) {
                    ps = 0;
                    pph ^= 1;
                }
                return true;
            };
            auto load_v = [&](int c, int bh) -> bool {
                int owner, idx;
                a.cm.home_of_global(c, owner, idx);
                const int y = idx * kC, z = owner * a.zs + bh;
                if (!mbar_wait(&bars.v_empty[vs], vph ^ 1, a.err, abort_word, lim)) return false;
                uint8_t *dst = smem + kOffV + vs * kTileBytes;
                mbar_arrive_expect_tx(&bars.v_full[vs], kTileBytes);
#pragma unroll
                for (int sub = 0; sub < K::kSub; ++sub)
                    tc::tma_load_3d(dst + sub * (kC * 128), &maps.v, 64 * sub, y, z, &bars.v_full[vs]);
                v_par[vs] = (int)vph;
                if (++vs == kVSlots) {
                    vs = 0;
                    vph ^= 1;
                }
                return true;
            };
            int ts = 0;
            uint32_t te_ph = 0;
            int t_next = blockIdx.x;
            const bool dynamic = a.tile_ctr != nullptr;
            while (ok) {
                // the CTA's next tile, published to the readers; the tile after
                // it is claimed now, so that the counter's round trip overlaps
                // this tile's loads
                const int t = t_next < T ? t_next : -1;
                if (t >= 0) {
                    t_next = dynamic ? (int)gridDim.x + atomicAdd(a.tile_ctr, 1) : t + gridDim.x;
                    // running behind the prep: the tile's head must be complete
                    // (its rows, chunk products and own-chunk outputs) before
                    // any role reads them; the tensor copies read after the
                    // acquire
                    if (a.ready) {
                        ok = counter_wait(a.ready + tile_of(t, a).bh, a.nloc, a.err, abort_word,
                                          lim);
                        if (!ok) break;
                        tc::fence_proxy_async_global();
                    }
                }
                ok = mbar_wait(&bars.tile_empty[ts], te_ph ^ 1, a.err, abort_word, lim);
                if (!ok) break;
                bars.tile_ring[ts] = t;
                mbar_arrive(&bars.tile_full[ts]);
                if (++ts == kTileRing) {
                    ts = 0;
                    te_ph ^= 1;
                }
                if (t < 0) break;
                const Tile tl = tile_of(t, a);
                const int b = tl.b, bh = tl.bh;
                // the row group starts the tile from the prep's own-chunk
                // output and log-sum-exp, a couple of steps from now: bring them
                // to L2 (they were written by the prep and have left it since)
                tc::bulk_prefetch_l2(a.OD + ((size_t)bh * a.Lq + tl.i * kC) * 128, kC * 128 * 2);
                tc::bulk_prefetch_l2(a.LSD + (size_t)bh * a.Lq + tl.i * kC, kC * 4);
                if (b == 0) continue;
                ok = mbar_wait(&bars.qb_empty, qe_ph ^ 1, a.err, abort_word, lim);
                qe_ph ^= 1;
                if (!ok) break;
                mbar_arrive_expect_tx(&bars.qb_tma_full, kTileBytes);
#pragma unroll
                for (int sub = 0; sub < K::kSub; ++sub)
                    tc::tma_load_3d(smem + kOffQb + sub * (kC * 128), &maps.qh, 64 * sub,
                                    tl.i * kC, bh, &bars.qb_tma_full);
                q_last_par = (int)(q_loads++ & 1);
                for (int c = b - 1; c >= 0 && ok; --c) {
                    ok = ok && load_pair(c, bh);
                    if (c < b - 1) ok = ok && load_v(c + 1, bh);
                }
                ok = ok && load_v(0, bh);
            }
            if (*abort_word) {
                // let every copy this thread issued land before the CTA exits
                for (int s = 0; s < kPairSlots; ++s)
                    if (pair_par[s] >= 0) mbar_wait(&bars.pair_full[s], pair_par[s], a.err, nullptr, lim);
                for (int s = 0; s < kVSlots; ++s)
                    if (v_par[s] >= 0) mbar_wait(&bars.v_full[s], v_par[s], a.err, nullptr, lim);
                if (q_last_par >= 0) mbar_wait(&bars.qb_tma_full, q_last_par, a.err, nullptr, lim);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ [U|S] issuer
        if (lane == 0) {
            int ps = 0;
            uint32_t pph = 0, qt_ph = 0, qc_ph = 0, se_ph = 0;
            const uint32_t qb_lo = tc::desc_lo(sQb, false);
            bool ok = true;
            int ts = 0;
            uint32_t tf_ph = 0;
            while (ok) {
                const int t = next_tile(bars, ts, tf_ph, 0, 1, true, a.err, abort_word);
                if (t < 0) break;
                const int b = tile_of(t, a).b;
                if (b == 0) continue;
                for (int c = b - 1; c >= 0 && ok; --c) {
                    const bool first = (c == b - 1);
                    // the carried rows of this step: Qh_b in shared memory, or
                    // the row group's conversion of the previous U
                    if (first) {
                        ok = mbar_wait(&bars.qb_tma_full, qt_ph, a.err, abort_word, lim);
                        qt_ph ^= 1;
                    } else {
                        ok = mbar_wait(&bars.qb_conv_full, qc_ph, a.err, abort_word, lim);
                        qc_ph ^= 1;
                    }
                    // the row group has read the previous S
                    ok = ok && mbar_wait(&bars.s_empty, se_ph ^ 1, a.err, abort_word, lim);
                    se_ph ^= 1;
                    ok = ok && mbar_wait(&bars.pair_full[ps], pph, a.err, abort_word, lim);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const uint32_t pair_lo = tc::desc_lo(sPair + ps * kPairBytes, false);
                    const uint32_t kh_lo = tc::desc_lo(sPair + ps * kPairBytes + D * 128, false);
                    if (c >= 1) {
                        if (first) gemm_us<D, true>(tmem + kColU, qb_lo, pair_lo);
                        else gemm_us<D, false>(tmem + kColU, tmem + kColQt, pair_lo);
                    } else {
                        if (first) gemm_s<D, true>(tmem + kColS, qb_lo, kh_lo);
                        else gemm_s<D, false>(tmem + kColS, tmem + kColQt, kh_lo);
                    }
                    tc::mma_commit(&bars.pair_empty[ps]);
                    if (++ps == kPairSlots) {
                        ps = 0;
                        pph ^= 1;
                    }
                    // U (when there is one) and S, for the row group
                    tc::mma_commit(&bars.s_full);
                    // Qh_b's tile is free once the first step's product completes
                    if (first) tc::mma_commit(&bars.qb_empty);
                }
            }
            // every MMA this thread issued has completed before TMEM is released
            tc::mma_commit(&bars.drain);
            mbar_wait(&bars.drain, 0, a.err, nullptr, lim);
        }
        __syncwarp();
    } else if (warp == 11) {
        // ------------------------------------------------------------ P V issuer
        if (lane == 0) {
            int vs = 0;
            uint32_t vph = 0, pf_ph = 0;
            bool ok = true;
            // V_{b-1}, ..., V_0 per tile; the tile's first P V writes O, the
            // rest accumulate (the chunk's own block joins in the epilogue)
            int ts = 0;
            uint32_t tf_ph = 0;
            while (ok) {
                const int t = next_tile(bars, ts, tf_ph, 0, 1, true, a.err, abort_word);
                if (t < 0) break;
                const int b = tile_of(t, a).b;
                for (int c = b - 1; c >= 0 && ok; --c) {
                    ok = mbar_wait(&bars.v_full[vs], vph, a.err, abort_word, lim) &&
                         mbar_wait(&bars.p_full, pf_ph, a.err, abort_word, lim);
                    if (!ok) break;
                    pf_ph ^= 1;
                    tc::fence_after_sync();
                    gemm_pv<D>(tmem + kColO, tmem + kColP, tc::desc_lo(sV + vs * kTileBytes, true),
                               c < b - 1);
                    tc::mma_commit(&bars.v_empty[vs]);
                    if (++vs == kVSlots) {
                        vs = 0;
                        vph ^= 1;
                    }
                    tc::mma_commit(&bars.o_done);
                }
            }
            tc::mma_commit(&bars.drain_pv);
            mbar_wait(&bars.drain_pv, 0, a.err, nullptr, lim);
        }
        __syncwarp();
      }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFox ? 184 : 192) : "memory");
      {
        // ------------------------------------------------------------ rows
        // Warps 0-7: warp w owns TMEM lane quadrant w & 3 (32 query rows) and
        // column half w >> 2.  Per step it turns its half of U into the next
        // carried rows, then runs the online softmax over its half of S; the
        // two warps of a quadrant exchange the row maximum through shared
        // memory (pair barrier 2 + quadrant, 64 threads) and keep partial row
        // sums until the epilogue.  Two warps per scheduler hide each other's
        // latency, where one warp per row ran the softmax alone.
        const int quad = warp & 3, hh = warp >> 2;
        const int r = quad * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
        constexpr int kOH = D / 2;  // columns of O (and of U) per half
        const int pair_bar = 2 + quad;
        const float sl2 = a.scale * kLog2e;
        constexpr bool fox = kFox;
        uint32_t sf_ph = 0, od_ph = 0;
        bool ok = true;
        int ts = 0;
        uint32_t tf_ph = 0;
        while (ok) {
            const int t = next_tile(bars, ts, tf_ph, 1, 256, threadIdx.x == 0, a.err, abort_word);
            if (t < 0) break;
            const Tile tl = tile_of(t, a);
            const int b = tl.b, bh = tl.bh;
            const float *Frow = fox ? a.F + (size_t)bh * a.Lp : nullptr;
            const float fi = fox ? Frow[b * kC + r] * kLog2e : 0.f;
            const int row = b * kC + r;       // in the whole sequence
            const int lrow = tl.i * kC + r;   // in the local rows
            // the prep's own-chunk output is 128 wide (head_dim 64 zero-padded)
            const __nv_bfloat16 *odrow = a.OD + ((size_t)bh * a.Lq + lrow) * 128 + hh * kOH;
            // OD and LSD through L2 only (.cg): the prep may have written
            // them while this grid ran
            const float lsd = __ldcg(a.LSD + (size_t)bh * a.Lq + lrow);
            if (b == 0) {
                // the chunk attends only to itself: the prep's result is final
                if (row < a.L) {
                    __nv_bfloat16 *orow = a.out + ((size_t)bh * a.Lout + lrow) * D + hh * kOH;
#pragma unroll
                    for (int j = 0; j < kOH / 8; ++j)
                        reinterpret_cast<uint4 *>(orow)[j] =
                            __ldcg(reinterpret_cast<const uint4 *>(odrow) + j);
                    if (hh == 0 && a.lse) a.lse[(size_t)bh * a.Lout + lrow] = lsd;
                }
                continue;
            }
            // the scan starts from an empty state (the tile's first P V writes O
            // without accumulating); the chunk's own block joins in the epilogue
            float m = -INFINITY, l = 0.f;
            // FoX: the prefixes of the step's key chunk, loaded one step ahead
            // (a load at the step's start would hold the group's barrier);
            // half 0 publishes them, one per thread
            float fcol_next = (fox && hh == 0) ? Frow[(b - 1) * kC + r] : 0.f;
            float fref_next = fox ? Frow[(b - 1) * kC] : 0.f;
            for (int c = b - 1; c >= 0; --c) {
                // FoX: the bias fi - F_j splits into a row term (fi - F_ref) and
                // a column term F_j - F_ref, F_ref the chunk's first prefix
                float dlt = 0.f;
                if (fox) {
                    const float fref = fref_next;
                    if (hh == 0) bars.fsm[r] = (fcol_next - fref) * kLog2e;
                    dlt = fi - fref * kLog2e;
                    if (c >= 1) {
                        if (hh == 0) fcol_next = Frow[(c - 1) * kC + r];
                        fref_next = Frow[(c - 1) * kC];
                    }
                }
                // [U|S]_c complete (the group barrier also publishes the prefixes)
                ok = group_all(1, 256, mbar_wait(&bars.s_full, sf_ph, a.err, abort_word, lim));
                if (!ok) break;
                sf_ph ^= 1;
                tc::fence_after_sync();
                if (c >= 1) {
                    // U -> the next carried rows (bf16), this half's columns; the
                    // product has read the current ones, so they may be overwritten
                    if (D == 128 || hh == 0) {
                        uint32_t u[64], pk[32];
                        tc::tmem_ld64(lane_addr + kColU + (D == 128 ? hh * 64 : 0), u);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            pk[j] = pack_bf16(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1]));
                        tc::tmem_st32(lane_addr + kColQt + (D == 128 ? hh * 32 : 0), pk);
                        tc::tmem_wait_st();
                    }
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.qb_conv_full);
                }
                // this half of the logit row, then S is released to the next MMA
                uint32_t v[64];
                tc::tmem_ld64(lane_addr + kColS + hh * 64, v);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.s_empty);
                // row extremes over interleaved partial results (exact in any order)
                float mx = -INFINITY;
                if (kFox) {
                    // the chunk's column prefixes, four per shared-memory load
                    const uint32_t fsm_s = smem_u32(bars.fsm + hh * 64);
                    float mp[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) mp[i] = -INFINITY;
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        const uint4 f4 = tc::lds128(fsm_s + 16 * j4);
                        const uint32_t fw[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e;
                            const float tt = fmaf(__uint_as_float(v[j]), sl2, -__uint_as_float(fw[e]));
                            v[j] = __float_as_uint(tt);
                            mp[e] = fmaxf(mp[e], tt);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, mp[i]);
                    mx += dlt;
                } else {
                    // max of the scaled logits from the raw extreme (min if scale < 0)
                    float mp[8];
                    if (sl2 >= 0.f) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
                        for (int j = 0; j < 64; ++j) mp[j & 7] = fmaxf(mp[j & 7], __uint_as_float(v[j]));
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx = fmaxf(mx, mp[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) mp[i] = INFINITY;
#pragma unroll
                        for (int j = 0; j < 64; ++j) mp[j & 7] = fminf(mp[j & 7], __uint_as_float(v[j]));
                        mx = INFINITY;
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx = fminf(mx, mp[i]);
                    }
                    mx *= sl2;
                }
                // the row maximum from both halves (the next write of this slot
                // comes after the next step's group barrier)
                bars.xm[hh][r] = mx;
                named_bar(pair_bar, 64);
                mx = fmaxf(bars.xm[0][r], bars.xm[1][r]);
                // lazy rescale: keep the reference max unless it grows by > 2^8.
                // The decision is made per warp (the O rescale uses warp-aligned
                // TMEM loads/stores) and is the same in both warps of a quadrant;
                // a lane that did not need it rescales by its exact factor, <= 1.
                const bool rescale = __any_sync(0xffffffffu, mx - m > kRescaleThreshold);
                const float mnew = rescale ? fmaxf(m, mx) : m;
                const float alpha = rescale ? exp2f(m - mnew) : 1.f;
                // probabilities, packed to bf16 pairs (the logits die as they go)
                // FoX rows already hold the scaled logits less the row term
                const float xs = kFox ? 1.f : sl2;
                const float off = kFox ? dlt - mnew : -mnew;
                float sum0 = 0.f, sum1 = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int j4 = 0; j4 < 16; ++j4) {
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
                    ok = group_all(1, 256, mbar_wait(&bars.o_done, od_ph, a.err, abort_word, lim));
                    if (!ok) break;
                    od_ph ^= 1;
                    tc::fence_after_sync();
                }
                // (the first step's P V overwrites O: nothing to rescale)
                if (rescale && c < b - 1) {
#pragma unroll
                    for (int cc = 0; cc < kOH / 32; ++cc) {
                        uint32_t o[32];
                        tc::tmem_ld32(lane_addr + kColO + hh * kOH + cc * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::tmem_st32(lane_addr + kColO + hh * kOH + cc * 32, o);
                    }
                }
                tc::tmem_st32(lane_addr + kColP + hh * 32, pk);
                tc::tmem_wait_st();
                l = l * alpha + (sum0 + sum1);
                m = mnew;
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full);
                // FoX: the first step has no group barrier between this step's
                // reads of the prefixes and the next step's writes
                if (fox && c == b - 1 && c >= 1) named_bar(1, 256);
            }
            if (!ok) break;
            // epilogue: the scan's state (O against the reference m, log2 units;
            // l the sum of the two halves' partial sums) merged with the chunk's
            // own block (OD normalised, LSD its log-sum-exp), weights 2^(m - M)
            // and 2^(LSD log2e - M), M the larger; lse = ln(2) * (M + log2 of
            // the summed weight).  This half's OD row is loaded before the wait
            // for the last P V.
            uint32_t od[kOH / 2];
#pragma unroll
            for (int j = 0; j < kOH / 8; ++j) {
                const uint4 u = __ldcg(reinterpret_cast<const uint4 *>(odrow) + j);
                od[4 * j] = u.x;
                od[4 * j + 1] = u.y;
                od[4 * j + 2] = u.z;
                od[4 * j + 3] = u.w;
            }
            ok = group_all(1, 256, mbar_wait(&bars.o_done, od_ph, a.err, abort_word, lim));
            if (!ok) break;
            od_ph ^= 1;
            tc::fence_after_sync();
            bars.xm[hh][r] = l;
            named_bar(pair_bar, 64);
            const float lt = bars.xm[0][r] + bars.xm[1][r];
            const float lsd2 = lsd * kLog2e;
            const float mm = fmaxf(m, lsd2);
            const float wa = exp2f(m - mm), wb = exp2f(lsd2 - mm);
            const float den = fmaf(lt, wa, wb);
            const float ia = wa / den, ib = wb / den;
            __nv_bfloat16 *orow = a.out + ((size_t)bh * a.Lout + lrow) * D + hh * kOH;
            {
                uint32_t v[kOH];
                __syncwarp();  // the ragged-row branch below diverges; the load is warp-aligned
                if constexpr (kOH == 64)
                    tc::tmem_ld64(lane_addr + kColO + hh * kOH, v);
                else
                    tc::tmem_ld32(lane_addr + kColO + hh * kOH, v);
                if (row < a.L) {
#pragma unroll
                    for (int q = 0; q < kOH / 8; ++q) {
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(
                                *reinterpret_cast<const __nv_bfloat162 *>(&od[q * 4 + e]));
                            y[2 * e] = fmaf(__uint_as_float(v[q * 8 + 2 * e]), ia, f.x * ib);
                            y[2 * e + 1] = fmaf(__uint_as_float(v[q * 8 + 2 * e + 1]), ia, f.y * ib);
                        }
                        uint4 u;
                        u.x = pack_bf16(y[0], y[1]);
                        u.y = pack_bf16(y[2], y[3]);
                        u.z = pack_bf16(y[4], y[5]);
                        u.w = pack_bf16(y[6], y[7]);
                        *reinterpret_cast<uint4 *>(orow + q * 8) = u;
                    }
                }
            }
            if (hh == 0 && a.lse && row < a.L)
                a.lse[(size_t)bh * a.Lout + lrow] = (mm + log2f(den)) * kLn2;
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
                            cudaStream_t st, bool after_prep) {
    const int T = a.nloc * a.BH;
    const int grid = T < num_sms ? T : num_sms;
    if (a.d != 128 && a.d != 64) return cudaErrorInvalidValue;
    void (*kern)(const FlashTcMaps, FlashTcArgs) =
        a.d == 64 ? (a.F ? flash_tc_kernel<true, 64> : flash_tc_kernel<false, 64>)
                  : (a.F ? flash_tc_kernel<true, 128> : flash_tc_kernel<false, 128>);
    const int smem = a.d == 64 ? smem_bytes<64>() : smem_bytes<128>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // Tile order: the CTAs of a head group stream the same key chunks a step
    // or so apart, so most tiles read chunks another CTA has just brought
    // into L2.  About ten CTAs per head (grid / 10 heads per group; at least
    // 2.5 grids of tiles per group, so that the group's light tiles still
    // balance the CTAs' ends), in groups of equal size (a small last group
    // balanced badly: B2 H12 L4096 in groups of 16 and 8 heads was 13%
    // slower than one group).  B8 H12 L4096 (6 groups of 16 heads against
    // all 96 interleaved): 0.533 -> 0.459 ms; B16: 1.39 -> 0.93 ms; up to
    // 24 heads, and B1 H12 L32768, one group, the order as before.
    FlashTcArgs ag = a;
    if (a.tile_group > 0) {
        ag.tile_group = a.tile_group < a.BH ? a.tile_group : a.BH;  // the caller's choice
    } else {
        long long g = (grid + 9) / 10;
        const long long gb = (5ll * grid + 2ll * a.nloc - 1) / (2ll * a.nloc);
        if (gb > g) g = gb;
        long long groups = a.BH / g;
        if (groups < 1) groups = 1;
        ag.tile_group = (int)((a.BH + groups - 1) / groups);
    }
    if (!after_prep) {
        if (a.tile_ctr) {
            e = cudaMemsetAsync(a.tile_ctr, 0, sizeof(int), st);
            if (e != cudaSuccess) return e;
        }
        kern<<<grid, kThreadsTC, smem, st>>>(maps, ag);
        return cudaGetLastError();
    }
    // behind the prep: each CTA may start on an SM the prep has left, and
    // its tiles wait on the prep's per-head counters
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps, ag);
}

}  // namespace path
