// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace path {

// Prefill workspace, per (batch*head) and padded length Lp = N * C:
//   Qh, Kh, Wt : [BH][Lp][d]    element type of the call
//   Sd         : [BH][N][C][C]  fp32 within-chunk logits (unscaled)
//   F          : [BH][Lp]       fp32 FoX prefix sums (PaTH-FoX calls only)
//   scratch    : [BH][N][5][C][C] fp32 (SIMT prep only)
struct PrepSimtArgs {
    const void *q, *k, *w;
    const float *beta;
    void *Qh, *Kh, *Wt;
    float *Sd, *scratch;
    int BH, L, Lp, N, C, d;
    int keys_only;  // 1: only Kh and Wt (q, Qh, Sd unused)
};

struct FlashSimtArgs {
    const void *Qh, *Kh, *Wt, *w, *v;
    const float *Sd, *F;
    void *out;
    float *lse;
    float scale;
    int BH, L, Lp, N, C, d;
};

size_t prep_simt_smem(int C);
size_t flash_simt_smem(int C, int d);
cudaError_t launch_prep_simt(const PrepSimtArgs &a, bool bf16_in, bool bf16_out,
                             cudaStream_t st);
cudaError_t launch_fox_prefix(const float *log_f, float *F, int L, int Lp, int BH,
                              cudaStream_t st);
// bf16_io: w, v and out in bf16 (the workspace stays fp32)
cudaError_t launch_flash_simt(const FlashSimtArgs &a, bool bf16_io, cudaStream_t st);

// Prefill backward (CUDA cores, fp32 arithmetic).  The forward prep's
// outputs (Qh, Kh, Wt fp32, Sd, F) come from launch_prep_simt on the same
// workspace.  Accumulators dKh, dV, dA, dF must be zero on entry.
struct BwdArgs {
    const void *q, *k, *v, *w, *out, *dout;  // [BH][L][d], element type of the call
    const float *beta, *lse, *dlse;          // [BH][L]; dlse may be null (zero)
    const float *Qh, *Kh, *Wt;               // forward prep (CUDA-core scan only)
    const float *F;                          // FoX prefix sums [BH][Lp], null for PaTH
    float *Qts;      // [BH][N(N-1)/2][C][d] carried query rows of every (b, c < b)
    float *dQh;      // [BH][Lp][d]
    float *dKh, *dV; // [BH][Lp][d] (atomic)
    float *dA;       // [BH][N][d][d] (atomic)
    float *dF;       // [BH][Lp] (atomic; PaTH-FoX only, else null)
    float *scratch;  // [BH][N][kBwdPrepCC][C][C] then [BH][N][2][C][d]
    void *dq, *dk, *dv, *dw;  // [BH][L][d], element type of the call
    float *dbeta;    // [BH][L]
    float *dlog_f;   // [BH][L] (PaTH-FoX only)
    float scale;
    int BH, L, Lp, N, C, d;
};

constexpr int kBwdPrepCC = 11;  // C x C scratch matrices per chunk of the backward prep
constexpr int kBwdBf16Tiles = 22, kBwdF32Tiles = 6;  // tensor-core backward prep intermediates
size_t bwd_scan_smem(int C, int d);
size_t bwd_prep_smem(int C);
// bf16_io: q, k, v, w, out, dout and the gradients dq, dk, dv, dw in bf16
cudaError_t launch_bwd(const BwdArgs &a, bool bf16_io, cudaStream_t st);

// Tensor-core backward scan (bf16, head_dim 128, chunk 128; PaTH, and
// PaTH-FoX when F is given).  Maps: 3-D bf16 tensors [BH][rows][128] in 64 x 128 boxes
// with the 128-byte swizzle: qh, kh, pm from the tensor-core prep (rows =
// Lp), v and dout (rows = L), qts the carried-row store (rows = 128 times
// the number of (query chunk, earlier key chunk) pairs of a head).
struct BwdTcMaps {
    CUtensorMap qh, kh, pm, v, dout, qts;
};

struct BwdTcArgs {
    const __nv_bfloat16 *out, *dout;  // [BH][L][128]
    const float *lse, *dlse;          // [BH][L]; dlse may be null
    float *dQh, *dKh, *dV;            // [BH][Lp][128] fp32
    float *dA;                        // [BH][N][128][128] fp32 (accumulated)
    const float *Dg;                  // [BH][Lp] dout . out - dlse per query row
    const float *F;                   // [BH][Lp] FoX prefix sums, or null (PaTH)
    float *dF;                        // [BH][Lp] FoX dF accumulator (with F; scale != 0)
    float scale;
    int BH, L, Lp, N;
    uint32_t *err;
};

cudaError_t launch_bwd_scan_tc(const BwdTcMaps &maps, const BwdTcArgs &a, int num_sms,
                               cudaStream_t st);
// Key side of the tensor-core backward (after launch_bwd_scan_tc): dV, dKh.
cudaError_t launch_bwd_kv_tc(const BwdTcMaps &maps, const BwdTcArgs &a, int num_sms,
                             cudaStream_t st);
// The CUDA-core backward prep alone (after a tensor-core scan).
cudaError_t launch_bwd_prep(const BwdArgs &a, bool bf16_io, cudaStream_t st);
// dlog f_s = sum_{i >= s} dF_i (PaTH-FoX backward, last step).
cudaError_t launch_fox_suffix(const float *dF, float *dlog_f, int L, int Lp, int BH,
                              cudaStream_t st);

// Batched 128 x 128 x 128 contraction over all chunks of all heads (tensor
// cores): per chunk, D = alpha * sum_p (+/-) op(A_p) op(B_p) (+ E), then an
// optional mask, written as fp32 and/or bf16.  Operands are bf16 tensors
// [BH][rows][128] through maps[a], maps[b] (the chunk's 128 rows); at / bt
// select the transposed operand.
struct ChunkGemmProd {
    int8_t a, b, at, bt, neg;
};
struct ChunkGemmMaps {
    CUtensorMap m[8];
};
struct ChunkGemmArgs {
    int np;
    ChunkGemmProd prod[6];
    float alpha;
    const float *E;            // [BH][Lp][128] added to the result, or null
    const float *rowscale;     // [BH][L]: bf16 output rows scaled by it, or null
    int mask;                  // 0 none, 1 keep j <= r, 2 keep j > r, 3 keep j < r
    float *out_f32;            // [BH][Lp][128] or null
    __nv_bfloat16 *out_bf16;   // [BH][Lp][128], or [BH][L][128] if out_final; or null
    int out_final;
    int BH, L, Lp, N;
    uint32_t *err;
};
cudaError_t launch_chunk_gemm_tc(const ChunkGemmMaps &maps, const ChunkGemmArgs &a,
                                 int num_sms, cudaStream_t st);

struct BwdDiagArgs {
    const float *Dg;  // [BH][Lp] dout . out - dlse (bwd_rowdot)
    const float *F;   // [BH][Lp] FoX prefix sums, or null (PaTH)
    float *dF;        // [BH][Lp] FoX dF accumulator (with F)
    const float *lse, *Sd, *dP;
    __nv_bfloat16 *P, *dSd;
    float scale;
    int BH, L, Lp, N;
};
cudaError_t launch_bwd_solve(const float *G, const float *beta, __nv_bfloat16 *T,
                             __nv_bfloat16 *Ti, int BH, int L, int Lp, int N, cudaStream_t st);
cudaError_t launch_bwd_diag(const BwdDiagArgs &a, cudaStream_t st);
cudaError_t launch_bwd_rowdot(const __nv_bfloat16 *out, const __nv_bfloat16 *dout,
                              const float *dlse, float *Dg, int BH, int L, int Lp,
                              cudaStream_t st);
cudaError_t launch_bwd_cvt(const float *x, __nv_bfloat16 *y, size_t n, cudaStream_t st);
cudaError_t launch_bwd_dbeta(const float *dX, const float *dLo, const float *G, float *dbeta,
                             int BH, int L, int Lp, int N, cudaStream_t st);

struct DecodeArgs {
    void *k_cache, *v_cache;
    const void *q_t, *k_t, *v_t, *w_t;
    const float *beta_t;
    void *out;
    float *partials;  // [BH][max_splits][d + 2]: m (log2 units), l, o[d]
    float scale;
    int BH, d, cap, cache_len, keys_per_split, max_splits;
    // PaTH-FoX: f_cache [BH][cap] holds F_j = sum_{s<=j} log f_s of the cached
    // tokens (slot cache_len is written by the step); log_f_t [BH].  Null for PaTH.
    float *f_cache = nullptr;
    const float *log_f_t = nullptr;
};

int decode_keys_per_split();
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);

// Key-cache build for a group of HB heads starting at global head h0.
struct KcacheArgs {
    const __nv_bfloat16 *w;  // raw w of the group, [HB][L][d]
    const float *Kh, *Wt;    // fp32 boundary-adjusted keys and T W, [HB][Lp][d]
    float *Pi, *Mout;        // [HB][S][d][d]
    __nv_bfloat16 *k_cache;  // full cache, [BH][cap][d]
    int h0, HB, cap, L, Lp, N, C, d, G, S;
};

size_t kcache_smem(int d, int C);
cudaError_t launch_kcache_sweep(const KcacheArgs &a, cudaStream_t st);

// Where each chunk of the sequence lives when the prefill is sharded over
// `world` ranks (sequence / context parallelism).  The N chunks form 2*world
// blocks of nb = ceil(N / (2*world)) chunks; rank r owns blocks r and
// 2*world-1-r (a zigzag, so that every rank gets early and late query chunks
// and the causal work is balanced).  A rank's local chunk i (its rows start
// at local row 128*i) is global chunk global_of_local(i); a global chunk c
// lives on rank owner at local index idx (home_of_global).  One GPU is
// world = 1, rank = 0, nb = N: local and global chunks coincide.
struct ChunkMap {
    int world, rank, nb;
    __host__ __device__ int global_of_local(int i) const {
        return i < nb ? rank * nb + i : (2 * world - 1 - rank) * nb + (i - nb);
    }
    __host__ __device__ void home_of_global(int c, int &owner, int &idx) const {
        const int blk = c / nb;
        owner = blk < world ? blk : 2 * world - 1 - blk;
        idx = (blk < world ? 0 : nb) + (c - blk * nb);
    }
};

// Tensor-core scan (bf16, head_dim 128, chunk 128).  Maps: 3-D bf16 tensors
// [BH][rows][128] in 64 x 128 boxes with 128-byte swizzle.
struct FlashTcMaps {
    CUtensorMap qh;          // local boundary-adjusted queries, rows = Lq
    // key side of every chunk: Kh, Pm^T (per chunk a d x d matrix, box of d
    // rows) and V, chunk c at row 128 * idx and z = owner * zs + bh (ChunkMap)
    CUtensorMap kh, pm, v;
};

struct FlashTcArgs {
    const __nv_bfloat16 *OD;  // [BH][Lq][128] each local chunk's own attention output (prep)
    const float *LSD;         // [BH][Lq] its log-sum-exp
    const float *F;           // [BH][Lp] FoX prefix sums over the whole sequence, or null
    __nv_bfloat16 *out;       // [BH][Lout][128] local rows
    float *lse;               // [BH][Lout] or null
    float scale;
    int BH, L, Lp, N;         // whole sequence: length, padded length, chunks
    ChunkMap cm;
    int nloc;                 // local chunks (query tiles) per head
    int Lq, Lout;             // local padded rows, local rows
    int zs;                   // z stride between owners in the key-side maps
    int d;                    // head dim of q, v, out: 128, or 64 (the workspace stays 128 wide)
    int *tile_ctr;            // device counter of the dynamic tile queue, or null: static
                              // round-robin tiles
    const int *ready;         // [BH] chunks of each head the prep has finished (the prep's
                              // PrepTcArgs::ready), when the scan overlaps the prep: a tile
                              // starts once its head counts nloc.  Null: the prep is complete
    int tile_group;           // heads per group of the tile order; 0: launch_flash_tc chooses
    uint32_t *err;
};

// after_prep = false: the launcher zeroes tile_ctr on the stream first and
// launches in stream order.  after_prep = true: the launch directly follows
// the prep's on the stream and may start while the prep runs (programmatic
// stream serialisation); the caller zeroed tile_ctr and a.ready before the
// prep launch.
cudaError_t launch_flash_tc(const FlashTcMaps &maps, const FlashTcArgs &a, int num_sms,
                            cudaStream_t st, bool after_prep = false);

// Tensor-core prep (bf16, head_dim 128, chunk 128): maps over the raw q, k, w,
// v inputs ([BH][L][128]) and over the Qh, Kh, Pm, OD outputs ([BH][Lp][128]),
// all with 64 x 128 boxes and the 128-byte swizzle.
struct PrepTcMaps {
    CUtensorMap q, k, w, v;      // inputs, rows = Lin
    CUtensorMap qh, kh, pm, od;  // outputs, rows = Lq
    CUtensorMap vx;              // copy of V's tiles (sharded prefill), rows = Lq
};

struct PrepTcArgs {
    const float *beta;   // [BH][Lin]
    const float *F;      // FoX prefix sums [BH][Lp] over the whole sequence (natural log
                         // units) or null
    float scale;
    // Qh, Kh, Pm (per chunk the 128 x 128 product I - W^T T W) and OD (each
    // chunk's own attention output, normalised) are written through the maps,
    // local chunk i at row 128 * i.
    float *LSD;          // [BH][Lq] log-sum-exp of the OD rows (natural log)
    int BH, L, Lp, N;    // whole sequence
    ChunkMap cm;
    int nloc;            // local chunks per head (the first nloc of the rank)
    int Lin, Lq;         // rows per head of the inputs and of the outputs
    int copy_v;          // also store each chunk's V tile through maps.vx
    int pm_transposed;   // store Pm^T (the forward scan) instead of Pm (the backward)
    int *ready;          // [BH] zeroed counters, each raised by one (release) once all
                         // of a chunk's outputs are in global memory; or null
    uint32_t *err;
};

cudaError_t launch_prep_tc(const PrepTcMaps &maps, const PrepTcArgs &a, int num_sms,
                           cudaStream_t st);

cudaError_t launch_selftest_wait(uint32_t *err_flag, uint64_t limit_ns, cudaStream_t st);

// bf16 rows [rows][d] <-> [rows][128] (zero-filled columns d..127); d a
// multiple of 8, both pointers 16-byte aligned.
cudaError_t launch_pad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st);
cudaError_t launch_unpad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st);

}  // namespace path
