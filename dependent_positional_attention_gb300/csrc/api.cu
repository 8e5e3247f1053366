// C ABI of libpath_attn: argument validation, workspace layout, dispatch.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "../../include/path_attn.h"
#include "common.cuh"
#include "ctx_symbol.h"
#include "kernels.h"
#include "tmap.h"

namespace path {

// Device-resident state of the library: this error flag, set by kernels
// whose bounded waits ran out, the fixed split-KV scratch of the
// allocation-free decode step (decode_noalloc.cu), and a counter that stays
// zero for the bounded-wait self-test (end of this file).
__device__ uint32_t g_error_flag;

namespace {

thread_local char g_msg[512];

path_status_t fail(path_status_t s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

path_status_t ok() {
    g_msg[0] = 0;
    return PATH_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Address of g_error_flag in the caller's current context (cached per
// context, ctx_symbol.h).
cudaError_t lookup_error_flag(void **p) { return cudaGetSymbolAddress(p, g_error_flag); }
PerContextAddress g_error_flag_addr(&lookup_error_flag);

uint32_t *error_flag_ptr() {
    void *p = nullptr;
    return g_error_flag_addr.get(&p) == cudaSuccess ? static_cast<uint32_t *>(p) : nullptr;
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cache[dev] = n;
    }
    return cache[dev];
}

// Offset of the per-head ready counters within the prefill's counter region.
constexpr size_t kReadyOff = 64;

struct PrefillPlan {
    int BH, L, Lp, N, C, d;
    int dk;     // head dim of the kernels (128 on the tensor-core route)
    bool bf16;  // bf16 inputs and output
    bool tc;    // the tensor-core route (bf16, chunk 128); else CUDA cores
    bool pad;   // tensor-core route for head_dim < 128: q, k, v, w, out zero-padded to 128
    bool d64;   // tensor-core route for head_dim 64 without padded copies: the prep reads
                // q, k, w, v directly (the second 64-column box of a row lies outside
                // the tensor and loads as zeros) and the scan runs at head_dim 64
    size_t esize;
    size_t off_Qh, off_Kh, off_Wt, off_Sd, off_F, off_scratch, off_pad, off_tile, total;
};

// Checks shared by the prefill forward and backward descriptors.
path_status_t check_prefill_desc(const path_prefill_desc_t *desc) {
    if (!desc) return fail(PATH_ERR_INVALID_ARG, "desc is NULL");
    if (desc->batch < 1 || desc->heads < 1 || desc->seq_len < 1 || desc->head_dim < 1)
        return fail(PATH_ERR_INVALID_ARG, "batch, heads, seq_len, head_dim must be >= 1");
    if (desc->dtype != PATH_F32 && desc->dtype != PATH_BF16)
        return fail(PATH_ERR_INVALID_ARG, "dtype must be PATH_F32 or PATH_BF16");
    if (!(desc->scale == desc->scale) || isinf(desc->scale))
        return fail(PATH_ERR_INVALID_ARG, "scale must be finite");
    if ((long long)desc->batch * desc->heads > 65535)
        return fail(PATH_ERR_UNSUPPORTED, "batch*heads must be <= 65535");
    if (desc->scan_group < 0) return fail(PATH_ERR_INVALID_ARG, "scan_group must be >= 0");
    return ok();
}

// Chunk of the CUDA-core route.  Default: 128 halves the per-step
// chunk-product work of 64 (d^2 per query per key chunk), and wins on every
// shape measured except small problems (batch*heads*seq_len <= 8192 with
// head_dim <= 64), where 64 keeps more blocks busy.
path_status_t cuda_core_chunk(const path_prefill_desc_t *desc, int *C) {
    const int d = desc->head_dim;
    if (d > 128 || d % 4)
        return fail(PATH_ERR_UNSUPPORTED, "head_dim must be 128, or <= 128 and a multiple of 4");
    const bool small = (long long)desc->batch * desc->heads * desc->seq_len <= 8192 && d <= 64;
    const int c = desc->chunk ? desc->chunk : (small ? 64 : 128);
    if (c != 16 && c != 32 && c != 64 && c != 128)
        return fail(PATH_ERR_UNSUPPORTED, "chunk must be 16, 32, 64 or 128");
    *C = c;
    return ok();
}

path_status_t plan_prefill(const path_prefill_desc_t *desc, PrefillPlan *p) {
    path_status_t st = check_prefill_desc(desc);
    if (st != PATH_OK) return st;
    const long long BH = (long long)desc->batch * desc->heads;
    p->bf16 = desc->dtype == PATH_BF16;
    p->d = desc->head_dim;
    // bf16 with head_dim a multiple of 8 below 128 takes the tensor-core route on
    // zero-padded copies (pad.cu) unless a chunk other than 128 is asked for
    const bool pad_ok = p->bf16 && p->d < 128 && p->d % 8 == 0 &&
                        (desc->chunk == 0 || desc->chunk == 128);
    p->tc = p->bf16 && (p->d == 128 || pad_ok);
    p->d64 = p->tc && p->d == 64;
    p->pad = p->tc && p->d < 128 && !p->d64;
    if (p->tc) {
        if (desc->chunk != 0 && desc->chunk != 128)
            return fail(PATH_ERR_UNSUPPORTED, "PATH_BF16 with head_dim 128 needs chunk 0 or 128");
        p->C = 128;
    } else {
        // CUDA-core route: fp32, or bf16 inputs/output with another head_dim
        st = cuda_core_chunk(desc, &p->C);
        if (st != PATH_OK) return st;
    }
    p->BH = (int)BH;
    p->L = desc->seq_len;
    p->N = (p->L + p->C - 1) / p->C;
    if ((long long)p->N * p->C > (1ll << 30)) return fail(PATH_ERR_UNSUPPORTED, "seq_len too large");
    p->Lp = p->N * p->C;
    p->esize = p->tc ? 2 : 4;  // the CUDA-core route keeps an fp32 workspace
    p->dk = p->tc ? 128 : p->d;
    const size_t rows = (size_t)p->BH * p->Lp;
    const size_t cc = (size_t)p->BH * p->N * p->C * p->C;
    size_t off = 0;
    p->off_Qh = off; off = align_up(off + rows * p->dk * p->esize, 256);
    p->off_Kh = off; off = align_up(off + rows * p->dk * p->esize, 256);
    p->off_Wt = off; off = align_up(off + rows * p->dk * p->esize, 256);
    p->off_Sd = off; off = align_up(off + cc * 4, 256);
    p->off_F = off; off = align_up(off + rows * 4, 256);
    // fp32 scratch of the SIMT prep (the tensor-core prep keeps it on chip)
    p->off_scratch = off; off = align_up(off + (p->tc ? 0 : cc * 5 * 4), 256);
    // padded q, k, w, v and out, [BH][L][128] bf16 each
    p->off_pad = off; off = align_up(off + (p->pad ? (size_t)5 * p->BH * p->L * 128 * 2 : 0), 256);
    // the tensor-core scan's tile counter, then (at kReadyOff) the prep's
    // per-head counts of finished chunks
    p->off_tile = off; off = align_up(off + (p->tc ? kReadyOff + (size_t)4 * p->BH : 0), 256);
    p->total = off;
    return ok();
}


// Backward workspace (all fp32): the forward prep's Qh, Kh, Wt, Sd, F and
// its scratch (shared with the backward prep's), the carried query rows Qts
// of every (query chunk, earlier key chunk) pair, dQh, then the atomically
// accumulated dKh, dV, dA, dF, zeroed by one memset.
struct BwdPlan {
    int BH, L, Lp, N, C, d;
    bool bf16;
    bool tc;  // bf16, head_dim 128, chunk 128: the tensor-core scan (PaTH calls)
    bool tc_only;  // tc and a nonzero scale: the CUDA-core route can never run, so the
                   // regions that route keeps in fp32 are sized for bf16
    size_t off_Qh, off_Kh, off_Wt, off_Sd, off_F, off_scratch, off_Qts, off_Dg, off_dQh;
    size_t off_dKh, off_dV, off_dA, off_dF, total;
};

path_status_t plan_bwd(const path_prefill_desc_t *desc, BwdPlan *p) {
    path_status_t st = check_prefill_desc(desc);
    if (st != PATH_OK) return st;
    st = cuda_core_chunk(desc, &p->C);
    if (st != PATH_OK) return st;
    p->bf16 = desc->dtype == PATH_BF16;
    p->BH = desc->batch * desc->heads;
    p->L = desc->seq_len;
    p->d = desc->head_dim;
    p->tc = p->bf16 && p->d == 128 && p->C == 128;
    // PaTH-FoX with scale 0 takes the CUDA-core route even when tc holds
    p->tc_only = p->tc && desc->scale != 0.f;
    p->N = (p->L + p->C - 1) / p->C;
    if ((long long)p->N * p->C > (1ll << 30)) return fail(PATH_ERR_UNSUPPORTED, "seq_len too large");
    p->Lp = p->N * p->C;
    const size_t BH = p->BH, N = p->N, C = p->C, d = p->d;
    const size_t rows = BH * p->Lp, cc = BH * N * C * C;
    // element size of Qh, Kh, Wt and the carried-row store: bf16 on the
    // tensor-core route, fp32 on the CUDA cores
    const size_t es = p->tc_only ? 2 : 4;
    size_t off = 0;
    p->off_Qh = off; off = align_up(off + rows * d * es, 256);
    p->off_Kh = off; off = align_up(off + rows * d * es, 256);
    p->off_Wt = off; off = align_up(off + rows * d * es, 256);
    // Sd: the CUDA-core route's within-chunk logits, or the tensor-core prep's
    // OD (bf16) and LSD (fp32)
    p->off_Sd = off;
    off = align_up(off + (p->tc_only ? rows * 128 * 2 + rows * 4 : cc * 4), 256);
    p->off_F = off; off = align_up(off + rows * 4, 256);
    // the CUDA-core backward prep's scratch, or the tensor-core one's tiles
    const size_t simt_scratch = p->tc_only ? 0 : (cc * kBwdPrepCC + BH * N * 2 * C * d) * 4;
    const size_t tc_tiles = p->tc ? rows * 128 * (kBwdBf16Tiles * 2 + kBwdF32Tiles * 4) : 0;
    p->off_scratch = off;
    off = align_up(off + (simt_scratch > tc_tiles ? simt_scratch : tc_tiles), 256);
    p->off_Qts = off; off = align_up(off + BH * (N * (N - 1) / 2) * C * d * es, 256);
    p->off_Dg = off; off = align_up(off + rows * 4, 256);
    // zeroed from here on
    p->off_dQh = off; off = align_up(off + rows * d * 4, 256);
    p->off_dKh = off; off = align_up(off + rows * d * 4, 256);
    p->off_dV = off; off = align_up(off + rows * d * 4, 256);
    p->off_dA = off; off = align_up(off + BH * N * d * d * 4, 256);
    p->off_dF = off; off = align_up(off + rows * 4, 256);
    p->total = off;
    return ok();
}

struct DecodePlan {
    int BH, keys_per_split, max_splits;
    size_t ws_bytes;
};

path_status_t plan_decode(const path_decode_desc_t *desc, DecodePlan *p) {
    if (!desc) return fail(PATH_ERR_INVALID_ARG, "desc is NULL");
    if (desc->batch < 1 || desc->heads < 1 || desc->head_dim < 1 || desc->cache_capacity < 1)
        return fail(PATH_ERR_INVALID_ARG, "batch, heads, head_dim, cache_capacity must be >= 1");
    if (desc->dtype != PATH_F32 && desc->dtype != PATH_BF16)
        return fail(PATH_ERR_INVALID_ARG, "dtype must be PATH_F32 or PATH_BF16");
    if (!(desc->scale == desc->scale) || isinf(desc->scale))
        return fail(PATH_ERR_INVALID_ARG, "scale must be finite");
    if (desc->dtype != PATH_BF16) return fail(PATH_ERR_UNSUPPORTED, "decode needs PATH_BF16");
    if (desc->head_dim != 64 && desc->head_dim != 128)
        return fail(PATH_ERR_UNSUPPORTED, "decode needs head_dim 64 or 128");
    const long long BH = (long long)desc->batch * desc->heads;
    if (BH > 65535) return fail(PATH_ERR_UNSUPPORTED, "batch*heads must be <= 65535");
    p->BH = (int)BH;
    p->keys_per_split = decode_keys_per_split();
    p->max_splits = (desc->cache_capacity + p->keys_per_split - 1) / p->keys_per_split;
    p->ws_bytes = align_up((size_t)p->BH * p->max_splits * (desc->head_dim + 2) * 4, 256);
    return ok();
}

struct KcachePlan {
    int BH, HB, L, Lp, N, C, d, G, S;
    size_t off_Kh, off_Wt, off_scratch, off_Pi, off_Mout, total;
};

path_status_t plan_kcache(const path_prefill_desc_t *desc, KcachePlan *p) {
    if (!desc) return fail(PATH_ERR_INVALID_ARG, "desc is NULL");
    if (desc->batch < 1 || desc->heads < 1 || desc->seq_len < 1 || desc->head_dim < 1)
        return fail(PATH_ERR_INVALID_ARG, "batch, heads, seq_len, head_dim must be >= 1");
    if (desc->dtype != PATH_BF16) return fail(PATH_ERR_UNSUPPORTED, "kcache build needs PATH_BF16");
    if (desc->head_dim > 128 || desc->head_dim % 8)
        return fail(PATH_ERR_UNSUPPORTED, "kcache build needs head_dim <= 128, multiple of 8");
    const long long BH = (long long)desc->batch * desc->heads;
    if (BH > 65535) return fail(PATH_ERR_UNSUPPORTED, "batch*heads must be <= 65535");
    p->BH = (int)BH;
    p->HB = p->BH < 16 ? p->BH : 16;
    p->d = desc->head_dim;
    p->C = 128;
    p->G = 16;
    p->L = desc->seq_len;
    p->N = (p->L + p->C - 1) / p->C;
    p->Lp = p->N * p->C;
    p->S = (p->N + p->G - 1) / p->G;
    const size_t rows = (size_t)p->HB * p->Lp;
    size_t off = 0;
    p->off_Kh = off; off = align_up(off + rows * p->d * 4, 256);
    p->off_Wt = off; off = align_up(off + rows * p->d * 4, 256);
    p->off_scratch = off; off = align_up(off + (size_t)p->HB * p->N * 5 * p->C * p->C * 4, 256);
    p->off_Pi = off; off = align_up(off + (size_t)p->HB * p->S * p->d * p->d * 4, 256);
    p->off_Mout = off; off = align_up(off + (size_t)p->HB * p->S * p->d * p->d * 4, 256);
    p->total = off;
    return ok();
}

// Sequence-sharded prefill: the partition of the N chunks over `world`
// ranks (ChunkMap) and one rank's local sizes and workspace.
struct CpPlan {
    int BH, L, Lp, N, nb, world, rank;
    int nloc;    // valid local chunks (a prefix of the rank's 2*nb)
    int Lr;      // valid local rows
    int Lq;      // padded local rows, 2 * nb * 128
    ChunkMap cm;
    size_t off_Qh, off_OD, off_LSD, off_F, off_tile, total;  // workspace
    size_t section;   // bytes of one of the three sections of an exchange block
    size_t exchange;  // bytes of one rank's exchange block
};

path_status_t plan_cp(const path_prefill_desc_t *desc, int32_t world, int32_t rank, CpPlan *p) {
    path_status_t st = check_prefill_desc(desc);
    if (st != PATH_OK) return st;
    if (desc->dtype != PATH_BF16 || desc->head_dim != 128 ||
        (desc->chunk != 0 && desc->chunk != 128))
        return fail(PATH_ERR_UNSUPPORTED,
                    "the sharded prefill needs PATH_BF16, head_dim 128 and chunk 0 or 128");
    if (world < 1 || world > 4096) return fail(PATH_ERR_INVALID_ARG, "world must be in 1..4096");
    if (rank < 0 || rank >= world) return fail(PATH_ERR_INVALID_ARG, "rank must be in [0, world)");
    p->BH = desc->batch * desc->heads;
    p->L = desc->seq_len;
    p->N = (p->L + 127) / 128;
    if ((long long)p->N * 128 > (1ll << 30)) return fail(PATH_ERR_UNSUPPORTED, "seq_len too large");
    p->Lp = p->N * 128;
    p->world = world;
    p->rank = rank;
    p->nb = (p->N + 2 * world - 1) / (2 * world);
    p->cm = ChunkMap{world, rank, p->nb};
    p->Lq = 2 * p->nb * 128;
    // valid local chunks: those whose global chunk exists (they form a prefix)
    p->nloc = 0;
    p->Lr = 0;
    for (int i = 0; i < 2 * p->nb; ++i) {
        const int c = p->cm.global_of_local(i);
        if (c >= p->N) break;
        ++p->nloc;
        p->Lr += (c + 1) * 128 <= p->L ? 128 : p->L - c * 128;
    }
    const size_t rows = (size_t)p->BH * p->Lq;
    size_t off = 0;
    p->off_Qh = off; off = align_up(off + rows * 128 * 2, 256);
    p->off_OD = off; off = align_up(off + rows * 128 * 2, 256);
    p->off_LSD = off; off = align_up(off + rows * 4, 256);
    p->off_F = off; off = align_up(off + (size_t)p->BH * p->Lp * 4, 256);
    p->off_tile = off; off = align_up(off + 4, 256);  // the scan's tile counter
    p->total = off;
    p->section = rows * 128 * 2;
    p->exchange = 3 * p->section;
    return ok();
}

// A prep over every chunk of the sequence on this GPU (no sharding).
void set_whole_sequence(PrepTcArgs &ta, int N, int L, int Lp) {
    ta.cm = ChunkMap{1, 0, N};
    ta.nloc = N;
    ta.Lin = L;
    ta.Lq = Lp;
    ta.copy_v = 0;
    ta.pm_transposed = 1;
    ta.ready = nullptr;
}

template <class T> T *at(void *base, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(base) + off);
}

// Address of padded array i (0 q, 1 k, 2 w, 3 v, 4 out) of a padded-route workspace.
char *pad_buf(void *workspace, const PrefillPlan &p, int i) {
    return at<char>(workspace, p.off_pad) + (size_t)i * p.BH * p.L * 128 * 2;
}

path_status_t cuda_status(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(PATH_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

// Builds one batched chunk contraction: operands are registered by map, up
// to eight distinct maps and six products.
struct GemmBuilder {
    ChunkGemmMaps maps;
    ChunkGemmArgs args;
    const CUtensorMap *ids[8];
    int nm = 0;
    explicit GemmBuilder(const ChunkGemmArgs &base) : args(base) {
        args.np = 0;
        args.alpha = 1.f;
        args.E = nullptr;
        args.rowscale = nullptr;
        args.mask = 0;
        args.out_f32 = nullptr;
        args.out_bf16 = nullptr;
        args.out_final = 0;
    }
    int map_of(const CUtensorMap *m) {
        for (int i = 0; i < nm; ++i)
            if (ids[i] == m) return i;
        ids[nm] = m;
        maps.m[nm] = *m;
        return nm++;
    }
    // D += (neg ? -1 : 1) * op(A) op(B), op = transpose when at / bt
    GemmBuilder &prod(const CUtensorMap *A, bool at, const CUtensorMap *B, bool bt,
                      bool neg = false) {
        ChunkGemmProd &p = args.prod[args.np++];
        p.a = (int8_t)map_of(A);
        p.b = (int8_t)map_of(B);
        p.at = at;
        p.bt = bt;
        p.neg = neg;
        return *this;
    }
};

// The backward prep of the tensor-core route (formulas: backward_simt.cu,
// bwd_prep_kernel; Ti as in backward_prep_tc.cu).  X^T is written Xt.
path_status_t run_bwd_prep_tc(const path_prefill_desc_t *desc, const BwdPlan &p,
                              const BwdArgs &ba, void *workspace, cudaStream_t st) {
    const size_t rows = (size_t)p.BH * p.Lp;
    char *u = at<char>(workspace, p.off_scratch);
    __nv_bfloat16 *bt[kBwdBf16Tiles];
    float *ft[kBwdF32Tiles];
    for (int i = 0; i < kBwdBf16Tiles; ++i)
        bt[i] = reinterpret_cast<__nv_bfloat16 *>(u + (size_t)i * rows * 256);
    for (int i = 0; i < kBwdF32Tiles; ++i)
        ft[i] = reinterpret_cast<float *>(u + (size_t)kBwdBf16Tiles * rows * 256 +
                                          (size_t)i * rows * 512);
    enum { a_, b_, T_, Ti_, Z_, Y_, Wt_, P_, dSd_, dQh_, dKh_, dA_, dWt_, R1_, da_, R2_, db_,
           R3_, R4_, dT_, dX_, dG_ };
    enum { G_, Sd_, dP_, dXf_, dLo_, dwp_ };
    static_assert(dG_ + 1 == kBwdBf16Tiles && dwp_ + 1 == kBwdF32Tiles, "tile counts");
    CUtensorMap mq, mk, mv, mw, mdo, mt[kBwdBf16Tiles];
    bool enc = encode_tmap_bf16_3d(&mq, ba.q, 128, p.L, p.BH, 64, 128) &&
               encode_tmap_bf16_3d(&mk, ba.k, 128, p.L, p.BH, 64, 128) &&
               encode_tmap_bf16_3d(&mv, ba.v, 128, p.L, p.BH, 64, 128) &&
               encode_tmap_bf16_3d(&mw, ba.w, 128, p.L, p.BH, 64, 128) &&
               encode_tmap_bf16_3d(&mdo, ba.dout, 128, p.L, p.BH, 64, 128);
    for (int i = 0; i < kBwdBf16Tiles && enc; ++i)
        enc = encode_tmap_bf16_3d(&mt[i], bt[i], 128, p.Lp, p.BH, 64, 128);
    if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
    ChunkGemmArgs base;
    base.BH = p.BH; base.L = p.L; base.Lp = p.Lp; base.N = p.N;
    base.err = error_flag_ptr();
    const int sms = num_sms();
    if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
    path_status_t s = ok();
    auto run = [&](GemmBuilder &g, const char *what) {
        if (s == PATH_OK) s = cuda_status(launch_chunk_gemm_tc(g.maps, g.args, sms, st), what);
    };
    const float *dQh = ba.dQh, *dKh = ba.dKh;
    {   // G = W Wt (fp32, for the solve and dbeta)
        GemmBuilder g(base); g.prod(&mw, false, &mw, true); g.args.out_f32 = ft[G_]; run(g, "G");
    }
    {   // a = M_le * (Q Wt)
        GemmBuilder g(base); g.prod(&mq, false, &mw, true); g.args.mask = 1;
        g.args.out_bf16 = bt[a_]; run(g, "a");
    }
    {   // b = M_gt * (K Wt)
        GemmBuilder g(base); g.prod(&mk, false, &mw, true); g.args.mask = 2;
        g.args.out_bf16 = bt[b_]; run(g, "b");
    }
    if (s != PATH_OK) return s;
    s = cuda_status(launch_bwd_solve(ft[G_], ba.beta, bt[T_], bt[Ti_], p.BH, p.L, p.Lp, p.N, st),
                    "solve");
    {   // Z = a T
        GemmBuilder g(base); g.prod(&mt[a_], false, &mt[T_], false); g.args.out_bf16 = bt[Z_];
        run(g, "Z");
    }
    {   // Y = b Tt
        GemmBuilder g(base); g.prod(&mt[b_], false, &mt[T_], true); g.args.out_bf16 = bt[Y_];
        run(g, "Y");
    }
    {   // Wt = T W
        GemmBuilder g(base); g.prod(&mt[T_], false, &mw, false); g.args.out_bf16 = bt[Wt_];
        run(g, "Wt");
    }
    {   // Sd = Q Kt - a Yt
        GemmBuilder g(base); g.prod(&mq, false, &mk, true).prod(&mt[a_], false, &mt[Y_], true, true);
        g.args.out_f32 = ft[Sd_]; run(g, "Sd");
    }
    {   // dP = dout Vt
        GemmBuilder g(base); g.prod(&mdo, false, &mv, true); g.args.out_f32 = ft[dP_];
        run(g, "dP");
    }
    if (s != PATH_OK) return s;
    BwdDiagArgs da;
    da.Dg = at<float>(workspace, p.off_Dg);
    da.F = ba.F;
    da.dF = ba.dF;
    da.lse = ba.lse; da.Sd = ft[Sd_]; da.dP = ft[dP_];
    da.P = bt[P_]; da.dSd = bt[dSd_]; da.scale = desc->scale;
    da.BH = p.BH; da.L = p.L; da.Lp = p.Lp; da.N = p.N;
    s = cuda_status(launch_bwd_diag(da, st), "diagonal block");
    if (s == PATH_OK) s = cuda_status(launch_bwd_cvt(dQh, bt[dQh_], rows * 128, st), "cvt");
    if (s == PATH_OK) s = cuda_status(launch_bwd_cvt(dKh, bt[dKh_], rows * 128, st), "cvt");
    if (s == PATH_OK) s = cuda_status(launch_bwd_cvt(ba.dA, bt[dA_], rows * 128, st), "cvt");
    {   // dv = dV (scan) + Pt dout
        GemmBuilder g(base); g.prod(&mt[P_], true, &mdo, false); g.args.E = ba.dV;
        g.args.out_bf16 = static_cast<__nv_bfloat16 *>(ba.dv); g.args.out_final = 1; run(g, "dv");
    }
    {   // dWt = -W dA
        GemmBuilder g(base); g.prod(&mw, false, &mt[dA_], false); g.args.alpha = -1.f;
        g.args.out_bf16 = bt[dWt_]; run(g, "dWt");
    }
    {   // R1 = dSd b
        GemmBuilder g(base); g.prod(&mt[dSd_], false, &mt[b_], false); g.args.out_bf16 = bt[R1_];
        run(g, "R1");
    }
    {   // da = M_le * -(R1 Tt + dQh Wtt)
        GemmBuilder g(base); g.prod(&mt[R1_], false, &mt[T_], true).prod(&mt[dQh_], false, &mt[Wt_], true);
        g.args.alpha = -1.f; g.args.mask = 1; g.args.out_bf16 = bt[da_]; run(g, "da");
    }
    {   // R2 = dSdt a + dKh Wt
        GemmBuilder g(base); g.prod(&mt[dSd_], true, &mt[a_], false).prod(&mt[dKh_], false, &mw, true);
        g.args.out_bf16 = bt[R2_]; run(g, "R2");
    }
    {   // db = M_gt * -(R2 T)
        GemmBuilder g(base); g.prod(&mt[R2_], false, &mt[T_], false); g.args.alpha = -1.f;
        g.args.mask = 2; g.args.out_bf16 = bt[db_]; run(g, "db");
    }
    {   // R3 = dSd b + dQh Wt
        GemmBuilder g(base); g.prod(&mt[dSd_], false, &mt[b_], false).prod(&mt[dQh_], false, &mw, true);
        g.args.out_bf16 = bt[R3_]; run(g, "R3");
    }
    {   // R4 = W dKht
        GemmBuilder g(base); g.prod(&mw, false, &mt[dKh_], true); g.args.out_bf16 = bt[R4_];
        run(g, "R4");
    }
    {   // dT = -at R3 - R4 b + dWt Wt
        GemmBuilder g(base);
        g.prod(&mt[a_], true, &mt[R3_], false, true).prod(&mt[R4_], false, &mt[b_], false, true)
            .prod(&mt[dWt_], false, &mw, true);
        g.args.out_bf16 = bt[dT_]; run(g, "dT");
    }
    {   // dX = Tit dT
        GemmBuilder g(base); g.prod(&mt[Ti_], true, &mt[dT_], false); g.args.out_f32 = ft[dXf_];
        g.args.out_bf16 = bt[dX_]; run(g, "dX");
    }
    {   // dLo = strict_lower(-dX Tt); dG = diag(beta) dLo
        GemmBuilder g(base); g.prod(&mt[dX_], false, &mt[T_], true); g.args.alpha = -1.f;
        g.args.mask = 3; g.args.out_f32 = ft[dLo_]; g.args.rowscale = ba.beta;
        g.args.out_bf16 = bt[dG_]; run(g, "dLo");
    }
    if (s != PATH_OK) return s;
    s = cuda_status(launch_bwd_dbeta(ft[dXf_], ft[dLo_], ft[G_], ba.dbeta, p.BH, p.L, p.Lp, p.N, st),
                    "dbeta");
    {   // dw (first half) = -Wt dAt - Zt dQh - Yt dKh + Tt dWt
        GemmBuilder g(base);
        g.prod(&mt[Wt_], false, &mt[dA_], true, true).prod(&mt[Z_], true, &mt[dQh_], false, true)
            .prod(&mt[Y_], true, &mt[dKh_], false, true).prod(&mt[T_], true, &mt[dWt_], false);
        g.args.out_f32 = ft[dwp_]; run(g, "dw1");
    }
    {   // dw = (first half) + dat Q + dbt K + dG W + dGt W
        GemmBuilder g(base);
        g.prod(&mt[da_], true, &mq, false).prod(&mt[db_], true, &mk, false)
            .prod(&mt[dG_], false, &mw, false).prod(&mt[dG_], true, &mw, false);
        g.args.E = ft[dwp_]; g.args.out_bf16 = static_cast<__nv_bfloat16 *>(ba.dw);
        g.args.out_final = 1; run(g, "dw");
    }
    {   // dq = dQh + dSd K + da W
        GemmBuilder g(base); g.prod(&mt[dSd_], false, &mk, false).prod(&mt[da_], false, &mw, false);
        g.args.E = dQh; g.args.out_bf16 = static_cast<__nv_bfloat16 *>(ba.dq); g.args.out_final = 1;
        run(g, "dq");
    }
    {   // dk = dKh + dSdt Q + db W
        GemmBuilder g(base); g.prod(&mt[dSd_], true, &mq, false).prod(&mt[db_], false, &mw, false);
        g.args.E = dKh; g.args.out_bf16 = static_cast<__nv_bfloat16 *>(ba.dk); g.args.out_final = 1;
        run(g, "dk");
    }
    return s;
}

}  // namespace

// Sets the message path_attn_last_error() returns on this host thread.
void record_last_error(const char *msg) {
    snprintf(g_msg, sizeof g_msg, "%s", msg ? msg : "");
}

// The descriptor of one backward pass over n (batch * head) slices, with the
// chunk resolved once for the whole call (the CUDA-core route's default chunk
// depends on batch * heads).
path_prefill_desc_t bwd_pass_desc(const path_prefill_desc_t *desc, int C, int n) {
    path_prefill_desc_t d = *desc;
    d.batch = 1;
    d.heads = n;
    d.chunk = C;
    return d;
}

// One pass of the backward over the p.BH heads the pointers start at (the
// workspace laid out by p).
path_status_t bwd_pass(const path_prefill_desc_t *desc, const BwdPlan &p, const void *q,
                       const void *k, const void *v, const void *w, const float *beta,
                       const float *log_f, const void *out, const float *lse, const void *dout,
                       const float *dlse, void *dq, void *dk, void *dv, void *dw, float *dbeta,
                       float *dlog_f, void *workspace, cudaStream_t st) {
    path_status_t s = PATH_OK;
    float *F = log_f ? at<float>(workspace, p.off_F) : nullptr;
    if (log_f) {
        s = cuda_status(launch_fox_prefix(log_f, F, p.L, p.Lp, p.BH, st), "fox prefix launch");
        if (s != PATH_OK) return s;
    }
    BwdArgs ba;
    ba.q = q; ba.k = k; ba.v = v; ba.w = w; ba.out = out; ba.dout = dout;
    ba.beta = beta; ba.lse = lse; ba.dlse = dlse;
    ba.Qh = at<float>(workspace, p.off_Qh);
    ba.Kh = at<float>(workspace, p.off_Kh);
    ba.Wt = at<float>(workspace, p.off_Wt);
    ba.F = F;
    ba.Qts = at<float>(workspace, p.off_Qts);
    ba.dQh = at<float>(workspace, p.off_dQh);
    ba.dKh = at<float>(workspace, p.off_dKh);
    ba.dV = at<float>(workspace, p.off_dV);
    ba.dA = at<float>(workspace, p.off_dA);
    ba.dF = log_f ? at<float>(workspace, p.off_dF) : nullptr;
    ba.scratch = at<float>(workspace, p.off_scratch);
    ba.dq = dq; ba.dk = dk; ba.dv = dv; ba.dw = dw; ba.dbeta = dbeta; ba.dlog_f = dlog_f;
    ba.scale = desc->scale;
    ba.BH = p.BH; ba.L = p.L; ba.Lp = p.Lp; ba.N = p.N; ba.C = p.C; ba.d = p.d;
    // PaTH-FoX takes the tensor-core route too, unless scale is 0 (its key-side
    // column sums are read back from the scaled bf16 dlogit tile)
    if (p.tc && (!log_f || desc->scale != 0.f)) {
        // tensor-core prep (bf16 Qh, Kh, Pm; its chunk outputs OD/LSD unused
        // here), then the tensor-core scan and key side, then the backward
        // prep (tensor-core contractions), then (PaTH-FoX) the dlog f suffix
        char *qh = at<char>(workspace, p.off_Qh), *kh = at<char>(workspace, p.off_Kh);
        char *pm = at<char>(workspace, p.off_Wt), *od = at<char>(workspace, p.off_Sd);
        char *qts = at<char>(workspace, p.off_Qts);
        const uint64_t npairs = (uint64_t)p.N * (p.N - 1) / 2;
        PrepTcMaps pm_maps;
        BwdTcMaps bm;
        const bool enc =
            encode_tmap_bf16_3d(&pm_maps.q, q, 128, p.L, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.k, k, 128, p.L, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.w, w, 128, p.L, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.v, v, 128, p.L, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.qh, qh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.kh, kh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.pm, pm, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&pm_maps.od, od, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&bm.qh, qh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&bm.kh, kh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&bm.pm, pm, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&bm.v, v, 128, p.L, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&bm.dout, dout, 128, p.L, p.BH, 64, 128) &&
            (npairs == 0 ||
             encode_tmap_bf16_3d(&bm.qts, qts, 128, npairs * 128, p.BH, 64, 128));
        if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
        const int sms = num_sms();
        if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
        memset(&pm_maps.vx, 0, sizeof pm_maps.vx);
        PrepTcArgs ta;
        ta.beta = beta;
        ta.F = nullptr;
        ta.scale = desc->scale;
        ta.LSD = reinterpret_cast<float *>(od + (size_t)p.BH * p.Lp * 128 * 2);
        ta.BH = p.BH; ta.L = p.L; ta.Lp = p.Lp; ta.N = p.N;
        set_whole_sequence(ta, p.N, p.L, p.Lp);
        ta.pm_transposed = 0;  // the backward's chain product reads Pm itself
        ta.err = error_flag_ptr();
        s = cuda_status(launch_prep_tc(pm_maps, ta, sms, st), "tensor-core prep launch");
        if (s != PATH_OK) return s;
        s = cuda_status(cudaMemsetAsync(at<char>(workspace, p.off_dQh), 0, p.total - p.off_dQh, st),
                        "accumulator clear");
        if (s != PATH_OK) return s;
        BwdTcArgs tb;
        tb.out = static_cast<const __nv_bfloat16 *>(out);
        tb.dout = static_cast<const __nv_bfloat16 *>(dout);
        tb.lse = lse; tb.dlse = dlse;
        tb.dQh = ba.dQh; tb.dKh = ba.dKh; tb.dV = ba.dV; tb.dA = ba.dA;
        tb.Dg = at<float>(workspace, p.off_Dg);
        tb.F = F;
        tb.dF = ba.dF;
        tb.scale = desc->scale;
        tb.BH = p.BH; tb.L = p.L; tb.Lp = p.Lp; tb.N = p.N;
        tb.err = error_flag_ptr();
        s = cuda_status(launch_bwd_rowdot(tb.out, tb.dout, dlse, at<float>(workspace, p.off_Dg),
                                          p.BH, p.L, p.Lp, st),
                        "row dot launch");
        if (s != PATH_OK) return s;
        s = cuda_status(launch_bwd_scan_tc(bm, tb, sms, st), "tensor-core backward scan launch");
        if (s != PATH_OK) return s;
        s = cuda_status(launch_bwd_kv_tc(bm, tb, sms, st), "tensor-core backward key-side launch");
        if (s != PATH_OK) return s;
        s = run_bwd_prep_tc(desc, p, ba, workspace, st);
        if (s != PATH_OK || !log_f) return s;
        return cuda_status(launch_fox_suffix(ba.dF, dlog_f, p.L, p.Lp, p.BH, st), "fox suffix launch");
    }
    PrepSimtArgs pa;
    pa.q = q; pa.k = k; pa.w = w; pa.beta = beta;
    pa.Qh = at<char>(workspace, p.off_Qh);
    pa.Kh = at<char>(workspace, p.off_Kh);
    pa.Wt = at<char>(workspace, p.off_Wt);
    pa.Sd = at<float>(workspace, p.off_Sd);
    pa.scratch = at<float>(workspace, p.off_scratch);
    pa.BH = p.BH; pa.L = p.L; pa.Lp = p.Lp; pa.N = p.N; pa.C = p.C; pa.d = p.d;
    pa.keys_only = 0;
    s = cuda_status(launch_prep_simt(pa, p.bf16, false, st), "backward prep launch");
    if (s != PATH_OK) return s;
    s = cuda_status(cudaMemsetAsync(at<char>(workspace, p.off_dQh), 0, p.total - p.off_dQh, st),
                    "accumulator clear");
    if (s != PATH_OK) return s;
    return cuda_status(launch_bwd(ba, p.bf16, st), "backward launch");
}

}  // namespace path

using namespace path;

extern "C" {

size_t path_attn_prefill_workspace_size(const path_prefill_desc_t *desc) {
    PrefillPlan p;
    if (plan_prefill(desc, &p) != PATH_OK) return 0;
    return p.total;
}

}  // extern "C"

namespace {

// overlap: the scan is launched next and may start while the prep runs (the
// fused forward); the prep then counts each head's finished chunks.
path_status_t prefill_prep(const path_prefill_desc_t *desc, const void *q, const void *k,
                           const void *v, const void *w, const float *beta, const float *log_f,
                           void *workspace, size_t workspace_bytes, path_stream_t stream,
                           bool overlap) {
    PrefillPlan p;
    path_status_t s = plan_prefill(desc, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {q, k, v, w, beta, workspace};
    const char *names[] = {"q", "k", "v", "w", "beta", "workspace"};
    for (int i = 0; i < 6; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (log_f && !aligned16(log_f)) return fail(PATH_ERR_INVALID_ARG, "log_f is not 16-byte aligned");
    if (workspace_bytes < p.total)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.total);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (log_f) {
        s = cuda_status(
            launch_fox_prefix(log_f, at<float>(workspace, p.off_F), p.L, p.Lp, p.BH, st),
            "fox prefix launch");
        if (s != PATH_OK) return s;
    }
    if (p.pad) {
        const void *src[4] = {q, k, w, v};
        for (int i = 0; i < 4 && s == PATH_OK; ++i)
            s = cuda_status(launch_pad_rows(src[i], pad_buf(workspace, p, i), (size_t)p.BH * p.L,
                                            p.d, st),
                            "pad launch");
        if (s != PATH_OK) return s;
        q = pad_buf(workspace, p, 0);
        k = pad_buf(workspace, p, 1);
        w = pad_buf(workspace, p, 2);
        v = pad_buf(workspace, p, 3);
    }
    if (p.tc) {
        PrepTcMaps maps;
        // head_dim 64: rows of 64, so that the second box of each row reads zeros
        const uint64_t din = p.d64 ? 64 : 128;
        const bool enc = encode_tmap_bf16_3d(&maps.q, q, din, p.L, p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.k, k, din, p.L, p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.w, w, din, p.L, p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.v, v, din, p.L, p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.qh, at<char>(workspace, p.off_Qh), 128, p.Lp,
                                             p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.kh, at<char>(workspace, p.off_Kh), 128, p.Lp,
                                             p.BH, 64, 128) &&
                         // the bf16 path keeps the chunk product where the fp32
                         // path keeps Wt, and each chunk's own attention block
                         // where the fp32 path keeps its within-chunk logits
                         encode_tmap_bf16_3d(&maps.pm, at<char>(workspace, p.off_Wt), 128, p.Lp,
                                             p.BH, 64, 128) &&
                         encode_tmap_bf16_3d(&maps.od, at<char>(workspace, p.off_Sd), 128, p.Lp,
                                             p.BH, 64, 128);
        if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
        memset(&maps.vx, 0, sizeof maps.vx);
        PrepTcArgs ta;
        ta.beta = beta;
        ta.F = log_f ? at<float>(workspace, p.off_F) : nullptr;
        ta.scale = desc->scale;
        ta.LSD = at<float>(workspace, p.off_Sd + (size_t)p.BH * p.Lp * 128 * 2);
        ta.BH = p.BH; ta.L = p.L; ta.Lp = p.Lp; ta.N = p.N;
        set_whole_sequence(ta, p.N, p.L, p.Lp);
        ta.err = error_flag_ptr();
        const int sms = num_sms();
        if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
        if (overlap) {
            // the scan's tile counter and the per-head counters, zeroed in
            // stream order before the prep
            s = cuda_status(cudaMemsetAsync(at<char>(workspace, p.off_tile), 0,
                                            kReadyOff + (size_t)4 * p.BH, st),
                            "counter reset");
            if (s != PATH_OK) return s;
            ta.ready = at<int>(workspace, p.off_tile + kReadyOff);
        }
        return cuda_status(launch_prep_tc(maps, ta, sms, st), "tensor-core prep launch");
    }
    PrepSimtArgs pa;
    pa.q = q; pa.k = k; pa.w = w; pa.beta = beta;
    pa.Qh = at<char>(workspace, p.off_Qh);
    pa.Kh = at<char>(workspace, p.off_Kh);
    pa.Wt = at<char>(workspace, p.off_Wt);
    pa.Sd = at<float>(workspace, p.off_Sd);
    pa.scratch = at<float>(workspace, p.off_scratch);
    pa.BH = p.BH; pa.L = p.L; pa.Lp = p.Lp; pa.N = p.N; pa.C = p.C; pa.d = p.d;
    pa.keys_only = 0;
    return cuda_status(launch_prep_simt(pa, p.bf16, false, st), "prep launch");
}

// overlap: launched directly after prefill_prep(..., overlap = true).
path_status_t prefill_scan(const path_prefill_desc_t *desc, const void *w, const void *v,
                           const float *log_f, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, path_stream_t stream, bool overlap) {
    PrefillPlan p;
    path_status_t s = plan_prefill(desc, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {w, v, out, workspace};
    const char *names[] = {"w", "v", "out", "workspace"};
    for (int i = 0; i < 4; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (lse && !aligned16(lse)) return fail(PATH_ERR_INVALID_ARG, "lse is not 16-byte aligned");
    if (workspace_bytes < p.total)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.total);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const void *Qh = at<char>(workspace, p.off_Qh), *Kh = at<char>(workspace, p.off_Kh);
    const void *Wt = at<char>(workspace, p.off_Wt);
    const float *Sd = at<float>(workspace, p.off_Sd);
    const float *F = log_f ? at<float>(workspace, p.off_F) : nullptr;
    void *out_user = out;
    if (p.pad) {
        v = pad_buf(workspace, p, 3);
        out = pad_buf(workspace, p, 4);
    }
    if (p.tc) {
        FlashTcMaps maps;
        // head_dim 64 scans at 64: the 64 x 64 corner of each chunk's Pm^T and
        // the first 64 columns of Qh and Kh, which are exact (the prep's padded
        // coordinates carry no weight)
        const int ds = p.d64 ? 64 : 128;
        const bool enc =
            encode_tmap_bf16_3d(&maps.qh, Qh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&maps.kh, Kh, 128, p.Lp, p.BH, 64, 128) &&
            encode_tmap_bf16_3d(&maps.pm, Wt, 128, p.Lp, p.BH, 64, ds) &&
            encode_tmap_bf16_3d(&maps.v, v, ds, p.L, p.BH, 64, 128);
        if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
        FlashTcArgs ta;
        ta.OD = reinterpret_cast<const __nv_bfloat16 *>(Sd);
        ta.LSD = reinterpret_cast<const float *>(reinterpret_cast<const char *>(Sd) +
                                                 (size_t)p.BH * p.Lp * 128 * 2);
        ta.F = F; ta.out = static_cast<__nv_bfloat16 *>(out); ta.lse = lse;
        ta.scale = desc->scale; ta.BH = p.BH; ta.L = p.L; ta.Lp = p.Lp; ta.N = p.N;
        ta.cm = ChunkMap{1, 0, p.N};
        ta.nloc = p.N; ta.Lq = p.Lp; ta.Lout = p.L; ta.zs = p.BH; ta.d = ds;
        ta.tile_ctr = at<int>(workspace, p.off_tile);
        ta.tile_group = desc->scan_group;
        ta.ready = overlap ? at<int>(workspace, p.off_tile + kReadyOff) : nullptr;
        ta.err = error_flag_ptr();
        const int sms = num_sms();
        if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
        s = cuda_status(launch_flash_tc(maps, ta, sms, st, overlap), "tensor-core scan launch");
        if (s != PATH_OK || !p.pad) return s;
        return cuda_status(launch_unpad_rows(out, out_user, (size_t)p.BH * p.L, p.d, st),
                           "unpad launch");
    }
    FlashSimtArgs fa;
    fa.Qh = Qh; fa.Kh = Kh; fa.Wt = Wt; fa.w = w; fa.v = v;
    fa.Sd = Sd; fa.F = F; fa.out = out; fa.lse = lse; fa.scale = desc->scale;
    fa.BH = p.BH; fa.L = p.L; fa.Lp = p.Lp; fa.N = p.N; fa.C = p.C; fa.d = p.d;
    return cuda_status(launch_flash_simt(fa, p.bf16, st), "scan launch");
}

}  // namespace

extern "C" {

path_status_t path_attn_prefill_prep(const path_prefill_desc_t *desc, const void *q,
                                     const void *k, const void *v, const void *w,
                                     const float *beta, const float *log_f, void *workspace,
                                     size_t workspace_bytes, path_stream_t stream) {
    return prefill_prep(desc, q, k, v, w, beta, log_f, workspace, workspace_bytes, stream, false);
}

path_status_t path_attn_prefill_scan(const path_prefill_desc_t *desc, const void *w,
                                     const void *v, const float *log_f, void *out, float *lse,
                                     void *workspace, size_t workspace_bytes,
                                     path_stream_t stream) {
    return prefill_scan(desc, w, v, log_f, out, lse, workspace, workspace_bytes, stream, false);
}

path_status_t path_attn_prefill_fwd(const path_prefill_desc_t *desc, const void *q,
                                    const void *k, const void *v, const void *w,
                                    const float *beta, const float *log_f, void *out,
                                    float *lse, void *workspace, size_t workspace_bytes,
                                    path_stream_t stream) {
    if (!v) return fail(PATH_ERR_INVALID_ARG, "v is NULL");
    if (!out) return fail(PATH_ERR_INVALID_ARG, "out is NULL");
    if (!aligned16(v)) return fail(PATH_ERR_INVALID_ARG, "v is not 16-byte aligned");
    if (!aligned16(out)) return fail(PATH_ERR_INVALID_ARG, "out is not 16-byte aligned");
    if (lse && !aligned16(lse)) return fail(PATH_ERR_INVALID_ARG, "lse is not 16-byte aligned");
    // the scan starts on the SMs the prep's last chunks leave idle
    path_status_t s = prefill_prep(desc, q, k, v, w, beta, log_f, workspace, workspace_bytes,
                                   stream, true);
    if (s != PATH_OK) return s;
    return prefill_scan(desc, w, v, log_f, out, lse, workspace, workspace_bytes, stream, true);
}

size_t path_attn_prefill_bwd_workspace_size(const path_prefill_desc_t *desc) {
    BwdPlan p;
    if (plan_bwd(desc, &p) != PATH_OK) return 0;
    return p.total;
}

path_status_t path_attn_prefill_bwd(const path_prefill_desc_t *desc, const void *q,
                                    const void *k, const void *v, const void *w,
                                    const float *beta, const float *log_f, const void *out,
                                    const float *lse, const void *dout, const float *dlse,
                                    void *dq, void *dk, void *dv, void *dw, float *dbeta,
                                    float *dlog_f, void *workspace, size_t workspace_bytes,
                                    path_stream_t stream) {
    BwdPlan full;
    path_status_t s = plan_bwd(desc, &full);
    if (s != PATH_OK) return s;
    const void *req[] = {q, k, v, w, beta, out, lse, dout, dq, dk, dv, dw, dbeta, workspace};
    const char *names[] = {"q", "k", "v", "w", "beta", "out", "lse", "dout", "dq", "dk",
                           "dv", "dw", "dbeta", "workspace"};
    for (int i = 0; i < 14; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    const void *opt[] = {log_f, dlse, dlog_f};
    const char *onames[] = {"log_f", "dlse", "dlog_f"};
    for (int i = 0; i < 3; ++i)
        if (opt[i] && !aligned16(opt[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", onames[i]);
    if (!log_f != !dlog_f)
        return fail(PATH_ERR_INVALID_ARG, "dlog_f must be given exactly when log_f is");
    // heads per pass: as many as the workspace holds (all of them for
    // path_attn_prefill_bwd_workspace_size bytes, one at the minimum)
    int hb = full.BH;
    if (workspace_bytes < full.total) {
        int lo = 0, hi = full.BH;  // lo fits (0 trivially), hi does not
        while (hi - lo > 1) {
            const int mid = lo + (hi - lo) / 2;
            BwdPlan pm;
            path_prefill_desc_t dm = bwd_pass_desc(desc, full.C, mid);
            if (plan_bwd(&dm, &pm) == PATH_OK && pm.total <= workspace_bytes) lo = mid;
            else hi = mid;
        }
        hb = lo;
        if (hb == 0) {
            BwdPlan p1;
            path_prefill_desc_t d1 = bwd_pass_desc(desc, full.C, 1);
            plan_bwd(&d1, &p1);
            return fail(PATH_ERR_INVALID_ARG,
                        "workspace too small: %zu bytes; one head per pass needs %zu "
                        "(path_attn_prefill_bwd_workspace_min)", workspace_bytes, p1.total);
        }
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t es = full.bf16 ? 2 : 4;
    const size_t act = (size_t)full.L * full.d * es;  // bytes per head of q, k, ..., dw
    const size_t vec = (size_t)full.L;                // floats per head of beta, lse, ...
    for (int h0 = 0; h0 < full.BH; h0 += hb) {
        const int n = full.BH - h0 < hb ? full.BH - h0 : hb;
        path_prefill_desc_t dn = bwd_pass_desc(desc, full.C, n);
        BwdPlan p;
        s = plan_bwd(&dn, &p);
        if (s != PATH_OK) return s;
        auto A = [&](const void *x) -> const void * {
            return static_cast<const char *>(x) + (size_t)h0 * act;
        };
        auto M = [&](void *x) -> void * { return static_cast<char *>(x) + (size_t)h0 * act; };
        auto Vc = [&](const float *x) -> const float * { return x ? x + (size_t)h0 * vec : x; };
        auto Vm = [&](float *x) -> float * { return x ? x + (size_t)h0 * vec : x; };
        s = bwd_pass(&dn, p, A(q), A(k), A(v), A(w), Vc(beta), Vc(log_f), A(out), Vc(lse),
                     A(dout), Vc(dlse), M(dq), M(dk), M(dv), M(dw), Vm(dbeta), Vm(dlog_f),
                     workspace, st);
        if (s != PATH_OK) return s;
    }
    return ok();
}

size_t path_attn_prefill_bwd_workspace_min(const path_prefill_desc_t *desc) {
    BwdPlan full;
    if (plan_bwd(desc, &full) != PATH_OK) return 0;
    path_prefill_desc_t d1 = bwd_pass_desc(desc, full.C, 1);
    BwdPlan p1;
    if (plan_bwd(&d1, &p1) != PATH_OK) return 0;
    return p1.total;
}

size_t path_attn_decode_workspace_size(const path_decode_desc_t *desc) {
    DecodePlan p;
    if (plan_decode(desc, &p) != PATH_OK) return 0;
    return p.ws_bytes;
}

path_status_t path_attn_decode_step(const path_decode_desc_t *desc, void *k_cache,
                                    void *v_cache, int32_t cache_len, const void *q_t,
                                    const void *k_t, const void *v_t, const void *w_t,
                                    const float *beta_t, void *out, void *workspace,
                                    size_t workspace_bytes, path_stream_t stream) {
    DecodePlan p;
    path_status_t s = plan_decode(desc, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {k_cache, v_cache, q_t, k_t, v_t, w_t, beta_t, out, workspace};
    const char *names[] = {"k_cache", "v_cache", "q_t", "k_t", "v_t", "w_t", "beta_t", "out",
                           "workspace"};
    for (int i = 0; i < 9; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (cache_len < 0 || cache_len >= desc->cache_capacity)
        return fail(PATH_ERR_INVALID_ARG, "cache_len %d outside [0, capacity %d)", cache_len,
                    desc->cache_capacity);
    if (workspace_bytes < p.ws_bytes)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.ws_bytes);
    DecodeArgs a;
    a.k_cache = k_cache; a.v_cache = v_cache; a.q_t = q_t; a.k_t = k_t; a.v_t = v_t;
    a.w_t = w_t; a.beta_t = beta_t; a.out = out;
    a.partials = static_cast<float *>(workspace);
    a.scale = desc->scale;
    a.BH = p.BH; a.d = desc->head_dim; a.cap = desc->cache_capacity; a.cache_len = cache_len;
    a.keys_per_split = p.keys_per_split; a.max_splits = p.max_splits;
    return cuda_status(launch_decode(a, reinterpret_cast<cudaStream_t>(stream)), "decode launch");
}

path_status_t path_attn_decode_step_fox(const path_decode_desc_t *desc, void *k_cache,
                                        void *v_cache, float *f_cache, int32_t cache_len,
                                        const void *q_t, const void *k_t, const void *v_t,
                                        const void *w_t, const float *beta_t,
                                        const float *log_f_t, void *out, void *workspace,
                                        size_t workspace_bytes, path_stream_t stream) {
    DecodePlan p;
    path_status_t s = plan_decode(desc, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {k_cache, v_cache, q_t, k_t, v_t, w_t, beta_t, out, workspace};
    const char *names[] = {"k_cache", "v_cache", "q_t", "k_t", "v_t", "w_t", "beta_t", "out",
                           "workspace"};
    for (int i = 0; i < 9; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (!f_cache) return fail(PATH_ERR_INVALID_ARG, "f_cache is NULL");
    if (!log_f_t) return fail(PATH_ERR_INVALID_ARG, "log_f_t is NULL");
    if ((reinterpret_cast<uintptr_t>(f_cache) & 3u) || (reinterpret_cast<uintptr_t>(log_f_t) & 3u))
        return fail(PATH_ERR_INVALID_ARG, "f_cache and log_f_t must be 4-byte aligned");
    if (cache_len < 0 || cache_len >= desc->cache_capacity)
        return fail(PATH_ERR_INVALID_ARG, "cache_len %d outside [0, capacity %d)", cache_len,
                    desc->cache_capacity);
    if (workspace_bytes < p.ws_bytes)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.ws_bytes);
    DecodeArgs a;
    a.k_cache = k_cache; a.v_cache = v_cache; a.q_t = q_t; a.k_t = k_t; a.v_t = v_t;
    a.w_t = w_t; a.beta_t = beta_t; a.out = out;
    a.partials = static_cast<float *>(workspace);
    a.scale = desc->scale;
    a.BH = p.BH; a.d = desc->head_dim; a.cap = desc->cache_capacity; a.cache_len = cache_len;
    a.keys_per_split = p.keys_per_split; a.max_splits = p.max_splits;
    a.f_cache = f_cache; a.log_f_t = log_f_t;
    return cuda_status(launch_decode(a, reinterpret_cast<cudaStream_t>(stream)),
                       "FoX decode launch");
}

path_status_t path_attn_fox_prefix(const float *log_f, float *f_out, int32_t heads_total,
                                   int32_t len, int32_t out_len, path_stream_t stream) {
    if (!log_f || !f_out) return fail(PATH_ERR_INVALID_ARG, "log_f and f_out must be non-NULL");
    if (heads_total < 1 || len < 1 || out_len < len)
        return fail(PATH_ERR_INVALID_ARG,
                    "need heads_total >= 1 and 1 <= len <= out_len (got %d, %d, %d)",
                    heads_total, len, out_len);
    return cuda_status(launch_fox_prefix(log_f, f_out, len, out_len, heads_total,
                                         reinterpret_cast<cudaStream_t>(stream)),
                       "FoX prefix launch");
}

size_t path_attn_build_kcache_workspace_size(const path_prefill_desc_t *desc) {
    KcachePlan p;
    if (plan_kcache(desc, &p) != PATH_OK) return 0;
    return p.total;
}

path_status_t path_attn_build_kcache(const path_prefill_desc_t *desc, const void *k,
                                     const void *w, const float *beta, void *k_cache,
                                     int32_t cache_capacity, void *workspace,
                                     size_t workspace_bytes, path_stream_t stream) {
    KcachePlan p;
    path_status_t s = plan_kcache(desc, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {k, w, beta, k_cache, workspace};
    const char *names[] = {"k", "w", "beta", "k_cache", "workspace"};
    for (int i = 0; i < 5; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (cache_capacity < desc->seq_len)
        return fail(PATH_ERR_INVALID_ARG, "cache_capacity %d < seq_len %d", cache_capacity,
                    desc->seq_len);
    if (workspace_bytes < p.total)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.total);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int d = p.d;
    for (int h0 = 0; h0 < p.BH; h0 += p.HB) {
        const int hb = (p.BH - h0 < p.HB) ? p.BH - h0 : p.HB;
        const size_t in_off = (size_t)h0 * p.L * d;
        PrepSimtArgs pa;
        pa.q = static_cast<const __nv_bfloat16 *>(k) + in_off;
        pa.k = static_cast<const __nv_bfloat16 *>(k) + in_off;
        pa.w = static_cast<const __nv_bfloat16 *>(w) + in_off;
        pa.beta = beta + (size_t)h0 * p.L;
        pa.Qh = at<float>(workspace, p.off_Kh);  // unused in keys-only mode
        pa.Kh = at<float>(workspace, p.off_Kh);
        pa.Wt = at<float>(workspace, p.off_Wt);
        pa.Sd = at<float>(workspace, p.off_scratch);  // unused in keys-only mode
        pa.scratch = at<float>(workspace, p.off_scratch);
        pa.BH = hb; pa.L = p.L; pa.Lp = p.Lp; pa.N = p.N; pa.C = p.C; pa.d = d;
        pa.keys_only = 1;
        s = cuda_status(launch_prep_simt(pa, true, false, st), "kcache prep launch");
        if (s != PATH_OK) return s;
        KcacheArgs ka;
        ka.w = static_cast<const __nv_bfloat16 *>(w) + in_off;
        ka.Kh = at<float>(workspace, p.off_Kh);
        ka.Wt = at<float>(workspace, p.off_Wt);
        ka.Pi = at<float>(workspace, p.off_Pi);
        ka.Mout = at<float>(workspace, p.off_Mout);
        ka.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
        ka.h0 = h0; ka.HB = hb; ka.cap = cache_capacity; ka.L = p.L; ka.Lp = p.Lp;
        ka.N = p.N; ka.C = p.C; ka.d = d; ka.G = p.G; ka.S = p.S;
        s = cuda_status(launch_kcache_sweep(ka, st), "kcache sweep launch");
        if (s != PATH_OK) return s;
    }
    return ok();
}

int32_t path_attn_cp_local_len(const path_prefill_desc_t *desc, int32_t world, int32_t rank) {
    CpPlan p;
    if (plan_cp(desc, world, rank, &p) != PATH_OK) return -1;
    return p.Lr;
}

path_status_t path_attn_cp_rows(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                int32_t *rows, int32_t capacity) {
    CpPlan p;
    path_status_t s = plan_cp(desc, world, rank, &p);
    if (s != PATH_OK) return s;
    if (p.Lr > 0 && !rows) return fail(PATH_ERR_INVALID_ARG, "rows is NULL");
    if (capacity < p.Lr)
        return fail(PATH_ERR_INVALID_ARG, "rows holds %d entries, the rank has %d rows", capacity,
                    p.Lr);
    int n = 0;
    for (int i = 0; i < p.nloc; ++i) {
        const int c = p.cm.global_of_local(i);
        for (int o = 0; o < 128 && c * 128 + o < p.L; ++o) rows[n++] = c * 128 + o;
    }
    return ok();
}

size_t path_attn_cp_exchange_bytes(const path_prefill_desc_t *desc, int32_t world) {
    CpPlan p;
    if (plan_cp(desc, world, 0, &p) != PATH_OK) return 0;
    return p.exchange;
}

size_t path_attn_cp_workspace_size(const path_prefill_desc_t *desc, int32_t world) {
    CpPlan p;
    if (plan_cp(desc, world, 0, &p) != PATH_OK) return 0;
    return p.total;
}

path_status_t path_attn_cp_prep(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                const void *q, const void *k, const void *v, const void *w,
                                const float *beta, const float *log_f, void *exchange,
                                void *workspace, size_t workspace_bytes, path_stream_t stream) {
    CpPlan p;
    path_status_t s = plan_cp(desc, world, rank, &p);
    if (s != PATH_OK) return s;
    const void *req[] = {q, k, v, w, beta, exchange, workspace};
    const char *names[] = {"q", "k", "v", "w", "beta", "exchange", "workspace"};
    for (int i = 0; i < 7; ++i) {
        if (i < 5 && p.Lr == 0) continue;  // a rank without rows reads no input
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (log_f && !aligned16(log_f)) return fail(PATH_ERR_INVALID_ARG, "log_f is not 16-byte aligned");
    if (workspace_bytes < p.total)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.total);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *F = at<float>(workspace, p.off_F);
    if (log_f) {
        // prefix sums over the whole sequence: the scan needs them at every chunk
        s = cuda_status(launch_fox_prefix(log_f, F, p.L, p.Lp, p.BH, st), "fox prefix launch");
        if (s != PATH_OK) return s;
    }
    if (p.nloc == 0) return ok();
    char *ex = static_cast<char *>(exchange);
    PrepTcMaps maps;
    const bool enc = encode_tmap_bf16_3d(&maps.q, q, 128, p.Lr, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.k, k, 128, p.Lr, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.w, w, 128, p.Lr, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.v, v, 128, p.Lr, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.qh, at<char>(workspace, p.off_Qh), 128, p.Lq,
                                         p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.od, at<char>(workspace, p.off_OD), 128, p.Lq,
                                         p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.kh, ex, 128, p.Lq, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.pm, ex + p.section, 128, p.Lq, p.BH, 64, 128) &&
                     encode_tmap_bf16_3d(&maps.vx, ex + 2 * p.section, 128, p.Lq, p.BH, 64, 128);
    if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
    PrepTcArgs ta;
    ta.beta = beta;
    ta.F = log_f ? F : nullptr;
    ta.scale = desc->scale;
    ta.LSD = at<float>(workspace, p.off_LSD);
    ta.BH = p.BH; ta.L = p.L; ta.Lp = p.Lp; ta.N = p.N;
    ta.cm = p.cm; ta.nloc = p.nloc; ta.Lin = p.Lr; ta.Lq = p.Lq; ta.copy_v = 1;
    ta.pm_transposed = 1; ta.ready = nullptr;
    ta.err = error_flag_ptr();
    const int sms = num_sms();
    if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
    return cuda_status(launch_prep_tc(maps, ta, sms, st), "tensor-core prep launch");
}

path_status_t path_attn_cp_scan(const path_prefill_desc_t *desc, int32_t world, int32_t rank,
                                const float *log_f, const void *exchange_all, void *out,
                                float *lse, void *workspace, size_t workspace_bytes,
                                path_stream_t stream) {
    CpPlan p;
    path_status_t s = plan_cp(desc, world, rank, &p);
    if (s != PATH_OK) return s;
    if (p.nloc == 0) return ok();
    const void *req[] = {exchange_all, out, workspace};
    const char *names[] = {"exchange_all", "out", "workspace"};
    for (int i = 0; i < 3; ++i) {
        if (!req[i]) return fail(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return fail(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (lse && !aligned16(lse)) return fail(PATH_ERR_INVALID_ARG, "lse is not 16-byte aligned");
    if (workspace_bytes < p.total)
        return fail(PATH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes,
                    p.total);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const char *ex = static_cast<const char *>(exchange_all);
    // the gathered blocks: [world][Kh, Pm, V][BH][Lq][128], so chunk c of head
    // bh in section s sits at z = owner * 3 * BH + s * BH + bh
    const uint64_t zall = (uint64_t)world * 3 * p.BH;
    FlashTcMaps maps;
    const bool enc =
        encode_tmap_bf16_3d(&maps.qh, at<char>(workspace, p.off_Qh), 128, p.Lq, p.BH, 64, 128) &&
        encode_tmap_bf16_3d(&maps.kh, ex, 128, p.Lq, zall, 64, 128) &&
        encode_tmap_bf16_3d(&maps.pm, ex + p.section, 128, p.Lq, zall - p.BH, 64, 128) &&
        encode_tmap_bf16_3d(&maps.v, ex + 2 * p.section, 128, p.Lq, zall - 2 * p.BH, 64, 128);
    if (!enc) return fail(PATH_ERR_CUDA, "TMA descriptor encoding failed");
    FlashTcArgs ta;
    ta.OD = at<const __nv_bfloat16>(workspace, p.off_OD);
    ta.LSD = at<const float>(workspace, p.off_LSD);
    ta.F = log_f ? at<const float>(workspace, p.off_F) : nullptr;
    ta.out = static_cast<__nv_bfloat16 *>(out);
    ta.lse = lse;
    ta.scale = desc->scale;
    ta.BH = p.BH; ta.L = p.L; ta.Lp = p.Lp; ta.N = p.N;
    ta.cm = p.cm; ta.nloc = p.nloc; ta.Lq = p.Lq; ta.Lout = p.Lr; ta.zs = 3 * p.BH; ta.d = 128;
    ta.tile_ctr = at<int>(workspace, p.off_tile);
    ta.tile_group = desc->scan_group;
    ta.ready = nullptr;
    ta.err = error_flag_ptr();
    const int sms = num_sms();
    if (sms <= 0) return fail(PATH_ERR_CUDA, "device query failed");
    return cuda_status(launch_flash_tc(maps, ta, sms, st), "tensor-core scan launch");
}

path_status_t path_attn_device_status(int32_t clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(PATH_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
    uint32_t *fp = error_flag_ptr();
    if (!fp) return fail(PATH_ERR_CUDA, "error flag lookup failed");
    uint32_t v = 0;
    e = cudaMemcpy(&v, fp, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(PATH_ERR_CUDA, "flag read: %s", cudaGetErrorString(e));
    if (clear) {
        uint32_t z = 0;
        e = cudaMemcpy(fp, &z, sizeof z, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(PATH_ERR_CUDA, "flag clear: %s", cudaGetErrorString(e));
    }
    if (v & kErrTimeout) return fail(PATH_ERR_TIMEOUT, "a device-side wait ran out");
    return ok();
}

path_status_t path_attn_selftest_bounded_wait(uint32_t limit_us, path_stream_t stream) {
    if (limit_us == 0 || limit_us > 10000000u)
        return fail(PATH_ERR_INVALID_ARG, "limit_us must be in 1..10000000");
    uint32_t *fp = error_flag_ptr();
    if (!fp) return fail(PATH_ERR_CUDA, "error flag lookup failed");
    return cuda_status(launch_selftest_wait(fp, (uint64_t)limit_us * 1000ull,
                                            reinterpret_cast<cudaStream_t>(stream)),
                       "selftest launch");
}

const char *path_attn_status_string(path_status_t status) {
    switch (status) {
    case PATH_OK: return "PATH_OK";
    case PATH_ERR_INVALID_ARG: return "PATH_ERR_INVALID_ARG";
    case PATH_ERR_UNSUPPORTED: return "PATH_ERR_UNSUPPORTED";
    case PATH_ERR_CUDA: return "PATH_ERR_CUDA";
    case PATH_ERR_TIMEOUT: return "PATH_ERR_TIMEOUT";
    }
    return "PATH_ERR_UNKNOWN";
}

const char *path_attn_last_error(void) { return g_msg; }

int32_t path_attn_version(void) { return 100; }

}  // extern "C"

// ------------------------------------------------------------ selftest kernel

namespace path {
namespace {
// A global counter nothing raises (the form of the scan's wait for the
// prep's chunks in the one-call forward).
__device__ int g_selftest_counter = 0;

// Lane 0 waits on an mbarrier that expects an arrival nobody makes; lane 1
// waits for the counter above to reach 1.  Each has its own abort word, so
// that each wait runs out on its own limit.
__global__ void selftest_wait_kernel(uint32_t *err_flag, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_word[2];
    if (threadIdx.x == 0) {
        abort_word[0] = abort_word[1] = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err_flag, &abort_word[0], limit_ns);
    if (threadIdx.x == 1) counter_wait(&g_selftest_counter, 1, err_flag, &abort_word[1], limit_ns);
}
}  // namespace

cudaError_t launch_selftest_wait(uint32_t *err_flag, uint64_t limit_ns, cudaStream_t st) {
    selftest_wait_kernel<<<1, 32, 0, st>>>(err_flag, limit_ns);
    return cudaGetLastError();
}
}  // namespace path
