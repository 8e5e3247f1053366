// Decode step that allocates nothing: path_attn_decode_step_noalloc.
//
// Some callers cannot hand the library a workspace: code loaded as a plugin
// into a host framework that owns every byte of device memory and offers
// its plugins no allocator, or a token loop that must never call cudaMalloc
// because an allocation can synchronise the device in the middle of
// generation.  For them this file keeps the split-KV partial results of the
// decode step in a fixed, file-scope device array instead of caller memory.
// The kernels are the ones path_attn_decode_step launches; only where their
// partials live differs.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include "../../include/path_attn.h"
#include "ctx_symbol.h"
#include "kernels.h"

namespace path {

void record_last_error(const char *msg);  // api.cu

namespace {

// 2 Mi floats = 8 MiB.  Every GPU that loads the library holds this array
// until the process exits.
constexpr size_t kScratchFloats = size_t(1) << 21;
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

// Host code may not use g_decode_scratch's name as an address (it is a host
// stand-in); its device address is looked up with the caller's context
// current and cached per context (ctx_symbol.h).
cudaError_t lookup_scratch(void **p) { return cudaGetSymbolAddress(p, g_decode_scratch); }
PerContextAddress g_scratch_addr(&lookup_scratch);

path_status_t reject(path_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    record_last_error(buf);
    return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace path

extern "C" path_status_t path_attn_decode_step_noalloc(
    const path_decode_desc_t *desc, void *k_cache, void *v_cache, int32_t cache_len,
    const void *q_t, const void *k_t, const void *v_t, const void *w_t, const float *beta_t,
    void *out, path_stream_t stream) {
    using namespace path;
    if (!desc) return reject(PATH_ERR_INVALID_ARG, "desc is NULL");
    if (desc->batch < 1 || desc->heads < 1 || desc->head_dim < 1 || desc->cache_capacity < 1)
        return reject(PATH_ERR_INVALID_ARG,
                      "batch, heads, head_dim, cache_capacity must be >= 1");
    if (desc->dtype != PATH_F32 && desc->dtype != PATH_BF16)
        return reject(PATH_ERR_INVALID_ARG, "dtype must be PATH_F32 or PATH_BF16");
    if (!(desc->scale == desc->scale) || isinf(desc->scale))
        return reject(PATH_ERR_INVALID_ARG, "scale must be finite");
    if (desc->dtype != PATH_BF16) return reject(PATH_ERR_UNSUPPORTED, "decode needs PATH_BF16");
    if (desc->head_dim != 64 && desc->head_dim != 128)
        return reject(PATH_ERR_UNSUPPORTED, "decode needs head_dim 64 or 128");
    const long long BH = (long long)desc->batch * desc->heads;
    if (BH > 65535) return reject(PATH_ERR_UNSUPPORTED, "batch*heads must be <= 65535");
    const void *req[] = {k_cache, v_cache, q_t, k_t, v_t, w_t, beta_t, out};
    const char *names[] = {"k_cache", "v_cache", "q_t", "k_t", "v_t", "w_t", "beta_t", "out"};
    for (int i = 0; i < 8; ++i) {
        if (!req[i]) return reject(PATH_ERR_INVALID_ARG, "%s is NULL", names[i]);
        if (!aligned16(req[i]))
            return reject(PATH_ERR_INVALID_ARG, "%s is not 16-byte aligned", names[i]);
    }
    if (cache_len < 0 || cache_len >= desc->cache_capacity)
        return reject(PATH_ERR_INVALID_ARG, "cache_len %d outside [0, capacity %d)", cache_len,
                      desc->cache_capacity);
    const int per = decode_keys_per_split();
    const int nsplit = (cache_len + per - 1) / per;
    const int slots = nsplit > 0 ? nsplit : 1;
    const size_t need = (size_t)BH * slots * (desc->head_dim + 2);
    if (need > kScratchFloats)
        return reject(PATH_ERR_INVALID_ARG,
                      "this step needs %zu bytes of split-KV scratch but the fixed scratch of "
                      "path_attn_decode_step_noalloc holds %zu bytes (batch*heads*ceil(cache_len/"
                      "%d)*(head_dim+2)*4); use path_attn_decode_step with a workspace",
                      need * 4, kScratchFloats * 4, per);
    void *scratch_v = nullptr;
    cudaError_t e = g_scratch_addr.get(&scratch_v);
    float *scratch = static_cast<float *>(scratch_v);
    if (e != cudaSuccess)
        return reject(PATH_ERR_CUDA, "scratch address lookup: %s", cudaGetErrorString(e));
    // Nothing in the scratch needs clearing: every partial the combine kernel
    // reads is written by the split kernel earlier in the same call.
    DecodeArgs a;
    a.k_cache = k_cache; a.v_cache = v_cache; a.q_t = q_t; a.k_t = k_t; a.v_t = v_t;
    a.w_t = w_t; a.beta_t = beta_t; a.out = out; a.partials = scratch;
    a.scale = desc->scale;
    a.BH = (int)BH; a.d = desc->head_dim; a.cap = desc->cache_capacity; a.cache_len = cache_len;
    a.keys_per_split = per; a.max_splits = slots;
    e = launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return reject(PATH_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    record_last_error("");
    return PATH_OK;
}
