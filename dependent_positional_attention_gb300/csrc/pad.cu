// Zero-padding of bf16 rows to head_dim 128 and back.
//
// PaTH is unchanged by zero-padding the head dimension: with w padded by
// zeros every transition H = I - beta w w^T is the identity on the added
// coordinates, zero-padded q and k leave every logit as it was, and
// zero-padded v only adds zero output columns.  bf16 calls with head_dim a
// multiple of 8 below 128 therefore run the head_dim-128 tensor-core kernels
// on padded copies of q, k, v, w (the caller's scale is kept) and copy the
// first head_dim columns of the output back.

#include "common.cuh"
#include "kernels.h"

namespace path {
namespace {

constexpr int kD = 128;

// dst[row][0..d) = src[row][0..d), dst[row][d..128) = 0; one thread per 16 bytes of dst.
__global__ void pad_rows_kernel(const __nv_bfloat16 *src, __nv_bfloat16 *dst, size_t rows, int d) {
    const size_t total = rows * (kD / 8);
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t row = e / (kD / 8);
        const int c = (int)(e % (kD / 8));
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (c * 8 < d) v = *reinterpret_cast<const uint4 *>(src + row * d + c * 8);
        *reinterpret_cast<uint4 *>(dst + row * kD + c * 8) = v;
    }
}

// dst[row][0..d) = src[row][0..d) for src rows of 128; one thread per 16 bytes of dst.
__global__ void unpad_rows_kernel(const __nv_bfloat16 *src, __nv_bfloat16 *dst, size_t rows, int d) {
    const int per = d / 8;
    const size_t total = rows * per;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t row = e / per;
        const int c = (int)(e % per);
        *reinterpret_cast<uint4 *>(dst + row * d + c * 8) =
            *reinterpret_cast<const uint4 *>(src + row * kD + c * 8);
    }
}

int blocks_for(size_t work) {
    const size_t b = (work + 255) / 256;
    return (int)(b < 8192 ? (b > 0 ? b : 1) : 8192);
}

}  // namespace

cudaError_t launch_pad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st) {
    pad_rows_kernel<<<blocks_for(rows * (kD / 8)), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(src), static_cast<__nv_bfloat16 *>(dst), rows, d);
    return cudaGetLastError();
}

cudaError_t launch_unpad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st) {
    unpad_rows_kernel<<<blocks_for(rows * (d / 8)), 256, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(src), static_cast<__nv_bfloat16 *>(dst), rows, d);
    return cudaGetLastError();
}

}  // namespace path
