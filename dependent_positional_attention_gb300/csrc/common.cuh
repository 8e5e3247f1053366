// Shared device-side helpers for libpath_attn (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace path {

// Device error flag bits (one 32-bit word owned by the library; its address
// is passed to every kernel that can wait).
enum : uint32_t { kErrTimeout = 1u };

// Element load/store helpers for the two supported element types.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_error(uint32_t *flag, uint32_t bits) {
    if (flag) atomicOr(flag, bits);
}

// ------------------------------------------------------------ mbarrier (CTA)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// One poll of the phase with the given parity, without a suspend-time hint
// (returns at once).
__device__ __forceinline__ bool mbar_poll(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// One wait of up to ~1 ms (the hardware may suspend the thread meanwhile).
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Slow path of mbar_wait: polls with the suspend hint and reads the global
// timer, which costs a few hundred cycles, so it is entered only after a
// first plain poll has failed.
__device__ __forceinline__ bool mbar_wait_slow(uint64_t *bar, uint32_t parity, uint32_t *err_flag,
                                            volatile int *abort_word, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_word && *abort_word) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            set_error(err_flag, kErrTimeout);
            if (abort_word) *abort_word = 1;
            return false;
        }
    }
}

// Bounded wait on the phase with the given parity.  Gives up after
// `limit_ns` of device time, sets the error flag and the CTA abort word, and
// returns false.  Also returns false once another role of the CTA has
// aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *err_flag,
                                          volatile int *abort_word, uint64_t limit_ns) {
    if (mbar_poll(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err_flag, abort_word, limit_ns);
}

constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s of device time

// ------------------------------------------------------ grid-level ordering

// Lets the grid launched after this one on the stream with programmatic
// stream serialisation start while this one still runs (a no-op otherwise).
// The dependent grid must then order its reads itself (counter_wait).
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Adds v to a global counter with release semantics at GPU scope: every write
// this thread has made or observed is visible to a thread that reads the new
// value with an acquire.
__device__ __forceinline__ void counter_release_add(int *p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int counter_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until the global counter *p reaches `target` (acquire at GPU
// scope).  Gives up like mbar_wait: after `limit_ns` of device time it sets
// the error flag and the CTA abort word and returns false; it also returns
// false once another role of the CTA has aborted.
__device__ __forceinline__ bool counter_wait(const int *p, int target, uint32_t *err_flag,
                                             volatile int *abort_word, uint64_t limit_ns) {
    if (counter_acquire(p) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(200);
        if (counter_acquire(p) >= target) return true;
        if (abort_word && *abort_word) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            set_error(err_flag, kErrTimeout);
            if (abort_word) *abort_word = 1;
            return false;
        }
    }
}

}  // namespace path
