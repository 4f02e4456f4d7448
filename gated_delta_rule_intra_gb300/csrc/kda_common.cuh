// Shared device helpers for the KDA intra-chunk backward kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int BT = 64;        // chunk length
constexpr int BC = 16;        // sub-block length
constexpr int KD = 128;       // head dimension
constexpr int NBLK = BT / BC; // 4 sub-blocks per chunk
constexpr float LN2 = 0.693147180559945309417232121458f;
constexpr int kMaxDev = 64;   // devices whose per-device launch state is cached

// Raise a kernel's dynamic shared-memory limit once per device (the attribute belongs
// to the device's copy of the function); `done` is the kernel's own per-device flag
// array.  Two threads racing here set the same value twice, which is harmless.
template <typename Kernel>
cudaError_t smem_limit_once(Kernel kern, int bytes, int dev, volatile int *done) {
    const bool cached = dev >= 0 && dev < kMaxDev;
    if (cached && done[dev]) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cached) done[dev] = 1;
    return e;
}

// 2^x on the SFU (MUFU.EX2), flush-to-zero.  Every argument passed here is <= 0 for
// inputs inside the method's premise (non-increasing chunk-local gate), so the
// result lies in [0, 1]; results below 2^-126 flush to 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <> __device__ __forceinline__ float to_f32<__half>(__half x) {
    return __half2float(x);
}

// Ampere-style 16-byte async global->shared copy (L2 only, bypassing L1).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Bounds-checked debug build (compiled with KDA_DEBUG_CHECKS): every global index a
// kernel computes is checked against its buffer's extent before the access; an index
// out of range sets `bit` in the caller's flag word (when one is set) and the access is
// skipped.  In the normal build the check is the constant true and compiles away.
constexpr unsigned DBG_STORE = 1u;  // an output index
constexpr unsigned DBG_LOAD = 2u;   // an input index
constexpr unsigned DBG_WAIT = 4u;   // a bounded wait gave up
#ifdef KDA_DEBUG_CHECKS
__device__ __forceinline__ bool dbg_ok(unsigned *flags, size_t idx, size_t n, unsigned bit) {
    if (idx < n) return true;
    if (flags) atomicOr(flags, bit);
    return false;
}
__device__ __forceinline__ void dbg_flag(unsigned *flags, bool fail, unsigned bit) {
    if (fail && flags) atomicOr(flags, bit);
}
#else
__device__ __forceinline__ bool dbg_ok(unsigned *, size_t, size_t, unsigned) { return true; }
__device__ __forceinline__ void dbg_flag(unsigned *, bool, unsigned) {}
#endif

// Decode a unit index into (b, h, chunk).  Heads vary fastest so that CTAs that
// run at the same time read neighbouring addresses of the [B, T, H, *] tensors.
struct Unit {
    int b, h, c;
};
// (The host rejects problems with 2^31 or more units, so 32-bit division suffices.)
__device__ __forceinline__ Unit decode_unit(long long u, int H, int NT) {
    const unsigned uu = (unsigned)u, q = uu / (unsigned)H;
    Unit x;
    x.h = (int)(uu - q * (unsigned)H);
    x.c = (int)(q % (unsigned)NT);
    x.b = (int)(q / (unsigned)NT);
    return x;
}

// Global row index of in-chunk row r of a unit in a [B, T, H, *] tensor.
__device__ __forceinline__ size_t grow(const Unit &x, int r, int T, int H) {
    return ((size_t)x.b * (size_t)T + (size_t)x.c * BT + (size_t)r) * (size_t)H +
           (size_t)x.h;
}

}  // namespace kda
