// common.cuh -- shared device helpers and the host launch wrapper of libdion.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>
#include <atomic>
#include <utility>

#include "../../include/dion.h"

namespace dion {

typedef __nv_bfloat16 bf16;

// Bits of the device status word (see dion_get_status).
enum : int { kStatusPivot = 1, kStatusNonFinite = 2 };

// A Gram matrix S = I + E with max|E| <= kNearIdentityTol takes the
// first-order inverse of its Cholesky factor, Z = I - F with
// F = strictly_lower(E) + diag(E)/2.  The result then has
// P^T P - I = -(F F + F F^T + F^T F^T) + O(E^3): entries of order sqrt(r) E^2
// (at most r E^2), below the float32 rounding the full factorization itself
// leaves at the ranks and row counts where E comes near the threshold
// (measured: max|P^T P - I| unchanged to three digits at ranks 512 to 4096
// with first-pass E up to 4.5e-4).
constexpr float kNearIdentityTol = 1e-3f;

// mu, lr and weight decay of a Dion step: given by value, or read on the device
// from hyper[0..2] when hyper is set, so that a captured CUDA graph of the
// step follows whatever the caller writes there between replays.  The derived
// factors 1 - mu, 1 - lr wd and lr sqrt(m/n) are formed on the device in both
// cases, each operation rounded once, so the two forms give the same bits.
struct StepHyper {
    float mu, lr, wd, sqrt_mn;
    const float* hyper;
    __device__ __forceinline__ void get(float& one_minus_mu, float& decay, float& scale) const
    {
        float mu_ = mu, lr_ = lr, wd_ = wd;
        if (hyper) {
            mu_ = hyper[0];
            lr_ = hyper[1];
            wd_ = hyper[2];
        }
        one_minus_mu = __fsub_rn(1.f, mu_);
        decay = __fsub_rn(1.f, __fmul_rn(lr_, wd_));
        scale = __fmul_rn(lr_, sqrt_mn);
    }
    __device__ __forceinline__ bool finite() const
    {
        return !hyper || (isfinite(hyper[0]) && isfinite(hyper[1]) && isfinite(hyper[2]));
    }
};

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

__host__ __device__ __forceinline__ long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---- host side: kernel launch with optional per-kernel event timing ----
int prof_begin(const char* name, cudaStream_t s);
void prof_end(int slot, cudaStream_t s);

template <typename... KArgs, typename... Args>
cudaError_t launch(const char* name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t s, Args&&... args)
{
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
    const int slot = prof_begin(name, s);
    kernel<<<grid, block, smem, s>>>(std::forward<Args>(args)...);
    cudaError_t e = cudaGetLastError();
    prof_end(slot, s);
    return e;
}

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device (the attribute is per device).  `done` is a bit mask of devices
// already set up; concurrent first calls may both set the attribute, which is
// harmless.  Devices beyond 63 are set up on every call.
inline cudaError_t smem_attr_once(const void* func, int bytes, std::atomic<unsigned long long>& done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

#define DION_TRY(expr)                                   \
    do {                                                 \
        cudaError_t _e = (expr);                         \
        if (_e != cudaSuccess) return DION_ERR_CUDA;     \
    } while (0)

}  // namespace dion
