// common.cuh -- shared device helpers and the host launch wrapper of libdion.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>
#include <utility>

#include "../../include/dion.h"

namespace dion {

typedef __nv_bfloat16 bf16;

// Bits of the device status word (see dion_get_status).
enum : int { kStatusPivot = 1, kStatusNonFinite = 2 };

// A Gram matrix S = I + E with max|E| <= kNearIdentityTol takes the
// first-order inverse of its Cholesky factor, I - strictly_lower(E) - diag(E)/2
// (error O(E^2), below float32 rounding).
constexpr float kNearIdentityTol = 1e-4f;

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

#define DION_TRY(expr)                                   \
    do {                                                 \
        cudaError_t _e = (expr);                         \
        if (_e != cudaSuccess) return DION_ERR_CUDA;     \
    } while (0)

}  // namespace dion
