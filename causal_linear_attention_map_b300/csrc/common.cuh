// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace la {

// Input/output element types.
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// elu(x) + 1 with alpha = 1: x + 1 for x > 0, exp(x) otherwise
// ("Transformers are RNNs", main results: the elu-based feature map).
__device__ __forceinline__ float phi_elu1(float x) { return x > 0.f ? x + 1.f : expf(x); }

// Same map with the fast exponential (MUFU ex2), for the bf16 paths whose
// rounding is far coarser than its error.
__device__ __forceinline__ float phi_elu1_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

__host__ __device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Random-feature maps with projections u_r = w_r . x (r < m) of a row x with
// |x|^2 = sq (review page "Stable, Fast and Accurate: Kernelized Attention
// with RPE", proposed method: PRF, TRF, Sphere-PRF, ORF, NPRF; Sphere-PRF and
// ORF are PRF with other distributions of W).  kind: 1 PRF, 2 NPRF, 3 TRF
// (the values of kernels.h's PHI_*).  Feature r of Dphi = rf_dim(kind, m):
//   PRF   exp(u_r - sq/2) / sqrt(m)
//   NPRF  PRF of x / |x|:  exp(u_r / |x| - 1/2) / sqrt(m)   (x = 0: 1 / sqrt(m))
//   TRF   exp(sq/2) / sqrt(m) * (cos u_r for r < m, sin u_{r-m} for r >= m)
__host__ __device__ __forceinline__ int rf_dim(int kind, int m) { return kind == 3 ? 2 * m : m; }
__host__ __device__ __forceinline__ int rf_m(int kind, int P) { return kind == 3 ? P / 2 : P; }
// the projection that feature r reads
__device__ __forceinline__ int rf_proj(int kind, int r, int m) { return kind == 3 && r >= m ? r - m : r; }
__device__ __forceinline__ float rf_value(int kind, int r, int m, float u, float sq)
{
    const float inv = rsqrtf((float)m);
    if (kind == 1) return expf(u - 0.5f * sq) * inv;
    if (kind == 2) return sq > 0.f ? expf(u * rsqrtf(sq) - 0.5f) * inv : inv;
    const float a = expf(0.5f * sq) * inv;
    return r < m ? a * cosf(u) : a * sinf(u);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per kernel and
// device (bit d of the mask: device d < 64; others set it on every call),
// so that a forward call does not pay for it again.
template <auto Kernel>
cudaError_t set_max_smem_once(int bytes)
{
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launch a kernel that depends on the previous launch in the stream as a
// programmatic dependent launch: it may start once every block of that
// launch has signalled (griddepcontrol.launch_dependents) or exited, and it
// must execute griddepcontrol.wait before it reads anything that launch
// wrote.  Its prologue then overlaps the previous kernel's tail.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace la
