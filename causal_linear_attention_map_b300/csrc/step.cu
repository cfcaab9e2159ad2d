// step.cu -- one recurrent decode step for a batch of heads (review page
// "Transformers are RNNs", proposed method b5: the causal transformer is an
// RNN with two memories S, z and a recurrent update):
//   S += phi(k) v^T ;  z += phi(k) ;  out = phi(q)^T S / phi(q)^T z
// in place.  The S read-modify-write is the whole cost: each CTA streams one
// head's Dphi x Dv fp32 block with 128-bit loads and stores, rows spread over
// the CTA's threads, and reduces phi(q)^T S across rows in shared memory.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxP = 256;

template <typename T>
__device__ __forceinline__ void phi_vec(const T *__restrict__ x, int D, int P, int kind,
                                        const float *__restrict__ W, float *f, float *red)
{
    const int tid = threadIdx.x;
    if (kind == PHI_ELU1) {
        for (int d = tid; d < D; d += blockDim.x) f[d] = phi_elu1(to_f32(x[d]));
        return;
    }
    // |x|^2 by one warp, then the P projections
    if (tid < 32) {
        float s = 0.f;
        for (int d = tid; d < D; d += 32) {
            float xv = to_f32(x[d]);
            s = fmaf(xv, xv, s);
        }
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (tid == 0) red[0] = s;
    }
    __syncthreads();
    const float sq = red[0];
    const int m = rf_m(kind, P);
    for (int r = tid; r < P; r += blockDim.x) {
        const float *wr = W + (long long)rf_proj(kind, r, m) * D;
        float u = 0.f;
        for (int d = 0; d < D; d++) u = fmaf(wr[d], to_f32(x[d]), u);
        f[r] = rf_value(kind, r, m, u, sq);
    }
    __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
step_kernel(float *__restrict__ S, float *__restrict__ z, const T *__restrict__ q,
            const T *__restrict__ k, const T *__restrict__ v, T *__restrict__ out, int D, int Dv,
            int P, int kind, const float *__restrict__ W)
{
    __shared__ float fk[kMaxP], fq[kMaxP], vv[128];
    __shared__ float red[32];
    __shared__ float part[4 * kThreads];   // den partials, then [row group][Dv] partials
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;

    phi_vec(k + h * D, D, P, kind, W, fk, red);
    phi_vec(q + h * D, D, P, kind, W, fq, red);
    for (int c = tid; c < Dv; c += blockDim.x) vv[c] = to_f32(v[h * Dv + c]);
    __syncthreads();

    // z += phi(k); den = phi(q) . z  (block reduction)
    float dpart = 0.f;
    for (int a = tid; a < P; a += blockDim.x) {
        float zn = z[h * P + a] + fk[a];
        z[h * P + a] = zn;
        dpart = fmaf(fq[a], zn, dpart);
    }
    part[tid] = dpart;

    // S += phi(k) v^T and num = phi(q)^T S_new, float4 per thread
    const int c4n = Dv / 4;              // float4 columns per row
    const int rg_n = blockDim.x / c4n;   // row groups
    const int c4 = tid % c4n, rg = tid / c4n;
    float4 *Sh = reinterpret_cast<float4 *>(S + h * (long long)P * Dv);
    const float4 v4 = make_float4(vv[4 * c4], vv[4 * c4 + 1], vv[4 * c4 + 2], vv[4 * c4 + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (rg < rg_n) {
#pragma unroll 8
        for (int a = rg; a < P; a += rg_n) {
            float4 s = Sh[(long long)a * c4n + c4];
            const float f = fk[a], g = fq[a];
            s.x = fmaf(f, v4.x, s.x);
            s.y = fmaf(f, v4.y, s.y);
            s.z = fmaf(f, v4.z, s.z);
            s.w = fmaf(f, v4.w, s.w);
            Sh[(long long)a * c4n + c4] = s;
            acc.x = fmaf(g, s.x, acc.x);
            acc.y = fmaf(g, s.y, acc.y);
            acc.z = fmaf(g, s.z, acc.z);
            acc.w = fmaf(g, s.w, acc.w);
        }
    }
    __syncthreads();
    // den: reduce part[]
    for (int o = blockDim.x / 2; o > 0; o >>= 1) {
        if (tid < o) part[tid] += part[tid + o];
        __syncthreads();
    }
    const float den = part[0];
    __syncthreads();
    // num: reduce acc over row groups, column by column (reuse part[] as [rg][Dv])
    if (rg < rg_n) {
        part[rg * Dv + 4 * c4 + 0] = acc.x;
        part[rg * Dv + 4 * c4 + 1] = acc.y;
        part[rg * Dv + 4 * c4 + 2] = acc.z;
        part[rg * Dv + 4 * c4 + 3] = acc.w;
    }
    __syncthreads();
    for (int c = tid; c < Dv; c += blockDim.x) {
        float s = 0.f;
        for (int r = 0; r < rg_n; r++) s += part[r * Dv + c];
        out[h * Dv + c] = from_f32<T>(s / den);
    }
}

}  // namespace

cudaError_t step(float *S, float *z, const void *q, const void *k, const void *v, void *out,
                 long long BH, int D, int Dv, int P, int kind, int m, const float *W, int dtype,
                 cudaStream_t s)
{
    (void)m;
    if (dtype == DT_F32)
        step_kernel<float><<<(unsigned)BH, kThreads, 0, s>>>(
            S, z, (const float *)q, (const float *)k, (const float *)v, (float *)out, D, Dv, P,
            kind, W);
    else
        step_kernel<__nv_bfloat16><<<(unsigned)BH, kThreads, 0, s>>>(
            S, z, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (__nv_bfloat16 *)out, D, Dv, P, kind, W);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace la
