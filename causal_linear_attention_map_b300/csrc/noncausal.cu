// noncausal.cu -- non-causal linear attention as two passes (review page
// "Transformers are RNNs", proposed method b2: by associativity phi(K)^T V is
// formed once and reused by every query):
//   pass 1: KV = sum_j phi(k_j) v_j^T, ksum = sum_j phi(k_j), split over N
//           with fp32 partials added into scratch;
//   pass 2: out_i = phi(q_i)^T KV / phi(q_i)^T ksum.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kC = 32;

template <typename T>
__device__ void phi_rows(const T *__restrict__ x, long long t0, int n, int D, int P, int kind,
                         const float *__restrict__ W, float *f, float *sq)
{
    const int tid = threadIdx.x;
    if (kind == PHI_ELU1) {
        for (int idx = tid; idx < kC * D; idx += blockDim.x) {
            int i = idx / D, d = idx % D;
            f[idx] = i < n ? phi_elu1(to_f32(x[(t0 + i) * D + d])) : 0.f;
        }
        return;
    }
    for (int i = tid; i < kC; i += blockDim.x) {
        float s = 0.f;
        if (i < n)
            for (int d = 0; d < D; d++) {
                float xv = to_f32(x[(t0 + i) * D + d]);
                s = fmaf(xv, xv, s);
            }
        sq[i] = s;
    }
    __syncthreads();
    const int m = rf_m(kind, P);
    for (int idx = tid; idx < kC * P; idx += blockDim.x) {
        int i = idx / P, r = idx % P;
        float val = 0.f;
        if (i < n) {
            const T *xr = x + (t0 + i) * D;
            const float *wr = W + (long long)rf_proj(kind, r, m) * D;
            float u = 0.f;
            for (int d = 0; d < D; d++) u = fmaf(wr[d], to_f32(xr[d]), u);
            val = rf_value(kind, r, m, u, sq[i]);
        }
        f[idx] = val;
    }
}

// grid (BH, splits); each CTA reduces rows [split * rows_per, ...) of one head.
template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_kv_kernel(const T *__restrict__ k, const T *__restrict__ v, int N, int D, int Dv, int P,
             int kind, const float *__restrict__ W, int rows_per, float *__restrict__ KV,
             float *__restrict__ ksum)
{
    extern __shared__ float sm[];
    float *acc = sm;                       // P * Dv
    float *ks = acc + (size_t)P * Dv;      // P
    float *fk = ks + P;                    // kC * P
    float *vv = fk + (size_t)kC * P;       // kC * Dv
    float *sq = vv + (size_t)kC * Dv;      // kC
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const long long r0 = (long long)blockIdx.y * rows_per;
    const long long r1 = min((long long)N, r0 + rows_per);
    for (int idx = tid; idx < P * Dv; idx += blockDim.x) acc[idx] = 0.f;
    for (int a = tid; a < P; a += blockDim.x) ks[a] = 0.f;
    __syncthreads();
    for (long long t0 = r0; t0 < r1; t0 += kC) {
        const int n = (int)min((long long)kC, r1 - t0);
        phi_rows(k + h * N * D, t0, n, D, P, kind, W, fk, sq);
        for (int idx = tid; idx < kC * Dv; idx += blockDim.x) {
            int i = idx / Dv, c = idx % Dv;
            vv[idx] = i < n ? to_f32(v[(h * N + t0 + i) * Dv + c]) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < P * Dv; idx += blockDim.x) {
            int a = idx / Dv, c = idx % Dv;
            float s = acc[idx];
            for (int j = 0; j < n; j++) s = fmaf(fk[j * P + a], vv[j * Dv + c], s);
            acc[idx] = s;
        }
        for (int a = tid; a < P; a += blockDim.x) {
            float s = ks[a];
            for (int j = 0; j < n; j++) s += fk[j * P + a];
            ks[a] = s;
        }
        __syncthreads();
    }
    for (int idx = tid; idx < P * Dv; idx += blockDim.x) atomicAdd(&KV[h * P * Dv + idx], acc[idx]);
    for (int a = tid; a < P; a += blockDim.x) atomicAdd(&ksum[h * P + a], ks[a]);
}

// grid (BH, row blocks); out_i = phi(q_i)^T KV / phi(q_i)^T ksum.
template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_out_kernel(const T *__restrict__ q, T *__restrict__ out, int N, int D, int Dv, int P, int kind,
              const float *__restrict__ W, int rows_per, const float *__restrict__ KV,
              const float *__restrict__ ksum)
{
    extern __shared__ float sm[];
    float *kv = sm;                        // P * Dv
    float *ks = kv + (size_t)P * Dv;       // P
    float *fq = ks + P;                    // kC * P
    float *den = fq + (size_t)kC * P;      // kC
    float *sq = den + kC;                  // kC
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const long long r0 = (long long)blockIdx.y * rows_per;
    const long long r1 = min((long long)N, r0 + rows_per);
    for (int idx = tid; idx < P * Dv; idx += blockDim.x) kv[idx] = KV[h * P * Dv + idx];
    for (int a = tid; a < P; a += blockDim.x) ks[a] = ksum[h * P + a];
    __syncthreads();
    for (long long t0 = r0; t0 < r1; t0 += kC) {
        const int n = (int)min((long long)kC, r1 - t0);
        phi_rows(q + h * N * D, t0, n, D, P, kind, W, fq, sq);
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x) {
            float s = 0.f;
            for (int a = 0; a < P; a++) s = fmaf(fq[i * P + a], ks[a], s);
            den[i] = s;
        }
        __syncthreads();
        for (int idx = tid; idx < n * Dv; idx += blockDim.x) {
            int i = idx / Dv, c = idx % Dv;
            float s = 0.f;
            for (int a = 0; a < P; a++) s = fmaf(fq[i * P + a], kv[a * Dv + c], s);
            out[(h * N + t0 + i) * Dv + c] = from_f32<T>(s / den[i]);
        }
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch(const Problem &p, float *KV, float *ks, cudaStream_t s)
{
    // Split N so that the reduction fills the GPU (~4 CTAs per SM worth).
    long long want = 148LL * 4;
    int splits = (int)max(1LL, min((long long)cdiv(p.N, kC), want / max(1LL, p.BH)));
    splits = max(1, min(splits, 65535));
    int rows_per = cdiv(cdiv(p.N, splits), kC) * kC;
    splits = cdiv(p.N, rows_per);
    size_t sm1 = ((size_t)p.P * p.Dv + p.P + (size_t)kC * p.P + (size_t)kC * p.Dv + kC) * 4;
    size_t sm2 = ((size_t)p.P * p.Dv + p.P + (size_t)kC * p.P + 2 * kC) * 4;
    cudaError_t e;
    // the opt-in limit once, at the largest size any launch of these kernels asks for
    if ((e = set_max_smem_once<nc_kv_kernel<T>>(227 * 1024)) != cudaSuccess) return e;
    if ((e = set_max_smem_once<nc_out_kernel<T>>(227 * 1024)) != cudaSuccess) return e;
    if (sm1 > 227 * 1024 || sm2 > 227 * 1024) return cudaErrorInvalidValue;
    nc_kv_kernel<T><<<dim3((unsigned)p.BH, splits), kThreads, sm1, s>>>(
        (const T *)p.k, (const T *)p.v, p.N, p.D, p.Dv, p.P, p.kind, p.W, rows_per, KV, ks);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(1);
    nc_out_kernel<T><<<dim3((unsigned)p.BH, splits), kThreads, sm2, s>>>(
        (const T *)p.q, (T *)p.out, p.N, p.D, p.Dv, p.P, p.kind, p.W, rows_per, KV, ks);
    if ((e = cudaGetLastError()) == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

size_t noncausal_scratch_bytes(const Problem &p)
{
    return (size_t)p.BH * ((size_t)p.P * p.Dv + p.P) * sizeof(float);
}

cudaError_t noncausal(const Problem &p, void *scratch, float *S_out, float *z_out, cudaStream_t s)
{
    float *KV = (float *)scratch;
    float *ks = KV + (size_t)p.BH * p.P * p.Dv;
    cudaError_t e = cudaMemsetAsync(scratch, 0, noncausal_scratch_bytes(p), s);
    if (e != cudaSuccess) return e;
    e = p.dtype == DT_F32 ? launch<float>(p, KV, ks, s) : launch<__nv_bfloat16>(p, KV, ks, s);
    if (e != cudaSuccess) return e;
    if (S_out &&
        (e = cudaMemcpyAsync(S_out, KV, (size_t)p.BH * p.P * p.Dv * 4, cudaMemcpyDeviceToDevice, s)) !=
            cudaSuccess)
        return e;
    if (z_out &&
        (e = cudaMemcpyAsync(z_out, ks, (size_t)p.BH * p.P * 4, cudaMemcpyDeviceToDevice, s)) !=
            cudaSuccess)
        return e;
    return cudaSuccess;
}

}  // namespace la
