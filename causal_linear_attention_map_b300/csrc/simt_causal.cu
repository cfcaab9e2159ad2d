// simt_causal.cu -- chunked causal linear attention on CUDA cores, fp32
// arithmetic, one CTA per head walking the sequence chunk by chunk.
//
// Per chunk of C positions (review page "Transformers are RNNs", proposed
// method b2-b3: associativity plus cumulative sums S_i, z_i):
//   A      = tril(phi(Q_c) phi(K_c)^T)            (diagonal included)
//   num    = A V_c + phi(Q_c) S_prev               den = rowsum(A) + phi(Q_c) z_prev
//   out    = num / den
//   S     += phi(K_c)^T V_c ,  z += colsum(phi(K_c))
// This is the fp32-input path (its error stays far under 1e-4) and the
// fallback for shapes the tensor-core kernel does not take.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kThreads = 256;

struct SimtSmem {
    int C;
    size_t S, z, fq, fk, vv, A, den, sq, total;
};

__host__ __device__ inline SimtSmem simt_layout(int P, int Dv, int C)
{
    SimtSmem L;
    L.C = C;
    size_t o = 0;
    L.S = o;   o += (size_t)P * Dv;
    L.z = o;   o += P;
    L.fq = o;  o += (size_t)C * P;
    L.fk = o;  o += (size_t)C * P;
    L.vv = o;  o += (size_t)C * Dv;
    L.A = o;   o += (size_t)C * C;
    L.den = o; o += C;
    L.sq = o;  o += C;
    L.total = o * sizeof(float);
    return L;
}

// phi of rows [t0, t0 + n) of x (a head's [N, D] block) into f [C, P];
// rows n..C-1 are zero so that they add nothing.
template <typename T>
__device__ void load_phi_rows(const T *__restrict__ x, int t0, int n, int C, int D, int P,
                              int kind, const float *__restrict__ W, float *f, float *sq)
{
    const int tid = threadIdx.x;
    if (kind == PHI_ELU1) {
        for (int idx = tid; idx < C * D; idx += blockDim.x) {
            int i = idx / D, d = idx % D;
            f[idx] = i < n ? phi_elu1(to_f32(x[(long long)(t0 + i) * D + d])) : 0.f;
        }
        return;
    }
    // random features: |x_i|^2 first, then each feature from its projection
    for (int i = tid; i < C; i += blockDim.x) {
        float s = 0.f;
        if (i < n)
            for (int d = 0; d < D; d++) {
                float xv = to_f32(x[(long long)(t0 + i) * D + d]);
                s = fmaf(xv, xv, s);
            }
        sq[i] = s;
    }
    __syncthreads();
    const int m = rf_m(kind, P);
    for (int idx = tid; idx < C * P; idx += blockDim.x) {
        int i = idx / P, r = idx % P;
        float val = 0.f;
        if (i < n) {
            const T *xr = x + (long long)(t0 + i) * D;
            const float *wr = W + (long long)rf_proj(kind, r, m) * D;
            float u = 0.f;
            for (int d = 0; d < D; d++) u = fmaf(wr[d], to_f32(xr[d]), u);
            val = rf_value(kind, r, m, u, sq[i]);
        }
        f[idx] = val;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
simt_causal_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   T *__restrict__ out, int N, int D, int Dv, int P, int C, int kind,
                   const float *__restrict__ W, float *__restrict__ S_out,
                   float *__restrict__ z_out)
{
    extern __shared__ float sm[];
    const SimtSmem L = simt_layout(P, Dv, C);
    float *S = sm + L.S, *z = sm + L.z, *fq = sm + L.fq, *fk = sm + L.fk;
    float *vv = sm + L.vv, *A = sm + L.A, *den = sm + L.den, *sq = sm + L.sq;

    const long long h = blockIdx.x;
    const T *qh = q + h * N * D;
    const T *kh = k + h * N * D;
    const T *vh = v + h * N * Dv;
    T *oh = out + h * N * Dv;
    const int tid = threadIdx.x;

    for (int idx = tid; idx < P * Dv; idx += blockDim.x) S[idx] = 0.f;
    for (int a = tid; a < P; a += blockDim.x) z[a] = 0.f;
    __syncthreads();

    for (int t0 = 0; t0 < N; t0 += C) {
        const int n = min(C, N - t0);
        load_phi_rows(qh, t0, n, C, D, P, kind, W, fq, sq);
        __syncthreads();
        load_phi_rows(kh, t0, n, C, D, P, kind, W, fk, sq);
        for (int idx = tid; idx < C * Dv; idx += blockDim.x) {
            int i = idx / Dv, c = idx % Dv;
            vv[idx] = i < n ? to_f32(vh[(long long)(t0 + i) * Dv + c]) : 0.f;
        }
        __syncthreads();

        // A = tril(phi(Q) phi(K)^T), j <= i
        for (int idx = tid; idx < C * C; idx += blockDim.x) {
            int i = idx / C, j = idx % C;
            float s = 0.f;
            if (j <= i)
                for (int a = 0; a < P; a++) s = fmaf(fq[i * P + a], fk[j * P + a], s);
            A[idx] = s;
        }
        __syncthreads();

        // den_i = rowsum(A)_i + phi(q_i) . z_prev
        for (int i = tid; i < C; i += blockDim.x) {
            float s = 0.f;
            for (int j = 0; j <= i; j++) s += A[i * C + j];
            float t = 0.f;
            for (int a = 0; a < P; a++) t = fmaf(fq[i * P + a], z[a], t);
            den[i] = s + t;
        }
        __syncthreads();

        // out_i = (A V + phi(Q) S_prev)_i / den_i
        for (int idx = tid; idx < n * Dv; idx += blockDim.x) {
            int i = idx / Dv, c = idx % Dv;
            float s = 0.f;
            for (int j = 0; j <= i; j++) s = fmaf(A[i * C + j], vv[j * Dv + c], s);
            float t = 0.f;
            for (int a = 0; a < P; a++) t = fmaf(fq[i * P + a], S[a * Dv + c], t);
            oh[(long long)(t0 + i) * Dv + c] = from_f32<T>((s + t) / den[i]);
        }
        __syncthreads();

        // S += phi(K)^T V ; z += colsum(phi(K))
        for (int idx = tid; idx < P * Dv; idx += blockDim.x) {
            int a = idx / Dv, c = idx % Dv;
            float s = S[idx];
            for (int j = 0; j < n; j++) s = fmaf(fk[j * P + a], vv[j * Dv + c], s);
            S[idx] = s;
        }
        for (int a = tid; a < P; a += blockDim.x) {
            float s = z[a];
            for (int j = 0; j < n; j++) s += fk[j * P + a];
            z[a] = s;
        }
        __syncthreads();
    }

    if (S_out)
        for (int idx = tid; idx < P * Dv; idx += blockDim.x) S_out[h * P * Dv + idx] = S[idx];
    if (z_out)
        for (int a = tid; a < P; a += blockDim.x) z_out[h * P + a] = z[a];
}

template <typename T>
cudaError_t launch(const Problem &p, float *S_out, float *z_out, cudaStream_t s)
{
    int C = 32;
    SimtSmem L = simt_layout(p.P, p.Dv, C);
    if (L.total > 227 * 1024) {
        C = 16;
        L = simt_layout(p.P, p.Dv, C);
    }
    auto kern = simt_causal_kernel<T>;
    if (L.total > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = set_max_smem_once<simt_causal_kernel<T>>(227 * 1024);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)p.BH, kThreads, L.total, s>>>(
        (const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.out, p.N, p.D, p.Dv, p.P, C,
        p.kind, p.W, S_out, z_out);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

cudaError_t simt_causal(const Problem &p, float *S_out, float *z_out, cudaStream_t s)
{
    if (p.dtype == DT_F32) return launch<float>(p, S_out, z_out, s);
    return launch<__nv_bfloat16>(p, S_out, z_out, s);
}

}  // namespace la
