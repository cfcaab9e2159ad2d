// rpe.cu -- kernelized attention with a Toeplitz relative-position weight
// (review page "Stable, Fast and Accurate: Kernelized Attention with
// Relative Positional Encoding", proposed method: the RPE matrix depends only
// on i - j and multiplies the kernelized attention elementwise):
//   out_i = sum_{j in J(i)} c_{i-j} (phi(q_i).phi(k_j)) v_j / sum_{j in J(i)} c_{i-j} phi(q_i).phi(k_j)
// with c_t = exp(b_t), b [H, 2N - 1] (index t + N - 1), J(i) = {0..i} when
// causal, else every position.
//
// The page multiplies by the Toeplitz matrix with FFTs (O(n log n) per
// feature-value column pair, i.e. Dphi * Dv convolutions per head).  Here the
// weighted form is computed chunk against chunk: the CUDA-core kernel below
// for every supported case, and (rpe_tc.cu) a tensor-core kernel for bf16
// elu+1 with D, Dv in {64, 128}, whose 2 N^2 (D + Dv + 16) flops per head on
// the tensor cores take less time than the D Dv FFTs of length 2N would on
// the CUDA cores at the sequence lengths used here.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kRT = 256;
constexpr int kRC = 32;   // positions per chunk

template <typename T>
__device__ void rpe_phi_rows(const T *__restrict__ x, int t0, int n, int D, int P, int kind,
                             const float *__restrict__ W, float *f, float *sq)
{
    if (kind == PHI_ELU1) {
        for (int idx = threadIdx.x; idx < kRC * D; idx += blockDim.x) {
            const int i = idx / D, d = idx % D;
            f[idx] = i < n ? phi_elu1(to_f32(x[(long long)(t0 + i) * D + d])) : 0.f;
        }
        return;
    }
    for (int i = threadIdx.x; i < kRC; i += blockDim.x) {
        float s = 0.f;
        if (i < n)
            for (int d = 0; d < D; d++) {
                const float xv = to_f32(x[(long long)(t0 + i) * D + d]);
                s = fmaf(xv, xv, s);
            }
        sq[i] = s;
    }
    __syncthreads();
    const int m = rf_m(kind, P);
    for (int idx = threadIdx.x; idx < kRC * P; idx += blockDim.x) {
        const int i = idx / P, r = idx % P;
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

// grid (query chunks, B*H): one chunk of kRC queries against every key chunk
template <typename T>
__global__ void __launch_bounds__(kRT)
rpe_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const float *__restrict__ bias, T *__restrict__ out, int N, int H, int D, int Dv, int P,
                int causal, int kind, const float *__restrict__ W)
{
    extern __shared__ float sm[];
    float *fq = sm, *fk = fq + kRC * P, *vv = fk + kRC * P, *A = vv + kRC * Dv, *num = A + kRC * kRC;
    float *den = num + kRC * Dv, *sq = den + kRC, *cw = sq + kRC;   // cw: 2 kRC - 1 weights
    const int NC = cdiv(N, kRC);
    const int qc = NC - 1 - (int)blockIdx.x;   // the longest rows first (causal)
    const long long h = blockIdx.y;
    const float *bh = bias + (h % H) * (2LL * N - 1);
    const int q0 = qc * kRC, nq = min(kRC, N - q0);
    for (int idx = threadIdx.x; idx < kRC * Dv; idx += blockDim.x) num[idx] = 0.f;
    for (int i = threadIdx.x; i < kRC; i += blockDim.x) den[i] = 0.f;
    rpe_phi_rows(q + h * N * D, q0, nq, D, P, kind, W, fq, sq);
    const int kend = causal ? qc : NC - 1;
    for (int kc = 0; kc <= kend; kc++) {
        const int k0 = kc * kRC, nk = min(kRC, N - k0);
        __syncthreads();
        rpe_phi_rows(k + h * N * D, k0, nk, D, P, kind, W, fk, sq);
        for (int idx = threadIdx.x; idx < kRC * Dv; idx += blockDim.x) {
            const int j = idx / Dv, c = idx % Dv;
            vv[idx] = j < nk ? to_f32(v[(h * N + k0 + j) * Dv + c]) : 0.f;
        }
        // weights for t = (q0 + i) - (k0 + j) = (q0 - k0) + u, u in [-(kRC-1), kRC-1]
        for (int u = threadIdx.x; u < 2 * kRC - 1; u += blockDim.x) {
            const long long t = (long long)(q0 - k0) + u - (kRC - 1);
            cw[u] = (t > -N && t < N) ? expf(bh[t + N - 1]) : 0.f;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < kRC * kRC; idx += blockDim.x) {
            const int i = idx / kRC, j = idx % kRC;
            float a = 0.f;
            if (i < nq && j < nk && !(causal && kc == qc && j > i)) {
                for (int x = 0; x < P; x++) a = fmaf(fq[i * P + x], fk[j * P + x], a);
                a *= cw[i - j + kRC - 1];
            }
            A[idx] = a;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < kRC * Dv; idx += blockDim.x) {
            const int i = idx / Dv, c = idx % Dv;
            float s = num[idx];
            for (int j = 0; j < kRC; j++) s = fmaf(A[i * kRC + j], vv[j * Dv + c], s);
            num[idx] = s;
        }
        for (int i = threadIdx.x; i < kRC; i += blockDim.x) {
            float s = den[i];
            for (int j = 0; j < kRC; j++) s += A[i * kRC + j];
            den[i] = s;
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nq * Dv; idx += blockDim.x) {
        const int i = idx / Dv;
        out[(h * N + q0) * Dv + idx] = from_f32<T>(num[idx] / den[i]);
    }
}

template <typename T>
cudaError_t launch_rpe_simt(const Problem &p, const float *bias, int H, bool causal, cudaStream_t s)
{
    const size_t smem = ((size_t)2 * kRC * p.P + 2 * kRC * p.Dv + kRC * kRC + 2 * kRC + 2 * kRC - 1) * sizeof(float);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = set_max_smem_once<rpe_simt_kernel<T>>(227 * 1024);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)cdiv(p.N, kRC), (unsigned)p.BH);
    rpe_simt_kernel<T><<<grid, kRT, smem, s>>>((const T *)p.q, (const T *)p.k, (const T *)p.v, bias, (T *)p.out,
                                               p.N, H, p.D, p.Dv, p.P, causal ? 1 : 0, p.kind, p.W);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

cudaError_t rpe_forward(const Problem &p, const float *bias, int H, bool causal, int *err, cudaStream_t s)
{
    if (rpe_tc_supported(p)) return rpe_tc_forward(p, bias, H, causal, err, s);
    if (p.dtype == DT_F32) return launch_rpe_simt<float>(p, bias, H, causal, s);
    return launch_rpe_simt<__nv_bfloat16>(p, bias, H, causal, s);
}

}  // namespace la
