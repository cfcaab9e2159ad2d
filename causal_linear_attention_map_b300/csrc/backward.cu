// backward.cu -- gradients of the linear-attention forward with respect to
// q, k and v, on CUDA cores (fp32 arithmetic), chunked and cut into segments
// like the forward: every dtype and feature map (bf16 elu+1 with D = Dv in
// {64, 128} goes to the tensor-core kernel of backward_tc.cu instead).
//
// Method (review page "Transformers are RNNs", proposed method b4: the
// gradients of forward and backward propagation are computed in linear time
// with the same cumulative sums).  With g_i = phi(q_i), f_j = phi(k_j),
// den_i = g_i . z_i, out_i = S_i^T g_i / den_i and the output cotangent dout:
//   dnum_i = dout_i / den_i,   dden_i = -(dout_i . out_i) / den_i
//   d g_i  = S_i dnum_i + z_i dden_i                      (forward direction)
//   d f_j  = R_j v_j + r_j,    dv_j = R_j^T f_j           (reverse direction)
//   R_j = sum_{i >= j} g_i dnum_i^T,   r_j = sum_{i >= j} g_i dden_i
// then dq and dk through phi.  In chunks of C positions, with the masked
// (j <= i) intra-chunk matrices A_ij = g_i . f_j and B_ij = dnum_i . v_j + dden_i:
//   dG = B F + dnum S_prev^T + dden z_prev^T
//   dF = B^T G + V R_next + 1 r_next^T,    dV = A^T dnum + F R_next
// Launches (causal): the segment sums of S, z; their exclusive prefix; the dq
// pass (which recomputes den and out, and also writes den, dden and the
// segment sums of R, r); their exclusive suffix; the dk/dv pass, whose
// segments walk their chunks backwards.  Non-causal: the same launches with
// per-head totals in place of prefixes and suffixes and no intra-chunk terms.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kBT = 256;

struct BwdGeo {
    int BH, N, C, NC, L, nseg;
    int D, Dv, P, kind, m, causal;
};

// Row-major fp32 shared-memory layout of the passes (offsets in floats).
struct BwdSmem {
    size_t S, z, R, r, G, F, V, O, Mn, X, dX, A, B, den, dd, sq, total;
};

__host__ __device__ inline BwdSmem bwd_layout(const BwdGeo &g, bool dq_pass)
{
    BwdSmem L;
    const size_t C = g.C, P = g.P, Dv = g.Dv, D = g.D;
    size_t o = 0;
    // state rows are Dv + 1 apart (no bank conflicts when threads walk the feature index)
    L.S = o;   o += P * (Dv + 1);   // forward memories (dq pass) or reverse memories (dk/dv pass)
    L.z = o;   o += P;
    L.R = o;   o += dq_pass ? P * (Dv + 1) : 0;   // dq pass: this segment's sums of R, r
    L.r = o;   o += dq_pass ? P : 0;
    L.G = o;   o += C * P;
    L.F = o;   o += C * P;
    L.V = o;   o += C * Dv;
    L.O = o;   o += C * Dv;   // dout (dq pass: then out)
    L.Mn = o;  o += C * Dv;   // dnum
    L.X = o;   o += g.kind != PHI_ELU1 ? C * D : 0;   // raw q (dq) or k (dk) rows for the random-feature chain rule
    L.dX = o;  o += C * P;    // dG or dF before the chain rule through phi
    L.A = o;   o += C * C;
    L.B = o;   o += C * C;
    L.den = o; o += C;
    L.dd = o;  o += C;
    L.sq = o;  o += 2 * C;   // |x|^2 per row, then the chain rule's two per-row sums
    L.total = o * sizeof(float);
    return L;
}

// phi of rows [t0, t0 + n) of a head's [N, D] block into f [C, P]; rows
// n..C-1 are zero.  PRF: |x|^2 into sq, and the raw rows into X (if given).
// Wt is W transposed ([D, m]): the threads of a warp take consecutive
// features, so their reads of it are consecutive.
template <typename T>
__device__ void phi_rows(const T *__restrict__ x, int t0, int n, const BwdGeo &g,
                         const float *__restrict__ Wt, float *f, float *sq, float *X)
{
    const int C = g.C, D = g.D, P = g.P;
    if (g.kind == PHI_ELU1) {
        for (int idx = threadIdx.x; idx < C * D; idx += blockDim.x) {
            const int i = idx / D, d = idx % D;
            f[idx] = i < n ? phi_elu1(to_f32(x[(long long)(t0 + i) * D + d])) : 0.f;
        }
        return;
    }
    for (int idx = threadIdx.x; idx < C * D; idx += blockDim.x) {
        const int i = idx / D, d = idx % D;
        X[idx] = i < n ? to_f32(x[(long long)(t0 + i) * D + d]) : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        float s = 0.f;
        for (int d = 0; d < D; d++) s = fmaf(X[i * D + d], X[i * D + d], s);
        sq[i] = s;
    }
    __syncthreads();
    const int m = rf_m(g.kind, P);
    for (int idx = threadIdx.x; idx < C * P; idx += blockDim.x) {
        const int i = idx / P, r = idx % P;
        float val = 0.f;
        if (i < n) {
            const float *wc = Wt + rf_proj(g.kind, r, m);
            float u = 0.f;
            for (int d = 0; d < D; d++) u = fmaf(wc[(long long)d * m], X[i * D + d], u);
            val = rf_value(g.kind, r, m, u, sq[i]);
        }
        f[idx] = val;
    }
}

template <typename T>
__device__ void load_rows(const T *__restrict__ x, int t0, int n, int C, int W, float *dst)
{
    for (int idx = threadIdx.x; idx < C * W; idx += blockDim.x) {
        const int i = idx / W, c = idx % W;
        dst[idx] = i < n ? to_f32(x[(long long)(t0 + i) * W + c]) : 0.f;
    }
}

// The chain rule through phi for rows [0, n): dx = J_phi(x)^T dphi, written
// to out rows [t0, t0 + n).  With t_r = dphi_r phi_r (and for TRF the pairs
// (cos, sin) of projection r):
//   elu + 1  d phi / dx = 1 (x > 0), exp(x) else, which is min(phi(x), 1)
//   PRF      dx = sum_r t_r w_r - x sum_r t_r
//   NPRF     dy = sum_r t_r w_r for y = x/|x|, then dx = (dy - y (y . dy)) / |x|
//   TRF      dx = x sum_r t_r + sum_r w_r (dsin_r phi_cos_r - dcos_r phi_sin_r)
// tmp holds 2 C floats.
template <typename T>
__device__ void phi_chain(const float *f, const float *dphi, const float *X, const BwdGeo &g,
                          const float *__restrict__ W, int t0, int n, float *tmp, T *__restrict__ out)
{
    const int C = g.C, D = g.D, P = g.P, kind = g.kind;
    if (kind == PHI_ELU1) {
        for (int idx = threadIdx.x; idx < n * D; idx += blockDim.x)
            out[(long long)t0 * D + idx] = from_f32<T>(dphi[idx] * fminf(f[idx], 1.f));
        return;
    }
    const int m = rf_m(kind, P);
    // per row: sum_r t_r and |x|^2
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        float s = 0.f, sq = 0.f;
        for (int r = 0; r < P; r++) s = fmaf(dphi[i * P + r], f[i * P + r], s);
        for (int d = 0; d < D; d++) sq = fmaf(X[i * D + d], X[i * D + d], sq);
        tmp[i] = s;
        tmp[C + i] = sq;
    }
    __syncthreads();
    if (kind == PHI_NPRF) {
        // dy into the out buffer's place is not available: form dy . y per row first
        for (int i = threadIdx.x; i < C; i += blockDim.x) {
            float dyy = 0.f;
            const float inv = tmp[C + i] > 0.f ? rsqrtf(tmp[C + i]) : 0.f;
            for (int d = 0; d < D; d++) {
                float dy = 0.f;
                for (int r = 0; r < m; r++) dy = fmaf(dphi[i * P + r] * f[i * P + r], W[(long long)r * D + d], dy);
                dyy = fmaf(dy, X[i * D + d] * inv, dyy);
            }
            tmp[i] = dyy;
        }
        __syncthreads();
    }
    for (int idx = threadIdx.x; idx < n * D; idx += blockDim.x) {
        const int i = idx / D, d = idx % D;
        float s = 0.f, val;
        if (kind == PHI_TRF) {
            for (int r = 0; r < m; r++)
                s = fmaf(dphi[i * P + m + r] * f[i * P + r] - dphi[i * P + r] * f[i * P + m + r],
                         W[(long long)r * D + d], s);
            val = s + tmp[i] * X[i * D + d];
        } else {
            for (int r = 0; r < m; r++) s = fmaf(dphi[i * P + r] * f[i * P + r], W[(long long)r * D + d], s);
            if (kind == PHI_PRF) {
                val = s - tmp[i] * X[i * D + d];
            } else {   // NPRF
                const float inv = tmp[C + i] > 0.f ? rsqrtf(tmp[C + i]) : 0.f;
                val = (s - tmp[i] * X[i * D + d] * inv) * inv;
            }
        }
        out[(long long)t0 * D + idx] = from_f32<T>(val);
    }
}

// acc[a][c] += sum_{j < n} X[j][a] Y[j][c]  (a < P, c < W), and when w1 is
// given, acc1[a] += sum_j X[j][a] w1[j] (the z / r column).
__device__ void accum_outer(float *acc, float *acc1, const float *X, const float *Y, const float *w1,
                            int n, int P, int W, int stride)
{
    for (int idx = threadIdx.x; idx < P * W; idx += blockDim.x) {
        const int a = idx / W, c = idx % W;
        float s = acc[a * stride + c];
        for (int j = 0; j < n; j++) s = fmaf(X[j * P + a], Y[j * W + c], s);
        acc[a * stride + c] = s;
    }
    for (int a = threadIdx.x; a < P; a += blockDim.x) {
        float s = acc1[a];
        for (int j = 0; j < n; j++) s = fmaf(X[j * P + a], w1 ? w1[j] : 1.f, s);
        acc1[a] = s;
    }
}

// ---- pass 1: per-segment sums of S = phi(K)^T V and z = colsum phi(K)
template <typename T>
__global__ void __launch_bounds__(kBT)
bwd_sums_kernel(const T *__restrict__ k, const T *__restrict__ v, const float *__restrict__ Wt, BwdGeo g,
                float *__restrict__ stS)
{
    extern __shared__ float sm[];
    const int h = blockIdx.x / g.nseg, s = blockIdx.x % g.nseg;
    const int P = g.P, Dv = g.Dv, C = g.C;
    float *acc = sm, *acc1 = acc + P * Dv, *F = acc1 + P, *V = F + C * P, *sq = V + C * Dv,
          *X = sq + C;
    for (int idx = threadIdx.x; idx < P * Dv + P; idx += blockDim.x) acc[idx] = 0.f;
    const T *kh = k + (long long)h * g.N * g.D;
    const T *vh = v + (long long)h * g.N * Dv;
    const int c0 = s * g.L, c1 = min(g.NC, c0 + g.L);
    for (int c = c0; c < c1; c++) {
        const int t0 = c * C, n = min(C, g.N - t0);
        __syncthreads();
        phi_rows(kh, t0, n, g, Wt, F, sq, X);
        load_rows(vh, t0, n, C, Dv, V);
        __syncthreads();
        accum_outer(acc, acc1, F, V, nullptr, n, P, Dv, Dv);
    }
    __syncthreads();
    float *dst = stS + ((long long)h * g.nseg + s) * (P * Dv + P);
    for (int idx = threadIdx.x; idx < P * Dv + P; idx += blockDim.x) dst[idx] = acc[idx];
}

// ---- scans over a head's segment slots (element-parallel):
//   mode 0: exclusive prefix   mode 1: exclusive suffix   mode 2: total in every slot
__global__ void bwd_scan_kernel(float *__restrict__ st, int nseg, int elems, int mode)
{
    // (a dependent launch after the tensor-core passes: wait for the sums)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long h = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= elems) return;
    float *p = st + h * nseg * (long long)elems + e;
    if (mode == 2) {
        float t = 0.f;
#pragma unroll 8
        for (int s = 0; s < nseg; s++) t += p[(long long)s * elems];
        for (int s = 0; s < nseg; s++) p[(long long)s * elems] = t;
        return;
    }
    // eight segments' loads in flight at a time, then their stores
    float run = 0.f;
    for (int i0 = 0; i0 < nseg; i0 += 8) {
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int i = i0 + j, s = mode == 0 ? i : nseg - 1 - i;
            x[j] = i < nseg ? p[(long long)s * elems] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int i = i0 + j, s = mode == 0 ? i : nseg - 1 - i;
            if (i < nseg) p[(long long)s * elems] = run;
            run += x[j];
        }
    }
}

// ---- pass 2: dq, plus den, dden per position and the segment sums of R, r
template <typename T>
__global__ void __launch_bounds__(kBT)
bwd_dq_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const T *__restrict__ dout, const float *__restrict__ W, const float *__restrict__ Wt, BwdGeo g,
              const float *__restrict__ stS, float *__restrict__ stR, float *__restrict__ den_out,
              float *__restrict__ dd_out, T *__restrict__ dq)
{
    extern __shared__ float sm[];
    const BwdSmem Ls = bwd_layout(g, true);
    float *S = sm + Ls.S, *z = sm + Ls.z, *R = sm + Ls.R, *r = sm + Ls.r, *G = sm + Ls.G, *F = sm + Ls.F;
    float *V = sm + Ls.V, *O = sm + Ls.O, *Mn = sm + Ls.Mn, *X = sm + Ls.X, *dX = sm + Ls.dX;
    float *A = sm + Ls.A, *Bm = sm + Ls.B, *den = sm + Ls.den, *dd = sm + Ls.dd, *sq = sm + Ls.sq;
    const int h = blockIdx.x / g.nseg, s = blockIdx.x % g.nseg;
    const int P = g.P, Dv = g.Dv, C = g.C, D = g.D;
    const long long slot = ((long long)h * g.nseg + s) * (P * Dv + P);
    const int SP = Dv + 1;
    for (int idx = threadIdx.x; idx < P * Dv; idx += blockDim.x) {
        // the prefix before this segment (or the totals)
        S[(idx / Dv) * SP + idx % Dv] = stS[slot + idx];
        R[(idx / Dv) * SP + idx % Dv] = 0.f;
    }
    for (int a = threadIdx.x; a < P; a += blockDim.x) {
        z[a] = stS[slot + P * Dv + a];
        r[a] = 0.f;
    }
    const T *qh = q + (long long)h * g.N * D, *kh = k + (long long)h * g.N * D;
    const T *vh = v + (long long)h * g.N * Dv, *oh = dout + (long long)h * g.N * Dv;
    T *dqh = dq + (long long)h * g.N * D;
    const int c0 = s * g.L, c1 = min(g.NC, c0 + g.L);
    for (int c = c0; c < c1; c++) {
        const int t0 = c * C, n = min(C, g.N - t0);
        __syncthreads();
        if (g.causal) phi_rows(kh, t0, n, g, Wt, F, sq, X);
        load_rows(vh, t0, n, C, Dv, V);
        load_rows(oh, t0, n, C, Dv, O);
        __syncthreads();
        phi_rows(qh, t0, n, g, Wt, G, sq, X);   // (X keeps the raw q rows for the chain rule)
        __syncthreads();
        if (g.causal)
            for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
                const int i = idx / C, j = idx % C;
                float t = 0.f;
                if (j <= i)
                    for (int a = 0; a < P; a++) t = fmaf(G[i * P + a], F[j * P + a], t);
                A[idx] = t;
            }
        __syncthreads();
        // den_i, then out_i (into O, after its dout . out dot product)
        for (int i = threadIdx.x; i < C; i += blockDim.x) {
            float t = 0.f;
            for (int a = 0; a < P; a++) t = fmaf(G[i * P + a], z[a], t);
            if (g.causal)
                for (int j = 0; j <= i; j++) t += A[i * C + j];
            den[i] = i < n ? t : 1.f;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < C * Dv; idx += blockDim.x) {
            const int i = idx / Dv, cc = idx % Dv;
            float t = 0.f;
            for (int a = 0; a < P; a++) t = fmaf(G[i * P + a], S[a * SP + cc], t);
            if (g.causal)
                for (int j = 0; j <= i; j++) t = fmaf(A[i * C + j], V[j * Dv + cc], t);
            const float o = O[idx];
            Mn[idx] = i < n ? o / den[i] : 0.f;   // dnum
            O[idx] = o * (t / den[i]);            // dout_ic * out_ic
        }
        __syncthreads();
        for (int i = threadIdx.x; i < C; i += blockDim.x) {
            float t = 0.f;
            for (int cc = 0; cc < Dv; cc++) t += O[i * Dv + cc];
            dd[i] = i < n ? -t / den[i] : 0.f;
            if (i < n) {
                den_out[(long long)h * g.N + t0 + i] = den[i];
                dd_out[(long long)h * g.N + t0 + i] = dd[i];
            }
        }
        __syncthreads();
        if (g.causal)
            for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
                const int i = idx / C, j = idx % C;
                float t = 0.f;
                if (j <= i) {
                    t = dd[i];
                    for (int cc = 0; cc < Dv; cc++) t = fmaf(Mn[i * Dv + cc], V[j * Dv + cc], t);
                }
                Bm[idx] = t;
            }
        __syncthreads();
        // dG = B F + dnum S_prev^T + dden z_prev^T
        for (int idx = threadIdx.x; idx < C * P; idx += blockDim.x) {
            const int i = idx / P, a = idx % P;
            float t = z[a] * dd[i];
            for (int cc = 0; cc < Dv; cc++) t = fmaf(S[a * SP + cc], Mn[i * Dv + cc], t);
            if (g.causal)
                for (int j = 0; j <= i; j++) t = fmaf(Bm[i * C + j], F[j * P + a], t);
            dX[idx] = t;
        }
        __syncthreads();
        phi_chain(G, dX, X, g, W, t0, n, sq, dqh);
        __syncthreads();
        if (g.causal) accum_outer(S, z, F, V, nullptr, n, P, Dv, SP);   // S += F^T V, z += colsum F
        accum_outer(R, r, G, Mn, dd, n, P, Dv, SP);                     // R += G^T dnum, r += G^T dden
    }
    __syncthreads();
    float *dst = stR + slot;
    for (int idx = threadIdx.x; idx < P * Dv; idx += blockDim.x) dst[idx] = R[(idx / Dv) * SP + idx % Dv];
    for (int a = threadIdx.x; a < P; a += blockDim.x) dst[P * Dv + a] = r[a];
}

// ---- pass 3: dk, dv; each segment walks its chunks from the last to the first
template <typename T>
__global__ void __launch_bounds__(kBT)
bwd_dkdv_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const T *__restrict__ dout, const float *__restrict__ W, const float *__restrict__ Wt, BwdGeo g,
                const float *__restrict__ stR, const float *__restrict__ den_in,
                const float *__restrict__ dd_in, T *__restrict__ dk, T *__restrict__ dv)
{
    extern __shared__ float sm[];
    const BwdSmem Ls = bwd_layout(g, false);
    float *R = sm + Ls.S, *r = sm + Ls.z, *G = sm + Ls.G, *F = sm + Ls.F, *V = sm + Ls.V;
    float *Mn = sm + Ls.Mn, *X = sm + Ls.X, *dX = sm + Ls.dX, *A = sm + Ls.A, *Bm = sm + Ls.B;
    float *dd = sm + Ls.dd, *sq = sm + Ls.sq, *den = sm + Ls.den;
    const int h = blockIdx.x / g.nseg, s = blockIdx.x % g.nseg;
    const int P = g.P, Dv = g.Dv, C = g.C, D = g.D;
    const long long slot = ((long long)h * g.nseg + s) * (P * Dv + P);
    const int SP = Dv + 1;
    for (int idx = threadIdx.x; idx < P * Dv; idx += blockDim.x)   // the sums after this segment (or the totals)
        R[(idx / Dv) * SP + idx % Dv] = stR[slot + idx];
    for (int a = threadIdx.x; a < P; a += blockDim.x) r[a] = stR[slot + P * Dv + a];
    const T *qh = q + (long long)h * g.N * D, *kh = k + (long long)h * g.N * D;
    const T *vh = v + (long long)h * g.N * Dv, *oh = dout + (long long)h * g.N * Dv;
    T *dkh = dk + (long long)h * g.N * D, *dvh = dv + (long long)h * g.N * Dv;
    const int c0 = s * g.L, c1 = min(g.NC, c0 + g.L);
    for (int c = c1 - 1; c >= c0; c--) {
        const int t0 = c * C, n = min(C, g.N - t0);
        __syncthreads();
        phi_rows(qh, t0, n, g, Wt, G, sq, X);
        load_rows(vh, t0, n, C, Dv, V);
        load_rows(oh, t0, n, C, Dv, Mn);
        for (int i = threadIdx.x; i < C; i += blockDim.x) {
            den[i] = i < n ? den_in[(long long)h * g.N + t0 + i] : 1.f;
            dd[i] = i < n ? dd_in[(long long)h * g.N + t0 + i] : 0.f;
        }
        __syncthreads();
        phi_rows(kh, t0, n, g, Wt, F, sq, X);   // (X keeps the raw k rows for the chain rule)
        for (int idx = threadIdx.x; idx < C * Dv; idx += blockDim.x) Mn[idx] /= den[idx / Dv];
        __syncthreads();
        if (g.causal)
            for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
                const int i = idx / C, j = idx % C;
                float a = 0.f, b = 0.f;
                if (j <= i) {
                    for (int x = 0; x < P; x++) a = fmaf(G[i * P + x], F[j * P + x], a);
                    b = dd[i];
                    for (int cc = 0; cc < Dv; cc++) b = fmaf(Mn[i * Dv + cc], V[j * Dv + cc], b);
                }
                A[idx] = a;
                Bm[idx] = b;
            }
        __syncthreads();
        // dF = B^T G + V R_next + r_next,   dV = A^T dnum + F R_next
        for (int idx = threadIdx.x; idx < C * P; idx += blockDim.x) {
            const int j = idx / P, a = idx % P;
            float t = r[a];
            for (int cc = 0; cc < Dv; cc++) t = fmaf(R[a * SP + cc], V[j * Dv + cc], t);
            if (g.causal)
                for (int i = j; i < C; i++) t = fmaf(Bm[i * C + j], G[i * P + a], t);
            dX[idx] = t;
        }
        for (int idx = threadIdx.x; idx < n * Dv; idx += blockDim.x) {
            const int j = idx / Dv, cc = idx % Dv;
            float t = 0.f;
            for (int a = 0; a < P; a++) t = fmaf(R[a * SP + cc], F[j * P + a], t);
            if (g.causal)
                for (int i = j; i < C; i++) t = fmaf(A[i * C + j], Mn[i * Dv + cc], t);
            dvh[(long long)t0 * Dv + idx] = from_f32<T>(t);
        }
        __syncthreads();
        phi_chain(F, dX, X, g, W, t0, n, sq, dkh);
        __syncthreads();
        if (g.causal) accum_outer(R, r, G, Mn, dd, n, P, Dv, SP);   // R += G^T dnum, r += G^T dden
    }
}

// W [m, D] -> Wt [D, m]
__global__ void bwd_wt_kernel(const float *__restrict__ W, float *__restrict__ Wt, int m, int D)
{
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < m * D) Wt[(long long)(idx % D) * m + idx / D] = W[idx];
}

BwdGeo bwd_plan(const Problem &p, bool causal, int sms)
{
    BwdGeo g;
    g.BH = (int)p.BH;
    g.N = p.N;
    g.D = p.D;
    g.Dv = p.Dv;
    g.P = p.P;
    g.kind = p.kind;
    g.m = p.m;
    g.causal = causal ? 1 : 0;
    g.C = p.P * p.Dv > 4096 || p.P > 128 ? 16 : 32;
    g.NC = cdiv(p.N, g.C);
    // at most two items per SM (one CTA fits an SM at a time: two waves, no
    // third one); fewer, longer segments when the heads alone fill the GPU
    const long long want = (2LL * sms) / p.BH;
    const int nseg = (int)(want < 1 ? 1 : want > g.NC ? g.NC : want);
    g.L = cdiv(g.NC, nseg);
    g.nseg = cdiv(g.NC, g.L);
    return g;
}

template <typename T>
cudaError_t launch_backward(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal,
                            void *scratch, cudaStream_t st)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const BwdGeo g = bwd_plan(p, causal, sms);
    const int elems = g.P * g.Dv + g.P;
    float *stS = (float *)scratch;
    float *stR = stS + (size_t)g.BH * g.nseg * elems;
    float *den = stR + (size_t)g.BH * g.nseg * elems;
    float *dd = den + (size_t)g.BH * g.N;
    float *Wt = dd + (size_t)g.BH * g.N;   // random features: W transposed
    const size_t sm_sum = ((size_t)elems + (size_t)g.C * (g.P + g.Dv + 1 + g.D)) * sizeof(float);
    const size_t sm_dq = bwd_layout(g, true).total, sm_dkdv = bwd_layout(g, false).total;
    if (sm_dq > 227 * 1024 || sm_sum > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = set_max_smem_once<bwd_sums_kernel<T>>(227 * 1024)) != cudaSuccess) return e;
    if ((e = set_max_smem_once<bwd_dq_kernel<T>>(227 * 1024)) != cudaSuccess) return e;
    if ((e = set_max_smem_once<bwd_dkdv_kernel<T>>(227 * 1024)) != cudaSuccess) return e;
    const unsigned items = (unsigned)(g.BH * g.nseg);
    const dim3 sgrid((unsigned)cdiv(elems, kBT), (unsigned)g.BH);
    const T *q = (const T *)p.q, *k = (const T *)p.k, *v = (const T *)p.v, *o = (const T *)dout;
    const int m = p.kind == PHI_ELU1 ? 0 : rf_m(p.kind, p.P);
    if (m > 0) bwd_wt_kernel<<<cdiv(m * g.D, kBT), kBT, 0, st>>>(p.W, Wt, m, g.D);
    bwd_sums_kernel<T><<<items, kBT, sm_sum, st>>>(k, v, Wt, g, stS);
    bwd_scan_kernel<<<sgrid, kBT, 0, st>>>(stS, g.nseg, elems, causal ? 0 : 2);
    bwd_dq_kernel<T><<<items, kBT, sm_dq, st>>>(q, k, v, o, p.W, Wt, g, stS, stR, den, dd, (T *)dq);
    bwd_scan_kernel<<<sgrid, kBT, 0, st>>>(stR, g.nseg, elems, causal ? 1 : 2);
    bwd_dkdv_kernel<T><<<items, kBT, sm_dkdv, st>>>(q, k, v, o, p.W, Wt, g, stR, den, dd, (T *)dk, (T *)dv);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(m > 0 ? 6 : 5);
    return e;
}

}  // namespace

bool backward_supported(const Problem &p) { return (long long)p.P * p.Dv <= 16384; }

cudaError_t backward_scan(float *st, long long BH, int nseg, int elems, int mode, cudaStream_t s)
{
    const dim3 sgrid((unsigned)cdiv(elems, kBT), (unsigned)BH);
    const cudaError_t e = launch_dependent(bwd_scan_kernel, sgrid, dim3(kBT), 0, s, st, nseg, elems, mode);
    if (e == cudaSuccess) note_launches(1);
    return e;
}

size_t backward_scratch_bytes(const Problem &p, bool causal)
{
    if (backward_tc_supported(p)) return backward_tc_scratch_bytes(p, causal);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const BwdGeo g = bwd_plan(p, causal, sms);
    const size_t elems = (size_t)g.P * g.Dv + g.P;
    const size_t wt = p.kind == PHI_ELU1 ? 0 : (size_t)rf_m(p.kind, p.P) * p.D;   // W transposed
    return (2 * (size_t)g.BH * g.nseg * elems + 2 * (size_t)g.BH * g.N + wt) * sizeof(float);
}

cudaError_t backward(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal,
                     void *scratch, int *err, cudaStream_t s)
{
    if (backward_tc_supported(p)) return backward_tc(p, dout, dq, dk, dv, causal, scratch, err, s);
    if (p.dtype == DT_F32) return launch_backward<float>(p, dout, dq, dk, dv, causal, scratch, s);
    return launch_backward<__nv_bfloat16>(p, dout, dq, dk, dv, causal, scratch, s);
}

}  // namespace la
