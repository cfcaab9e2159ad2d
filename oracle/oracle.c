/*
 * oracle.c -- the oracle for kernelized (linear) attention: a plain, slow,
 * obviously correct CPU implementation in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file.  It is used by the test suite, by the package smoke check
 * and by the timed CPU baseline of the benchmark, and by nothing else.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * What it follows (review pages of the papers, by title and section):
 *  - "Transformers are RNNs: Fast Autoregressive Transformers with Linear
 *    Attention", section "proposed method" (제안 방법), bullets 1-5: softmax
 *    is replaced by a feature map phi so that sim(q, k) = phi(q).phi(k);
 *    associativity gives phi(Q)(phi(K)^T V); causal masking is enforced with
 *    cumulative sums S_i, z_i updated step by step; the causal transformer is
 *    an RNN with two memories (S, z) and a recurrent update.
 *  - same page, section "main results" (주요 결과), bullet 2: the feature map
 *    is elu based.  Reading taken: phi(x) = elu(x) + 1 with alpha = 1, i.e.
 *    x + 1 for x > 0 and exp(x) otherwise.
 *  - "Stable, Fast and Accurate: Kernelized Attention with Relative
 *    Positional Encoding", section "proposed method", bullet 6: positive
 *    random features (PRF) are one of the supported feature maps.  The page
 *    names PRF without a formula; the formula used is the standard positive
 *    random feature map phi_r(x) = exp(w_r.x - |x|^2/2) / sqrt(m),
 *    r = 1..m, with W (m x D) passed in as data.
 *
 * The quantities, for one head with inputs q_i, k_i (D), v_i (Dv):
 *   S_i = sum_{j<=i} phi(k_j) v_j^T      (Dphi x Dv)
 *   z_i = sum_{j<=i} phi(k_j)            (Dphi)
 *   out_i = phi(q_i)^T S_i / phi(q_i)^T z_i
 * The non-causal form uses the sums over all j.  No epsilon is added to the
 * denominator: phi > 0 and z_i contains the term j = i, so it is positive.
 *
 * Layouts (row-major, heads flattened bh = b * H + h):
 *   q, k    [BH, N, D]       v, out  [BH, N, Dv]
 *   S       [BH, Dphi, Dv]   z       [BH, Dphi]
 *   W       [m, D]           (PRF only; NULL for elu+1)
 * Dphi = D for elu+1 and m for PRF.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PHI_ELU1 0
#define ORACLE_PHI_PRF 1
#define ORACLE_PHI_NPRF 2
#define ORACLE_PHI_TRF 3

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_phi_dim(int D, int kind, int m)
{
    if (kind == ORACLE_PHI_ELU1)
        return D;
    return kind == ORACLE_PHI_TRF ? 2 * m : m;
}

/* elu(x) + 1 with alpha = 1 ("Transformers are RNNs", main results b2). */
static double elu_plus_one(double x)
{
    if (x > 0.0)
        return x + 1.0;
    return exp(x);
}

/* phi of one D-vector x into f (Dphi values). */
void oracle_phi(const double *x, int D, int kind, const double *W, int m,
                double *f)
{
    if (kind == ORACLE_PHI_ELU1) {
        for (int d = 0; d < D; d++)
            f[d] = elu_plus_one(x[d]);
        return;
    }
    double sq = 0.0;
    for (int d = 0; d < D; d++)
        sq += x[d] * x[d];
    double inv_sqrt_m = 1.0 / sqrt((double)m);
    /* NPRF reads the direction x / |x| (x = 0 reads as 0) */
    double scale = (kind == ORACLE_PHI_NPRF && sq > 0.0) ? 1.0 / sqrt(sq) : 1.0;
    for (int r = 0; r < m; r++) {
        double wx = 0.0;
        for (int d = 0; d < D; d++)
            wx += W[(long)r * D + d] * x[d];
        wx *= scale;
        if (kind == ORACLE_PHI_PRF) {
            /* positive random features: exp(w_r . x - |x|^2 / 2) / sqrt(m) */
            f[r] = exp(wx - 0.5 * sq) * inv_sqrt_m;
        } else if (kind == ORACLE_PHI_NPRF) {
            /* PRF of the unit vector: exp(w_r . x/|x| - 1/2) / sqrt(m) (0 for x = 0: -0) */
            f[r] = exp(wx - (sq > 0.0 ? 0.5 : 0.0)) * inv_sqrt_m;
        } else {
            /* trigonometric: exp(|x|^2 / 2) / sqrt(m) [cos(w_r . x), sin(w_r . x)] */
            double a = exp(0.5 * sq) * inv_sqrt_m;
            f[r] = a * cos(wx);
            f[m + r] = a * sin(wx);
        }
    }
}

/* The two memories' update with one key/value pair:
 *   S += phi(k) v^T ;  z += phi(k)                                        */
static void update_state(double *S, double *z, const double *fk,
                         const double *v, int P, int Dv)
{
    for (int a = 0; a < P; a++) {
        z[a] += fk[a];
        for (int c = 0; c < Dv; c++)
            S[(long)a * Dv + c] += fk[a] * v[c];
    }
}

/* The readout: out = phi(q)^T S / phi(q)^T z. */
static void readout(const double *S, const double *z, const double *fq,
                    double *out, int P, int Dv)
{
    double den = 0.0;
    for (int a = 0; a < P; a++)
        den += fq[a] * z[a];
    for (int c = 0; c < Dv; c++) {
        double num = 0.0;
        for (int a = 0; a < P; a++)
            num += fq[a] * S[(long)a * Dv + c];
        out[c] = num / den;
    }
}

/*
 * Causal forward by the recurrence: for each head start from S = 0, z = 0
 * and for i = 0..N-1 first add (k_i, v_i) to the memories, then read out
 * with q_i (the sums include j = i).
 * S_out / z_out (nullable) receive the final memories S_N, z_N.
 */
void oracle_causal(const double *q, const double *k, const double *v,
                   double *out, long BH, long N, int D, int Dv, int kind,
                   const double *W, int m, double *S_out, double *z_out)
{
    int P = oracle_phi_dim(D, kind, m);
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        double *S = calloc((size_t)P * Dv, sizeof(double));
        double *z = calloc((size_t)P, sizeof(double));
        double *fk = malloc((size_t)P * sizeof(double));
        double *fq = malloc((size_t)P * sizeof(double));
        for (long i = 0; i < N; i++) {
            const double *ki = k + (h * N + i) * D;
            const double *qi = q + (h * N + i) * D;
            const double *vi = v + (h * N + i) * Dv;
            oracle_phi(ki, D, kind, W, m, fk);
            update_state(S, z, fk, vi, P, Dv);
            oracle_phi(qi, D, kind, W, m, fq);
            readout(S, z, fq, out + (h * N + i) * Dv, P, Dv);
        }
        if (S_out)
            memcpy(S_out + h * (long)P * Dv, S, (size_t)P * Dv * sizeof(double));
        if (z_out)
            memcpy(z_out + h * (long)P, z, (size_t)P * sizeof(double));
        free(S);
        free(z);
        free(fk);
        free(fq);
    }
}

/*
 * Non-causal forward ("Transformers are RNNs", proposed method b2): the
 * memories are summed over all N positions once, then every query reads
 * them out.
 */
void oracle_noncausal(const double *q, const double *k, const double *v,
                      double *out, long BH, long N, int D, int Dv, int kind,
                      const double *W, int m)
{
    int P = oracle_phi_dim(D, kind, m);
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        double *S = calloc((size_t)P * Dv, sizeof(double));
        double *z = calloc((size_t)P, sizeof(double));
        double *f = malloc((size_t)P * sizeof(double));
        for (long j = 0; j < N; j++) {
            oracle_phi(k + (h * N + j) * D, D, kind, W, m, f);
            update_state(S, z, f, v + (h * N + j) * Dv, P, Dv);
        }
        for (long i = 0; i < N; i++) {
            oracle_phi(q + (h * N + i) * D, D, kind, W, m, f);
            readout(S, z, f, out + (h * N + i) * Dv, P, Dv);
        }
        free(S);
        free(z);
        free(f);
    }
}

/*
 * One recurrent step for BH independent heads ("Transformers are RNNs",
 * proposed method b5): S, z [BH, Dphi, Dv] / [BH, Dphi] are updated in place
 * with (k, v) and then read out with q.  q, k [BH, D]; v, out [BH, Dv].
 */
void oracle_step(double *S, double *z, const double *q, const double *k,
                 const double *v, double *out, long BH, int D, int Dv,
                 int kind, const double *W, int m)
{
    int P = oracle_phi_dim(D, kind, m);
#pragma omp parallel for schedule(static)
    for (long h = 0; h < BH; h++) {
        double *f = malloc((size_t)P * sizeof(double));
        double *Sh = S + h * (long)P * Dv;
        double *zh = z + h * (long)P;
        oracle_phi(k + h * D, D, kind, W, m, f);
        update_state(Sh, zh, f, v + h * Dv, P, Dv);
        oracle_phi(q + h * D, D, kind, W, m, f);
        readout(Sh, zh, f, out + h * Dv, P, Dv);
        free(f);
    }
}

/*
 * The masked quadratic form, written out directly, for the listed rows of
 * ONE head (q, k [N, D]; v [N, Dv]):
 *   out_i = sum_{j in J(i)} (phi(q_i).phi(k_j)) v_j / sum_{j in J(i)} phi(q_i).phi(k_j)
 * with J(i) = {0..i} when causal and {0..N-1} otherwise.  rows[r] = i.
 * out_rows [count, Dv].  O(count * N * Dphi); used as brute force on tiny
 * inputs and on sampled rows of large ones.
 */
void oracle_quadratic_rows(const double *q, const double *k, const double *v,
                           double *out_rows, long N, int D, int Dv,
                           int causal, int kind, const double *W, int m,
                           const long *rows, long count)
{
    int P = oracle_phi_dim(D, kind, m);
    double *fk = malloc((size_t)N * P * sizeof(double));
#pragma omp parallel for schedule(static)
    for (long j = 0; j < N; j++)
        oracle_phi(k + j * D, D, kind, W, m, fk + j * P);
#pragma omp parallel for schedule(dynamic, 1)
    for (long r = 0; r < count; r++) {
        long i = rows[r];
        double *fq = malloc((size_t)P * sizeof(double));
        oracle_phi(q + i * D, D, kind, W, m, fq);
        double den = 0.0;
        double *num = calloc((size_t)Dv, sizeof(double));
        long last = causal ? i : N - 1;
        for (long j = 0; j <= last; j++) {
            double w = 0.0;
            for (int a = 0; a < P; a++)
                w += fq[a] * fk[j * P + a];
            den += w;
            for (int c = 0; c < Dv; c++)
                num[c] += w * v[j * Dv + c];
        }
        for (int c = 0; c < Dv; c++)
            out_rows[r * Dv + c] = num[c] / den;
        free(num);
        free(fq);
    }
    free(fk);
}

/*
 * The chain rule through phi: dx = J_phi(x)^T df for one D-vector x, given
 * the cotangent df (Dphi values).  f is scratch for Dphi values.
 *   elu + 1:  d phi / dx = 1 for x > 0, exp(x) otherwise (elementwise).
 *   PRF:      d phi_r / dx = phi_r(x) (w_r - x), so
 *             dx = sum_r df_r phi_r(x) w_r - x sum_r df_r phi_r(x).
 */
static void phi_vjp(const double *x, const double *df, int D, int kind,
                    const double *W, int m, double *dx, double *f)
{
    if (kind == ORACLE_PHI_ELU1) {
        for (int d = 0; d < D; d++)
            dx[d] = (x[d] > 0.0 ? 1.0 : exp(x[d])) * df[d];
        return;
    }
    oracle_phi(x, D, kind, W, m, f);
    double sq = 0.0;
    for (int d = 0; d < D; d++) {
        sq += x[d] * x[d];
        dx[d] = 0.0;
    }
    if (kind == ORACLE_PHI_PRF) {
        /* d phi_r / dx = phi_r (w_r - x) */
        double s = 0.0;
        for (int r = 0; r < m; r++) {
            double c = df[r] * f[r];
            s += c;
            for (int d = 0; d < D; d++)
                dx[d] += c * W[(long)r * D + d];
        }
        for (int d = 0; d < D; d++)
            dx[d] -= s * x[d];
    } else if (kind == ORACLE_PHI_NPRF) {
        /* with y = x/|x|: d phi_r / dy = phi_r w_r, and dy/dx = (I - y y^T) / |x| */
        if (sq == 0.0)
            return;
        double n = sqrt(sq), dy_y = 0.0;
        for (int r = 0; r < m; r++) {
            double c = df[r] * f[r];
            for (int d = 0; d < D; d++)
                dx[d] += c * W[(long)r * D + d];
        }
        for (int d = 0; d < D; d++)
            dy_y += dx[d] * x[d] / n;
        for (int d = 0; d < D; d++)
            dx[d] = (dx[d] - dy_y * x[d] / n) / n;
    } else {
        /* phi_c = a cos(u), phi_s = a sin(u), a = exp(|x|^2/2)/sqrt(m), u = W x:
         * dx = x sum_r (dc_r phi_c + ds_r phi_s) + sum_r w_r (ds_r phi_c - dc_r phi_s) */
        double s = 0.0;
        for (int r = 0; r < m; r++) {
            s += df[r] * f[r] + df[m + r] * f[m + r];
            double c = df[m + r] * f[r] - df[r] * f[m + r];
            for (int d = 0; d < D; d++)
                dx[d] += c * W[(long)r * D + d];
        }
        for (int d = 0; d < D; d++)
            dx[d] += s * x[d];
    }
}

/* R += g dn^T ;  r += g dd  (the reverse memories, one query's terms) */
static void accumulate_reverse(double *R, double *r, const double *g,
                               const double *dn, double dd, int P, int Dv)
{
    for (int a = 0; a < P; a++) {
        r[a] += g[a] * dd;
        for (int c = 0; c < Dv; c++)
            R[(long)a * Dv + c] += g[a] * dn[c];
    }
}

/*
 * Gradients of L = sum_i dout_i . out_i with respect to q, k and v
 * ("Transformers are RNNs", proposed method b4: the gradients of the
 * forward and backward propagation are computed in linear time, with
 * cumulative sums like the forward pass).  With g_i = phi(q_i),
 * f_j = phi(k_j), num_i = S_i^T g_i, den_i = z_i . g_i, out = num / den:
 *   dnum_i = dout_i / den_i,   dden_i = -(dout_i . out_i) / den_i
 *   d g_i  = S_i dnum_i + z_i dden_i                 (forward sweep)
 *   R_j = sum_{i >= j} g_i dnum_i^T,  r_j = sum_{i >= j} g_i dden_i
 *   d f_j  = R_j v_j + r_j,   dv_j = R_j^T f_j       (reverse sweep)
 * then dq, dk through phi (phi_vjp).  The non-causal form uses the sums over
 * all positions for S, z, R and r.
 * Layouts as for the forward: q, k, dq, dk [BH, N, D]; v, dout, dv [BH, N, Dv].
 */
void oracle_backward(const double *q, const double *k, const double *v,
                     const double *dout, double *dq, double *dk, double *dv,
                     long BH, long N, int D, int Dv, int causal, int kind,
                     const double *W, int m)
{
    int P = oracle_phi_dim(D, kind, m);
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        double *S = calloc((size_t)P * Dv, sizeof(double));
        double *z = calloc((size_t)P, sizeof(double));
        double *R = calloc((size_t)P * Dv, sizeof(double));
        double *r = calloc((size_t)P, sizeof(double));
        double *f = malloc((size_t)P * sizeof(double));
        double *g = malloc((size_t)P * sizeof(double));
        double *dphi = malloc((size_t)P * sizeof(double));
        double *tmp = malloc((size_t)P * sizeof(double));
        double *dnum = malloc((size_t)N * Dv * sizeof(double));
        double *dden = malloc((size_t)N * sizeof(double));
        const double *qh = q + h * N * D, *kh = k + h * N * D;
        const double *vh = v + h * N * Dv, *oh = dout + h * N * Dv;
        if (!causal) {
            for (long j = 0; j < N; j++) {
                oracle_phi(kh + j * D, D, kind, W, m, f);
                update_state(S, z, f, vh + j * Dv, P, Dv);
            }
        }
        /* forward sweep: the memories S_i, z_i, the readout and d g_i */
        for (long i = 0; i < N; i++) {
            if (causal) {
                oracle_phi(kh + i * D, D, kind, W, m, f);
                update_state(S, z, f, vh + i * Dv, P, Dv);
            }
            oracle_phi(qh + i * D, D, kind, W, m, g);
            double den = 0.0;
            for (int a = 0; a < P; a++)
                den += g[a] * z[a];
            double dot = 0.0;
            for (int c = 0; c < Dv; c++) {
                double s = 0.0;
                for (int a = 0; a < P; a++)
                    s += g[a] * S[(long)a * Dv + c];
                dot += oh[i * Dv + c] * (s / den);
            }
            dden[i] = -dot / den;
            for (int c = 0; c < Dv; c++)
                dnum[i * Dv + c] = oh[i * Dv + c] / den;
            for (int a = 0; a < P; a++) {
                double s = z[a] * dden[i];
                for (int c = 0; c < Dv; c++)
                    s += S[(long)a * Dv + c] * dnum[i * Dv + c];
                dphi[a] = s;
            }
            phi_vjp(qh + i * D, dphi, D, kind, W, m, dq + (h * N + i) * D, tmp);
        }
        if (!causal) {
            for (long i = 0; i < N; i++) {
                oracle_phi(qh + i * D, D, kind, W, m, g);
                accumulate_reverse(R, r, g, dnum + i * Dv, dden[i], P, Dv);
            }
        }
        /* reverse sweep: R_j, r_j over i >= j, then d f_j and dv_j */
        for (long j = N - 1; j >= 0; j--) {
            if (causal) {
                oracle_phi(qh + j * D, D, kind, W, m, g);
                accumulate_reverse(R, r, g, dnum + j * Dv, dden[j], P, Dv);
            }
            oracle_phi(kh + j * D, D, kind, W, m, f);
            for (int a = 0; a < P; a++) {
                double s = r[a];
                for (int c = 0; c < Dv; c++)
                    s += R[(long)a * Dv + c] * vh[j * Dv + c];
                dphi[a] = s;
            }
            for (int c = 0; c < Dv; c++) {
                double s = 0.0;
                for (int a = 0; a < P; a++)
                    s += R[(long)a * Dv + c] * f[a];
                dv[(h * N + j) * Dv + c] = s;
            }
            phi_vjp(kh + j * D, dphi, D, kind, W, m, dk + (h * N + j) * D, tmp);
        }
        free(S); free(z); free(R); free(r); free(f); free(g); free(dphi);
        free(tmp); free(dnum); free(dden);
    }
}

/*
 * Softmax attention as an RNN ("Attention as an RNN", proposed method: a
 * learned query token q reads keys and values as a many-to-one RNN; its
 * many-to-many outputs are the outputs after every prefix).  Per head, with
 * s_i = q . k_i:
 *     o_k = sum_{i<=k} exp(s_i) v_i / sum_{i<=k} exp(s_i)
 * evaluated as the RNN cell over the state (m, u, w) = (running max of s,
 * sum of exp(s_i - m), sum of exp(s_i - m) v_i):
 *     m' = max(m, s),  u' = u exp(m - m') + exp(s - m'),
 *     w' = w exp(m - m') + exp(s - m') v,     o = w' / u'.
 * The initial state is m = -infinity, u = 0, w = 0.  No 1/sqrt(D) factor is
 * applied to s (the caller scales q).
 * q [BH, D]; k [BH, N, D]; v, out [BH, N, Dv]; state [BH, Dv + 2] as
 * (m, u, w_0..w_{Dv-1}): in/out for oracle_prefix_step, out (nullable) for
 * oracle_prefix_attention.
 */
static void prefix_cell(double *st, const double *q, const double *k,
                        const double *v, double *o, int D, int Dv)
{
    double s = 0.0;
    for (int d = 0; d < D; d++)
        s += q[d] * k[d];
    double m = st[0];
    double mn = s > m ? s : m;
    double a = (m == -INFINITY) ? 0.0 : exp(m - mn);
    double b = exp(s - mn);
    st[0] = mn;
    st[1] = st[1] * a + b;
    for (int c = 0; c < Dv; c++) {
        st[2 + c] = st[2 + c] * a + b * v[c];
        o[c] = st[2 + c] / st[1];
    }
}

void oracle_prefix_attention(const double *q, const double *k, const double *v,
                             double *out, long BH, long N, int D, int Dv,
                             double *state_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        double *st = malloc((size_t)(Dv + 2) * sizeof(double));
        st[0] = -INFINITY;
        st[1] = 0.0;
        for (int c = 0; c < Dv; c++)
            st[2 + c] = 0.0;
        for (long i = 0; i < N; i++)
            prefix_cell(st, q + h * D, k + (h * N + i) * D, v + (h * N + i) * Dv,
                        out + (h * N + i) * Dv, D, Dv);
        if (state_out)
            memcpy(state_out + h * (long)(Dv + 2), st, (size_t)(Dv + 2) * sizeof(double));
        free(st);
    }
}

void oracle_prefix_step(double *state, const double *q, const double *k,
                        const double *v, double *out, long BH, int D, int Dv)
{
#pragma omp parallel for schedule(static)
    for (long h = 0; h < BH; h++)
        prefix_cell(state + h * (long)(Dv + 2), q + h * D, k + h * D, v + h * Dv,
                    out + h * Dv, D, Dv);
}

/*
 * Kernelized attention with relative positional encoding ("Stable, Fast and
 * Accurate: Kernelized Attention with Relative Positional Encoding",
 * proposed method: the RPE matrix is Toeplitz - its entry depends only on
 * i - j - and multiplies the kernelized attention elementwise):
 *   out_i = sum_{j in J(i)} c_{i-j} (phi(q_i).phi(k_j)) v_j
 *           / sum_{j in J(i)} c_{i-j} phi(q_i).phi(k_j),      c_t = exp(b_t)
 * with J(i) = {0..i} (causal) or all positions.  b [H, 2N - 1] holds the
 * log-weights of head h at index t + N - 1 for t = i - j in [-(N-1), N-1]
 * (heads bh = b_idx * H + h share row h).  Written out directly, O(N^2).
 */
void oracle_rpe(const double *q, const double *k, const double *v,
                const double *b, double *out, long BH, long N, int H, int D,
                int Dv, int causal, int kind, const double *W, int m)
{
    int P = oracle_phi_dim(D, kind, m);
#pragma omp parallel for schedule(dynamic, 1)
    for (long h = 0; h < BH; h++) {
        const double *bh = b + (h % H) * (2 * N - 1);
        double *fk = malloc((size_t)N * P * sizeof(double));
        double *fq = malloc((size_t)P * sizeof(double));
        double *num = malloc((size_t)Dv * sizeof(double));
        for (long j = 0; j < N; j++)
            oracle_phi(k + (h * N + j) * D, D, kind, W, m, fk + j * P);
        for (long i = 0; i < N; i++) {
            oracle_phi(q + (h * N + i) * D, D, kind, W, m, fq);
            double den = 0.0;
            for (int c = 0; c < Dv; c++)
                num[c] = 0.0;
            long last = causal ? i : N - 1;
            for (long j = 0; j <= last; j++) {
                double a = 0.0;
                for (int x = 0; x < P; x++)
                    a += fq[x] * fk[j * P + x];
                a *= exp(bh[i - j + N - 1]);
                den += a;
                for (int c = 0; c < Dv; c++)
                    num[c] += a * v[(h * N + j) * Dv + c];
            }
            for (int c = 0; c < Dv; c++)
                out[(h * N + i) * Dv + c] = num[c] / den;
        }
        free(fk);
        free(fq);
        free(num);
    }
}
