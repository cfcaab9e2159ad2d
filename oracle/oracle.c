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
    return kind == ORACLE_PHI_PRF ? m : D;
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
    /* positive random features: exp(w_r . x - |x|^2 / 2) / sqrt(m) */
    double sq = 0.0;
    for (int d = 0; d < D; d++)
        sq += x[d] * x[d];
    double inv_sqrt_m = 1.0 / sqrt((double)m);
    for (int r = 0; r < m; r++) {
        double wx = 0.0;
        for (int d = 0; d < D; d++)
            wx += W[(long)r * D + d] * x[d];
        f[r] = exp(wx - 0.5 * sq) * inv_sqrt_m;
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
