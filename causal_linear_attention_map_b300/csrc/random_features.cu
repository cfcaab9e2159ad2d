// random_features.cu -- host-side draws of the random-feature projection W
// for the maps that differ from plain PRF only in how W is drawn (review
// page "Stable, Fast and Accurate: Kernelized Attention with RPE", proposed
// method: PRF, TRF, Sphere-PRF, ORF).
//
// The stream of N(0, 1) draws: draw t uses the SplitMix64 outputs of the
// counters 2t and 2t + 1 (seeded by `seed`), turned into two uniforms in
// (0, 1] and into one normal by the Box-Muller transform (its cosine branch).
// The draws are consumed in row-major order of the matrices named below.
#include <math.h>
#include <stdint.h>

#include <vector>

#include "linattn.h"

namespace {

uint64_t splitmix64(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

struct Normals {
    uint64_t seed, t = 0;
    double next()
    {
        const uint64_t a = splitmix64(seed + 2 * t), b = splitmix64(seed + 2 * t + 1);
        t++;
        const double u1 = ((a >> 11) + 1.0) * 0x1.0p-53;   // (0, 1]
        const double u2 = ((b >> 11) + 1.0) * 0x1.0p-53;
        return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
    }
};

}  // namespace

extern "C" int la_random_features(int w_kind, int m, int D, unsigned long long seed, float *W)
{
    if (!W) return LA_ERR_NULL;
    if (m < 1 || D < 1) return LA_ERR_DIM;
    if (w_kind != LA_W_GAUSSIAN && w_kind != LA_W_ORTHOGONAL && w_kind != LA_W_SPHERE) return LA_ERR_FEATURE;
    Normals g{seed};
    std::vector<double> row(D);
    if (w_kind == LA_W_GAUSSIAN || w_kind == LA_W_SPHERE) {
        for (int r = 0; r < m; r++) {
            double n2 = 0.0;
            for (int d = 0; d < D; d++) {
                row[d] = g.next();
                n2 += row[d] * row[d];
            }
            const double s = w_kind == LA_W_SPHERE ? sqrt((double)D / n2) : 1.0;
            for (int d = 0; d < D; d++) W[(long long)r * D + d] = (float)(row[d] * s);
        }
        return LA_OK;
    }
    // orthogonal blocks: a Gaussian D x D matrix, rows orthonormalised by
    // modified Gram-Schmidt, then D norms of fresh Gaussian D-vectors
    std::vector<double> Q((size_t)D * D);
    for (int r0 = 0; r0 < m; r0 += D) {
        for (size_t i = 0; i < Q.size(); i++) Q[i] = g.next();
        for (int i = 0; i < D; i++) {
            double *qi = &Q[(size_t)i * D];
            for (int j = 0; j < i; j++) {
                const double *qj = &Q[(size_t)j * D];
                double dot = 0.0;
                for (int d = 0; d < D; d++) dot += qi[d] * qj[d];
                for (int d = 0; d < D; d++) qi[d] -= dot * qj[d];
            }
            double n2 = 0.0;
            for (int d = 0; d < D; d++) n2 += qi[d] * qi[d];
            const double inv = 1.0 / sqrt(n2);
            for (int d = 0; d < D; d++) qi[d] *= inv;
        }
        for (int i = 0; i < D; i++) {
            double n2 = 0.0;
            for (int d = 0; d < D; d++) {
                const double x = g.next();
                n2 += x * x;
            }
            if (r0 + i >= m) continue;
            const double s = sqrt(n2);
            for (int d = 0; d < D; d++) W[(long long)(r0 + i) * D + d] = (float)(Q[(size_t)i * D + d] * s);
        }
    }
    return LA_OK;
}
