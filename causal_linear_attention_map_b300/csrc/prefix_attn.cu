// prefix_attn.cu -- softmax attention of one query token per head over every
// prefix of the sequence, as an RNN (review page "Attention as an RNN",
// proposed method: attention is a many-to-one RNN whose many-to-many outputs
// come from a parallel prefix scan).  Per head, with s_i = q . k_i:
//     o_k = sum_{i<=k} exp(s_i) v_i / sum_{i<=k} exp(s_i)
// The scan's state is (m, u, w): the largest score so far, and the sums of
// exp(s_i - m) and exp(s_i - m) v_i.  Two states combine associatively
// (left a, right b): m = max(m_a, m_b), u = u_a e^(m_a - m) + u_b e^(m_b - m),
// w likewise.
//
// One pass over K and V: the sequence is cut into tiles of kTile positions,
// handed out in order from a ticket counter.  A tile computes its scores, its
// own aggregate state, and publishes it (flag 1); one warp then looks back
// over the earlier tiles of its head, combining published aggregates until
// it meets a published inclusive state (flag 2) - decoupled look-back - and
// publishes its own inclusive state.  The outputs are then formed from the
// exclusive prefix and the tile's running sums (a second read of the tile's
// V, from L2).  The page names Hillis-Steele; on this GPU the work-efficient
// single pass with look-back reads K and V from HBM once, which is what
// bounds the operation.  Waits on other tiles' flags are bounded: on expiry
// the library's error word is set and the kernel finishes without waiting.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kPT = 256;      // threads per CTA
constexpr int kTile = 256;    // positions per tile
constexpr long long kSpinLimit = 1LL << 26;   // flag polls before a wait gives up
constexpr int kErrTimeout = 1;

struct PrefixGeo {
    int BH, N, D, Dv, tph;    // tph: tiles per head
};

__device__ __forceinline__ int ld_flag(const int *f)
{
    return *reinterpret_cast<const volatile int *>(f);
}

// (ma, ua) (+) (mb, ub) into (mb, ub), returning the two rescale factors
// (ea for the left side, eb for the right) for the w columns.  An empty side
// (m = -inf) contributes nothing.
__device__ __forceinline__ void combine_mu(float ma, float ua, float &mb, float &ub, float &ea, float &eb)
{
    if (ma == -INFINITY) {
        ea = 0.f;
        eb = 1.f;
        return;
    }
    if (mb == -INFINITY) {
        ea = 1.f;
        eb = 0.f;
        mb = ma;
        ub = ua;
        return;
    }
    const float m = fmaxf(ma, mb);
    ea = __expf(ma - m);
    eb = __expf(mb - m);
    ub = ua * ea + ub * eb;
    mb = m;
}

template <typename T>
__global__ void __launch_bounds__(kPT)
prefix_attn_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   T *__restrict__ out, float *__restrict__ state_out, PrefixGeo g, int *ticket,
                   int *flags, float *agg, float *incl, int *err)
{
    // Rows of a tile are split into G = kPT / Dv groups of R rows; thread
    // (grp, col) owns column col of group grp.  Within a group the state is
    // carried with the group's running maximum (factors a_r, b_r per row), so
    // no exponential is taken of a score far below a later one.
    __shared__ int s_tile;
    __shared__ float s_s[kTile];              // scores
    __shared__ float s_a[kTile], s_b[kTile];  // per-row rescale of the carried sums, weight of row r
    __shared__ float s_m[kTile], s_U[kTile];  // group-running max and u after row r
    __shared__ float s_w[kPT];                // per-(group, column) w: the group's sums, then its offset
    __shared__ float s_gm[16], s_gu[16];      // per group: its (m, u), then its exclusive offset
    __shared__ float s_al[kTile], s_be[kTile], s_rd[kTile];   // output factors per row
    __shared__ float s_X[2 + 128];            // exclusive prefix of the tile (m, u, w)
    __shared__ float s_T[2 + 128];            // the tile's aggregate (m, u, w)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_tile = atomicAdd(ticket, 1);
    __syncthreads();
    const long long tile = s_tile;
    const int h = (int)(tile / g.tph), t = (int)(tile % g.tph);
    const int i0 = t * kTile, n = min(kTile, g.N - i0);
    const int D = g.D, Dv = g.Dv, SW = Dv + 2;
    const int G = kPT / Dv, R = kTile / G, grp = tid / Dv, col = tid % Dv;
    const T *kh = k + ((long long)h * g.N + i0) * D;
    const T *vh = v + ((long long)h * g.N + i0) * Dv;
    T *oh = out + ((long long)h * g.N + i0) * Dv;

    // scores s_i = q . k_i: one warp per row, lanes over the features (coalesced rows)
    float qr[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int d = lane + 32 * j;
        qr[j] = d < D ? to_f32(q[(long long)h * D + d]) : 0.f;
    }
    for (int i = warp; i < kTile; i += kPT / 32) {
        float s = 0.f;
        if (i < n) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int d = lane + 32 * j;
                if (d < D) s = fmaf(qr[j], to_f32(kh[(long long)i * D + d]), s);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) s_s[i] = s;
    }
    __syncthreads();
    // per group: the RNN cell's (m, u) row by row, and the factors a_r, b_r
    if (tid < G) {
        float m = -INFINITY, u = 0.f;
        for (int r = tid * R; r < tid * R + R; r++) {
            float a = 1.f, b = 0.f;
            if (r < n) {
                const float s = s_s[r], mn = fmaxf(m, s);
                a = m == -INFINITY ? 0.f : __expf(m - mn);
                b = __expf(s - mn);
                m = mn;
                u = u * a + b;
            }
            s_a[r] = a;
            s_b[r] = b;
            s_m[r] = m;
            s_U[r] = u;
        }
        s_gm[tid] = m;
        s_gu[tid] = u;
    }
    __syncthreads();
    // per (group, column): the group's w
    float w = 0.f;
    for (int r = grp * R; r < grp * R + R && r < n; r++) w = w * s_a[r] + s_b[r] * to_f32(vh[(long long)r * Dv + col]);
    s_w[tid] = w;
    __syncthreads();
    // exclusive offsets of the groups within the tile, and the tile's aggregate
    if (tid < Dv) {
        float om = -INFINITY, ou = 0.f, ow = 0.f;
        for (int gg = 0; gg < G; gg++) {
            const float gm = s_gm[gg], gu = s_gu[gg], gw = s_w[gg * Dv + tid];
            s_w[gg * Dv + tid] = ow;   // (offset of group gg, column tid)
            float ea, eb, m2 = gm, u2 = gu;
            combine_mu(om, ou, m2, u2, ea, eb);   // (om, ou, ow) (+) group gg
            ow = ow * ea + gw * eb;
            om = m2;
            ou = u2;
        }
        s_T[2 + tid] = ow;
        if (tid == 0) {
            s_T[0] = om;
            s_T[1] = ou;
        }
    }
    __syncthreads();
    if (tid == 0) {   // the groups' (m, u) offsets
        float om = -INFINITY, ou = 0.f;
        for (int gg = 0; gg < G; gg++) {
            const float gm = s_gm[gg], gu = s_gu[gg];
            s_gm[gg] = om;
            s_gu[gg] = ou;
            float ea, eb, m2 = gm, u2 = gu;
            combine_mu(om, ou, m2, u2, ea, eb);
            om = m2;
            ou = u2;
        }
    }

    // publish and look back (warp 0): X = the states of every earlier tile of this head
    if (warp == 0) {
        float *myagg = agg + tile * SW, *myincl = incl + tile * SW;
        float xm = -INFINITY, xu = 0.f, xw[4] = {0.f, 0.f, 0.f, 0.f};
        if (t > 0) {
            for (int c = lane; c < SW; c += 32) __stcg(myagg + c, s_T[c]);
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                atomicExch(flags + tile, 1);
            }
            long long pred = tile - 1;
            while (true) {
                int f = 0;
                if (lane == 0) {
                    long long spins = 0;
                    while ((f = ld_flag(flags + pred)) == 0) {
                        if (++spins > kSpinLimit) {   // give up: report, and finish without the prefix
                            atomicExch(err, kErrTimeout);
                            f = -1;
                            break;
                        }
                    }
                }
                f = __shfl_sync(0xffffffffu, f, 0);
                if (f < 0) break;
                __threadfence();
                const float *src = (f == 2 ? incl : agg) + pred * SW;
                float pm = __ldcg(src), pu = __ldcg(src + 1), ea, eb;
                combine_mu(pm, pu, xm, xu, ea, eb);   // X = pred (+) X
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int c = lane + 32 * j;
                    if (c < Dv) xw[j] = __ldcg(src + 2 + c) * ea + xw[j] * eb;
                }
                if (f == 2) break;
                pred--;
            }
        }
        // inclusive = X (+) T, published with flag 2
        float im = s_T[0], iu = s_T[1], ea, eb, iw[4];
        const float m0 = xm, u0 = xu;
        combine_mu(m0, u0, im, iu, ea, eb);
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = lane + 32 * j;
            iw[j] = c < Dv ? xw[j] * ea + s_T[2 + c] * eb : 0.f;
            if (c < Dv) s_X[2 + c] = xw[j];
        }
        if (lane == 0) {
            __stcg(myincl, im);
            __stcg(myincl + 1, iu);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = lane + 32 * j;
            if (c < Dv) __stcg(myincl + 2 + c, iw[j]);
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            atomicExch(flags + tile, 2);
        }
        if (state_out && t == g.tph - 1) {   // the head's final RNN state
            float *so = state_out + (long long)h * SW;
            if (lane == 0) {
                so[0] = im;
                so[1] = iu;
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int c = lane + 32 * j;
                if (c < Dv) so[2 + c] = iw[j];
            }
        }
        if (lane == 0) {
            s_X[0] = xm;
            s_X[1] = xu;
        }
    }
    __syncthreads();
    // per group: Xg = X (+) the group's offset (m, u in s_gm, s_gu); per column: its w
    const float xm = s_X[0], xu = s_X[1];
    float gm = s_gm[grp], gu = s_gu[grp], ea, eb;
    combine_mu(xm, xu, gm, gu, ea, eb);
    const float gw = s_X[2 + col] * ea + s_w[tid] * eb;
    // per row: o_r = (Xg.w al + w_r be) / (Xg.u al + U_r be), al = e^(Xg.m - mu), be = e^(m_r - mu)
    if (tid < kTile) {
        const int r = tid, rg = r / R;
        float m2 = s_gm[rg], u2 = s_gu[rg], e1, e2;
        combine_mu(xm, xu, m2, u2, e1, e2);   // Xg of row r's group
        float mr = s_m[r], ur = s_U[r], al, be;
        combine_mu(m2, u2, mr, ur, al, be);
        s_al[r] = al;
        s_be[r] = be;
        s_rd[r] = r < n ? 1.f / ur : 0.f;
    }
    __syncthreads();
    float run = 0.f;
    for (int r = grp * R; r < grp * R + R && r < n; r++) {
        run = run * s_a[r] + s_b[r] * to_f32(vh[(long long)r * Dv + col]);
        oh[(long long)r * Dv + col] = from_f32<T>((gw * s_al[r] + run * s_be[r]) * s_rd[r]);
    }
}

// One RNN step per head: state (m, u, w) [BH, Dv + 2] fp32 in place; one warp per head.
template <typename T>
__global__ void prefix_step_kernel(float *__restrict__ state, const T *__restrict__ q, const T *__restrict__ k,
                                   const T *__restrict__ v, T *__restrict__ out, long long BH, int D, int Dv)
{
    const long long h = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (h >= BH) return;
    float s = 0.f;
    for (int d = lane; d < D; d += 32) s = fmaf(to_f32(q[h * D + d]), to_f32(k[h * D + d]), s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    float *st = state + h * (Dv + 2);
    const float m = st[0], mn = fmaxf(m, s);
    const float a = m == -INFINITY ? 0.f : __expf(m - mn), b = __expf(s - mn);
    const float u = st[1] * a + b;
    for (int c = lane; c < Dv; c += 32) {
        const float w = st[2 + c] * a + b * to_f32(v[h * Dv + c]);
        st[2 + c] = w;
        out[h * Dv + c] = from_f32<T>(w / u);
    }
    __syncwarp();
    if (lane == 0) {
        st[0] = mn;
        st[1] = u;
    }
}

__global__ void prefix_empty_kernel(float *state, long long BH, int Dv)
{
    const long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (i >= BH * (Dv + 2)) return;
    state[i] = i % (Dv + 2) == 0 ? -INFINITY : 0.f;
}

template <typename T>
cudaError_t launch_prefix(const void *q, const void *k, const void *v, void *out, float *state_out, long long BH,
                          int N, int D, int Dv, void *scratch, int *err, cudaStream_t s)
{
    PrefixGeo g;
    g.BH = (int)BH;
    g.N = N;
    g.D = D;
    g.Dv = Dv;
    g.tph = cdiv(N, kTile);
    const long long tiles = BH * g.tph;
    const size_t SW = (size_t)Dv + 2;
    unsigned char *b = (unsigned char *)scratch;
    int *ticket = (int *)b;
    int *flags = (int *)(b + 256);
    float *agg = (float *)(b + 256 + ((tiles * 4 + 255) & ~255LL));
    float *incl = agg + tiles * SW;
    cudaError_t e = cudaMemsetAsync(scratch, 0, 256 + tiles * 4, s);
    if (e != cudaSuccess) return e;
    prefix_attn_kernel<T><<<(unsigned)tiles, kPT, 0, s>>>((const T *)q, (const T *)k, (const T *)v, (T *)out,
                                                          state_out, g, ticket, flags, agg, incl, err);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

size_t prefix_scratch_bytes(long long BH, int N, int Dv)
{
    const long long tiles = BH * cdiv(N, kTile);
    return 256 + ((tiles * 4 + 255) & ~255LL) + 2 * (size_t)tiles * (Dv + 2) * sizeof(float);
}

cudaError_t prefix_attention(const void *q, const void *k, const void *v, void *out, float *state_out,
                             long long BH, int N, int D, int Dv, int dtype, void *scratch, int *err,
                             cudaStream_t s)
{
    if (dtype == DT_F32) return launch_prefix<float>(q, k, v, out, state_out, BH, N, D, Dv, scratch, err, s);
    return launch_prefix<__nv_bfloat16>(q, k, v, out, state_out, BH, N, D, Dv, scratch, err, s);
}

cudaError_t prefix_empty_state(float *state, long long BH, int Dv, cudaStream_t s)
{
    const long long n = BH * (Dv + 2);
    prefix_empty_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(state, BH, Dv);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

cudaError_t prefix_step(float *state, const void *q, const void *k, const void *v, void *out, long long BH,
                        int D, int Dv, int dtype, cudaStream_t s)
{
    const unsigned grid = (unsigned)((BH + 7) / 8);
    if (dtype == DT_F32)
        prefix_step_kernel<float><<<grid, 256, 0, s>>>(state, (const float *)q, (const float *)k,
                                                       (const float *)v, (float *)out, BH, D, Dv);
    else
        prefix_step_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            state, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (__nv_bfloat16 *)out, BH, D, Dv);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace la
