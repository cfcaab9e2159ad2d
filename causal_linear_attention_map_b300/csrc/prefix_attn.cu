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
// handed out in order from a ticket counter (round the heads).  A tile computes its scores, its
// own aggregate state, and publishes it (flag 1); one warp then looks back
// over the earlier tiles of its head, combining published aggregates until
// it meets a published inclusive state (flag 2) - decoupled look-back - and
// publishes its own inclusive state.  The outputs are then formed from the
// exclusive prefix and the tile's running sums.  Within a tile the rows form
// one group of 32 per warp: the group's running (m, u) is an inclusive warp
// scan of (m, u) pairs, and the group sums of the w columns are short serial
// recurrences (32 rows) whose V loads do not depend on them (the outputs read
// the tile's V again, from L2).  The page names Hillis-Steele; on this GPU the work-efficient
// single pass with look-back reads K and V from HBM once, which is what
// bounds the operation.  Waits on other tiles' flags are bounded: on expiry
// the library's error word is set and the kernel finishes without waiting.
#include "common.cuh"
#include "kernels.h"

namespace la {
namespace {

constexpr int kPT = 256;      // threads per CTA
constexpr int kTile = 256;    // positions per tile (one per thread)
constexpr int kGroups = kPT / 32;      // groups of rows, one per warp
constexpr int kGR = kTile / kGroups;   // rows per group
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

// columns [c0, c0 + cpl) (cpl in {1, 2, 4}) of row `row` of a [rows, Dv] block as fp32
template <typename T>
__device__ __forceinline__ void load_cols(const T *base, long long row, int Dv, int c0, int cpl, bool ok, float (&o)[4])
{
    o[0] = o[1] = o[2] = o[3] = 0.f;
    if (!ok) return;
    const T *p = base + row * Dv + c0;
    if constexpr (sizeof(T) == 2) {
        if (cpl == 4) {
            const uint2 x = *reinterpret_cast<const uint2 *>(p);
            o[0] = __uint_as_float(x.x << 16);
            o[1] = __uint_as_float(x.x & 0xffff0000u);
            o[2] = __uint_as_float(x.y << 16);
            o[3] = __uint_as_float(x.y & 0xffff0000u);
        } else if (cpl == 2) {
            const uint32_t x = *reinterpret_cast<const uint32_t *>(p);
            o[0] = __uint_as_float(x << 16);
            o[1] = __uint_as_float(x & 0xffff0000u);
        } else {
            o[0] = to_f32(p[0]);
        }
    } else {
        if (cpl == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(p);
            o[0] = x.x;
            o[1] = x.y;
            o[2] = x.z;
            o[3] = x.w;
        } else if (cpl == 2) {
            const float2 x = *reinterpret_cast<const float2 *>(p);
            o[0] = x.x;
            o[1] = x.y;
        } else {
            o[0] = to_f32(p[0]);
        }
    }
}

// q . (16 bytes of a k row), q in fp32 from shared memory
template <typename T> __device__ __forceinline__ float dot_piece(uint4 x, const float *qs);
template <> __device__ __forceinline__ float dot_piece<float>(uint4 x, const float *qs)
{
    return __uint_as_float(x.x) * qs[0] + __uint_as_float(x.y) * qs[1] + __uint_as_float(x.z) * qs[2] +
           __uint_as_float(x.w) * qs[3];
}
template <> __device__ __forceinline__ float dot_piece<__nv_bfloat16>(uint4 x, const float *qs)
{
    // a bf16 is the top half of an fp32
    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        acc = fmaf(__uint_as_float(u[i] << 16), qs[2 * i], acc);
        acc = fmaf(__uint_as_float(u[i] & 0xffff0000u), qs[2 * i + 1], acc);
    }
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kPT, 4)
prefix_attn_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   T *__restrict__ out, float *__restrict__ state_out, PrefixGeo g, int *ticket,
                   int *flags, float *agg, float *incl, int *err)
{
    // Rows of a tile form kGroups groups of kGR rows, one per warp.  Within a
    // group the state is carried relative to the group's running maximum
    // (factors a_r, b_r per row), so no exponential is taken of a score far
    // below a later one.
    __shared__ int s_tile;
    __shared__ float s_a[kTile], s_b[kTile];  // per-row rescale of the carried sums, weight of row r
    __shared__ float s_m[kTile], s_U[kTile];  // group-running max and u after row r
    __shared__ float s_w[kGroups * 128];      // per (group, column): the group's w, then its offset
    __shared__ float s_gm[kGroups], s_gu[kGroups];     // per group: its (m, u), then its exclusive offset
    __shared__ float s_ge1[kGroups], s_ge2[kGroups];   // per group: factors of X and of the offset in Xg
    __shared__ float s_xgm[kGroups], s_xgu[kGroups];   // per group: Xg = X (+) offset, its (m, u)
    __shared__ float s_al[kTile], s_be[kTile], s_rd[kTile];   // output factors per row
    __shared__ float s_X[2 + 128];            // exclusive prefix of the tile (m, u, w)
    __shared__ float s_T[2 + 128];            // the tile's aggregate (m, u, w)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_tile = atomicAdd(ticket, 1);
    __syncthreads();
    const long long tile = s_tile;
    // tickets go round the heads (tile t of head h is ticket t * BH + h), so the
    // tiles in flight spread over every head and each look-back stays short
    const int h = (int)(tile % g.BH), t = (int)(tile / g.BH);
    const int i0 = t * kTile, n = min(kTile, g.N - i0);
    const int D = g.D, Dv = g.Dv, SW = Dv + 2;
    const T *kh = k + ((long long)h * g.N + i0) * D;
    const T *vh = v + ((long long)h * g.N + i0) * Dv;
    T *oh = out + ((long long)h * g.N + i0) * Dv;

    // the tile's K and V rows into L2 in bulk, so that the V rows are on chip by
    // the time the group sums read them (the scores read K meanwhile)
    if (tid == 0) {
        const unsigned kb = (unsigned)((long long)n * D * sizeof(T)), vb = (unsigned)((long long)n * Dv * sizeof(T));
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kh), "r"(kb) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vh), "r"(vb) : "memory");
    }
    // q -> shared memory (fp32)
    __shared__ float s_q[128];
    for (int d = tid; d < D; d += kPT) s_q[d] = to_f32(q[(long long)h * D + d]);
    __syncthreads();
    // scores: lane l computes the score of row r = r0 + l from 16-byte pieces of
    // its k row, eight pieces in flight at a time
    const int r0 = warp * kGR, r = r0 + lane;
    float my_s = -INFINITY;
    if (r < n) {
        constexpr int EP = 16 / (int)sizeof(T);
        const int np = D / EP;
        const uint4 *kr = reinterpret_cast<const uint4 *>(kh + (long long)r * D);
        float acc = 0.f;
        for (int p0 = 0; p0 < np; p0 += 8) {
            uint4 x[8];
#pragma unroll
            for (int j = 0; j < 8; j++) x[j] = p0 + j < np ? __ldg(kr + p0 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < 8; j++)
                if (p0 + j < np) acc += dot_piece<T>(x[j], s_q + (p0 + j) * EP);
        }
        my_s = acc;
    }
    // the group's RNN cell row by row, as an inclusive warp scan of (m, u)
    // pairs: m = the running maximum, u = sum of exp(s - m)
    float m = my_s, uu = r < n ? 1.f : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float pm = __shfl_up_sync(0xffffffffu, m, off), pu = __shfl_up_sync(0xffffffffu, uu, off);
        if (lane >= off) {
            float ea, eb;
            combine_mu(pm, pu, m, uu, ea, eb);   // (row - off's prefix) (+) this
        }
    }
    {
        const float mprev = __shfl_up_sync(0xffffffffu, m, 1);
        const float a = lane == 0 || mprev == -INFINITY ? 0.f : __expf(mprev - m);
        const float b = my_s == -INFINITY ? 0.f : __expf(my_s - m);
        s_a[r] = r < n ? a : 1.f;   // rows past the end carry the sums unchanged
        s_b[r] = r < n ? b : 0.f;
        s_m[r] = m;
        s_U[r] = uu;
        if (lane == 31) {
            s_gm[warp] = m;
            s_gu[warp] = uu;
        }
    }
    __syncthreads();
    // per (group, column): the group's w.  Warp g takes group g, lane l the
    // columns [l cpl, l cpl + cpl); eight rows' loads in flight at a time
    const int cpl = Dv >= 32 ? Dv / 32 : 1, c0 = lane * cpl;
    const bool lane_on = c0 < Dv;
    {
        const int rb = warp * kGR;
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = 0; i < kGR; i += 8) {
            float vv[8][4];
#pragma unroll
            for (int ii = 0; ii < 8; ii++) load_cols<T>(vh, rb + i + ii, Dv, c0, cpl, lane_on && rb + i + ii < n, vv[ii]);
#pragma unroll
            for (int ii = 0; ii < 8; ii++) {
                const float a = s_a[rb + i + ii], b = s_b[rb + i + ii];
#pragma unroll
                for (int c = 0; c < 4; c++) w[c] = w[c] * a + b * vv[ii][c];
            }
        }
        if (lane_on)
            for (int c = 0; c < cpl; c++) s_w[warp * Dv + c0 + c] = w[c];
    }
    __syncthreads();
    // exclusive offsets of the groups within the tile, and the tile's aggregate
    if (tid < Dv) {
        float om = -INFINITY, ou = 0.f, ow = 0.f;
        for (int gg = 0; gg < kGroups; gg++) {
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
        for (int gg = 0; gg < kGroups; gg++) {
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
            // up to 32 earlier tiles of the head at a time: lane l waits for the
            // flag of the l-th tile back; the nearest published inclusive state
            // ends the walk, and the states up to it are combined in order
            long long base = tile - g.BH;   // this head's previous tile
            int left = t;                   // earlier tiles of the head not yet combined
            bool done = false;
            while (!done && left > 0) {
                const int win = min(32, left);
                int f = 0;
                if (lane < win) {
                    const int *fp = flags + (base - (long long)lane * g.BH);
                    long long spins = 0;
                    while ((f = ld_flag(fp)) == 0) {
                        if (++spins > kSpinLimit) {   // give up: report, and finish without the prefix
                            atomicExch(err, kErrTimeout);
                            f = -1;
                            break;
                        }
                    }
                }
                if (__any_sync(0xffffffffu, f < 0)) break;
                const unsigned inc = __ballot_sync(0xffffffffu, lane < win && f == 2);
                const int L = inc ? __ffs(inc) - 1 : win - 1;
                done = inc != 0;
                __threadfence();
                for (int j0 = 0; j0 <= L; j0 += 4) {   // four states' loads in flight, then their combines
                    float pm[4], pu[4], pw[4][4];
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        const int j = j0 + jj;
                        const int fj = __shfl_sync(0xffffffffu, f, j & 31);
                        pm[jj] = -INFINITY;
                        pu[jj] = 0.f;
#pragma unroll
                        for (int c4 = 0; c4 < 4; c4++) pw[jj][c4] = 0.f;
                        if (j <= L) {
                            const float *src = (fj == 2 ? incl : agg) + (base - (long long)j * g.BH) * SW;
                            pm[jj] = __ldcg(src);
                            pu[jj] = __ldcg(src + 1);
#pragma unroll
                            for (int c4 = 0; c4 < 4; c4++) {
                                const int c = lane + 32 * c4;
                                if (c < Dv) pw[jj][c4] = __ldcg(src + 2 + c);
                            }
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        if (j0 + jj > L) break;
                        float ea, eb;
                        combine_mu(pm[jj], pu[jj], xm, xu, ea, eb);   // X = (j-th tile back) (+) X
#pragma unroll
                        for (int c4 = 0; c4 < 4; c4++) xw[c4] = pw[jj][c4] * ea + xw[c4] * eb;
                    }
                }
                base -= (long long)win * g.BH;
                left -= win;
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
    // per group: Xg = X (+) the group's offset (m, u in s_gm, s_gu), with the
    // factors of X and of the offset in it
    const float xm = s_X[0], xu = s_X[1];
    if (tid < kGroups) {
        float m2 = s_gm[tid], u2 = s_gu[tid], e1, e2;
        combine_mu(xm, xu, m2, u2, e1, e2);
        s_ge1[tid] = e1;
        s_ge2[tid] = e2;
        s_xgm[tid] = m2;
        s_xgu[tid] = u2;
    }
    __syncthreads();
    // per row: o_r = (Xg.w al + w_r be) / (Xg.u al + U_r be), al = e^(Xg.m - mu), be = e^(m_r - mu)
    {
        const int rg = tid / kGR;
        float m2 = s_xgm[rg], u2 = s_xgu[rg];
        float mr = s_m[tid], ur = s_U[tid], al, be;
        combine_mu(m2, u2, mr, ur, al, be);
        s_al[tid] = al;
        s_be[tid] = be;
        s_rd[tid] = tid < n ? 1.f / ur : 0.f;
    }
    __syncthreads();
    {
        const int rb = warp * kGR;
        float gw[4], run[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; c++) {   // Xg.w of this lane's columns
            const int cc = min(c0 + c, Dv - 1);
            gw[c] = s_X[2 + cc] * s_ge1[warp] + s_w[warp * Dv + cc] * s_ge2[warp];
        }
        for (int i = 0; i < kGR; i += 8) {
            float vv[8][4];
#pragma unroll
            for (int ii = 0; ii < 8; ii++)   // (from L2)
                load_cols<T>(vh, rb + i + ii, Dv, c0, cpl, lane_on && rb + i + ii < n, vv[ii]);
#pragma unroll
            for (int ii = 0; ii < 8; ii++) {
                const int rr = rb + i + ii;
                const float a = s_a[rr], b = s_b[rr], al = s_al[rr], be = s_be[rr], rd = s_rd[rr];
                float o[4];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    run[c] = run[c] * a + b * vv[ii][c];
                    o[c] = (gw[c] * al + run[c] * be) * rd;
                }
                if (lane_on && rr < n) {
                    T *dst = oh + (long long)rr * Dv + c0;
                    for (int c = 0; c < cpl; c++) dst[c] = from_f32<T>(o[c]);
                }
            }
        }
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
