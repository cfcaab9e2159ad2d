// backward_tc.cu -- the backward of kernelized attention on the sm_103a
// tensor cores (review page "Transformers are RNNs", proposed method b4:
// linear-time gradients with the same cumulative sums), bf16 inputs, elu+1,
// D = Dv in {64, 128}.
//
// The algebra is that of backward.cu: with G = phi(Q), F = phi(K) of a chunk
// of 128 positions, M = [dnum | dden] (dnum = dout / den, dden = -(dout .
// out) / den), Vx = [V | 1] and the masked (j <= i) intra-chunk matrices
// A = tril(G F^T), B = tril(M Vx^T):
//   dq pass (chunks in order, from the forward memories S, z before the chunk):
//     X  = G F^T                          -> P = tril X                 (TMEM)
//     X  = G [S|z] + P [V|1]              -> den, out, dnum, dden -> M  (shared)
//     X  = M Vx^T                         -> B = tril X                 (TMEM)
//     X  = B F + M [S|z]^T                -> dG -> dq = dG o min(G, 1)
//     S|z += F^T [V|1],  R|r += G^T M     (R|r: this segment's reverse sums)
//   dk/dv pass (chunks in reverse, from the reverse memories R, r after it):
//     X  = F G^T                          -> P^T = triu X
//     X  = P^T dnum + F R                 -> dV
//     X  = Vx M^T                         -> B^T = triu X
//     X  = B^T G + Vx [R|r]^T             -> dF -> dk = dF o min(F, 1)
//     R|r += G^T M
// Every product is a group of tcgen05.mma (kind::f16, M = 128, fp32 in TMEM).
//
// Precision.  The gradients of q and k are small differences: g_i . dg_i = 0
// exactly (num . dnum + den . dden = 0), so the constant part of dG that
// phi ~ 1 + x puts in every component cancels, and what is left depends on
// the small part x.  bf16 operands (8 significant bits) lose it: a model of
// this chunk algebra with bf16 operands and exact sums missed the fp64
// oracle by 2-42% row-relative on dq.  Here the operands are fp16 (11
// significant bits) and M, whose rounding matters most for dq, is carried as
// an fp16 hi + lo pair in the products of the dq pass that give dG (the R
// updates and the dk/dv pass use its hi part alone); the same model then
// stays within 6.7e-3 on dq, 6.4e-3 on dk and 7e-4 on dv (N up to 16384,
// scaled and unscaled inputs, causal and not).  fp16's range is handled by
// exact powers of two, chosen per chunk:
//   mu   = 2^floor(log2(min den of the chunk's rows)): M is stored as mu M
//          (so |mu dnum| <= |dout|), and every product with M is divided by
//          mu in fp32;
//   2^-k on the carried memory tile ([S|z] or mu [R|r]) so that its largest
//          entry stays below 2^14, and the same 2^-k on P and B, so that the
//          products that share an accumulator carry the same factor.
// Inputs with a q, k or v entry of magnitude >= 2^16 (whose phi or value has
// no finite fp16) or not finite, whose scaled scores or intra-chunk B
// overflow fp16, or whose denominators underflow set the library's error
// word (reported by la_check as LA_ERR_RANGE); they belong on the fp32
// CUDA-core backward.
//
// Tiles: Q, K, dout in 128-byte swizzle (64-column boxes), converted in
// place (phi to fp16 for Q and K); V, M and the memories in 32-byte swizzle
// blocks of 16 columns followed by a 16-column side block: ONES after V
// (columns 0-7 one), z hi | lo after S (columns 0-7 | 8-15), r and dden as
// hi | lo pairs (columns 0, 1 and 8, 9) after R and dnum.  In the dq pass
// the lo part of dnum takes the dout tile's place once M is formed.  The stages of a chunk
// run one after another (one thread issues, every thread waits on the
// commit).  The next chunk's F and V tiles are loaded as soon as the chunk's
// products no longer read them, its G and dout tiles after the last product,
// and the chunk after it is prefetched into L2.
//
// Launches: the forward memories' segment sums (this file's kernel in its
// sums-only form), their exclusive prefix, the dq pass (which writes den,
// dden per position and the segment sums of R, r), their exclusive suffix,
// the dk/dv pass.  Non-causal: per-head totals instead of prefix and suffix,
// and no intra-chunk products.  Every wait is bounded (error word, no trap).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kBC = 128;                     // chunk
constexpr int kBThreads = 256;               // 8 warps: TMEM lane quadrant w % 4, column half w / 4
constexpr long long kBBudget = 4000000000LL;
constexpr int kBErr = 1;                     // a bounded wait ran out
constexpr int kBErrRange = 2;                // an operand outside fp16's range

template <int DD>
struct BtcPlan {
    static constexpr int E = DD + 16;                 // value width with the side block
    static constexpr int QB = kBC * DD * 2;           // G, F, dout tiles (64-column boxes, 128-byte swizzle)
    static constexpr int VB = kBC * E * 2;            // V and its ONES block (16-column boxes, 32-byte swizzle)
    static constexpr int MB = kBC * E * 2;            // M tile (hi), same form
    static constexpr int ZB = DD * E * 2;             // the carried memory tile, DD rows, same form
    static constexpr int G0 = 0, F0 = QB, O0 = 2 * QB, V0 = 3 * QB, M0 = V0 + VB, Z0 = M0 + MB;
    static constexpr int RED = Z0 + ZB;               // 2 x 128 floats (row-sum halves) + 8 (block reductions)
    // Gradient rows are staged as bf16 (row stride RS, padded against bank
    // conflicts) and copied out by the whole block in full rows.  At D = 128
    // the memory tile's region serves for dq and dk (it is dead by then) and
    // dv goes out directly; at D = 64 a region of its own serves all three.
    static constexpr int RS = DD * 2 + 16;
    static constexpr int STG = RED + 2048;
    static constexpr int STGB = DD == 64 ? kBC * RS : 0;
    static constexpr int TILES = STG + STGB;
    static constexpr int STAGE_QK = DD == 64 ? STG : Z0;
    static constexpr int STAGE_V = DD == 64 ? STG : -1;
    static_assert(DD == 64 || kBC * RS <= ZB, "the memory tile's region holds a staged gradient chunk");
    static constexpr int RAW = TILES + 1024 + 1024;   // + alignment + barriers
    static constexpr int SMEM = RAW > 116 * 1024 ? RAW : 116 * 1024;   // one CTA per SM (all of TMEM)
    static constexpr int XW = E > 128 ? E : 128;
    static constexpr int T_SZ = 0, T_RR = E, T_X = 2 * E, T_P = 2 * E + XW;   // TMEM columns
    static_assert(T_P + 64 <= 512, "TMEM plan");
    static_assert(SMEM <= 227 * 1024, "shared memory plan");
    static_assert(QB == (DD / 16) * kBC * 32, "the lo part of dnum fills the dout tile exactly");
};

struct BtcGeo {
    int BH, N, NC, L, nseg;
};

// kind::f16 instruction descriptor with fp16 A and B, fp32 accumulation
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn)
{
    return (1u << 4)                      // D format: f32
           | ((uint32_t)a_mn << 15)       // A major (A, B format fields 0: f16)
           | ((uint32_t)b_mn << 16)       // B major
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t u)
{
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
}

// x rounds to +-inf in fp16 although it is finite
__device__ __forceinline__ bool f16_overflows(float x) { return fabsf(x) >= 65520.f && fabsf(x) < INFINITY; }

__device__ __forceinline__ float f16_round(float x) { return __half2float(__float2half_rn(x)); }

// 2^floor(log2 x) for a positive normal float
__device__ __forceinline__ float pow2_floor(float x) { return __int_as_float(__float_as_int(x) & 0x7f800000); }

// 2^-k with k >= 0 the least that brings |x| below 2^14
__device__ __forceinline__ float down_scale(float mx)
{
    if (!(mx >= 16384.f)) return 1.f;
    const int e = ((__float_as_int(mx) >> 23) & 0xff) - 127;   // floor(log2 mx) >= 14
    return __int_as_float((127 - (e - 13)) << 23);
}

__device__ __forceinline__ uint32_t b_align1k(uint32_t a) { return (a + 1023u) & ~1023u; }

// 16 B chunk j of row r of a [128 x cols] tile in 128-byte swizzle (64-column boxes)
__device__ __forceinline__ uint32_t b_toff(int r, int j) { return (uint32_t)(j >> 3) * (kBC * 128) + sw128_off(r, j & 7); }

// 16 B chunk of column col (a multiple of 8) of row r in a 32-byte-swizzle block tile whose blocks are `bs` bytes apart
__device__ __forceinline__ uint32_t b_soff(int r, int col, int bs)
{
    return (uint32_t)(col >> 4) * bs + sw32_off(r, (col >> 3) & 1);
}

__device__ __forceinline__ void tld32(uint32_t a, uint32_t (&r)[32]) { tmem_ld32x2_nowait(a, r); }

// 8 fp32 values -> fp16 into columns [c0, c0 + 8) of row r of a 32-byte block tile
__device__ __forceinline__ void put8_f16(uint32_t tile, int bs, int r, int c0, const float *v)
{
    sts128(tile + b_soff(r, c0, bs), make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]),
                                                pack_f16x2(v[4], v[5]), pack_f16x2(v[6], v[7])));
}

// the side block of row r: (hi, lo) of x in columns 0-1 and 8-9, zeros elsewhere
__device__ __forceinline__ void put_side16(uint32_t tile, int bs, int r, int c0, float x)
{
    const float hi = f16_round(x);
    const uint32_t p = pack_f16x2(hi, x - hi);
    sts128(tile + b_soff(r, c0, bs), make_uint4(p, 0, 0, 0));
    sts128(tile + b_soff(r, c0 + 8, bs), make_uint4(p, 0, 0, 0));
}

// the z side block of [S|z]: z hi in columns 0-7, lo in 8-15
__device__ __forceinline__ void put_zside16(uint32_t tile, int bs, int r, int c0, float z)
{
    const float hi = f16_round(z);
    const uint32_t h = pack_f16x2(hi, hi), l = pack_f16x2(z - hi, z - hi);
    sts128(tile + b_soff(r, c0, bs), make_uint4(h, h, h, h));
    sts128(tile + b_soff(r, c0 + 8, bs), make_uint4(l, l, l, l));
}

// The largest |x| seen, as packed bf16 magnitudes: a bf16 of magnitude >= 2^16
// (bits >= 0x4780, the first above 65280) has no finite fp16, nor has
// phi = x + 1 of it; every smaller bf16 and its phi fit.
constexpr uint32_t kBf16TooBig = 0x4780u;
__device__ __forceinline__ bool bf16_max_too_big(uint32_t amax)
{
    return (amax >> 16) >= kBf16TooBig || (amax & 0xffffu) >= kBf16TooBig;
}

// phi = elu + 1 = max(x, 0) + 2^(min(x, 0) log2 e) of 8 bf16 -> 8 fp16, in
// half2 arithmetic (x is exact in fp16; x + 1 rounds once; the exponential
// of a negative x is within a few fp16 ulps of it, and below 1 in size)
__device__ __forceinline__ uint4 phi_f16x8(uint4 x, uint32_t &amax)
{
    const uint32_t in[4] = {x.x, x.y, x.z, x.w};
    const __half2 zero = __float2half2_rn(0.f), l2e = __float2half2_rn(1.4426950408889634f);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        amax = __vmaxu2(amax, in[i] & 0x7fff7fffu);
        const float2 t = unpack_bf16x2(in[i]);
        const __half2 hx = __floats2half2_rn(t.x, t.y);
        const __half2 p = __hadd2(__hmax2(hx, zero), h2exp2(__hmul2(__hmin2(hx, zero), l2e)));
        o[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 bf16 -> 8 fp16
__device__ __forceinline__ uint4 bf16_to_f16x8(uint4 x, uint32_t &amax)
{
    const uint32_t in[4] = {x.x, x.y, x.z, x.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        amax = __vmaxu2(amax, in[i] & 0x7fff7fffu);
        const float2 t = unpack_bf16x2(in[i]);
        o[i] = pack_f16x2(t.x, t.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// PASS 0: sums only (S, z per segment); 1: dq pass; 2: dk/dv pass
template <int DD, int PASS>
__global__ void __launch_bounds__(kBThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, BtcGeo g,
              int causal, float *__restrict__ stS, float *__restrict__ stR, float *__restrict__ den_g,
              float *__restrict__ dd_g, __nv_bfloat16 *__restrict__ grad_a, __nv_bfloat16 *__restrict__ grad_b,
              int *err)
{
    using PL = BtcPlan<DD>;
    constexpr int E = PL::E, HALF = DD / 2, ZBS = DD * 32;   // ZBS: block stride of the memory tile
    constexpr int MBS = kBC * 32;                            // block stride of V, M and the lo part of dnum
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = b_align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *ld = bar, *mb = bar + 1, *ldb = bar + 4;   // ld: G, dout tiles; ldb: F, V tiles
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(bar + 3);
    float *red = reinterpret_cast<float *>(gbase + PL::RED);
    float *red8 = red + 2 * kBC;

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int qd = warp & 3, hg = warp >> 2, r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const int h = blockIdx.x % g.BH, s = blockIdx.x / g.BH;
    const int c0 = s * g.L, c1 = min(g.NC, c0 + g.L);
    const uint32_t G0 = base + PL::G0, F0 = base + PL::F0, O0 = base + PL::O0, V0 = base + PL::V0;
    const uint32_t M0 = base + PL::M0, Z0 = base + PL::Z0;
    const uint32_t ML0 = O0;   // the lo part of mu dnum, once dout has been read
    const long long slot = ((long long)h * g.nseg + s) * (DD * DD + DD);

    if (tid == 0) {
        mbar_init(ld, 1);
        mbar_init(ldb, 1);
        mbar_init(mb, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    {   // the ONES block after V's boxes (rows: keys; columns 0-7 one)
        const uint32_t one = pack_f16x2(1.f, 1.f);
        const uint32_t blk = V0 + (DD / 16) * MBS;
        if (tid < kBC) {
            sts128(blk + sw32_off(tid, 0), make_uint4(one, one, one, one));
            sts128(blk + sw32_off(tid, 1), make_uint4(0, 0, 0, 0));
        }
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    bool ok = true, pend_a = false, pend_b = false;   // thread 0 issued tile loads not yet waited for
    bool big = false;                     // this thread saw a value outside fp16's range
    uint32_t ldph = 0, ldbph = 0, mbph = 0;
    // bounded wait by every thread, made block-uniform
    auto wait_all = [&](uint64_t *b, uint32_t parity) {
        bool w = !*abort_cta;
        if (w && !mbar_try_wait(b, parity)) {
            const long long t0 = clock64();
            while (!mbar_try_wait(b, parity)) {
                if (*abort_cta) {
                    w = false;
                    break;
                }
                if (clock64() - t0 > kBBudget) {
                    atomicExch(err, kBErr);
                    *abort_cta = 1;
                    w = false;
                    break;
                }
            }
        }
        return __syncthreads_and(w) != 0;
    };
    // shared-memory and TMEM writes of every thread are visible to the tensor cores
    auto publish = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    };
    // thread 0 issued a group of MMAs: commit and wait for it
    auto finish_mma = [&]() {
        if (tid == 0) mma_commit(mb);
        ok = ok && wait_all(mb, mbph);
        mbph ^= 1;
        tc_fence_after();
    };
    // the largest value over the block (every thread calls it)
    auto block_max = [&](float v) {
#pragma unroll
        for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
        __syncthreads();
        if (lane == 0) red8[warp] = v;
        __syncthreads();
        float m = red8[0];
#pragma unroll
        for (int i = 1; i < kBThreads / 32; i++) m = fmaxf(m, red8[i]);
        return m;
    };

    // the next launch (a scan) may start; this pass reads the previous one's
    // results only after it has completed (dependent launches)
    griddep_launch();
    if constexpr (PASS != 0) griddep_wait();
    // ---- the memory at the segment's start (dq: S|z prefix; dk/dv: R|r suffix) -> TMEM
    if constexpr (PASS != 0) {
        const float *src = (PASS == 1 ? stS : stR) + slot;
        const uint32_t tcol = PASS == 1 ? PL::T_SZ : PL::T_RR;
        if (r < DD) {
#pragma unroll 1
            for (int cb = 0; cb < HALF; cb += 32) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; i++) w[i] = __float_as_uint(src[(long long)r * DD + hg * HALF + cb + i]);
                tmem_st32x2_nowait(tmem + lane_base + tcol + hg * HALF + cb, w);
            }
            if (hg == 0) {
                const float zr = src[(long long)DD * DD + r];
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; i++) w[i] = PASS == 1 ? (i < 8 ? __float_as_uint(zr) : 0u) : (i == 0 ? __float_as_uint(zr) : 0u);
                tmem_st16_nowait(tmem + lane_base + tcol + DD, w);
            }
        }
        tmem_st_wait();
    }
    if constexpr (PASS != 2) {   // sums that start at zero: S|z (sums-only form), R|r (dq pass)
        const uint32_t tcol = PASS == 0 ? PL::T_SZ : PL::T_RR;
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; i++) w[i] = 0u;
        for (int cb = 0; cb < HALF; cb += 32) tmem_st32x2_nowait(tmem + lane_base + tcol + hg * HALF + cb, w);
        if (hg == 0) {
            uint32_t w16[16];
#pragma unroll
            for (int i = 0; i < 16; i++) w16[i] = 0u;
            tmem_st16_nowait(tmem + lane_base + tcol + DD, w16);
        }
        tmem_st_wait();
    }
    publish();

    // The carried memory (dq: S|z from T_SZ; dk/dv: mul * R|r from T_RR) -> its
    // fp16 tile, scaled by a power of two that keeps it below 2^14; returns the scale.
    auto memory_tile = [&](float mul) {
        const uint32_t tcol = PASS == 1 ? PL::T_SZ : PL::T_RR;
        float v[HALF], side = 0.f, mx = 0.f;
        tc_fence_after();
        if (r < DD) {
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 32) {
                uint32_t x[32];
                tld32(tmem + lane_base + tcol + hg * HALF + cb, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    v[cb + i] = __uint_as_float(x[i]) * mul;
                    mx = fmaxf(mx, fabsf(v[cb + i]));
                }
            }
            if (hg == 0) {
                uint32_t d[16];
                tmem_ld16_nowait(tmem + lane_base + tcol + DD, d);
                tmem_ld_wait();
                // z: column 0 of the side block; r: columns 0 + 1 (the hi | lo pair of dden)
                side = (PASS == 1 ? __uint_as_float(d[0]) : __uint_as_float(d[0]) + __uint_as_float(d[1])) * mul;
                mx = fmaxf(mx, fabsf(side));
            }
        }
        const float sc = down_scale(block_max(mx));
        if (r < DD) {
#pragma unroll
            for (int i = 0; i < HALF; i++) v[i] *= sc;
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 8) put8_f16(Z0, ZBS, r, hg * HALF + cb, v + cb);
            if (hg == 0) {
                if (PASS == 1) put_zside16(Z0, ZBS, r, DD, side * sc);
                else put_side16(Z0, ZBS, r, DD, side * sc);
            }
        }
        return sc;
    };

    const int cfirst = PASS == 2 ? c1 - 1 : c0, cstep = PASS == 2 ? -1 : 1;
    const int nchunks = c1 - c0;
    // tile loads (thread 0): G and dout of chunk cc on `ld`; F and V on `ldb`, with the
    // tiles of the chunk after it (the cidx + 1-th of the segment) prefetched into L2
    auto issue_a = [&](int cc) {
        if constexpr (PASS != 0) {
            mbar_arrive_expect_tx(ld, 2 * PL::QB);
            pend_a = true;
            for (int b = 0; b < DD / 64; b++) {
                tma_load_3d(gbase + PL::G0 + b * (kBC * 128), &tm_q, ld, b * 64, cc * kBC, h);
                tma_load_3d(gbase + PL::O0 + b * (kBC * 128), &tm_o, ld, b * 64, cc * kBC, h);
            }
        }
    };
    auto issue_b = [&](int cc, int cidx) {
        mbar_arrive_expect_tx(ldb, PL::QB + kBC * DD * 2);
        pend_b = true;
        for (int b = 0; b < DD / 64; b++)
            tma_load_3d(gbase + PL::F0 + b * (kBC * 128), &tm_k, ldb, b * 64, cc * kBC, h);
        for (int b = 0; b < DD / 16; b++)
            tma_load_3d(gbase + PL::V0 + b * MBS, &tm_v, ldb, b * 16, cc * kBC, h);
        if (cidx + 1 < nchunks) {
            const int nrow = (cc + cstep) * kBC;
            for (int b = 0; b < DD / 64; b++) {
                if (PASS != 0) tma_prefetch_3d(&tm_q, b * 64, nrow, h);
                tma_prefetch_3d(&tm_k, b * 64, nrow, h);
                if (PASS != 0) tma_prefetch_3d(&tm_o, b * 64, nrow, h);
            }
            for (int b = 0; b < DD / 16; b++) tma_prefetch_3d(&tm_v, b * 16, nrow, h);
        }
    };
    for (int ci = 0; ci < nchunks && ok; ci++) {
        const int c = cfirst + ci * cstep;
        const int row0 = c * kBC;
        const bool valid = row0 + r < g.N;
        // ---- tiles: the first chunk's here; a later chunk's F, V (and G, dout) are
        //      issued by the previous chunk as soon as its products no longer read them
        if (ci == 0 && tid == 0) {
            issue_a(c);
            issue_b(c, ci);
        }
        float dnv = 0.f, ddv = 0.f;  // this row's den and dden (dk/dv pass: read back from the dq pass)
        if constexpr (PASS == 2) {   // (their loads in flight while the tiles are converted)
            if (valid) {
                dnv = den_g[(long long)h * g.N + row0 + r];
                ddv = dd_g[(long long)h * g.N + row0 + r];
            }
        }
        ok = ok && wait_all(ldb, ldbph);
        ldbph ^= 1;
        pend_b = false;
        if constexpr (PASS != 0) {
            ok = ok && wait_all(ld, ldph);
            ldph ^= 1;
            pend_a = false;
        }
        if (!ok) break;
        // ---- phi in place on this thread's half row of G and F (F rows past N become zero), as fp16;
        //      V as fp16 (all loads of a tile issued before its math)
        {
            constexpr int JH = DD / 16;
            uint32_t amax = 0u;
            uint4 x[JH];
            if constexpr (PASS != 0) {
#pragma unroll
                for (int j = 0; j < JH; j++) x[j] = lds128(G0 + b_toff(r, hg * JH + j));
#pragma unroll
                for (int j = 0; j < JH; j++) sts128(G0 + b_toff(r, hg * JH + j), phi_f16x8(x[j], amax));
            }
#pragma unroll
            for (int j = 0; j < JH; j++) x[j] = lds128(F0 + b_toff(r, hg * JH + j));
#pragma unroll
            for (int j = 0; j < JH; j++) {
                const uint4 f = phi_f16x8(x[j], amax);   // (rows past N are zero-filled: phi = 1, then dropped)
                sts128(F0 + b_toff(r, hg * JH + j), valid ? f : make_uint4(0, 0, 0, 0));
            }
            constexpr int NV = kBC * DD / 8 / kBThreads;   // the V boxes, 16 B at a time
            uint4 y[NV];
#pragma unroll
            for (int i = 0; i < NV; i++) y[i] = lds128(V0 + 16 * (tid + i * kBThreads));
#pragma unroll
            for (int i = 0; i < NV; i++) sts128(V0 + 16 * (tid + i * kBThreads), bf16_to_f16x8(y[i], amax));
            big |= bf16_max_too_big(amax);
        }
        float mu = 1.f, zsc = 1.f;   // the chunk's M scale and memory-tile scale
        if constexpr (PASS == 1) {
            zsc = memory_tile(1.f);
        }
        if constexpr (PASS == 2) {
            const float mind = -block_max(valid ? -dnv : -INFINITY);
            big |= mind < 1e-30f;
            mu = mind < INFINITY && mind >= 1e-30f ? pow2_floor(mind) : 1.f;
            const float fm = valid ? mu / dnv : 0.f;
            // mu M = [mu dout / den (hi; lo into the dout tile) | mu dden (hi | lo side block)]
            constexpr int JH = DD / 16;
            float f[HALF];
#pragma unroll
            for (int j = 0; j < JH; j++) {
                const uint4 x = lds128(O0 + b_toff(r, hg * JH + j));
                const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float2 t = unpack_bf16x2(u[i]);
                    f[8 * j + 2 * i] = t.x * fm;
                    f[8 * j + 2 * i + 1] = t.y * fm;
                }
            }
            // (a single fp16 part here: the dk/dv pass is not sensitive to it)
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 8) {
#pragma unroll
                for (int i = 0; i < 8; i++) big |= f16_overflows(f[cb + i]);
                put8_f16(M0, MBS, r, hg * HALF + cb, f + cb);
            }
            if (hg == 0) put_side16(M0, MBS, r, DD, valid ? ddv * mu : 0.f);
            zsc = memory_tile(mu);
        }
        publish();

        constexpr uint32_t lboT = DD >= 128 ? kBC * 128 : 0;   // MN-major 128-byte tiles: the second 64-wide block
        if constexpr (PASS == 0) {
            // S|z += F^T [V|1]
            if (tid == 0 && ok) {
                tc_fence_after();
                constexpr uint32_t id = idesc_f16(128, E, 1, 1);
#pragma unroll
                for (int kk = 0; kk < kBC; kk += 16)
                    mma_bf16_ss(tmem + PL::T_SZ, sw128_desc(F0 + (kk / 8) * 1024, lboT, 1024),
                                sw32_desc(V0 + (kk / 8) * 256, MBS, 256), id, 1u);
            }
            finish_mma();
            if (tid == 0 && ok && ci + 1 < nchunks) issue_b(c + cstep, ci + 1);
            continue;
        }

        // ---- the masked intra-chunk product of the pass, times zsc, as fp16 in TMEM
        auto tril_to_p = [&](bool upper) {
            uint32_t a0[32], a1[32], pk[32];
            tld32(tmem + lane_base + PL::T_X + hg * 64, a0);
            tld32(tmem + lane_base + PL::T_X + hg * 64 + 32, a1);
            tmem_ld_wait();
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int cc = hg * 64 + 2 * i;
                auto keep = [&](int col) { return upper ? col >= r : col <= r; };
                const float x0 = keep(cc) ? __uint_as_float(a0[2 * i]) * zsc : 0.f;
                const float x1 = keep(cc + 1) ? __uint_as_float(a0[2 * i + 1]) * zsc : 0.f;
                const float x2 = keep(cc + 32) ? __uint_as_float(a1[2 * i]) * zsc : 0.f;
                const float x3 = keep(cc + 33) ? __uint_as_float(a1[2 * i + 1]) * zsc : 0.f;
                mx = fmaxf(fmaxf(mx, fmaxf(fabsf(x0), fabsf(x1))), fmaxf(fabsf(x2), fabsf(x3)));
                pk[i] = pack_f16x2(x0, x1);
                pk[16 + i] = pack_f16x2(x2, x3);
            }
            big |= f16_overflows(mx);
            tmem_st32x2_nowait(tmem + lane_base + PL::T_P + hg * 32, pk);
            tmem_st_wait();
            publish();
        };
        // X = G^T (mu M), M's hi part only (the R|r update; X then holds mu times it)
        auto issue_r_update = [&](bool first) {
            constexpr uint32_t id = idesc_f16(128, E, 1, 1);
#pragma unroll
            for (int kk = 0; kk < kBC; kk += 16)
                mma_bf16_ss(tmem + PL::T_X, sw128_desc(G0 + (kk / 8) * 1024, lboT, 1024),
                            sw32_desc(M0 + (kk / 8) * 256, MBS, 256), id, (!first || kk > 0) ? 1u : 0u);
        };
        // T_RR += X / mu (rows < DD)
        auto add_r_update = [&]() {
            if (r < DD) {
                const float inv = 1.f / mu;
#pragma unroll 1
                for (int cb = 0; cb < HALF; cb += 32) {
                    uint32_t x[32], y[32];
                    tld32(tmem + lane_base + PL::T_X + hg * HALF + cb, x);
                    tld32(tmem + lane_base + PL::T_RR + hg * HALF + cb, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        y[i] = __float_as_uint(fmaf(__uint_as_float(x[i]), inv, __uint_as_float(y[i])));
                    tmem_st32x2_nowait(tmem + lane_base + PL::T_RR + hg * HALF + cb, y);
                }
                if (hg == 0) {
                    uint32_t x[16], y[16];
                    tmem_ld16_nowait(tmem + lane_base + PL::T_X + DD, x);
                    tmem_ld16_nowait(tmem + lane_base + PL::T_RR + DD, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        y[i] = __float_as_uint(fmaf(__uint_as_float(x[i]), inv, __uint_as_float(y[i])));
                    tmem_st16_nowait(tmem + lane_base + PL::T_RR + DD, y);
                }
                tmem_st_wait();
            }
        };
        // fp32 TMEM rows of X times `f` -> the bf16 gradient rows (times min(phi, 1) of `phi_tile` when
        // given), staged in shared memory at byte offset `stage` and copied out in full rows (stage < 0:
        // stored by each thread directly)
        auto store_grad = [&](__nv_bfloat16 *dst_base, float f, uint32_t phi_tile, int stage) {
            constexpr int JH = DD / 16;
            const uint32_t stg = base + (uint32_t)stage;
            uint32_t x[32];
#pragma unroll
            for (int cb = 0; cb < HALF; cb += 32) {
                tld32(tmem + lane_base + PL::T_X + hg * HALF + cb, x);
                tmem_ld_wait();
                if (stage >= 0 || valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(dst_base + ((long long)h * g.N + row0 + r) * DD + hg * HALF + cb);
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        float w[8];
                        if (phi_tile) {
                            const uint4 gq = lds128(phi_tile + b_toff(r, hg * JH + cb / 8 + j));
                            const uint32_t u[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
                            for (int i = 0; i < 4; i++) {
                                const float2 t = unpack_f16x2(u[i]);
                                w[2 * i] = f * fminf(t.x, 1.f);
                                w[2 * i + 1] = f * fminf(t.y, 1.f);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; i++) w[i] = f;
                        }
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; i++)
                            o[i] = pack_bf16x2(__uint_as_float(x[8 * j + 2 * i]) * w[2 * i],
                                               __uint_as_float(x[8 * j + 2 * i + 1]) * w[2 * i + 1]);
                        if (stage >= 0)
                            sts128(stg + r * PL::RS + (hg * HALF + cb + 8 * j) * 2, make_uint4(o[0], o[1], o[2], o[3]));
                        else
                            dst[j] = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
            if (stage >= 0) {
                __syncthreads();
                constexpr int CPR = DD / 8;   // 16 B pieces per row
                const int nrows = min(kBC, g.N - row0);
#pragma unroll
                for (int i = tid; i < kBC * CPR; i += kBThreads) {
                    const int row = i / CPR, pc = i % CPR;
                    if (row < nrows)
                        *reinterpret_cast<uint4 *>(dst_base + ((long long)h * g.N + row0 + row) * DD + pc * 8) =
                            lds128(stg + row * PL::RS + pc * 16);
                }
            }
        };

        if constexpr (PASS == 1) {
            // (1) X = G F^T -> P; and S|z += F^T [V|1] for the next chunk (the memory
            //     tile of this chunk is made), so that F and V are free after (4)
            if (causal) {
                if (tid == 0 && ok) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc_f16(128, kBC, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < DD; kk += 16) {
                        const uint32_t off = (kk / 64) * (kBC * 128) + (kk % 64) * 2;
                        mma_bf16_ss(tmem + PL::T_X, sw128_desc(G0 + off, 16, 1024), sw128_desc(F0 + off, 16, 1024), id,
                                    kk > 0 ? 1u : 0u);
                    }
                    constexpr uint32_t id_s = idesc_f16(128, E, 1, 1);
#pragma unroll
                    for (int kk = 0; kk < kBC; kk += 16)
                        mma_bf16_ss(tmem + PL::T_SZ, sw128_desc(F0 + (kk / 8) * 1024, lboT, 1024),
                                    sw32_desc(V0 + (kk / 8) * 256, MBS, 256), id_s, 1u);
                }
                finish_mma();
                tril_to_p(false);
            }
            // (2) X = G [S|z] zsc (+ zsc P [V|1]) = zsc [NUM | DEN]
            if (tid == 0 && ok) {
                tc_fence_after();
                constexpr uint32_t id = idesc_f16(128, E, 0, 1);
#pragma unroll
                for (int kk = 0; kk < DD; kk += 16) {
                    const uint32_t off = (kk / 64) * (kBC * 128) + (kk % 64) * 2;
                    mma_bf16_ss(tmem + PL::T_X, sw128_desc(G0 + off, 16, 1024), sw32_desc(Z0 + (kk / 8) * 256, ZBS, 256),
                                id, kk > 0 ? 1u : 0u);
                }
                if (causal) {
#pragma unroll
                    for (int kk = 0; kk < kBC; kk += 16)
                        mma_bf16_ts(tmem + PL::T_X, tmem + PL::T_P + kk / 2, sw32_desc(V0 + (kk / 8) * 256, MBS, 256),
                                    id, 1u);
                }
            }
            finish_mma();
            // den, out, dnum, dden -> mu M (hi and lo); den, dden -> global
            {
                uint32_t d[16], n0[32];
                tmem_ld16_nowait(tmem + lane_base + PL::T_X + DD, d);
                float den = 0.f, part = 0.f;
                float dn[HALF];
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    tld32(tmem + lane_base + PL::T_X + hg * HALF + cb, n0);
                    tmem_ld_wait();
                    const float xden = __uint_as_float(d[0]) + __uint_as_float(d[8]);   // zsc den
                    den = xden * (1.f / zsc);
                    const float inv_n = 1.f / xden;   // NUM = X / zsc; out = NUM / den = X / (zsc den)
                    const float rden = valid ? 1.f / den : 0.f;
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint4 x = lds128(O0 + b_toff(r, (hg * HALF + cb) / 8 + j));
                        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const float2 t = unpack_bf16x2(u[i]);
                            const int k2 = 8 * j + 2 * i;
                            part = fmaf(t.x, __uint_as_float(n0[k2]) * inv_n, part);
                            part = fmaf(t.y, __uint_as_float(n0[k2 + 1]) * inv_n, part);
                            dn[cb + k2] = t.x * rden;
                            dn[cb + k2 + 1] = t.y * rden;
                        }
                    }
                }
                red[hg * kBC + r] = part;
                __syncthreads();   // (also: every row of dout has been read)
                const float dd = valid ? -(red[r] + red[kBC + r]) / den : 0.f;
                const float mind = -block_max(valid ? -den : -INFINITY);
                big |= mind < 1e-30f;
                mu = mind < INFINITY && mind >= 1e-30f ? pow2_floor(mind) : 1.f;
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 8) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float f = dn[cb + i] * mu;
                        hi[i] = f16_round(f);
                        lo[i] = f - hi[i];
                        big |= f16_overflows(f);
                    }
                    put8_f16(M0, MBS, r, hg * HALF + cb, hi);
                    put8_f16(ML0, MBS, r, hg * HALF + cb, lo);
                }
                if (hg == 0) {
                    put_side16(M0, MBS, r, DD, dd * mu);
                    if (valid) {
                        den_g[(long long)h * g.N + row0 + r] = den;
                        dd_g[(long long)h * g.N + row0 + r] = dd;
                    }
                }
            }
            publish();
            // (3) X = mu M Vx^T -> zsc mu B
            if (causal) {
                if (tid == 0 && ok) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc_f16(128, kBC, 0, 0);
#pragma unroll
                    for (int kb = 0; kb < E / 16; kb++)
                        mma_bf16_ss(tmem + PL::T_X, sw32_desc(M0 + kb * MBS, 16, 256), sw32_desc(V0 + kb * MBS, 16, 256),
                                    id, kb > 0 ? 1u : 0u);
#pragma unroll
                    for (int kb = 0; kb < DD / 16; kb++)
                        mma_bf16_ss(tmem + PL::T_X, sw32_desc(ML0 + kb * MBS, 16, 256), sw32_desc(V0 + kb * MBS, 16, 256),
                                    id, 1u);
                }
                finish_mma();
                tril_to_p(false);
            }
            // (4) X = zsc mu B F + mu M (zsc [S|z])^T = zsc mu dG -> dq
            if (tid == 0 && ok) {
                tc_fence_after();
                constexpr uint32_t id_b = idesc_f16(128, DD, 0, 1), id_s = idesc_f16(128, DD, 0, 0);
                if (causal) {
#pragma unroll
                    for (int kk = 0; kk < kBC; kk += 16)
                        mma_bf16_ts(tmem + PL::T_X, tmem + PL::T_P + kk / 2, sw128_desc(F0 + (kk / 8) * 1024, lboT, 1024),
                                    id_b, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kb = 0; kb < E / 16; kb++)
                    mma_bf16_ss(tmem + PL::T_X, sw32_desc(M0 + kb * MBS, 16, 256), sw32_desc(Z0 + kb * ZBS, 16, 256),
                                id_s, (causal || kb > 0) ? 1u : 0u);
#pragma unroll
                for (int kb = 0; kb < DD / 16; kb++)
                    mma_bf16_ss(tmem + PL::T_X, sw32_desc(ML0 + kb * MBS, 16, 256), sw32_desc(Z0 + kb * ZBS, 16, 256),
                                id_s, 1u);
            }
            finish_mma();
            if (tid == 0 && ok && ci + 1 < nchunks) issue_b(c + cstep, ci + 1);   // F and V are free
            store_grad(grad_a, 1.f / (zsc * mu), G0, PL::STAGE_QK);
            tc_fence_before();
            __syncthreads();   // X has been read
            // X = mu G^T M (-> R|r)
            if (tid == 0 && ok) {
                tc_fence_after();
                issue_r_update(true);
            }
            finish_mma();
            if (tid == 0 && ok && ci + 1 < nchunks) issue_a(c + cstep);   // G and dout are free
            add_r_update();
        }

        if constexpr (PASS == 2) {
            // (1) X = F G^T -> zsc P^T (i >= j)
            if (causal) {
                if (tid == 0 && ok) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc_f16(128, kBC, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < DD; kk += 16) {
                        const uint32_t off = (kk / 64) * (kBC * 128) + (kk % 64) * 2;
                        mma_bf16_ss(tmem + PL::T_X, sw128_desc(F0 + off, 16, 1024), sw128_desc(G0 + off, 16, 1024), id,
                                    kk > 0 ? 1u : 0u);
                    }
                }
                finish_mma();
                tril_to_p(true);
            }
            // (2) X = zsc P^T (mu dnum) + F (zsc mu R) = zsc mu dV
            if (tid == 0 && ok) {
                tc_fence_after();
                constexpr uint32_t id = idesc_f16(128, DD, 0, 1);
                if (causal) {
#pragma unroll
                    for (int kk = 0; kk < kBC; kk += 16)
                        mma_bf16_ts(tmem + PL::T_X, tmem + PL::T_P + kk / 2, sw32_desc(M0 + (kk / 8) * 256, MBS, 256),
                                    id, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < DD; kk += 16) {
                    const uint32_t off = (kk / 64) * (kBC * 128) + (kk % 64) * 2;
                    mma_bf16_ss(tmem + PL::T_X, sw128_desc(F0 + off, 16, 1024), sw32_desc(Z0 + (kk / 8) * 256, ZBS, 256), id,
                                (causal || kk > 0) ? 1u : 0u);
                }
            }
            finish_mma();
            store_grad(grad_b, 1.f / (zsc * mu), 0u, PL::STAGE_V);
            tc_fence_before();
            __syncthreads();   // (X is read before the next product overwrites it)
            // (3) X = Vx (mu M)^T -> zsc mu B^T (i >= j)
            if (causal) {
                if (tid == 0 && ok) {
                    tc_fence_after();
                    constexpr uint32_t id = idesc_f16(128, kBC, 0, 0);
#pragma unroll
                    for (int kb = 0; kb < E / 16; kb++)
                        mma_bf16_ss(tmem + PL::T_X, sw32_desc(V0 + kb * MBS, 16, 256), sw32_desc(M0 + kb * MBS, 16, 256),
                                    id, kb > 0 ? 1u : 0u);
                }
                finish_mma();
                tril_to_p(true);
            }
            // (4) X = zsc mu B^T G + Vx (zsc mu [R|r])^T = zsc mu dF -> dk
            if (tid == 0 && ok) {
                tc_fence_after();
                constexpr uint32_t id_b = idesc_f16(128, DD, 0, 1), id_r = idesc_f16(128, DD, 0, 0);
                if (causal) {
#pragma unroll
                    for (int kk = 0; kk < kBC; kk += 16)
                        mma_bf16_ts(tmem + PL::T_X, tmem + PL::T_P + kk / 2, sw128_desc(G0 + (kk / 8) * 1024, lboT, 1024),
                                    id_b, kk > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int kb = 0; kb < E / 16; kb++)
                    mma_bf16_ss(tmem + PL::T_X, sw32_desc(V0 + kb * MBS, 16, 256), sw32_desc(Z0 + kb * ZBS, 16, 256),
                                id_r, (causal || kb > 0) ? 1u : 0u);
            }
            finish_mma();
            store_grad(grad_a, 1.f / (zsc * mu), F0, PL::STAGE_QK);
            tc_fence_before();
            __syncthreads();   // X and F have been read
            if (tid == 0 && ok && ci + 1 < nchunks) issue_b(c + cstep, ci + 1);   // F and V are free
            // R|r += G^T M (causal)
            if (causal) {
                if (tid == 0 && ok) {
                    tc_fence_after();
                    issue_r_update(true);
                }
                finish_mma();
            }
            if (tid == 0 && ok && ci + 1 < nchunks) issue_a(c + cstep);   // G and dout are free
            if (causal) add_r_update();
        }
        publish();
    }

    // ---- segment sums out: sums-only pass S|z -> stS; dq pass R|r -> stR
    if constexpr (PASS != 2) {
        if (ok && r < DD) {
            const uint32_t tcol = PASS == 0 ? PL::T_SZ : PL::T_RR;
            float *dst = (PASS == 0 ? stS : stR) + slot;
            tc_fence_after();
            uint32_t x[32];
#pragma unroll 1
            for (int cb = 0; cb < HALF; cb += 32) {
                tld32(tmem + lane_base + tcol + hg * HALF + cb, x);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i++) dst[(long long)r * DD + hg * HALF + cb + i] = __uint_as_float(x[i]);
            }
            if (hg == 0) {
                uint32_t d[16];
                tmem_ld16_nowait(tmem + lane_base + tcol + DD, d);
                tmem_ld_wait();
                // z is the side block's column 0; r is columns 0 + 1 (the hi | lo pair of dden)
                dst[(long long)DD * DD + r] =
                    PASS == 0 ? __uint_as_float(d[0]) : __uint_as_float(d[0]) + __uint_as_float(d[1]);
            }
        }
    }
    if (big) atomicExch(err, kBErrRange);
    // nothing of this CTA in flight at exit (only possible after a wait gave up):
    // every issued MMA completes, and tile loads land, before TMEM and shared memory go
    if (tid == 0) {
        mma_commit(mb);
        mbar_wait(mb, mbph, nullptr, 0, kBBudget);
        if (pend_a) mbar_wait(ld, ldph, nullptr, 0, kBBudget);
        if (pend_b) mbar_wait(ldb, ldbph, nullptr, 0, kBBudget);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 btc_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool btc_map(CUtensorMap *m, const void *base, long long BH, long long N, int cols, int sw)
{
    auto enc = btc_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)N * cols * 2};
    cuuint32_t box[3] = {sw == 32 ? 16u : 64u, (cuuint32_t)kBC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

BtcGeo btc_plan(long long BH, int N, int sms)
{
    BtcGeo g;
    g.BH = (int)BH;
    g.N = N;
    g.NC = cdiv(N, kBC);
    const int want = BH >= sms ? 1 : (int)(sms / BH);
    g.L = cdiv(g.NC, max(1, min(want, g.NC)));
    g.nseg = cdiv(g.NC, g.L);
    return g;
}

int btc_sms()
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int DD>
cudaError_t launch_btc(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal, void *scratch,
                       int *err, cudaStream_t s)
{
    using PL = BtcPlan<DD>;
    const BtcGeo g = btc_plan(p.BH, p.N, btc_sms());
    const int elems = DD * DD + DD;
    float *stS = (float *)scratch;
    float *stR = stS + (size_t)g.BH * g.nseg * elems;
    float *den = stR + (size_t)g.BH * g.nseg * elems;
    float *dd = den + (size_t)g.BH * g.N;
    CUtensorMap tq, tk, tv, to;
    if (!btc_map(&tq, p.q, p.BH, p.N, DD, 128) || !btc_map(&tk, p.k, p.BH, p.N, DD, 128) ||
        !btc_map(&tv, p.v, p.BH, p.N, DD, 32) || !btc_map(&to, dout, p.BH, p.N, DD, 128))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = set_max_smem_once<bwd_tc_kernel<DD, 0>>(PL::SMEM)) != cudaSuccess) return e;
    if ((e = set_max_smem_once<bwd_tc_kernel<DD, 1>>(PL::SMEM)) != cudaSuccess) return e;
    if ((e = set_max_smem_once<bwd_tc_kernel<DD, 2>>(PL::SMEM)) != cudaSuccess) return e;
    const unsigned items = (unsigned)(g.BH * g.nseg);
    const int c = causal ? 1 : 0;
    auto *bq = (__nv_bfloat16 *)dq, *bk = (__nv_bfloat16 *)dk, *bv = (__nv_bfloat16 *)dv;
    bwd_tc_kernel<DD, 0><<<items, kBThreads, PL::SMEM, s>>>(tq, tk, tv, to, g, c, stS, stR, den, dd, nullptr, nullptr, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(1);
    if ((e = backward_scan(stS, g.BH, g.nseg, elems, causal ? 0 : 2, s)) != cudaSuccess) return e;
    if ((e = launch_dependent(bwd_tc_kernel<DD, 1>, dim3(items), dim3(kBThreads), PL::SMEM, s, tq, tk, tv, to, g, c,
                              stS, stR, den, dd, bq, (__nv_bfloat16 *)nullptr, err)) != cudaSuccess)
        return e;
    note_launches(1);
    if ((e = backward_scan(stR, g.BH, g.nseg, elems, causal ? 1 : 2, s)) != cudaSuccess) return e;
    if ((e = launch_dependent(bwd_tc_kernel<DD, 2>, dim3(items), dim3(kBThreads), PL::SMEM, s, tq, tk, tv, to, g, c,
                              stS, stR, den, dd, bk, bv, err)) != cudaSuccess)
        return e;
    note_launches(1);
    return cudaSuccess;
}

}  // namespace

bool backward_tc_supported(const Problem &p)
{
    return p.dtype == DT_BF16 && p.kind == PHI_ELU1 && p.D == p.Dv && (p.D == 64 || p.D == 128) &&
           p.BH * (long long)p.N < (1LL << 31) - kBC;
}

size_t backward_tc_scratch_bytes(const Problem &p, bool)
{
    const BtcGeo g = btc_plan(p.BH, p.N, btc_sms());
    const size_t elems = (size_t)p.D * p.D + p.D;
    return (2 * (size_t)g.BH * g.nseg * elems + 2 * (size_t)g.BH * g.N) * sizeof(float);
}

cudaError_t backward_tc(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal, void *scratch,
                        int *err, cudaStream_t s)
{
    if (p.D == 64) return launch_btc<64>(p, dout, dq, dk, dv, causal, scratch, err, s);
    return launch_btc<128>(p, dout, dq, dk, dv, causal, scratch, err, s);
}

}  // namespace la
