// tc_causal.cu -- chunked causal linear attention on the sm_103a tensor
// cores (tcgen05, TMEM accumulators, TMA loads), bf16 inputs, fp32 state.
//
// The method (review page "Transformers are RNNs", proposed method b2-b3,
// b5): with phi applied to q and k, out_i = phi(q_i)^T S_i / phi(q_i)^T z_i
// where S_i, z_i are cumulative sums over j <= i.  A sequence is cut into
// chunks of C = 128 positions; with S_prev, z_prev the sums before a chunk,
//   A    = tril(phi(Q_c) phi(K_c)^T)                      (j <= i)
//   out  = (A V_c + phi(Q_c) S_prev) / (rowsum(A) + phi(Q_c) z_prev)
//   S   += phi(K_c)^T V_c,   z += colsum(phi(K_c)).
// To fill the GPU when B*H is small each head's chunks are split into
// segments handled by different CTAs, and the segment states are joined by
// an exclusive prefix over segments:
//   1. state pass: each (head, segment) CTA computes its segment's
//      sum of phi(K)^T V and colsum(phi(K)) (tensor-core contractions per
//      chunk, accumulated in TMEM) and writes them to scratch;
//   2. scan: exclusive prefix of those states over segments, per head;
//   3. output pass: each (head, segment) CTA starts from its prefix state
//      and runs the chunk recurrence above, writing out.
// With a single segment per head, passes 1 and 2 are skipped.
//
// Every contraction of a chunk is a tcgen05.mma with fp32 accumulation in
// TMEM; the denominators and z ride along as narrow (N = 16) products with a
// constant tile ONES (columns 0-7 = 1, 8-15 = 0) and a tile ZP holding
// z_prev split into bf16 hi (columns 0-7) and lo (columns 8-15):
//   MMA1   A    = phiQ . phiK^T        M=C,    N=C,  K=Dphi
//   MMA3   NUM  = phiQ . S_prev        M=C,    N=Dv, K=Dphi   (bf16 copy of S)
//   MMA3b  DEN  = phiQ . ZP            M=C,    N=16, K=Dphi
//   MMA4   S   += phiK^T . V           M=Dphi, N=Dv, K=C
//   MMA4b  Z   += phiK^T . ONES        M=Dphi, N=16, K=C      (Z[:,0] = z)
//   MMA2   NUM += P . V                M=C,    N=Dv, K=C      (P from TMEM)
//   MMA2b  DEN += P . ONES             M=C,    N=16, K=C
// with P = bf16(tril(A)) written back into TMEM by the math warps, and
// out = NUM / (DEN[:,0] + DEN[:,8]).  phi is applied in place on the
// TMA-loaded Q/K tiles in shared memory; it never goes back to HBM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;          // chunk length (MMA M)
constexpr int kErrTimeout = 1;

// Output pass: 16 math warps (4 column groups x 4 TMEM lane quadrants), a
// TMA producer warp and an MMA warp.
constexpr int kOutMathWarps = 16;
constexpr int kOutThreads = (kOutMathWarps + 2) * 32;
// State pass: 8 math warps (2 column groups x 4 quadrants) + producer + MMA.
constexpr int kStateMathWarps = 8;
constexpr int kStateThreads = (kStateMathWarps + 2) * 32;

constexpr int ONES_BYTES = kC * 32;  // [C x 16] bf16, 32-byte swizzle

template <int DP, int DV>
struct OutPlan {
    static constexpr int QB = kC * DP * 2;  // one Q or K chunk tile (bytes)
    static constexpr int VB = kC * DV * 2;  // one V chunk tile
    static constexpr int SB = DP * DV * 2;  // S_prev (bf16)
    static constexpr int ZB = DP * 32 < 1024 ? 1024 : DP * 32;   // ZP [DP x 16]
    static constexpr int kRest = 2 * QB + 2 * VB + SB + ZB + ONES_BYTES;
    static constexpr int NQ = (2 * QB + kRest + 3072 <= 227 * 1024) ? 2 : 1;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + NQ * QB;
    static constexpr int V0 = K0 + 2 * QB;
    static constexpr int S0 = V0 + 2 * VB;
    static constexpr int Z0 = S0 + SB;
    static constexpr int O0 = Z0 + ZB;
    static constexpr int TILES = O0 + ONES_BYTES;
    static constexpr int SMEM = TILES + 1024 /* align */ + 1024 /* barriers */;
    // TMEM columns (32-aligned regions)
    static constexpr int T_S = 0, T_Z = DV, T_NUM = DV + 32, T_DEN = 2 * DV + 32,
                         T_A = 2 * DV + 64, T_P = 2 * DV + 192;
    static constexpr int TMEM_COLS = 512;
    static_assert(T_P + 64 <= 512, "TMEM plan too large");
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
};

template <int DP, int DV>
struct StatePlan {
    static constexpr int QB = kC * DP * 2;
    static constexpr int VB = kC * DV * 2;
    static constexpr int NS = ((QB + VB) * 3 + ONES_BYTES + 3072 <= 227 * 1024) ? 3 : 2;
    static constexpr int K0 = 0;
    static constexpr int V0 = NS * QB;
    static constexpr int O0 = V0 + NS * VB;
    static constexpr int TILES = O0 + ONES_BYTES;
    static constexpr int SMEM = TILES + 1024 + 1024;
    static constexpr int T_S = 0, T_Z = DV;
    static constexpr int TMEM_COLS = DV + 32 <= 128 ? 128 : 256;
};

struct Geometry {
    int N, nchunks, cps, nseg;
};

__device__ __forceinline__ unsigned char *align1k(unsigned char *p)
{
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                             ~uintptr_t(1023));
}

template <int NTHREADS>
__device__ __forceinline__ void math_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// Bounded wait that turns into a no-op once the CTA has aborted.  Threads
// never leave their loops early: after an abort they run on without waiting
// (computing garbage that is never trusted) so that every named barrier is
// still reached by all of its threads.
__device__ __forceinline__ bool wait_ok(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                        int *err)
{
    if (*abort_flag) return false;
    if (!mbar_wait(bar, parity, err, kErrTimeout)) {
        *abort_flag = 1;
        return false;
    }
    return true;
}

// phi(x) = elu(x) + 1 on 8 packed bf16.
__device__ __forceinline__ uint4 phi8(uint4 raw)
{
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int t = 0; t < 4; t++) {
        float2 p = unpack_bf16x2(w[t]);
        w[t] = pack_bf16x2(phi_elu1_fast(p.x), phi_elu1_fast(p.y));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// phi in place on row `r` of a [kC x DP] 128B-swizzled tile, the 16 B chunks
// j = g, g + NG, g + 2 NG, ... of the row (column group g of NG).  Rows past
// the sequence end (`zero`) are cleared instead.
template <int DP, int NG>
__device__ __forceinline__ void phi_row_part(unsigned char *tile, int r, int g, bool zero)
{
#pragma unroll
    for (int j = g; j < DP / 8; j += NG) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + (j / 8) * (kC * 128) + sw128_off(r, j % 8));
        *p = zero ? make_uint4(0, 0, 0, 0) : phi8(*p);
    }
}

// TMEM load of NCOL (16 or 32) 32-bit columns, no wait.
template <int NCOL>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[NCOL])
{
    if constexpr (NCOL == 32)
        tmem_ld32_nowait(taddr, r);
    else
        tmem_ld16_nowait(taddr, r);
}

// Write NCOL fp32 values as bf16 into row r, columns [c0, c0 + NCOL) of a
// 128B-swizzled MN-major tile with `rows` rows per 64-column block.
template <int NCOL>
__device__ __forceinline__ void store_row_bf16(unsigned char *tile, int rows, int r, int c0,
                                               const uint32_t (&v)[NCOL])
{
#pragma unroll
    for (int j = 0; j < NCOL / 8; j++) {
        const int col = c0 + 8 * j;
        unsigned char *blk = tile + (col / 64) * (rows * 128);
        *reinterpret_cast<uint4 *>(blk + sw128_off(r, (col % 64) / 8)) = make_uint4(
            pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
            pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
            pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
            pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
    }
}

// z (fp32) -> one row of the ZP tile: columns 0-7 bf16(z), 8-15 bf16(z - bf16(z)).
__device__ __forceinline__ void store_zp_row(unsigned char *zp, int r, float z)
{
    const float hi = __bfloat162float(__float2bfloat16_rn(z));
    const uint32_t h = pack_bf16x2(hi, hi), l = pack_bf16x2(z - hi, z - hi);
    *reinterpret_cast<uint4 *>(zp + sw32_off(r, 0)) = make_uint4(h, h, h, h);
    *reinterpret_cast<uint4 *>(zp + sw32_off(r, 1)) = make_uint4(l, l, l, l);
}

// The constant ONES tile [kC x 16]: columns 0-7 = 1, 8-15 = 0.
__device__ __forceinline__ void fill_ones(unsigned char *ones, int tid, int nthreads)
{
    const uint32_t one = pack_bf16x2(1.f, 1.f);
    for (int r = tid; r < kC; r += nthreads) {
        *reinterpret_cast<uint4 *>(ones + sw32_off(r, 0)) = make_uint4(one, one, one, one);
        *reinterpret_cast<uint4 *>(ones + sw32_off(r, 1)) = make_uint4(0, 0, 0, 0);
    }
}

// ------------------------------------------------------------ state pass

template <int DP, int DV>
__global__ void __launch_bounds__(kStateThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                Geometry g, float *__restrict__ dS, float *__restrict__ dz, int *err)
{
    using PL = StatePlan<DP, DV>;
    constexpr int NS = PL::NS;
    constexpr int NMATH = kStateMathWarps * 32;
    constexpr int NG = kStateMathWarps / 4;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1k(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + PL::TILES);
    uint64_t *full = bars, *phi_done = bars + NS, *empty = bars + 2 * NS, *final_bar = bars + 3 * NS;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 3 * NS + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

    const int seg = blockIdx.x, head = blockIdx.y;
    const int c_begin = seg * g.cps;
    const int nc = min(c_begin + g.cps, g.nchunks) - c_begin;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int PRODUCER = kStateMathWarps, MMAW = kStateMathWarps + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&phi_done[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp < kStateMathWarps) fill_ones(sm + PL::O0, threadIdx.x, NMATH);
    fence_proxy_async_smem();
    if (warp == MMAW) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == PRODUCER) {
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int c = 0; c < nc; c++) {
                const int st = c % NS;
                if (c >= NS && !wait_ok(&empty[st], ((c / NS) - 1) & 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(&full[st], PL::QB + PL::VB);
                const int row = (c_begin + c) * kC;
                for (int b = 0; b < DP / 64; b++)
                    tma_load_3d(sm + PL::K0 + st * PL::QB + b * kC * 128, &tm_k, &full[st], b * 64,
                                row, head);
                for (int b = 0; b < DV / 64; b++)
                    tma_load_3d(sm + PL::V0 + st * PL::VB + b * kC * 128, &tm_v, &full[st], b * 64,
                                row, head);
                issued = c + 1;
            }
            for (int c = max(0, issued - NS); c < issued; c++)   // drain in-flight loads
                mbar_wait(&full[c % NS], (c / NS) & 1, err, kErrTimeout);
        }
    } else if (warp == MMAW) {
        if (lane == 0) {
            constexpr uint32_t id_kv = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t id_z = idesc_bf16(128, 16, 1, 1);
            const uint32_t ones = smem_u32(sm + PL::O0);
            for (int c = 0; c < nc; c++) {
                const int st = c % NS;
                if (!wait_ok(&phi_done[st], (c / NS) & 1, abort_flag, err)) continue;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm + PL::K0 + st * PL::QB);
                const uint32_t va = smem_u32(sm + PL::V0 + st * PL::VB);
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    const uint64_t ad =
                        sw128_desc(ka + (k / 8) * 1024, DP == 128 ? kC * 128 : 0, 1024);
                    const uint32_t acc = (c > 0 || k > 0) ? 1u : 0u;
                    mma_bf16_ss(tmem + PL::T_S, ad, sw128_desc(va + (k / 8) * 1024, kC * 128, 1024),
                                id_kv, acc);
                    mma_bf16_ss(tmem + PL::T_Z, ad, sw32_desc(ones + (k / 8) * 256, 256, 256), id_z,
                                acc);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(final_bar);   // also drains every MMA issued above
            mbar_wait(final_bar, 0, err, kErrTimeout);
        }
    } else {
        const int q = warp & 3, grp = warp >> 2;
        const int row = q * 32 + lane;
        for (int c = 0; c < nc; c++) {
            const int st = c % NS;
            wait_ok(&full[st], (c / NS) & 1, abort_flag, err);
            const int n_valid = min(kC, g.N - (c_begin + c) * kC);
            phi_row_part<DP, NG>(sm + PL::K0 + st * PL::QB, row, grp, row >= n_valid);
            fence_proxy_async_smem();
            math_bar<NMATH>();
            if (threadIdx.x == 0) mbar_arrive(&phi_done[st]);
        }
        // final state -> scratch (warp-uniform condition: tcgen05.ld is warp-collective)
        const bool done = wait_ok(final_bar, 0, abort_flag, err);
        if (__all_sync(0xffffffffu, done) && row < DP) {
            tc_fence_after();
            const long long base = ((long long)head * g.nseg + seg);
            constexpr int CW = DV / NG;   // columns per group
            float *dst = dS + base * DP * DV + (long long)row * DV + grp * CW;
#pragma unroll
            for (int c0 = 0; c0 < CW; c0 += 32) {
                uint32_t v[32];
                tmem_ld32_nowait(tmem + ((uint32_t)(q * 32) << 16) + PL::T_S + grp * CW + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4 *>(dst + c0 + i) =
                        make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                    __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            }
            if (grp == 0) {
                uint32_t zv[16];
                tmem_ld16_nowait(tmem + ((uint32_t)(q * 32) << 16) + PL::T_Z, zv);
                tmem_ld_wait();
                dz[base * DP + row] = __uint_as_float(zv[0]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMAW) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// ------------------------------------------------------------ scan

// Exclusive prefix over segments of the per-segment states, in place.  Each
// thread owns one state element of one head; loads are batched in registers.
__global__ void seg_scan_kernel(float *__restrict__ dS, float *__restrict__ dz, int nseg, int sz_S,
                                int sz_z)
{
    const long long head = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    float *p;
    long long stride;
    if (e < sz_S) {
        p = dS + head * nseg * (long long)sz_S + e;
        stride = sz_S;
    } else if (e < sz_S + sz_z) {
        p = dz + head * nseg * (long long)sz_z + (e - sz_S);
        stride = sz_z;
    } else {
        return;
    }
    float run = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += 16) {
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; i++) x[i] = s0 + i < nseg ? p[(s0 + i) * stride] : 0.f;
#pragma unroll
        for (int i = 0; i < 16; i++)
            if (s0 + i < nseg) {
                p[(s0 + i) * stride] = run;
                run += x[i];
            }
    }
}

// ------------------------------------------------------------ output pass

template <int DP, int DV>
__global__ void __launch_bounds__(kOutThreads, 1)
tc_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, Geometry g,
              const float *__restrict__ preS, const float *__restrict__ prez,
              __nv_bfloat16 *__restrict__ out, float *__restrict__ S_out, float *__restrict__ z_out,
              int *err)
{
    using PL = OutPlan<DP, DV>;
    constexpr int NQ = PL::NQ;
    constexpr int NMATH = kOutMathWarps * 32;
    constexpr int NG = kOutMathWarps / 4;   // column groups
    constexpr int CW = DV / NG;             // NUM / S columns per thread (16 or 32)
    constexpr int PRODUCER = kOutMathWarps, MMAW = kOutMathWarps + 1;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1k(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + PL::TILES);
    uint64_t *qfull = bars;             // [2]
    uint64_t *qempty = bars + 2;        // [2]
    uint64_t *kvfull = bars + 4;        // [2]
    uint64_t *kvempty = bars + 6;       // [2]
    uint64_t *ops_ready = bars + 8;
    uint64_t *p_ready = bars + 9;
    uint64_t *mma1_bar = bars + 10;
    uint64_t *mma4_bar = bars + 11;
    uint64_t *mma2_bar = bars + 12;
    uint64_t *drain_bar = bars + 13;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 14);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

    const int seg = blockIdx.x, head = blockIdx.y;
    const int c_begin = seg * g.cps;
    const int nc = min(c_begin + g.cps, g.nchunks) - c_begin;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1);
            mbar_init(&kvfull[i], 1);
            mbar_init(&kvempty[i], 1);
        }
        mbar_init(ops_ready, 1);
        mbar_init(p_ready, 1);
        mbar_init(mma1_bar, 1);
        mbar_init(mma4_bar, 1);
        mbar_init(mma2_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == MMAW) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == PRODUCER) {
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued_q = 0, issued_kv = 0;
            for (int c = 0; c < nc; c++) {
                const int row = (c_begin + c) * kC;
                const int sq = c % NQ, skv = c % 2;
                if (c >= NQ && !wait_ok(&qempty[sq], ((c / NQ) - 1) & 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(&qfull[sq], PL::QB);
                for (int b = 0; b < DP / 64; b++)
                    tma_load_3d(sm + PL::Q0 + sq * PL::QB + b * kC * 128, &tm_q, &qfull[sq],
                                b * 64, row, head);
                issued_q = c + 1;
                if (c >= 2 && !wait_ok(&kvempty[skv], ((c / 2) - 1) & 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(&kvfull[skv], PL::QB + PL::VB);
                for (int b = 0; b < DP / 64; b++)
                    tma_load_3d(sm + PL::K0 + skv * PL::QB + b * kC * 128, &tm_k, &kvfull[skv],
                                b * 64, row, head);
                for (int b = 0; b < DV / 64; b++)
                    tma_load_3d(sm + PL::V0 + skv * PL::VB + b * kC * 128, &tm_v, &kvfull[skv],
                                b * 64, row, head);
                issued_kv = c + 1;
            }
            for (int c = max(0, issued_q - NQ); c < issued_q; c++)   // drain in-flight loads
                mbar_wait(&qfull[c % NQ], (c / NQ) & 1, err, kErrTimeout);
            for (int c = max(0, issued_kv - 2); c < issued_kv; c++)
                mbar_wait(&kvfull[c % 2], (c / 2) & 1, err, kErrTimeout);
        }
    } else if (warp == MMAW) {
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t id_qs = idesc_bf16(128, DV, 0, 1);
            constexpr uint32_t id_q16 = idesc_bf16(128, 16, 0, 1);
            constexpr uint32_t id_kv = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t id_k16 = idesc_bf16(128, 16, 1, 1);
            const uint32_t s_addr = smem_u32(sm + PL::S0), zp_addr = smem_u32(sm + PL::Z0),
                           ones = smem_u32(sm + PL::O0);
            for (int c = 0; c < nc; c++) {
                const int sq = c % NQ, skv = c % 2;
                if (!wait_ok(ops_ready, c & 1, abort_flag, err)) continue;
                tc_fence_after();
                const uint32_t qa = smem_u32(sm + PL::Q0 + sq * PL::QB);
                const uint32_t ka = smem_u32(sm + PL::K0 + skv * PL::QB);
                const uint32_t va = smem_u32(sm + PL::V0 + skv * PL::VB);
                // MMA1: A = phiQ phiK^T
#pragma unroll
                for (int k = 0; k < DP; k += 16) {
                    const uint32_t off = (k / 64) * (kC * 128) + (k % 64) * 2;
                    mma_bf16_ss(tmem + PL::T_A, sw128_desc(qa + off, 16, 1024),
                                sw128_desc(ka + off, 16, 1024), id_qk, k > 0 ? 1u : 0u);
                }
                mma_commit(mma1_bar);
                // MMA3 / MMA3b: NUM = phiQ S_prev, DEN = phiQ ZP
#pragma unroll
                for (int k = 0; k < DP; k += 16) {
                    const uint64_t ad = sw128_desc(qa + (k / 64) * (kC * 128) + (k % 64) * 2, 16, 1024);
                    mma_bf16_ss(tmem + PL::T_NUM, ad,
                                sw128_desc(s_addr + (k / 8) * 1024, DP * 128, 1024), id_qs,
                                k > 0 ? 1u : 0u);
                    mma_bf16_ss(tmem + PL::T_DEN, ad, sw32_desc(zp_addr + (k / 8) * 256, 256, 256),
                                id_q16, k > 0 ? 1u : 0u);
                }
                // MMA4 / MMA4b: S += phiK^T V, Z += phiK^T ONES
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    const uint64_t ad =
                        sw128_desc(ka + (k / 8) * 1024, DP == 128 ? kC * 128 : 0, 1024);
                    mma_bf16_ss(tmem + PL::T_S, ad, sw128_desc(va + (k / 8) * 1024, kC * 128, 1024),
                                id_kv, 1u);
                    mma_bf16_ss(tmem + PL::T_Z, ad, sw32_desc(ones + (k / 8) * 256, 256, 256),
                                id_k16, 1u);
                }
                mma_commit(mma4_bar);
                mma_commit(&qempty[sq]);
                // MMA2 / MMA2b: NUM += P V, DEN += P ONES  (P in TMEM)
                if (!wait_ok(p_ready, c & 1, abort_flag, err)) continue;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    const uint32_t pa = tmem + PL::T_P + k / 2;
                    mma_bf16_ts(tmem + PL::T_NUM, pa,
                                sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_qs, 1u);
                    mma_bf16_ts(tmem + PL::T_DEN, pa, sw32_desc(ones + (k / 8) * 256, 256, 256),
                                id_q16, 1u);
                }
                mma_commit(mma2_bar);
                mma_commit(&kvempty[skv]);
            }
            mma_commit(drain_bar);   // every MMA issued above has completed
            mbar_wait(drain_bar, 0, err, kErrTimeout);
        }
    } else {
        // ---------------- math warps: thread (row, grp), row = TMEM lane
        const int q = warp & 3, grp = warp >> 2;
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        unsigned char *St = sm + PL::S0;
        unsigned char *Zt = sm + PL::Z0;
        const long long pre_base = ((long long)head * g.nseg + seg);
        const int srow = row % DP;   // state row (rows >= DP duplicate rows - DP)

        fill_ones(sm + PL::O0, threadIdx.x, NMATH);
        // initial state: TMEM S and Z, the bf16 S_prev copy, ZP
        {
            uint32_t v[CW];
            const float *src = preS ? preS + pre_base * DP * DV + (long long)srow * DV + grp * CW
                                    : nullptr;
#pragma unroll
            for (int i = 0; i < CW; i += 4) {
                const float4 x = src ? *reinterpret_cast<const float4 *>(src + i)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                v[i] = __float_as_uint(x.x);
                v[i + 1] = __float_as_uint(x.y);
                v[i + 2] = __float_as_uint(x.z);
                v[i + 3] = __float_as_uint(x.w);
            }
#pragma unroll
            for (int c0 = 0; c0 < CW; c0 += 16) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; i++) w[i] = v[c0 + i];
                tmem_st16_nowait(tmem + lane_base + PL::T_S + grp * CW + c0, w);
            }
            if (row < DP) store_row_bf16<CW>(St, DP, row, grp * CW, v);
            if (grp == 0) {
                const float z0 = prez ? prez[pre_base * DP + srow] : 0.f;
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; i++) w[i] = i < 8 ? __float_as_uint(z0) : 0u;
                tmem_st16_nowait(tmem + lane_base + PL::T_Z, w);
                if (row < DP) store_zp_row(Zt, row, z0);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        math_bar<NMATH>();

        for (int c = 0; c < nc; c++) {
            const int sq = c % NQ, skv = c % 2;
            const int n_valid = min(kC, g.N - (c_begin + c) * kC);
            // 1. phi in place on this chunk's Q and K tiles
            wait_ok(&qfull[sq], (c / NQ) & 1, abort_flag, err);
            phi_row_part<DP, NG>(sm + PL::Q0 + sq * PL::QB, row, grp, false);
            wait_ok(&kvfull[skv], (c / 2) & 1, abort_flag, err);
            phi_row_part<DP, NG>(sm + PL::K0 + skv * PL::QB, row, grp, row >= n_valid);
            // 2. S_prev and ZP from the state after the previous chunk
            if (c > 0) {
                wait_ok(mma4_bar, (c - 1) & 1, abort_flag, err);
                tc_fence_after();
                if (q * 32 < DP) {   // warp-uniform
                    uint32_t v[CW];
                    tmem_ld_cols<CW>(tmem + lane_base + PL::T_S + grp * CW, v);
                    uint32_t zv[16];
                    if (grp == 0) tmem_ld16_nowait(tmem + lane_base + PL::T_Z, zv);
                    tmem_ld_wait();
                    store_row_bf16<CW>(St, DP, row, grp * CW, v);
                    if (grp == 0) store_zp_row(Zt, row, __uint_as_float(zv[0]));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            math_bar<NMATH>();
            if (threadIdx.x == 0) mbar_arrive(ops_ready);
            // 3. P = bf16(tril(A)) into TMEM
            wait_ok(mma1_bar, c & 1, abort_flag, err);
            tc_fence_after();
            {
                uint32_t a[32], pk[16];
                tmem_ld32_nowait(tmem + lane_base + PL::T_A + grp * 32, a);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const int col = grp * 32 + 2 * i;
                    pk[i] = pack_bf16x2(col <= row ? __uint_as_float(a[2 * i]) : 0.f,
                                        col + 1 <= row ? __uint_as_float(a[2 * i + 1]) : 0.f);
                }
                tmem_st16_nowait(tmem + lane_base + PL::T_P + grp * 16, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            math_bar<NMATH>();
            if (threadIdx.x == 0) mbar_arrive(p_ready);
            // 4. out = NUM / (DEN[0] + DEN[8])
            const bool ok = wait_ok(mma2_bar, c & 1, abort_flag, err);
            tc_fence_after();
            {
                uint32_t v[CW], d[16];
                tmem_ld_cols<CW>(tmem + lane_base + PL::T_NUM + grp * CW, v);
                tmem_ld16_nowait(tmem + lane_base + PL::T_DEN, d);
                tmem_ld_wait();
                const float inv = 1.f / (__uint_as_float(d[0]) + __uint_as_float(d[8]));
                if (ok && row < n_valid) {
                    __nv_bfloat16 *orow =
                        out + ((long long)head * g.N + (long long)(c_begin + c) * kC + row) * DV +
                        grp * CW;
#pragma unroll
                    for (int j = 0; j < CW / 8; j++)
                        *reinterpret_cast<uint4 *>(orow + 8 * j) = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * j]) * inv, __uint_as_float(v[8 * j + 1]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv, __uint_as_float(v[8 * j + 3]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv, __uint_as_float(v[8 * j + 5]) * inv),
                            pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv, __uint_as_float(v[8 * j + 7]) * inv));
                }
            }
            tc_fence_before();
        }
        // final state of the last segment -> S_out, z_out
        const bool aborted = __any_sync(0xffffffffu, *abort_flag != 0);   // warp-uniform
        if (seg == g.nseg - 1 && (S_out || z_out) && !aborted && q * 32 < DP) {
            tc_fence_after();
            uint32_t v[CW], zv[16];
            tmem_ld_cols<CW>(tmem + lane_base + PL::T_S + grp * CW, v);
            tmem_ld16_nowait(tmem + lane_base + PL::T_Z, zv);
            tmem_ld_wait();
            if (S_out) {
                float *dst = S_out + ((long long)head * DP + row) * DV + grp * CW;
#pragma unroll
                for (int i = 0; i < CW; i += 4)
                    *reinterpret_cast<float4 *>(dst + i) =
                        make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                    __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            }
            if (z_out && grp == 0) z_out[(long long)head * DP + row] = __uint_as_float(zv[0]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMAW) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D map over a [BH, N, cols] bf16 tensor; box = 64 columns x 128 rows x 1 head,
// 128-byte swizzle; rows past N read as zero.
bool make_map(CUtensorMap *m, const void *base, long long BH, int N, int cols)
{
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)N * cols * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

Geometry plan(const Problem &p, int num_sms)
{
    Geometry g;
    g.N = p.N;
    g.nchunks = cdiv(p.N, kC);
    long long want = num_sms / max(1LL, p.BH);
    int nseg = (int)max(1LL, min((long long)g.nchunks, want));
    g.cps = cdiv(g.nchunks, nseg);
    g.nseg = cdiv(g.nchunks, g.cps);
    return g;
}

int g_num_sms = 0;

int num_sms()
{
    if (!g_num_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    return g_num_sms;
}

template <int DP, int DV>
cudaError_t run(const Problem &p, void *scratch, float *S_out, float *z_out, int *err,
                cudaStream_t s)
{
    using OP = OutPlan<DP, DV>;
    using SP = StatePlan<DP, DV>;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, p.q, p.BH, p.N, p.D) || !make_map(&tk, p.k, p.BH, p.N, p.D) ||
        !make_map(&tv, p.v, p.BH, p.N, p.Dv))
        return cudaErrorInvalidValue;
    Geometry g = plan(p, num_sms());
    float *dS = nullptr, *dz = nullptr;
    cudaError_t e;
    int launches = 0;
    if (g.nseg > 1) {
        dS = (float *)scratch;
        dz = dS + (size_t)p.BH * g.nseg * DP * DV;
        if ((e = cudaFuncSetAttribute(tc_state_kernel<DP, DV>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, SP::SMEM)) !=
            cudaSuccess)
            return e;
        tc_state_kernel<DP, DV><<<dim3(g.nseg, (unsigned)p.BH), kStateThreads, SP::SMEM, s>>>(
            tk, tv, g, dS, dz, err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int sz = DP * DV + DP;
        seg_scan_kernel<<<dim3(cdiv(sz, 256), (unsigned)p.BH), 256, 0, s>>>(dS, dz, g.nseg,
                                                                          DP * DV, DP);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        launches += 2;
    }
    if ((e = cudaFuncSetAttribute(tc_out_kernel<DP, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  OP::SMEM)) != cudaSuccess)
        return e;
    tc_out_kernel<DP, DV><<<dim3(g.nseg, (unsigned)p.BH), kOutThreads, OP::SMEM, s>>>(
        tq, tk, tv, g, dS, dz, (__nv_bfloat16 *)p.out, S_out, z_out, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(launches + 1);
    return cudaSuccess;
}

}  // namespace

bool tc_causal_supported(const Problem &p)
{
    return p.dtype == DT_BF16 && p.kind == PHI_ELU1 && (p.D == 64 || p.D == 128) &&
           (p.Dv == 64 || p.Dv == 128);
}

size_t tc_causal_scratch_bytes(const Problem &p)
{
    Geometry g = plan(p, num_sms());
    if (g.nseg <= 1) return 0;
    return (size_t)p.BH * g.nseg * ((size_t)p.P * p.Dv + p.P) * sizeof(float);
}

cudaError_t tc_causal(const Problem &p, void *scratch, float *S_out, float *z_out, int *err,
                      cudaStream_t s)
{
    if (p.D == 64 && p.Dv == 64) return run<64, 64>(p, scratch, S_out, z_out, err, s);
    if (p.D == 64 && p.Dv == 128) return run<64, 128>(p, scratch, S_out, z_out, err, s);
    if (p.D == 128 && p.Dv == 64) return run<128, 64>(p, scratch, S_out, z_out, err, s);
    return run<128, 128>(p, scratch, S_out, z_out, err, s);
}

}  // namespace la
