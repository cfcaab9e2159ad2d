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
//      sum of phi(K)^T V and colsum(phi(K)) (one tensor-core contraction per
//      chunk, accumulated in TMEM) and writes them to scratch;
//   2. scan: exclusive prefix of those states over segments, per head;
//   3. output pass: each (head, segment) CTA starts from its prefix state
//      and runs the chunk recurrence above, writing out.
// With a single segment per head, passes 1 and 2 are skipped.
//
// Per chunk (output pass) the four contractions are tcgen05.mma with fp32
// accumulation in TMEM:
//   MMA1  A    = phiQ . phiK^T        M=C, N=C,  K=Dphi  (both K-major)
//   MMA3  num  = phiQ . S_prev        M=C, N=Dv, K=Dphi  (S_prev MN-major, bf16 copy)
//   MMA4  S   += phiK^T . V           M=Dphi, N=Dv, K=C  (both MN-major)
//   MMA2  num += P . V                M=C, N=Dv, K=C     (P = bf16 masked A)
// phi is applied in place on the TMA-loaded Q/K tiles by the math warps
// (phi never goes back to HBM), which also form the denominators on CUDA
// cores: phi(q_i).z_prev while transforming row i, rowsum(A) while
// extracting P.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;            // chunk length (MMA M)
constexpr int kMathThreads = 128;  // warps 0-3: TMEM lane quadrants 0-3
constexpr int kThreads = kMathThreads + 64;  // + producer warp 4, MMA warp 5
constexpr int kErrTimeout = 1;

// Shared-memory plan of the output pass for one (DP, DV).
template <int DP, int DV>
struct OutPlan {
    static constexpr int QB = kC * DP * 2;  // one Q or K chunk tile (bytes)
    static constexpr int VB = kC * DV * 2;  // one V chunk tile
    static constexpr int PB = kC * kC * 2;  // masked scores P (bf16)
    static constexpr int SB = DP * DV * 2;  // S_prev (bf16)
    static constexpr int kBase = 2 * QB + 2 * QB + 2 * VB + PB + SB;
    static constexpr int NQ = (kBase + 4096 <= 227 * 1024) ? 2 : 1;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + NQ * QB;
    static constexpr int V0 = K0 + 2 * QB;
    static constexpr int P0 = V0 + 2 * VB;
    static constexpr int S0 = P0 + PB;
    static constexpr int TILES = S0 + SB;
    static constexpr int SMEM = TILES + 1024 /* align */ + 1024 /* barriers, z */;
    static constexpr int TMEM_S = 0, TMEM_NUM = DV, TMEM_A = 2 * DV;
    static constexpr int TMEM_COLS = (2 * DV + kC) <= 256 ? 256 : 512;
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
};

template <int DP, int DV>
struct StatePlan {
    static constexpr int QB = kC * DP * 2;
    static constexpr int VB = kC * DV * 2;
    static constexpr int NS = ((QB + VB) * 3 + 2048 <= 227 * 1024) ? 3 : 2;
    static constexpr int K0 = 0;
    static constexpr int V0 = NS * QB;
    static constexpr int TILES = V0 + NS * VB;
    static constexpr int SMEM = TILES + 1024 + 1024;
    static constexpr int TMEM_COLS = DV <= 32 ? 32 : (DV <= 64 ? 64 : 128);
};

struct Geometry {
    int N, nchunks, cps, nseg;
};

__device__ __forceinline__ unsigned char *align1k(unsigned char *p)
{
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                             ~uintptr_t(1023));
}

__device__ __forceinline__ void math_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

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

// phi(x) = elu(x) + 1 on 8 packed bf16, in place; returns them as floats.
__device__ __forceinline__ uint4 phi8(uint4 raw, float (&f)[8])
{
    uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int t = 0; t < 4; t++) {
        float2 p = unpack_bf16x2(w[t]);
        f[2 * t] = phi_elu1_fast(p.x);
        f[2 * t + 1] = phi_elu1_fast(p.y);
        w[t] = pack_bf16x2(f[2 * t], f[2 * t + 1]);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Transform row `r` of a [kC x DP] swizzled tile in place.  If `zero`, the
// row is cleared (positions past the end of the sequence).  If zs != null,
// returns phi(row) . zs using the bf16-rounded phi values.
template <int DP>
__device__ __forceinline__ float phi_row(unsigned char *tile, int r, bool zero, const float *zs)
{
    float dot = 0.f;
#pragma unroll
    for (int b = 0; b < DP / 64; b++) {
        unsigned char *blk = tile + b * (kC * 128);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            uint4 *p = reinterpret_cast<uint4 *>(blk + sw128_off(r, j));
            if (zero) {
                *p = make_uint4(0, 0, 0, 0);
                continue;
            }
            float f[8];
            uint4 o = phi8(*p, f);
            *p = o;
            if (zs) {
                const float *zz = zs + b * 64 + j * 8;
                uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    float2 q = unpack_bf16x2(w[t]);
                    dot = fmaf(q.x, zz[2 * t], dot);
                    dot = fmaf(q.y, zz[2 * t + 1], dot);
                }
            }
        }
    }
    return dot;
}

// Column sum of column d of a [kC x DP] swizzled bf16 tile.
template <int DP>
__device__ __forceinline__ float col_sum(const unsigned char *tile, int d)
{
    const unsigned char *blk = tile + (d / 64) * (kC * 128);
    const int cc = d % 64, j = cc / 8, e = cc % 8;
    float s = 0.f;
#pragma unroll 8
    for (int r = 0; r < kC; r++) {
        const __nv_bfloat16 *p =
            reinterpret_cast<const __nv_bfloat16 *>(blk + sw128_off(r, j)) + e;
        s += __bfloat162float(*p);
    }
    return s;
}

// ------------------------------------------------------------ state pass

template <int DP, int DV>
__global__ void __launch_bounds__(kThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                Geometry g, float *__restrict__ dS, float *__restrict__ dz, int *err)
{
    using PL = StatePlan<DP, DV>;
    constexpr int NS = PL::NS;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1k(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + PL::TILES);
    uint64_t *full = bars, *phi_done = bars + NS, *empty = bars + 2 * NS, *final_bar = bars + 3 * NS;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 3 * NS + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

    const int seg = blockIdx.x, head = blockIdx.y;
    const int c_begin = seg * g.cps;
    const int c_end = min(c_begin + g.cps, g.nchunks);
    const int nc = c_end - c_begin;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&phi_done[i], 1);
            mbar_init(&empty[i], 2);   // MMA commit + math (colsum done)
        }
        mbar_init(final_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 4) {
        // ---------------- TMA producer
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
            // drain: the loads issued last into each stage have landed
            for (int c = max(0, issued - NS); c < issued; c++)
                mbar_wait(&full[c % NS], (c / NS) & 1, err, kErrTimeout);
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer: S += phiK^T V
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(128, DV, 1, 1);
            for (int c = 0; c < nc; c++) {
                const int st = c % NS;
                if (!wait_ok(&phi_done[st], (c / NS) & 1, abort_flag, err)) continue;
                tc_fence_after();
                const uint32_t ka = smem_u32(sm + PL::K0 + st * PL::QB);
                const uint32_t va = smem_u32(sm + PL::V0 + st * PL::VB);
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    uint64_t ad = sw128_desc(ka + (k / 8) * 1024, DP == 128 ? kC * 128 : 0, 1024);
                    uint64_t bd = sw128_desc(va + (k / 8) * 1024, kC * 128, 1024);
                    mma_bf16_ss(tmem, ad, bd, idesc, (c > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&empty[st]);
            }
            mma_commit(final_bar);   // also the drain: every MMA issued above has completed
            mbar_wait(final_bar, 0, err, kErrTimeout);
        }
    } else {
        // ---------------- math warps: phi(K) in place, colsum for z
        const int t = threadIdx.x;
        float zacc = 0.f;
        for (int c = 0; c < nc; c++) {
            const int st = c % NS;
            wait_ok(&full[st], (c / NS) & 1, abort_flag, err);
            const int n_valid = min(kC, g.N - (c_begin + c) * kC);
            unsigned char *ktile = sm + PL::K0 + st * PL::QB;
            phi_row<DP>(ktile, t, t >= n_valid, nullptr);
            fence_proxy_async_smem();
            math_bar();
            if (t == 0) mbar_arrive(&phi_done[st]);
            if (t < DP) zacc += col_sum<DP>(ktile, t);
            math_bar();
            if (t == 0) mbar_arrive(&empty[st]);   // colsum reads done: stage may be refilled
        }
        // final state -> scratch (warp-uniform condition: tcgen05.ld is warp-collective)
        const bool done = wait_ok(final_bar, 0, abort_flag, err);
        if (__all_sync(0xffffffffu, done)) {
            tc_fence_after();
            const long long base = ((long long)head * g.nseg + seg);
            if (t < DP) {
                float *dst = dS + base * DP * DV + (long long)t * DV;
#pragma unroll
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + i) =
                            make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                }
                dz[base * DP + t] = zacc;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// ------------------------------------------------------------ scan

// Exclusive prefix over segments of the per-segment states, in place.
__global__ void seg_scan_kernel(float *__restrict__ dS, float *__restrict__ dz, int nseg, int sz_S,
                                int sz_z)
{
    const long long head = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e < sz_S) {
        float *p = dS + head * nseg * (long long)sz_S + e;
        float run = 0.f;
        for (int s = 0; s < nseg; s++) {
            float x = p[(long long)s * sz_S];
            p[(long long)s * sz_S] = run;
            run += x;
        }
    } else if (e < sz_S + sz_z) {
        float *p = dz + head * nseg * (long long)sz_z + (e - sz_S);
        float run = 0.f;
        for (int s = 0; s < nseg; s++) {
            float x = p[(long long)s * sz_z];
            p[(long long)s * sz_z] = run;
            run += x;
        }
    }
}

// ------------------------------------------------------------ output pass

template <int DP, int DV>
__global__ void __launch_bounds__(kThreads, 1)
tc_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, Geometry g,
              const float *__restrict__ preS, const float *__restrict__ prez,
              __nv_bfloat16 *__restrict__ out, float *__restrict__ S_out, float *__restrict__ z_out,
              int *err)
{
    using PL = OutPlan<DP, DV>;
    constexpr int NQ = PL::NQ;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1k(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + PL::TILES);
    uint64_t *qfull = bars;             // [NQ]
    uint64_t *qempty = bars + 2;        // [NQ]
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
    float *zs = reinterpret_cast<float *>(bars + 16);   // [DP]

    const int seg = blockIdx.x, head = blockIdx.y;
    const int c_begin = seg * g.cps;
    const int c_end = min(c_begin + g.cps, g.nchunks);
    const int nc = c_end - c_begin;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool last_seg = (seg == g.nseg - 1);

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
    if (warp == 5) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 4) {
        // ---------------- TMA producer
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
            // drain: the loads issued last into each stage have landed
            for (int c = max(0, issued_q - NQ); c < issued_q; c++)
                mbar_wait(&qfull[c % NQ], (c / NQ) & 1, err, kErrTimeout);
            for (int c = max(0, issued_kv - 2); c < issued_kv; c++)
                mbar_wait(&kvfull[c % 2], (c / 2) & 1, err, kErrTimeout);
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t id_qs = idesc_bf16(128, DV, 0, 1);
            constexpr uint32_t id_kv = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t id_pv = idesc_bf16(128, DV, 0, 1);
            const uint32_t t_S = tmem + PL::TMEM_S, t_num = tmem + PL::TMEM_NUM,
                           t_A = tmem + PL::TMEM_A;
            const uint32_t p_addr = smem_u32(sm + PL::P0), s_addr = smem_u32(sm + PL::S0);
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
                    mma_bf16_ss(t_A, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024),
                                id_qk, k > 0 ? 1u : 0u);
                }
                mma_commit(mma1_bar);
                // MMA3: num = phiQ S_prev
#pragma unroll
                for (int k = 0; k < DP; k += 16) {
                    const uint32_t aoff = (k / 64) * (kC * 128) + (k % 64) * 2;
                    mma_bf16_ss(t_num, sw128_desc(qa + aoff, 16, 1024),
                                sw128_desc(s_addr + (k / 8) * 1024, DP * 128, 1024), id_qs,
                                k > 0 ? 1u : 0u);
                }
                // MMA4: S += phiK^T V
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    mma_bf16_ss(t_S, sw128_desc(ka + (k / 8) * 1024, DP == 128 ? kC * 128 : 0, 1024),
                                sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_kv, 1u);
                }
                mma_commit(mma4_bar);
                mma_commit(&qempty[sq]);
                // MMA2: num += P V
                if (!wait_ok(p_ready, c & 1, abort_flag, err)) continue;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kC; k += 16) {
                    const uint32_t aoff = (k / 64) * (kC * 128) + (k % 64) * 2;
                    mma_bf16_ss(t_num, sw128_desc(p_addr + aoff, 16, 1024),
                                sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_pv, 1u);
                }
                mma_commit(mma2_bar);
                mma_commit(&kvempty[skv]);
            }
            // drain: every MMA issued above has completed before TMEM is freed
            mma_commit(drain_bar);
            mbar_wait(drain_bar, 0, err, kErrTimeout);
        }
    } else {
        // ---------------- math warps (thread t owns query row t / state row t)
        const int t = threadIdx.x;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        unsigned char *Pt = sm + PL::P0;
        unsigned char *St = sm + PL::S0;
        const long long pre_base = ((long long)head * g.nseg + seg);

        // initial state: TMEM S (all 128 lanes; rows >= DP duplicate rows - DP),
        // S_prev bf16 copy, z_prev.
        {
            const int r = t % DP;
            const float *src = preS ? preS + pre_base * DP * DV + (long long)r * DV : nullptr;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 x = src ? *reinterpret_cast<const float4 *>(src + c0 + i)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
                }
                tmem_st32(tmem + lane_base + PL::TMEM_S + c0, v);
                if (t < DP) {
                    unsigned char *blk = St + (c0 / 64) * (DP * 128);
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int chunk = (c0 % 64) / 8 + j;
                        *reinterpret_cast<uint4 *>(blk + sw128_off(t, chunk)) =
                            make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                       pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                       pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                       pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                    }
                }
            }
            if (t < DP) zs[t] = prez ? prez[pre_base * DP + t] : 0.f;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        math_bar();

        for (int c = 0; c < nc; c++) {
            const int sq = c % NQ, skv = c % 2;
            const int n_valid = min(kC, g.N - (c_begin + c) * kC);
            unsigned char *qt = sm + PL::Q0 + sq * PL::QB;
            unsigned char *kt = sm + PL::K0 + skv * PL::QB;
            // 1. phi(Q) (+ phi(q_t) . z_prev) and phi(K) in place
            wait_ok(&qfull[sq], (c / NQ) & 1, abort_flag, err);
            const float den_inter = phi_row<DP>(qt, t, false, zs);
            wait_ok(&kvfull[skv], (c / 2) & 1, abort_flag, err);
            phi_row<DP>(kt, t, t >= n_valid, nullptr);
            fence_proxy_async_smem();
            math_bar();
            if (t < DP) zs[t] += col_sum<DP>(kt, t);   // z for the next chunk
            // 2. S_prev for this chunk from S after the previous chunk
            if (c > 0) {
                wait_ok(mma4_bar, (c - 1) & 1, abort_flag, err);
                tc_fence_after();
                if (warp < (DP + 31) / 32) {
#pragma unroll
                    for (int c0 = 0; c0 < DV; c0 += 32) {
                        float v[32];
                        tmem_ld32(tmem + lane_base + PL::TMEM_S + c0, v);
                        unsigned char *blk = St + (c0 / 64) * (DP * 128);
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const int chunk = (c0 % 64) / 8 + j;
                            *reinterpret_cast<uint4 *>(blk + sw128_off(t, chunk)) =
                                make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]),
                                           pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                                           pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                                           pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
                        }
                    }
                    fence_proxy_async_smem();
                }
            }
            tc_fence_before();
            math_bar();
            if (t == 0) mbar_arrive(ops_ready);
            // 3. P = bf16(tril(A)), den_intra = rowsum
            wait_ok(mma1_bar, c & 1, abort_flag, err);
            tc_fence_after();
            float den_intra = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < kC; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + lane_base + PL::TMEM_A + c0, v);
                unsigned char *blk = Pt + (c0 / 64) * (kC * 128);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int col = c0 + 8 * j + 2 * e;
                        float a0 = col <= t ? v[8 * j + 2 * e] : 0.f;
                        float a1 = col + 1 <= t ? v[8 * j + 2 * e + 1] : 0.f;
                        w[e] = pack_bf16x2(a0, a1);
                        float2 r = unpack_bf16x2(w[e]);
                        den_intra += r.x + r.y;
                    }
                    const int chunk = (c0 % 64) / 8 + j;
                    *reinterpret_cast<uint4 *>(blk + sw128_off(t, chunk)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            math_bar();
            if (t == 0) mbar_arrive(p_ready);
            // 4. out = num / den
            const bool ok = wait_ok(mma2_bar, c & 1, abort_flag, err);
            tc_fence_after();
            const float inv = 1.f / (den_intra + den_inter);
            __nv_bfloat16 *orow =
                out + ((long long)head * g.N + (long long)(c_begin + c) * kC + t) * DV;
#pragma unroll
            for (int c0 = 0; c0 < DV; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + lane_base + PL::TMEM_NUM + c0, v);
                if (ok && t < n_valid) {
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        *reinterpret_cast<uint4 *>(orow + c0 + 8 * j) =
                            make_uint4(pack_bf16x2(v[8 * j] * inv, v[8 * j + 1] * inv),
                                       pack_bf16x2(v[8 * j + 2] * inv, v[8 * j + 3] * inv),
                                       pack_bf16x2(v[8 * j + 4] * inv, v[8 * j + 5] * inv),
                                       pack_bf16x2(v[8 * j + 6] * inv, v[8 * j + 7] * inv));
                }
            }
            tc_fence_before();
        }
        // final state of the last segment -> S_out, z_out
        const bool aborted = __any_sync(0xffffffffu, *abort_flag != 0);   // warp-uniform
        if (last_seg && (S_out || z_out) && !aborted) {
            tc_fence_after();
            if (warp < (DP + 31) / 32) {
#pragma unroll
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + PL::TMEM_S + c0, v);
                    if (S_out) {
                        float *dst = S_out + ((long long)head * DP + t) * DV + c0;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) =
                                make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    }
                }
                if (z_out && t < DP) z_out[(long long)head * DP + t] = zs[t];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
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
        tc_state_kernel<DP, DV><<<dim3(g.nseg, (unsigned)p.BH), kThreads, SP::SMEM, s>>>(
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
    tc_out_kernel<DP, DV><<<dim3(g.nseg, (unsigned)p.BH), kThreads, OP::SMEM, s>>>(
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
