// rpe_tc.cu -- kernelized attention with a Toeplitz relative-position weight
// on the sm_103a tensor cores (review page "Stable, Fast and Accurate:
// Kernelized Attention with Relative Positional Encoding", proposed method):
//   out_i = sum_j c_{i-j} (phi(q_i).phi(k_j)) v_j / sum_j c_{i-j} phi(q_i).phi(k_j),
//   c_t = exp(b_t), j <= i when causal.
// bf16 inputs, phi = elu + 1, D, Dv in {64, 128}.
//
// One CTA per (head, chunk of 128 queries); it walks the key chunks (those
// at or before its own when causal).  Per key chunk, with fp32 accumulation
// in TMEM:
//   A          = phiQ . phiK^T                 (tcgen05, M = N = 128, K = D)
//   P          = bf16(A o c_{i-j})             (TMEM warps; causal mask on the diagonal chunk)
//   NUM | DEN += P . [V | ONES]               (tcgen05, N = Dv + 16, K = 128; P from TMEM)
// and finally out = NUM / DEN.  ONES is a constant [128 x 16] block after
// each V slot (columns 0-7 one, 8-15 zero), so the denominator is the
// product's column Dv.  A lands in one of two TMEM regions that alternate
// between key chunks, so the product of chunk kc + 1 runs while the TMEM
// warps turn chunk kc into P.
//
// Roles (18 warps): warps 0-15 TMEM warps (phi in place on the Q tile and on
// each K tile, P, the epilogue; warp w owns TMEM lanes 32 (w % 4).. and
// column quarter w / 4), warp 16 the TMA producer, warp 17 the MMA thread.
// The K / V ring is as deep as shared memory allows (4 slots at D = Dv =
// 64): with two, the load of key chunk kc + 2 waited for the product of
// chunk kc, and the TMEM warps waited for that load.
// Every wait is bounded: on expiry the library's error word is set and all
// roles finish without waiting.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kRC = 128;                 // chunk (queries and keys)
constexpr int kRWarps = 16;              // TMEM warps: 4 lane quadrants x 4 column groups
constexpr int kRGroups = kRWarps / 4;
constexpr int kRProd = kRWarps, kRMma = kRWarps + 1;
constexpr int kRThreads = (kRWarps + 2) * 32;
constexpr long long kRBudget = 4000000000LL;
constexpr int kRErr = 1;

template <int D, int DV>
struct RpePlan {
    static constexpr int QB = kRC * D * 2;            // Q or K tile (128-byte swizzle, 64-column boxes)
    static constexpr int VB = kRC * (DV + 16) * 2;    // V slot: DV / 16 boxes of 16 columns + ONES
    // K / V ring depth: as deep as shared memory allows, up to 4 (the load of key
    // chunk kc + NS is issued once the product of chunk kc has read its slot)
    static constexpr int kFix = QB + 2 * 256 * 4 + 2048;
    static constexpr int NS = kFix + 4 * (QB + VB) <= 227 * 1024 ? 4 : kFix + 3 * (QB + VB) <= 227 * 1024 ? 3 : 2;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + QB;
    static constexpr int V0 = K0 + NS * QB;
    static constexpr int CW = V0 + NS * VB;           // weights window [2][256] fp32
    static constexpr int TILES = CW + 2 * 256 * 4;
    // at least 116 KB, so that one CTA holds an SM (it allocates all 512 TMEM columns)
    static constexpr int SMEM = TILES + 2048 > 116 * 1024 ? TILES + 2048 : 116 * 1024;
    static constexpr int NQ16 = DV + 16;
    static constexpr int T_NUM = 0, T_P = 160, T_A0 = 256;   // TMEM columns; A regions at 256 and 384
    // P slots: two (at 96 and 160) when NUM | DEN leaves room (Dv = 64), so that
    // P of chunk kc + 1 is written while the product of chunk kc reads P(kc)
    static constexpr int NP = NQ16 <= 96 ? 2 : 1;
    static constexpr int T_P1 = 96;
    static_assert(NQ16 <= T_P && T_P + 64 <= T_A0, "TMEM plan");
    static_assert(NP == 1 || (NQ16 <= T_P1 && T_P1 + 64 <= T_P), "TMEM plan");
    static_assert(SMEM <= 227 * 1024, "shared memory plan");
};

__device__ __forceinline__ uint32_t r_align1k(uint32_t a) { return (a + 1023u) & ~1023u; }

__device__ __forceinline__ uint32_t r_tile_off(int r, int j)
{
    return (uint32_t)(j >> 3) * (kRC * 128) + sw128_off(r, j & 7);
}

template <int D, int DV>
__global__ void __launch_bounds__(kRThreads, 1)
rpe_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ bias,
              __nv_bfloat16 *__restrict__ out, int BH, int N, int H, int causal, int *err)
{
    using PL = RpePlan<D, DV>;
    constexpr int QTR = DV / kRGroups;   // NUM columns per thread in the epilogue
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = r_align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *q_full = bar, *q_ready = bar + 1, *a_full = bar + 10, *a_free = bar + 12, *num_full = bar + 16;
    uint64_t *k_full = bar + 24, *k_ready = bar + 28, *v_full = bar + 32, *kv_empty = bar + 36;   // [NS] each
    uint64_t *p_ready = bar + 20, *p_free = bar + 22;   // [NP] each
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 17);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(bar + 18);
    float *cw = reinterpret_cast<float *>(gbase + PL::CW);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int NC = cdiv(N, kRC);
    const int h = blockIdx.x % BH, qc = NC - 1 - (int)(blockIdx.x / BH);
    const int nkc = causal ? qc + 1 : NC;   // key chunks this CTA reads
    const float *bh = bias + (long long)(h % H) * (2LL * N - 1);

    auto wait = [&](uint64_t *b, uint32_t parity) -> bool {
        if (*abort_cta) return false;
        if (mbar_try_wait(b, parity)) return true;
        const long long t0 = clock64();
        while (!mbar_try_wait(b, parity)) {
            if (*abort_cta) return false;
            if (clock64() - t0 > kRBudget) {
                atomicExch(err, kRErr);
                *abort_cta = 1;
                return false;
            }
        }
        return true;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_ready, kRWarps);
        for (int i = 0; i < PL::NS; i++) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_ready[i], kRWarps);
            mbar_init(&v_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_free[i], kRWarps);
        }
        for (int i = 0; i < PL::NP; i++) {
            mbar_init(&p_ready[i], kRWarps);
            mbar_init(&p_free[i], 1);
        }
        mbar_init(num_full, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp < kRWarps) {   // the ONES block after each V slot's DV / 16 boxes
        const uint32_t one = pack_bf16x2(1.f, 1.f);
        for (int i = threadIdx.x; i < PL::NS * kRC; i += kRWarps * 32) {
            const int st = i / kRC, r = i % kRC;
            const uint32_t blk = base + PL::V0 + st * PL::VB + (DV / 16) * (kRC * 32);
            sts128(blk + sw32_off(r, 0), make_uint4(one, one, one, one));
            sts128(blk + sw32_off(r, 1), make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
    }
    if (warp == kRMma) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kRProd) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            const uint64_t keep = policy_evict_last();   // K, V chunks are read by every later query chunk
            mbar_arrive_expect_tx(q_full, PL::QB);
            for (int b = 0; b < D / 64; b++)
                tma_load_3d(gbase + PL::Q0 + b * (kRC * 128), &tm_q, q_full, b * 64, qc * kRC, h);
            int issued = 0;
            for (int kc = 0; kc < nkc; kc++) {
                const int st = kc % PL::NS;
                if (kc >= PL::NS && !wait(&kv_empty[st], ((kc / PL::NS) - 1) & 1)) break;
                mbar_arrive_expect_tx(&k_full[st], PL::QB);
                for (int b = 0; b < D / 64; b++)
                    tma_load_3d_hint(gbase + PL::K0 + st * PL::QB + b * (kRC * 128), &tm_k, &k_full[st], b * 64,
                                     kc * kRC, h, keep);
                mbar_arrive_expect_tx(&v_full[st], kRC * DV * 2);
                for (int b = 0; b < DV / 16; b++)
                    tma_load_3d_hint(gbase + PL::V0 + st * PL::VB + b * (kRC * 32), &tm_v, &v_full[st], b * 16,
                                     kc * kRC, h, keep);
                issued = kc + 1;
            }
            // loads still in flight after an abort land before the CTA exits
            mbar_wait(q_full, 0, nullptr, 0, kRBudget);
            for (int kc = issued > PL::NS ? issued - PL::NS : 0; kc < issued; kc++) {
                mbar_wait(&k_full[kc % PL::NS], (kc / PL::NS) & 1, nullptr, 0, kRBudget);
                mbar_wait(&v_full[kc % PL::NS], (kc / PL::NS) & 1, nullptr, 0, kRBudget);
            }
        }
    } else if (warp == kRMma) {
        // --------------------------------------------------- MMA thread
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kRC, 0, 0);
            constexpr uint32_t id_pv = idesc_bf16(128, PL::NQ16, 0, 1);
            bool ok = wait(q_ready, 0);
            auto mma1 = [&](int kc) {
                const int st = kc % PL::NS, rg = kc & 1;
                if (kc >= 2) ok = ok && wait(&a_free[rg], ((kc >> 1) - 1) & 1);
                ok = ok && wait(&k_ready[st], (kc / PL::NS) & 1);
                tc_fence_after();
                if (ok) {
                    const uint32_t qa = base + PL::Q0, ka = base + PL::K0 + st * PL::QB;
#pragma unroll
                    for (int kk = 0; kk < D; kk += 16) {
                        const uint32_t off = (kk / 64) * (kRC * 128) + (kk % 64) * 2;
                        mma_bf16_ss(tmem + PL::T_A0 + rg * 128, sw128_desc(qa + off, 16, 1024),
                                    sw128_desc(ka + off, 16, 1024), id_qk, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&a_full[rg]);
            };
            if (ok) mma1(0);
            for (int kc = 0; kc < nkc && ok; kc++) {
                if (kc + 1 < nkc) mma1(kc + 1);
                const int st = kc % PL::NS, ps = kc % PL::NP;
                const uint32_t tp = ps ? PL::T_P1 : PL::T_P;
                ok = ok && wait(&p_ready[ps], (kc / PL::NP) & 1) && wait(&v_full[st], (kc / PL::NS) & 1);
                tc_fence_after();
                if (ok) {
                    const uint32_t va = base + PL::V0 + st * PL::VB;
#pragma unroll
                    for (int kk = 0; kk < kRC; kk += 16)
                        mma_bf16_ts(tmem + PL::T_NUM, tmem + tp + kk / 2,
                                    sw32_desc(va + (kk / 8) * 256, kRC * 32, 256), id_pv,
                                    (kc > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&p_free[ps]);
                mma_commit(&kv_empty[st]);
            }
            mma_commit(num_full);
            mbar_wait(num_full, 0, nullptr, 0, kRBudget);
        }
    } else {
        // ---------------------------------------------------- TMEM warps
        const int qd = warp & 3, grp = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        constexpr int JH = D / 8 / kRGroups;   // 16 B chunks per quarter row
        // phi in place on this thread's quarter row of a tile; `zero`: the row is past the sequence
        auto phi_half = [&](uint32_t t, bool zero) {
            uint4 x[JH];
#pragma unroll
            for (int j = 0; j < JH; j++) x[j] = lds128(t + r_tile_off(r, grp * JH + j));
#pragma unroll
            for (int j = 0; j < JH; j++)
                sts128(t + r_tile_off(r, grp * JH + j), zero ? make_uint4(0, 0, 0, 0) : phi_elu1_bf16x8(x[j]));
            fence_proxy_async_smem();
            __syncwarp();
        };
        // (every wait result is made warp-uniform: the tcgen05.ld / st below
        // and the __syncwarp in phi_half are warp-collective)
        auto wait_w = [&](uint64_t *b, uint32_t parity) { return __all_sync(0xffffffffu, wait(b, parity)); };
        bool ok = wait_w(q_full, 0);
        if (ok) phi_half(base + PL::Q0, false);   // (query rows past N are never stored)
        if (lane == 0) mbar_arrive(q_ready);
        const int q0 = qc * kRC;
        auto phi_k = [&](int kc) {
            const int st = kc % PL::NS;
            ok = ok && wait_w(&k_full[st], (kc / PL::NS) & 1);
            if (ok) phi_half(base + PL::K0 + st * PL::QB, kc * kRC + r >= N);
            if (lane == 0) mbar_arrive(&k_ready[st]);
        };
        if (nkc > 0) phi_k(0);
        // the log-weight b_t of this thread's window offset u = threadIdx.x for key
        // chunk kc: t = (q0 - k0) + u - 127 (read one chunk ahead, off the critical path)
        auto bias_at = [&](int kc) {
            const long long t = (long long)(q0 - kc * kRC) + threadIdx.x - (kRC - 1);
            return threadIdx.x < 2 * kRC - 1 && t > -N && t < N ? bh[t + N - 1] : -INFINITY;
        };
        float bnext = nkc > 0 ? bias_at(0) : -INFINITY;
        for (int kc = 0; kc < nkc; kc++) {
            const float bcur = bnext;
            if (kc + 1 < nkc) bnext = bias_at(kc + 1);
            if (kc + 1 < nkc) phi_k(kc + 1);
            const int rg = kc & 1;
            // weights c_t for t = (q0 - k0) + u - 127, u in [0, 255)
            float *w = cw + (kc & 1) * 256;
            if (threadIdx.x < 2 * kRC - 1) w[threadIdx.x] = bcur == -INFINITY ? 0.f : __expf(bcur);
            asm volatile("bar.sync 1, %0;" ::"n"(kRWarps * 32) : "memory");
            ok = ok && wait_w(&a_full[rg], (kc >> 1) & 1);
            tc_fence_after();
            uint32_t a0[32];
            const uint32_t ra = tmem + lane_base + PL::T_A0 + rg * 128 + grp * 32;
            tmem_ld32_nowait(ra, a0);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_free[rg]);
            const bool diag = causal && kc == qc;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int c = grp * 32 + 2 * i;   // key index in the chunk
                const float w0 = w[r - c + kRC - 1], w1 = w[r - c - 1 + kRC - 1];
                pk[i] = pack_bf16x2(diag && c > r ? 0.f : __uint_as_float(a0[2 * i]) * w0,
                                    diag && c + 1 > r ? 0.f : __uint_as_float(a0[2 * i + 1]) * w1);
            }
            const int ps = kc % PL::NP;   // the P slot of this chunk, free once the product of kc - NP has read it
            if (kc >= PL::NP) ok = ok && wait_w(&p_free[ps], ((kc / PL::NP) - 1) & 1);
            tc_fence_after();
            tmem_st16_nowait(tmem + lane_base + (ps ? PL::T_P1 : PL::T_P) + grp * 16, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_ready[ps]);
        }
        // out = NUM / DEN for this thread's row and column half
        ok = ok && wait_w(num_full, 0);
        tc_fence_after();
        // the loads by the whole warp; only the stores depend on the row
        uint32_t d[16], n0[32];
        tmem_ld16_nowait(tmem + lane_base + PL::T_NUM + DV, d);
        if constexpr (QTR == 32)
            tmem_ld32_nowait(tmem + lane_base + PL::T_NUM + grp * QTR, n0);
        else
            tmem_ld16_nowait(tmem + lane_base + PL::T_NUM + grp * QTR, *reinterpret_cast<uint32_t(*)[16]>(n0));
        tmem_ld_wait();
        if (ok && q0 + r < N) {
            const float inv = 1.f / __uint_as_float(d[0]);
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((long long)h * N + q0 + r) * DV + grp * QTR);
#pragma unroll
            for (int j = 0; j < QTR / 8; j++)
                dst[j] = make_uint4(pack_bf16x2(__uint_as_float(n0[8 * j]) * inv, __uint_as_float(n0[8 * j + 1]) * inv),
                                    pack_bf16x2(__uint_as_float(n0[8 * j + 2]) * inv, __uint_as_float(n0[8 * j + 3]) * inv),
                                    pack_bf16x2(__uint_as_float(n0[8 * j + 4]) * inv, __uint_as_float(n0[8 * j + 5]) * inv),
                                    pack_bf16x2(__uint_as_float(n0[8 * j + 6]) * inv, __uint_as_float(n0[8 * j + 7]) * inv));
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == kRMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 rpe_encode()
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

// 3-D map over a [BH, N, cols] bf16 tensor: 64 x 128 boxes in 128-byte
// swizzle, or (sw = 32) 16 x 128 boxes in 32-byte swizzle; rows past N read as zero
bool rpe_map(CUtensorMap *m, const void *base, long long BH, long long N, int cols, int sw)
{
    auto enc = rpe_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)N * cols * 2};
    cuuint32_t box[3] = {sw == 32 ? 16u : 64u, (cuuint32_t)kRC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int DV>
cudaError_t launch_rpe_tc(const Problem &p, const float *bias, int H, bool causal, int *err, cudaStream_t s)
{
    using PL = RpePlan<D, DV>;
    CUtensorMap tq, tk, tv;
    if (!rpe_map(&tq, p.q, p.BH, p.N, D, 128) || !rpe_map(&tk, p.k, p.BH, p.N, D, 128) ||
        !rpe_map(&tv, p.v, p.BH, p.N, DV, 32))
        return cudaErrorInvalidValue;
    cudaError_t e = set_max_smem_once<rpe_tc_kernel<D, DV>>(PL::SMEM);
    if (e != cudaSuccess) return e;
    const long long ctas = p.BH * cdiv(p.N, kRC);
    rpe_tc_kernel<D, DV><<<(unsigned)ctas, kRThreads, PL::SMEM, s>>>(tq, tk, tv, bias, (__nv_bfloat16 *)p.out,
                                                                    (int)p.BH, p.N, H, causal ? 1 : 0, err);
    e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

}  // namespace

bool rpe_tc_supported(const Problem &p)
{
    return p.dtype == DT_BF16 && p.kind == PHI_ELU1 && (p.D == 64 || p.D == 128) && (p.Dv == 64 || p.Dv == 128) &&
           p.BH * (long long)cdiv(p.N, kRC) < (1LL << 31);
}

cudaError_t rpe_tc_forward(const Problem &p, const float *bias, int H, bool causal, int *err, cudaStream_t s)
{
    if (p.D == 64 && p.Dv == 64) return launch_rpe_tc<64, 64>(p, bias, H, causal, err, s);
    if (p.D == 64 && p.Dv == 128) return launch_rpe_tc<64, 128>(p, bias, H, causal, err, s);
    if (p.D == 128 && p.Dv == 64) return launch_rpe_tc<128, 64>(p, bias, H, causal, err, s);
    return launch_rpe_tc<128, 128>(p, bias, H, causal, err, s);
}

}  // namespace la
