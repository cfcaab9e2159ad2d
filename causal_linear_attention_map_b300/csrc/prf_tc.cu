// prf_tc.cu -- causal linear attention with positive random features formed
// inside the chunk kernel (sm_103a: tcgen05, TMEM, TMA): phi(q) and phi(k)
// never leave the SM.
//
// The method.  phi(x) = exp(W x - |x|^2 / 2) / sqrt(m) (positive random
// features: review page "Rethinking Attention with Performers", FAVOR+; and
// its normalised form NPRF, phi(x / |x|), review page "Stable, Fast and
// Accurate: Kernelized Attention with Relative Positional Encoding",
// proposed method), with the causal recurrence of "Transformers are RNNs"
// (proposed method b2-b3, b5) cut into chunks of C = 128 positions:
//   A    = tril(phi(Q_c) phi(K_c)^T)
//   out  = (A V_c + phi(Q_c) S_prev) / (rowsum(A) + phi(Q_c) z_prev)
//   S   += phi(K_c)^T V_c,   z += colsum(phi(K_c)).
//
// Shapes: D = 64, Dv = 64, m = 128 or 256 features, bf16 in and out.  The
// features are taken in blocks of 128 (a pass per block).  Sums over
// features split exactly over blocks, so with m = 256 the first pass writes
// its un-normalised NUM, DEN to fp32 scratch (column-major per chunk, so that
// each warp access is 128 contiguous bytes) and the second adds its own and
// divides.
//
// Passes.  A row-norm pass writes |k|^2 (NPRF: and |q|^2) of every row.
// Then, as in the elu+1 kernels, each head's chunks are cut into segments so
// that every SM has a (head, segment) item: a segment-sum pass (AGG; one item
// per head, feature block and segment but the last) sums phi(K)^T V and
// colsum phi(K) over a segment, a scan turns those into exclusive prefixes
// over segments, and the output pass starts each segment from its prefix.
// Items are assigned statically: CTA b takes items b, b + grid, ...
//
// A q row's PRF factor exp(-|q|^2 / 2) multiplies every feature of the row
// and cancels between phi(q)^T S and phi(q)^T z, so the q tiles leave it out
// (NPRF normalises u by |x|, which is no such factor, and keeps it).
//
// Per tile of 128 rows of q or k (x, one 64-column box), on chip:
//   U      = X W_blk^T       tcgen05, M = 128 rows, N = 128 features, K = 64,
//                            W as bf16 hi + lo (W_hi = bf16(W),
//                            W_lo = bf16(W - W_hi), both products into one
//                            fp32 accumulator), into a 128-column TMEM buffer
//   phi    = exp(U - s)      exp warps: U from TMEM, |x|^2 from the norm
//                            pass, bf16 phi written over the tile's
//                            shared-memory slot (x sits in the slot's first
//                            box and is dead once U is complete)
// Per chunk (output pass), tcgen05.mma kind::f16, fp32 accumulation in TMEM:
//   MMA1   A         = phiQ . phiK^T               N = 128, K = 128
//   MMA3   NUM | DEN = phiQ . [S_prev | ZP]        N = 80,  K = 128
//   MMA4   S | z    += phiK^T . [V | ONES]         N = 80,  K = 128 (M = features)
//   MMA2   NUM | DEN += P . [V | ONES]             N = 80,  K = 128 (P bf16 in TMEM)
// ONES is a constant [C x 16] block (columns 0-7 one, 8-15 zero) after each V
// tile and ZP holds z_prev as bf16 hi (columns 0-7) and lo (8-15) after
// S_prev, so that z, rowsum(P) and phiQ . z_prev ride on the N = 80 products:
// DEN = column 64 + column 72.
//
// TMEM (512 columns): S | z [0, 80), A [96, 224), NUM | DEN [224, 304),
// P [320, 384), U [384, 512).  A and NUM have regions of their own, so MMA1
// of the next chunk needs only the masked P of this one, and MMA3 only the
// epilogue of the previous one.  The segment-sum form keeps two S | z
// regions (0 and 96) that alternate between items.  Rings: two chunks deep
// in the output passes, three in the segment-sum pass.
//
// Warp roles (20 warps, five per SM sub-partition: 96 registers):
//   warps 0-7    exp warps: warp w owns TMEM lane quadrant w % 4 (tile rows
//                32 (w % 4) ..) and features 64 (w / 4) .. of each U
//   warps 8-15   TMEM warps, lane quadrant w % 4, column half (w - 8) / 4:
//                the segment's prefix, S_prev | ZP, the masked P, the
//                epilogue (and the state export); in the segment-sum form
//                the segment's sums to scratch
//   warp 16      TMA producer of the q and k tiles (L2 prefetch two chunks ahead)
//   warp 17      lane 0: TMA producer of the V tiles; lane 1: TMA store of
//                the output tiles (staged in the V slot, dead after MMA2)
//   warp 18      chunk MMA issuer: MMA3(j), MMA4(j), MMA2(j), MMA1(j + 1)
//   warp 19      projection issuer: U of every tile as soon as it has landed
//                and the exp warps have read the previous U, so that the next
//                chunk's projections and exps run while this chunk's products do
//
// Every wait is bounded (clock64 budget); on expiry the kernel sets the
// library's error word and the CTA runs to its end without waiting.
#include <cuda.h>
#include <cmath>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "prf_tc.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;     // chunk length (rows of a tile; MMA M)
constexpr int kD = 64;      // q, k width
constexpr int kDV = 64;     // v width
constexpr int kFB = 128;    // features per pass
constexpr int kNQ = kDV + 16;   // N of the products with [V | ONES] or [S_prev | ZP]
constexpr int kPrefetch = 2;  // chunks of L2 prefetch of q, k ahead of their tile loads
constexpr int kErrTimeout = 1;
constexpr long long kWaitBudget = 4000000000LL;   // SM cycles (~2 s)

constexpr int kExpWarps = 8;
constexpr int kTmWarps = 8;
constexpr int kQKWarp = kExpWarps + kTmWarps;   // 16
constexpr int kVWarp = kQKWarp + 1;             // 17
constexpr int kMmaWarp = kVWarp + 1;            // 18
constexpr int kProjWarp = kMmaWarp + 1;         // 19
constexpr int kThreads = (kProjWarp + 1) * 32;  // 640 (five warps per SM sub-partition: 96 registers)

// What a launch computes.
//   kAgg   segment sums of one feature block
//   kFull  output pass of a single-block map (m = 128): out = NUM / DEN
//   kPart  output pass of block 0 of m = 256: NUM, DEN -> fp32 scratch
//   kComb  output pass of block 1: out = (NUM + part) / (DEN + part)
enum { kAgg = 0, kFull = 1, kPart = 2, kComb = 3 };

template <int MODE, int M>
struct PrfPlan {
    static constexpr bool AGG = MODE == kAgg;
    static constexpr int NB = M / kFB;                  // feature blocks
    static constexpr int XB = kC * kD * 2;              // one raw q or k tile (one box)
    static constexpr int WB = kFB * kD * 2;             // W_hi (or W_lo) of one block
    static constexpr int PB = kC * kFB * 2;             // one phi slot: two 64-feature boxes
    static constexpr int VB = kC * kNQ * 2;             // one V slot: 4 blocks of 16 columns + ONES
    static constexpr int SPB = kFB * kNQ * 2;           // S_prev | ZP
    // W: hi and lo of every block the launch uses (the segment-sum form takes
    // items of any block; an output pass uses one)
    static constexpr int NWB = AGG ? NB : 1;
    // ring depth: two chunks in the output passes; three in the segment-sum
    // pass, which holds no q tiles or S_prev
    static constexpr int NS = AGG ? 3 : 2;
    static constexpr int W0 = 0;
    static constexpr int Q0 = W0 + 2 * NWB * WB;
    static constexpr int K0 = Q0 + (AGG ? 0 : NS * PB);
    static constexpr int V0 = K0 + NS * PB;
    static constexpr int SP0 = V0 + NS * VB;
    static constexpr int TILES = SP0 + (AGG ? 0 : SPB);
    static constexpr int SMEM = TILES + 1024 /* alignment */ + 1024 /* barriers */;
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
    static_assert(52 * 8 <= 1024, "barrier map exceeds its 1 KB");
    static_assert(SMEM > 114 * 1024, "one CTA per SM: the kernel holds all 512 TMEM columns");
};

// TMEM columns: S | z, A, NUM | DEN, P, U; the segment-sum form's second S | z region
constexpr int T_S = 0, T_A = 96, T_N = 224, T_P = 320, T_U = 384, T_S1 = 96;

struct PrfGeo {
    int BH, N, NC;    // heads, positions, chunks per head
    int L, nseg;      // chunks per segment, segments per head
    int nb;           // feature blocks of the map (1 or 2)
    int blk;          // output pass: its feature block
    int n_items;
};

struct PrfArgs {
    const float *sqk, *sqq;   // [BH, N]: |k|^2, |q|^2 (NPRF) of every row, from the norm pass
    const float *W;   // [m, 64] fp32
    float *preS;      // [BH, nb, nseg, 128, 64]: segment sums, then exclusive prefixes
    float *prez;      // [BH, nb, nseg, 128]
    float *num_part;  // [BH, NC, 64, 128]: block 0's NUM (m = 256), column-major per chunk
    float *den_part;  // [BH, NC, 128]
    float *S_out;     // [BH, m, 64] or null: the state after the last position
    float *z_out;     // [BH, m]
    float log_scale;  // ln(m) / 2
    int normalize;    // NPRF
    int *err;
};

struct Ctl {
    volatile int *cta;   // shared abort word of this CTA
    int *err;            // library error word
};

__device__ __forceinline__ void raise_abort(const Ctl &c)
{
    atomicExch(c.err, kErrTimeout);
    *c.cta = 1;
}

// Bounded wait on a phase of an mbarrier; false once this CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *b, uint32_t parity, const Ctl &c)
{
    if (*c.cta) return false;
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*c.cta) return false;
        if (clock64() - t0 > kWaitBudget) {
            raise_abort(c);
            return false;
        }
    }
    return true;
}

// wait_bar for a lane that shares its warp with another waiting role.
__device__ __forceinline__ bool wait_bar_nap(uint64_t *b, uint32_t parity, const Ctl &c)
{
    if (*c.cta) return false;
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (*c.cta) return false;
        if (clock64() - t0 > kWaitBudget) {
            raise_abort(c);
            return false;
        }
        __nanosleep(128);
    }
    return true;
}

__device__ __forceinline__ uint32_t align1k(uint32_t a) { return (a + 1023u) & ~1023u; }

// 2^x on the SFU (the PTX instruction ex2.approx).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One 32-bit TMEM column of this thread's lane (no wait).
__device__ __forceinline__ uint32_t tmem_ld1_nowait(uint32_t taddr)
{
    uint32_t r;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
    return r;
}

// 32 fp32 state values -> bf16 at row r, columns [c0, c0 + 32) of the
// MN-major S_prev operand in 32-byte swizzle (16-column blocks kFB * 32 bytes apart).
__device__ __forceinline__ void sprev_store32(uint32_t st, int r, int c0, const uint32_t (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int col = c0 + 8 * j;
        const uint32_t a = st + (uint32_t)(col >> 4) * (kFB * 32) + sw32_off(r, (col >> 3) & 1);
        sts128(a, make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                             pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                             pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                             pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]))));
    }
}

// z (fp32) -> row r of ZP: columns 0-7 bf16(z), 8-15 bf16(z - bf16(z)).
__device__ __forceinline__ void zp_store(uint32_t zp, int r, float z)
{
    const float hi = __bfloat162float(__float2bfloat16_rn(z));
    const uint32_t h = pack_bf16x2(hi, hi), l = pack_bf16x2(z - hi, z - hi);
    sts128(zp + sw32_off(r, 0), make_uint4(h, h, h, h));
    sts128(zp + sw32_off(r, 1), make_uint4(l, l, l, l));
}

// Item -> (head, segment, feature block).  Output passes: items are
// (segment, head) with heads fastest; segment-sum pass: (segment, head,
// block) with blocks fastest.
struct Item {
    int bh, s, blk, c0, nc;
};
template <bool AGG>
__device__ __forceinline__ Item decode(int item, const PrfGeo &g)
{
    Item it;
    if constexpr (AGG) {
        const int per = g.BH * g.nb;
        it.s = item / per;
        it.bh = (item % per) / g.nb;
        it.blk = item % g.nb;
    } else {
        it.s = item / g.BH;
        it.bh = item % g.BH;
        it.blk = g.blk;
    }
    it.c0 = it.s * g.L;
    it.nc = min(g.L, g.NC - it.c0);
    return it;
}

// This CTA's chunks in order: items blockIdx.x, blockIdx.x + grid, ...
template <bool AGG>
struct Walk {
    int item;
    Item it;
    int c;
    bool valid;
    __device__ __forceinline__ void start(const PrfGeo &g)
    {
        item = blockIdx.x;
        c = 0;
        valid = item < g.n_items;
        if (valid) it = decode<AGG>(item, g);
    }
    __device__ __forceinline__ void advance(const PrfGeo &g)
    {
        if (++c < it.nc) return;
        item += gridDim.x;
        c = 0;
        valid = item < g.n_items;
        if (valid) it = decode<AGG>(item, g);
    }
    __device__ __forceinline__ int row0() const { return (it.c0 + c) * kC; }
};

// ---------------------------------------------------------------- kernel

template <int MODE, int M>
__global__ void __launch_bounds__(kThreads, 1)
prf_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, PrfGeo g,
                 PrfArgs a)
{
    using PL = PrfPlan<MODE, M>;
    constexpr bool AGG = PL::AGG;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    constexpr int NS = PL::NS;
    // [kind * 4 + slot], kind 0 q, 1 k
    uint64_t *x_full = bar, *phi_ready = bar + 8, *slot_free = bar + 16;
    uint64_t *v_full = bar + 24, *v_empty = bar + 28;        // [slot]
    uint64_t *u_full = bar + 32, *u_free = bar + 33;
    uint64_t *a_full = bar + 34, *a_free = bar + 35, *p_ready = bar + 36, *sp_ready = bar + 37,
             *s_done = bar + 38, *num_full = bar + 39, *num_free = bar + 40;
    uint64_t *out_ready = bar + 41;                          // [slot]
    uint64_t *sum_done = bar + 45, *sum_read = bar + 47;     // [2] segment-sum form
    uint64_t *drain = bar + 49;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 50);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(bar + 51);

    const Ctl ctl{abort_cta, a.err};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // the next launch in the chain (scan, or the second feature block's
    // pass) may be scheduled now; it waits for this grid before reading its output
    griddep_launch();

    if (threadIdx.x == 0) {
        for (int i = 0; i < 8; i++) {
            mbar_init(&x_full[i], 1);
            mbar_init(&phi_ready[i], kExpWarps);
            mbar_init(&slot_free[i], 1);
        }
        for (int i = 0; i < 4; i++) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&out_ready[i], kTmWarps);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&sum_done[i], 1);
            mbar_init(&sum_read[i], kTmWarps);
        }
        mbar_init(u_full, 1);
        mbar_init(u_free, kExpWarps);
        mbar_init(a_full, 1);
        mbar_init(a_free, kTmWarps);
        mbar_init(p_ready, kTmWarps);
        mbar_init(sp_ready, kTmWarps);
        mbar_init(s_done, 1);
        mbar_init(num_full, 1);
        mbar_init(num_free, kTmWarps);
        mbar_init(drain, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp < kExpWarps + kTmWarps) {
        // W rows of the block(s) this launch uses -> W_hi, W_lo: K-major
        // [128 features x 64] operands in 128-byte swizzle
        constexpr int NT = (kExpWarps + kTmWarps) * 32;
        for (int i = threadIdx.x; i < PL::NWB * kFB; i += NT) {
            const int wb = i / kFB, row = i % kFB;
            const int blk = AGG ? wb : g.blk;
            const float *src = a.W + (long long)(blk * kFB + row) * kD;
            const uint32_t hi_base = base + PL::W0 + wb * 2 * PL::WB, lo_base = hi_base + PL::WB;
#pragma unroll 1
            for (int c = 0; c < kD / 8; c++) {
                const float4 x0 = __ldg(reinterpret_cast<const float4 *>(src + 8 * c));
                const float4 x1 = __ldg(reinterpret_cast<const float4 *>(src + 8 * c + 4));
                const float w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                float hi[8], lo[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    hi[e] = __bfloat162float(__float2bfloat16_rn(w[e]));
                    lo[e] = w[e] - hi[e];
                }
                sts128(hi_base + sw128_off(row, c), make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                                               pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7])));
                sts128(lo_base + sw128_off(row, c), make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                               pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7])));
            }
        }
        // the constant ONES block after each V slot's four 16-column blocks
        const uint32_t one = pack_bf16x2(1.f, 1.f);
        for (int i = threadIdx.x; i < NS * kC; i += NT) {
            const int sl = i / kC, r = i % kC;
            const uint32_t blk = base + PL::V0 + sl * PL::VB + (kDV / 16) * (kC * 32);
            sts128(blk + sw32_off(r, 0), make_uint4(one, one, one, one));
            sts128(blk + sw32_off(r, 1), make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kQKWarp) {
        // ------------------------------------------------ q, k tile producer
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            const uint64_t pol = policy_evict_first();
            // tiles kPrefetch chunks ahead of the loads go into L2 first
            auto prefetch = [&](const Walk<AGG> &p) {
                if (!AGG) tma_prefetch_3d(&tm_q, 0, p.row0(), p.it.bh);
                tma_prefetch_3d(&tm_k, 0, p.row0(), p.it.bh);
            };
            Walk<AGG> w, pf;
            w.start(g);
            pf = w;
            for (int i = 0; i < kPrefetch && pf.valid; i++) {
                if (i > 0) prefetch(pf);
                pf.advance(g);
            }
            uint32_t issued[2] = {0, 0};   // loads issued per kind
            for (uint32_t j = 0; w.valid && !*abort_cta; j++) {
                if (pf.valid) {
                    prefetch(pf);
                    pf.advance(g);
                }
                const int sl = j % NS;
#pragma unroll
                for (int kind = AGG ? 1 : 0; kind < 2; kind++) {
                    if (j >= NS && !wait_bar(&slot_free[kind * 4 + sl], ((j / NS) - 1) & 1, ctl)) break;
                    const uint32_t dst = (kind == 0 ? PL::Q0 : PL::K0) + sl * PL::PB;
                    mbar_arrive_expect_tx(&x_full[kind * 4 + sl], PL::XB);
                    tma_load_3d_hint(gbase + dst, kind == 0 ? &tm_q : &tm_k, &x_full[kind * 4 + sl], 0, w.row0(),
                                     w.it.bh, pol);
                    issued[kind]++;
                }
                w.advance(g);
            }
            // loads still in flight (only after an abort)
            for (int kind = AGG ? 1 : 0; kind < 2; kind++)
                for (uint32_t m = issued[kind] > NS ? issued[kind] - NS : 0; m < issued[kind]; m++)
                    mbar_wait(&x_full[kind * 4 + m % NS], (m / NS) & 1, nullptr, 0);
        }
    } else if (warp == kVWarp) {
        if (lane == 0) {
            // ------------------------------------------------ V tile producer
            prefetch_tmap(&tm_v);
            const uint64_t pol = policy_evict_first();
            Walk<AGG> w;
            w.start(g);
            uint32_t j = 0;   // loads issued
            for (; w.valid; j++, w.advance(g)) {
                const int sl = j % NS;
                if (j >= NS && !wait_bar_nap(&v_empty[sl], ((j / NS) - 1) & 1, ctl)) break;
                mbar_arrive_expect_tx(&v_full[sl], kC * kDV * 2);
#pragma unroll
                for (int b = 0; b < kDV / 16; b++)
                    tma_load_3d_hint(gbase + PL::V0 + sl * PL::VB + b * (kC * 32), &tm_v, &v_full[sl], b * 16,
                                     w.row0(), w.it.bh, pol);
            }
            for (uint32_t m = j > NS ? j - NS : 0; m < j; m++) mbar_wait(&v_full[m % NS], (m / NS) & 1, nullptr, 0);
        } else if (lane == 1 && !AGG) {
            // ------------------------------------------ output tile stores
            prefetch_tmap(&tm_o);
            Walk<AGG> w;
            w.start(g);
            for (uint32_t j = 0; w.valid; j++, w.advance(g)) {
                const int sl = j % NS;
                const bool ok = wait_bar_nap(&out_ready[sl], (j / NS) & 1, ctl);
                if (ok && MODE != kPart) {
                    tma_store_3d(&tm_o, base + PL::V0 + sl * PL::VB, 0, w.row0(), w.it.bh);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
                mbar_arrive(&v_empty[sl]);
            }
            bulk_wait_all();
        }
    } else if (warp == kProjWarp) {
        // --------------------------------------------- projection issuer
        // U = X W_blk^T for every tile in the order the exp warps take them
        // (q then k of each chunk), as soon as the tile has landed and the exp
        // warps have read the previous U
        if (lane == 0) {
            constexpr uint32_t id_u = idesc_bf16(128, kFB, 0, 0);
            uint32_t nu = 0;
            Walk<AGG> w;
            w.start(g);
            for (uint32_t j = 0; w.valid; j++, w.advance(g)) {
                const int sl = j % NS;
#pragma unroll 1
                for (int kind = AGG ? 1 : 0; kind < 2; kind++) {
                    const uint32_t xa = base + (kind == 0 ? PL::Q0 : PL::K0) + sl * PL::PB;
                    wait_bar(&x_full[kind * 4 + sl], (j / NS) & 1, ctl);
                    if (nu > 0) wait_bar(u_free, (nu - 1) & 1, ctl);
                    tc_fence_after();
                    const uint32_t wh = base + PL::W0 + (AGG ? w.it.blk : 0) * 2 * PL::WB, wl = wh + PL::WB;
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kD; kk += 16) {
                            const uint64_t ad = sw128_desc(xa + kk * 2, 16, 1024);
                            mma_bf16_ss(tmem + T_U, ad, sw128_desc(wh + kk * 2, 16, 1024), id_u, kk > 0 ? 1u : 0u);
                            mma_bf16_ss(tmem + T_U, ad, sw128_desc(wl + kk * 2, 16, 1024), id_u, 1u);
                        }
                    }
                    mma_commit(u_full);   // (the exp warps wait for every U: nothing is left in flight at exit)
                    nu++;
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------- chunk MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t id_qs = idesc_bf16(128, kNQ, 0, 1);
            constexpr uint32_t id_kv = idesc_bf16(128, kNQ, 1, 1);
            constexpr uint32_t lbo_v = kC * 32, lbo_s = kFB * 32, lbo_kT = kC * 128;
            Walk<AGG> cur, nx;
            cur.start(g);
            nx = cur;
            if (nx.valid) nx.advance(g);
            if constexpr (AGG) {
                uint32_t ii = 0;   // items begun
                int rr = 0;
                for (uint32_t j = 0; cur.valid; j++) {
                    const int sl = j % NS;
                    if (cur.c == 0) {   // this item's sums go to region ii % 2, once item ii - 2's were read
                        rr = ii & 1;
                        if (ii >= 2) wait_bar(&sum_read[rr], ((ii >> 1) - 1) & 1, ctl);
                        ii++;
                    }
                    wait_bar(&phi_ready[4 + sl], (j / NS) & 1, ctl);
                    wait_bar(&v_full[sl], (j / NS) & 1, ctl);
                    tc_fence_after();
                    const uint32_t ka = base + PL::K0 + sl * PL::PB, va = base + PL::V0 + sl * PL::VB;
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kC; kk += 16)
                            mma_bf16_ss(tmem + T_S + rr * T_S1, sw128_desc(ka + (kk / 8) * 1024, lbo_kT, 1024),
                                        sw32_desc(va + (kk / 8) * 256, lbo_v, 256), id_kv,
                                        (cur.c > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&slot_free[4 + sl]);
                    mma_commit(&v_empty[sl]);
                    if (cur.c + 1 == cur.it.nc) mma_commit(&sum_done[rr]);
                    cur = nx;
                    if (nx.valid) nx.advance(g);
                }
            } else {
                const uint32_t sp = base + PL::SP0;
                // MMA1(j): A = phiQ phiK^T
                auto mma1 = [&](uint32_t j) {
                    const int sl = j % NS;
                    wait_bar(&phi_ready[sl], (j / NS) & 1, ctl);
                    wait_bar(&phi_ready[4 + sl], (j / NS) & 1, ctl);
                    if (j > 0) wait_bar(a_free, (j - 1) & 1, ctl);
                    tc_fence_after();
                    const uint32_t qa = base + PL::Q0 + sl * PL::PB, ka = base + PL::K0 + sl * PL::PB;
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kFB; kk += 16) {
                            const uint32_t off = (kk / 64) * (kC * 128) + (kk % 64) * 2;
                            mma_bf16_ss(tmem + T_A, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024),
                                        id_qk, kk > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(a_full);
                };
                if (cur.valid) mma1(0);
                for (uint32_t j = 0; cur.valid; j++) {
                    const bool more = nx.valid;
                    const int sl = j % NS;
                    const uint32_t qa = base + PL::Q0 + sl * PL::PB, ka = base + PL::K0 + sl * PL::PB;
                    const uint32_t va = base + PL::V0 + sl * PL::VB;
                    // MMA3: NUM | DEN = phiQ [S_prev | ZP]
                    wait_bar(sp_ready, j & 1, ctl);
                    if (j > 0) wait_bar(num_free, (j - 1) & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kFB; kk += 16)
                            mma_bf16_ss(tmem + T_N, sw128_desc(qa + (kk / 64) * (kC * 128) + (kk % 64) * 2, 16, 1024),
                                        sw32_desc(sp + (kk / 8) * 256, lbo_s, 256), id_qs, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&slot_free[sl]);
                    // MMA4: S | z += phiK^T [V | ONES]
                    wait_bar(&v_full[sl], (j / NS) & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kC; kk += 16)
                            mma_bf16_ss(tmem + T_S, sw128_desc(ka + (kk / 8) * 1024, lbo_kT, 1024),
                                        sw32_desc(va + (kk / 8) * 256, lbo_v, 256), id_kv, 1u);
                    }
                    mma_commit(s_done);
                    mma_commit(&slot_free[4 + sl]);
                    // MMA2: NUM | DEN += P [V | ONES]
                    wait_bar(p_ready, j & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kC; kk += 16)
                            mma_bf16_ts(tmem + T_N, tmem + T_P + kk / 2, sw32_desc(va + (kk / 8) * 256, lbo_v, 256),
                                        id_qs, 1u);
                    }
                    mma_commit(num_full);
                    if (more) mma1(j + 1);
                    cur = nx;
                    if (nx.valid) nx.advance(g);
                }
            }
            mma_commit(drain);   // every MMA issued above has completed
            mbar_wait(drain, 0, nullptr, 0);
        }
    } else if (warp < kExpWarps) {
        // ------------------------------------------------------- exp warps
        const int qd = warp & 3, eh = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        constexpr float kLog2e = 1.4426950408889634f;
        uint32_t nt = 0;   // projections consumed
        // |x|^2 of row r of a chunk's k (and, for NPRF, q) tile, from the norm
        // pass, loaded a chunk ahead of its use.  A q row's PRF factor
        // exp(-|q|^2 / 2) multiplies every feature of that row, so it cancels
        // between the numerator phi(q)^T S and the denominator phi(q)^T z: PRF
        // q tiles leave it out (NPRF's u / |x| is no such factor)
        auto load_sq = [&](const Walk<AGG> &p, float &k2, float &q2) {
            const long long grow = (long long)p.it.bh * g.N + p.row0() + r;
            const bool in = r < g.N - p.row0();
            k2 = in ? __ldcg(a.sqk + grow) : 0.f;
            q2 = in && a.normalize && !AGG ? __ldcg(a.sqq + grow) : 0.f;
        };
        Walk<AGG> w;
        w.start(g);
        float nsq_k = 0.f, nsq_q = 0.f;
        if (w.valid) load_sq(w, nsq_k, nsq_q);
        for (uint32_t j = 0; w.valid; j++, w.advance(g)) {
            const int sl = j % NS;
            const int nvalid = g.N - w.row0();   // rows of this chunk inside the sequence
            const float sq_k = nsq_k, sq_q = nsq_q;
            {
                Walk<AGG> nx = w;
                nx.advance(g);
                if (nx.valid) load_sq(nx, nsq_k, nsq_q);
            }
#pragma unroll 1
            for (int kind = AGG ? 1 : 0; kind < 2; kind++) {
                const uint32_t t = base + (kind == 0 ? PL::Q0 : PL::K0) + sl * PL::PB;
                const float sq = kind == 1 ? sq_k : sq_q;
                // PRF: exp(u - |x|^2/2 - ln(m)/2); NPRF: exp(u / |x| - 1/2 - ln(m)/2), as 2^(u a - b)
                const float us = a.normalize ? (sq > 0.f ? rsqrtf(sq) : 0.f) : 1.f;
                const float sh = a.normalize ? (sq > 0.f ? 0.5f : 0.f) + a.log_scale : 0.5f * sq + a.log_scale;
                // (PRF q rows: sq = 0 here, the factor left out as above)
                const float ua = us * kLog2e, ub = sh * kLog2e;
                const bool zero = kind == 1 && r >= nvalid;   // k rows past the end add nothing
                // (U complete means the projection has read x: the slot's first box can take phi)
                wait_bar(u_full, nt & 1, ctl);
                tc_fence_after();
                uint32_t v0[32], v1[32];
                tmem_ld32_nowait(tmem + lane_base + T_U + eh * 64, v0);
                tmem_ld32_nowait(tmem + lane_base + T_U + eh * 64 + 32, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(u_free);
                nt++;
                auto emit = [&](const uint32_t(&v)[32], int h) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++) {
                        uint32_t o[4];
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const float e0 = ex2_approx(fmaf(__uint_as_float(v[8 * q4 + 2 * i]), ua, -ub));
                            const float e1 = ex2_approx(fmaf(__uint_as_float(v[8 * q4 + 2 * i + 1]), ua, -ub));
                            o[i] = zero ? 0u : pack_bf16x2(e0, e1);
                        }
                        // features 64 eh + 32 h + 8 q4 .. : 16 B chunk (32 h + 8 q4) / 8 of box eh
                        sts128(t + eh * (kC * 128) + sw128_off(r, 4 * h + q4), make_uint4(o[0], o[1], o[2], o[3]));
                    }
                };
                emit(v0, 0);
                emit(v1, 1);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&phi_ready[kind * 4 + sl]);
            }
        }
    } else {
        // ----------------------------------------------------- TMEM warps
        const int qd = warp & 3, grp = (warp - kExpWarps) >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        if constexpr (AGG) {
            // each item's sums S | z (region ii % 2) -> its slot in scratch
            uint32_t ii = 0;
            for (int item = blockIdx.x; item < g.n_items; item += gridDim.x, ii++) {
                const Item it = decode<true>(item, g);
                const int rr = ii & 1;
                wait_bar(&sum_done[rr], (ii >> 1) & 1, ctl);
                tc_fence_after();
                const uint32_t src = tmem + lane_base + T_S + rr * T_S1;
                uint32_t v[32], zv[16];
                tmem_ld32_nowait(src + grp * 32, v);
                if (grp == 0) tmem_ld16_nowait(src + kDV, zv);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sum_read[rr]);
                const long long slot = ((long long)it.bh * g.nb + it.blk) * g.nseg + it.s;
                float4 *dst = reinterpret_cast<float4 *>(a.preS + slot * (kFB * kDV) + (long long)r * kDV + grp * 32);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    __stcg(dst + i, make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3])));
                if (grp == 0) __stcg(a.prez + slot * kFB + r, __uint_as_float(zv[0]));
            }
        } else {
            const uint32_t sp = base + PL::SP0, zp = sp + (kDV / 16) * (kFB * 32);
            uint32_t nsd = 0;   // s_done phases consumed
            auto wait_sdone = [&](uint32_t upto) {
                while (nsd <= upto) {
                    wait_bar(s_done, nsd & 1, ctl);
                    nsd++;
                }
            };
            // the state in T_S -> S_out, z_out rows 128 blk + r of head bh
            auto export_state = [&](int bh) {
                tc_fence_after();
                uint32_t v[32], zv[16];
                tmem_ld32_nowait(tmem + lane_base + T_S + grp * 32, v);
                if (grp == 0) tmem_ld16_nowait(tmem + lane_base + T_S + kDV, zv);
                tmem_ld_wait();
                const long long row = (long long)bh * (g.nb * kFB) + g.blk * kFB + r;
                float4 *dst = reinterpret_cast<float4 *>(a.S_out + row * kDV + grp * 32);
#pragma unroll
                for (int i = 0; i < 8; i++)
                    dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                         __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                if (grp == 0) a.z_out[row] = __uint_as_float(zv[0]);
            };
            // NUM | DEN of chunk jj (rows row0 + r of head bh) -> the output
            // tile in the chunk's V slot, or (first block of two) to scratch
            auto epilogue = [&](uint32_t jj, int bh, int row0) {
                wait_bar(num_full, jj & 1, ctl);
                tc_fence_after();
                uint32_t n[32];
                const uint32_t d0 = tmem_ld1_nowait(tmem + lane_base + T_N + kDV);       // phiQ z_prev hi + rowsum P
                const uint32_t d8 = tmem_ld1_nowait(tmem + lane_base + T_N + kDV + 8);   // phiQ z_prev lo
                tmem_ld32_nowait(tmem + lane_base + T_N + grp * 32, n);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(num_free);
                // the first block's sums of this chunk: [64 columns][128 rows]
                // fp32, so that a warp's access to one column is 128 contiguous bytes
                const long long cid = (long long)bh * g.NC + row0 / kC;
                float *part = a.num_part + cid * (kDV * kC) + (long long)(grp * 32) * kC + r;
                float den = __uint_as_float(d0) + __uint_as_float(d8);
                float o[32];
#pragma unroll
                for (int i = 0; i < 32; i++) o[i] = __uint_as_float(n[i]);
                if constexpr (MODE == kPart) {
#pragma unroll
                    for (int i = 0; i < 32; i++) __stcg(part + i * kC, o[i]);
                    if (grp == 0) __stcg(a.den_part + cid * kC + r, den);
                } else {
                    if constexpr (MODE == kComb) {
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] += __ldcg(part + i * kC);
                        den += __ldcg(a.den_part + cid * kC + r);
                    }
                    const float inv = 1.f / den;
                    const uint32_t vs = base + PL::V0 + (jj % NS) * PL::VB;
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++)
                        sts128(vs + sw128_off(r, grp * 4 + q4),
                               make_uint4(pack_bf16x2(o[8 * q4] * inv, o[8 * q4 + 1] * inv),
                                          pack_bf16x2(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv),
                                          pack_bf16x2(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv),
                                          pack_bf16x2(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv)));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&out_ready[jj % NS]);
            };
            Walk<false> w;
            w.start(g);
            bool first = true;
            int pbh = 0, prow0 = 0;
            bool plast = false;   // the previous chunk ended its head's last segment
            uint32_t j = 0;
            for (; w.valid; j++, w.advance(g)) {
                const Item it = w.it;
                const int row0 = w.row0();
                if (w.c == 0) {
                    // ---- the state before this segment (its prefix; zero for
                    // the first) -> T_S, and S_prev | ZP of its first chunk
                    if (j > 0) {
                        wait_sdone(j - 1);   // MMA3, MMA4 of the previous chunk have completed
                        if (plast && a.S_out) export_state(pbh);
                    }
                    if (first) {   // the prefixes (and block 0's sums) come from the launches before
                        griddep_wait();
                        first = false;
                    }
                    const long long slot = ((long long)it.bh * g.nb + g.blk) * g.nseg + it.s;
                    const float4 *src =
                        reinterpret_cast<const float4 *>(a.preS + slot * (kFB * kDV) + (long long)r * kDV + grp * 32);
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float4 pv = it.s > 0 ? __ldcg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[4 * i] = __float_as_uint(pv.x);
                        v[4 * i + 1] = __float_as_uint(pv.y);
                        v[4 * i + 2] = __float_as_uint(pv.z);
                        v[4 * i + 3] = __float_as_uint(pv.w);
                    }
                    tmem_st32_nowait(tmem + lane_base + T_S + grp * 32, v);
                    sprev_store32(sp, r, grp * 32, v);
                    if (grp == 0) {
                        const float z = it.s > 0 ? __ldcg(a.prez + slot * kFB + r) : 0.f;
                        uint32_t zw[16];
#pragma unroll
                        for (int i = 0; i < 16; i++) zw[i] = i < 8 ? __float_as_uint(z) : 0u;
                        tmem_st16_nowait(tmem + lane_base + T_S + kDV, zw);
                        zp_store(zp, r, z);
                    }
                    tmem_st_wait();
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sp_ready);
                }
                if constexpr (MODE == kComb) {   // the first block's sums for this chunk (32 KB): into L2 now
                    const long long cid = (long long)it.bh * g.NC + row0 / kC;
                    const int t = (warp - kExpWarps) * 32 + lane;   // 0 .. 255: one 128-byte line each
                    prefetch_l2(a.num_part + cid * (kDV * kC) + t * 32);
                    if (t < kC / 32) prefetch_l2(a.den_part + cid * kC + t * 32);
                }
                if (j > 0) epilogue(j - 1, pbh, prow0);
                // ---- A(j) -> the masked bf16 P -> T_P (P(j - 1) has been read:
                // the epilogue waited for MMA2(j - 1))
                wait_bar(a_full, j & 1, ctl);
                tc_fence_after();
                // (in two halves of 32 keys, which keeps the P step within the registers)
                uint32_t pk[32];
                const int cb = grp * 64;
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t av[32];
                    tmem_ld32_nowait(tmem + lane_base + T_A + cb + 32 * hh, av);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int col = cb + 32 * hh + 2 * i;
                        pk[16 * hh + i] = pack_bf16x2(col <= r ? __uint_as_float(av[2 * i]) : 0.f,
                                                      col + 1 <= r ? __uint_as_float(av[2 * i + 1]) : 0.f);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(a_free);
                tmem_st32_nowait(tmem + lane_base + T_P + grp * 32, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
                // ---- S_prev | ZP for the item's next chunk, once MMA4(j) has completed
                if (w.c + 1 < it.nc) {
                    wait_sdone(j);
                    tc_fence_after();
                    uint32_t v[32], zv[16];
                    tmem_ld32_nowait(tmem + lane_base + T_S + grp * 32, v);
                    if (grp == 0) tmem_ld16_nowait(tmem + lane_base + T_S + kDV, zv);
                    tmem_ld_wait();
                    sprev_store32(sp, r, grp * 32, v);
                    if (grp == 0) zp_store(zp, r, __uint_as_float(zv[0]));
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sp_ready);
                }
                pbh = it.bh;
                prow0 = row0;
                plast = it.s == g.nseg - 1 && w.c + 1 == it.nc;
            }
            if (j > 0) {
                epilogue(j - 1, pbh, prow0);
                if (plast && a.S_out) {
                    wait_sdone(j - 1);
                    export_state(pbh);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// |x|^2 of every row of a [rows, 64] bf16 tensor: a warp takes 32 rows (4 KB
// in a row) as 8 coalesced 512-byte pieces, lanes 8t .. 8t + 7 of piece i
// holding row 4i + t, and lane l writes row l's sum.
__global__ void prf_norm_kernel(const __nv_bfloat16 *__restrict__ x, float *__restrict__ sq, long long rows)
{
    const int lane = threadIdx.x % 32;
    const long long r0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32 * 32;
    if (r0 >= rows) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r0 * kD);
    const long long n = rows - r0;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = 4 * i + lane / 8 < n ? __ldg(src + 32 * i + lane) : make_uint4(0, 0, 0, 0);
    float mine = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        float p = 0.f;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const float lo = __uint_as_float(u[e] << 16), hi = __uint_as_float(u[e] & 0xffff0000u);
            p = fmaf(lo, lo, p);
            p = fmaf(hi, hi, p);
        }
        p += __shfl_xor_sync(0xffffffffu, p, 1);
        p += __shfl_xor_sync(0xffffffffu, p, 2);
        p += __shfl_xor_sync(0xffffffffu, p, 4);
        const float t = __shfl_sync(0xffffffffu, p, 8 * (lane % 4));   // row 4i + lane % 4
        if (i == lane / 4) mine = t;
    }
    if (lane < n) sq[r0 + lane] = mine;
}

// Exclusive prefix over a (head, feature block)'s segments of the segment
// sums, in place: slot s then holds the sums over segments 0 .. s - 1 (zero
// for s = 0).  The last segment's own sums are never computed or read.
__global__ void prf_seg_scan_kernel(float *__restrict__ preS, float *__restrict__ prez, int nseg)
{
    griddep_launch();
    griddep_wait();   // the segment sums are complete
    constexpr int szS = kFB * kDV, szz = kFB;
    const long long row = blockIdx.y;   // head * blocks + block
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    float *p;
    int stride;
    if (e < szS) {
        p = preS + row * nseg * (long long)szS + e;
        stride = szS;
    } else if (e < szS + szz) {
        p = prez + row * nseg * (long long)szz + (e - szS);
        stride = szz;
    } else {
        return;
    }
    float run = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += 8) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; i++) x[i] = s0 + i < nseg - 1 ? p[(long long)(s0 + i) * stride] : 0.f;
#pragma unroll
        for (int i = 0; i < 8; i++)
            if (s0 + i < nseg) {
                p[(long long)(s0 + i) * stride] = run;
                run += x[i];
            }
    }
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 prf_encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D map over a [BH, N, 64] bf16 tensor: box = 64 columns x 128 rows x 1
// head in 128-byte swizzle, or (sw32) 16 columns x 128 rows in 32-byte
// swizzle; rows past N read as zero (and are not written by a store).
bool prf_map(CUtensorMap *m, const void *base, long long BH, long long N, bool sw32)
{
    auto enc = prf_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {64 * 2, (cuuint64_t)N * 64 * 2};
    cuuint32_t box[3] = {sw32 ? 16u : 64u, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int prf_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

// Segments per head: enough (head, segment) items to give every SM one, and
// no segmentation once B*H alone fills the GPU.
PrfGeo prf_plan(long long BH, int N, int nb, int sms)
{
    PrfGeo g;
    g.BH = (int)BH;
    g.N = N;
    g.NC = cdiv(N, kC);
    g.nb = nb;
    g.blk = 0;
    const int want = BH >= sms ? 1 : (int)(sms / BH);
    g.L = cdiv(g.NC, max(1, min(want, g.NC)));
    g.nseg = cdiv(g.NC, g.L);
    g.n_items = (int)(BH * g.nseg);
    return g;
}

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

struct PrfLayout {
    size_t preS, prez, num_part, den_part, sqk, sqq, total;
};

PrfLayout prf_layout(const Problem &p)
{
    const PrfGeo g = prf_plan(p.BH, p.N, p.m / kFB, prf_sms());
    const size_t slots = g.nseg > 1 ? (size_t)g.BH * g.nb * g.nseg : 0;
    PrfLayout L;
    L.preS = 0;
    L.prez = L.preS + up256(slots * kFB * kDV * 4);
    L.num_part = L.prez + up256(slots * kFB * 4);
    const size_t rows = g.nb > 1 ? (size_t)g.BH * g.NC * kC : 0;   // whole chunks
    L.den_part = L.num_part + up256(rows * kDV * 4);
    L.sqk = L.den_part + up256(rows * 4);
    const size_t nrows = (size_t)g.BH * g.N;
    L.sqq = L.sqk + up256(nrows * 4);
    L.total = L.sqq + up256(p.kind == PHI_NPRF ? nrows * 4 : 0);
    return L;
}

template <int M>
cudaError_t prf_run(const Problem &p, void *scratch, float *S_out, float *z_out, int *err, cudaStream_t s)
{
    constexpr int NB = M / kFB;
    const int sms = prf_sms();
    PrfGeo g = prf_plan(p.BH, p.N, NB, sms);
    const PrfLayout L = prf_layout(p);
    unsigned char *b = (unsigned char *)scratch;
    CUtensorMap tq, tk, tv, to;
    if (!prf_map(&tq, p.q, p.BH, p.N, false) || !prf_map(&tk, p.k, p.BH, p.N, false) ||
        !prf_map(&tv, p.v, p.BH, p.N, true) || !prf_map(&to, p.out, p.BH, p.N, false))
        return cudaErrorInvalidValue;
    PrfArgs a;
    a.sqk = (const float *)(b + L.sqk);
    a.sqq = (const float *)(b + L.sqq);
    a.W = p.W;
    a.preS = (float *)(b + L.preS);
    a.prez = (float *)(b + L.prez);
    a.num_part = (float *)(b + L.num_part);
    a.den_part = (float *)(b + L.den_part);
    a.S_out = S_out;
    a.z_out = z_out;
    a.log_scale = (float)(0.5 * std::log((double)M));
    a.normalize = p.kind == PHI_NPRF ? 1 : 0;
    a.err = err;
    constexpr int kOut0 = NB == 1 ? kFull : kPart;
    cudaError_t e;
    if ((e = set_max_smem_once<prf_chunk_kernel<kAgg, M>>(PrfPlan<kAgg, M>::SMEM)) != cudaSuccess ||
        (e = set_max_smem_once<prf_chunk_kernel<kOut0, M>>(PrfPlan<kOut0, M>::SMEM)) != cudaSuccess ||
        (NB > 1 && (e = set_max_smem_once<prf_chunk_kernel<kComb, M>>(PrfPlan<kComb, M>::SMEM)) != cudaSuccess))
        return e;
    int launches = 0;
    const long long rows = p.BH * (long long)p.N;
    const unsigned nblk = (unsigned)((rows + 255) / 256);
    prf_norm_kernel<<<nblk, 256, 0, s>>>((const __nv_bfloat16 *)p.k, (float *)a.sqk, rows);
    if (p.kind == PHI_NPRF) prf_norm_kernel<<<nblk, 256, 0, s>>>((const __nv_bfloat16 *)p.q, (float *)a.sqq, rows);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    launches += p.kind == PHI_NPRF ? 2 : 1;
    const bool seg = g.nseg > 1;
    if (seg) {
        PrfGeo ga = g;
        ga.n_items = g.BH * NB * (g.nseg - 1);
        prf_chunk_kernel<kAgg, M><<<min(ga.n_items, sms), kThreads, PrfPlan<kAgg, M>::SMEM, s>>>(tq, tk, tv, to, ga,
                                                                                                 a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_dependent(prf_seg_scan_kernel, dim3(cdiv(kFB * kDV + kFB, 256), (unsigned)(g.BH * NB)),
                                  dim3(256), 0, s, a.preS, a.prez, g.nseg)) != cudaSuccess)
            return e;
        launches += 2;
    }
    const dim3 grid(min(g.n_items, sms));
    if (seg)
        e = launch_dependent(prf_chunk_kernel<kOut0, M>, grid, dim3(kThreads), PrfPlan<kOut0, M>::SMEM, s, tq, tk,
                             tv, to, g, a);
    else {
        prf_chunk_kernel<kOut0, M><<<grid, kThreads, PrfPlan<kOut0, M>::SMEM, s>>>(tq, tk, tv, to, g, a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    launches++;
    if constexpr (NB > 1) {
        PrfGeo g1 = g;
        g1.blk = 1;
        if ((e = launch_dependent(prf_chunk_kernel<kComb, M>, grid, dim3(kThreads), PrfPlan<kComb, M>::SMEM, s, tq,
                                  tk, tv, to, g1, a)) != cudaSuccess)
            return e;
        launches++;
    }
    note_launches(launches);
    return cudaSuccess;
}

}  // namespace

bool prf_fused_supported(const Problem &p, bool causal)
{
    return causal && p.dtype == DT_BF16 && (p.kind == PHI_PRF || p.kind == PHI_NPRF) && p.D == kD &&
           p.Dv == kDV && (p.m == 128 || p.m == 256) && p.N > 0 && p.BH > 0 &&
           p.BH * (long long)p.N < (1LL << 31) - kC;
}

size_t prf_fused_scratch_bytes(const Problem &p) { return prf_layout(p).total; }

cudaError_t prf_fused_forward(const Problem &p, void *scratch, float *S_out, float *z_out, int *err, cudaStream_t s)
{
    return p.m == 256 ? prf_run<256>(p, scratch, S_out, z_out, err, s) : prf_run<128>(p, scratch, S_out, z_out, err, s);
}

}  // namespace la
