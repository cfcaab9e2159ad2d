// tc_causal.cu -- linear attention on the sm_103a tensor cores (tcgen05,
// TMEM accumulators, TMA loads and stores), bf16 inputs, fp32 state: the
// chunked causal kernel, the non-causal readout, and the random-feature
// projection.
//
// The method (review page "Transformers are RNNs", proposed method b2-b3,
// b5): with phi applied to q and k, out_i = phi(q_i)^T S_i / phi(q_i)^T z_i
// where S_i, z_i are cumulative sums over j <= i.  A sequence is cut into
// chunks of C = 128 positions; with S_prev, z_prev the sums before a chunk,
//   A    = tril(phi(Q_c) phi(K_c)^T)                      (j <= i)
//   out  = (A V_c + phi(Q_c) S_prev) / (rowsum(A) + phi(Q_c) z_prev)
//   S   += phi(K_c)^T V_c,   z += colsum(phi(K_c)).
//
// Work items.  When B*H is below the number of SMs, each head's chunks are
// cut into segments so that every SM gets one (head, segment) item; an item
// needs the state (S, z) after the previous segments of its head.  That
// prefix comes from a separate pass over K, V: the kernel runs first in its
// aggregate form (AGG = true: each item only sums phi(K)^T V and colsum
// phi(K) over its segment, into scratch), a small scan turns those sums into
// exclusive prefixes over segments, and the output form (AGG = false) starts
// each segment's chunk recurrence from its prefix.  CTA b takes item b first;
// further items (when there are more items than CTAs) come from a global
// ticket counter.  (Chaining the segment states from CTA to CTA in
// one pass was measured slower: under a full HBM load every link costs
// several microseconds of global-memory round trips, and the chain advances
// one segment per link.)
//
// Warp roles (16 warps, 4 per SM sub-partition, so 128 registers):
//   warps 0-7   TMEM warps: phi(Q) in place on the Q tile, masked scores P,
//               the state copy S_prev / ZP for the next chunk, the epilogue,
//               phase B.  Warp w owns TMEM lane quadrant w % 4 (rows 32 (w%4)
//               ..) and column half w / 4.  (Aggregate form: two thirds of
//               each K tile's phi, then the segment's sums to scratch.)
//   warps 8-11  phi warps, one per lane quadrant (one tile row per thread):
//               phi(K) in place on the K tile in shared memory.
//   warp 12     TMA producer of Q tiles and item scheduler (in the
//               aggregate form, which reads no Q, warp 13 hands out items).
//   warp 13     TMA producer of K tiles.
//   warp 14     TMA producer of V tiles (lane 0) and TMA store of the output
//               tiles (lane 1).
//   warp 15     MMA issuer (one thread).
// The epilogue writes each output tile into the shared-memory slot of that
// chunk's V tile (V is dead once MMA2 has read it), and one thread stores it
// with a TMA tile store, releasing the V slot once the store has read it.
// The producers prefetch a tile ahead into L2.  Q, K and V have their own
// rings because they free up at different points: Q after MMA3, K after
// MMA4, V after the output store.
//
// Per chunk, four groups of tcgen05.mma (kind::f16, M = 128, K = 16 per
// instruction) with fp32 accumulation in TMEM:
//   MMA1   A         = phiQ . phiK^T              N = C,       K = Dphi
//   MMA3   NUM | DEN = phiQ . [S_prev | ZP]       N = Dv + 16, K = Dphi
//   MMA4   S   | z  += phiK^T . [V | ONES]        N = Dv + 16, K = C  (M = Dphi)
//   MMA2   NUM | DEN += P . [V | ONES]            N = Dv + 16, K = C  (P bf16 in TMEM)
// ONES is a constant [C x 16] block (columns 0-7 = 1, 8-15 = 0) after each V
// slot, and ZP holds z_prev split into bf16 hi (columns 0-7) and lo (8-15)
// after S_prev: V and S_prev are kept in 32-byte swizzle (16-column blocks)
// so that these blocks are simply the next block of the operand, and
// out = NUM / (DEN[:,0] + DEN[:,8]).  (A separate N = 16 product per K step
// would cost about as much as the full one.)  phi never goes back to HBM.
// TMEM holds two regions R0, R1 that chunks use alternately: chunk k's
// scores A(k) land in R[k % 2], and once the TMEM warps have read them into
// registers (as the masked bf16 P, which gets its own slot) the same region
// takes NUM(k) | DEN(k).  So MMA3(k) never waits for the epilogue of k - 1;
// only MMA1(k + 2) needs R[k % 2] back.  The issue order per chunk is
// MMA3(k), MMA4(k), MMA1(k+1), MMA2(k), which keeps independent work in the
// tensor pipe while the TMEM warps convert A(k + 1) and drain NUM(k).  At
// D = Dv = 128 S_prev is staged in two 64-row halves (the second written
// once MMA3 has read the first), which leaves shared memory for two-deep Q,
// K and V rings.
//
// Every wait is bounded (clock64 budget).  On expiry the kernel sets the
// library's device error word and a per-launch abort word (the other CTAs
// take no further item once they see it; their own waits are bounded too),
// and all roles of the CTA run to the end without waiting.
#include <cuda.h>
#include <cmath>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;               // chunk length (MMA M)
constexpr int kErrTimeout = 1;
constexpr long long kWaitBudget = 4000000000LL;   // SM cycles (~2 s)

constexpr int kTmemWarps = 8;
constexpr int kPhiWarps = 4;
constexpr int kProducerWarp = kTmemWarps + kPhiWarps;   // 12: Q tiles, items
constexpr int kKWarp = kProducerWarp + 1;               // 13: K tiles
constexpr int kVWarp = kKWarp + 1;                      // 14: V tiles
constexpr int kMmaWarp = kVWarp + 1;                    // 15
constexpr int kThreads = (kMmaWarp + 1) * 32;           // 512
constexpr int kPrefetch = 1;                            // chunks of L2 prefetch ahead
constexpr int kItemConsumers = kTmemWarps + kPhiWarps + 4;

// Column-chunk split of the phi(K) work in the segment-sum form: phi warps
// [0, kAggSplit1), TMEM warps of column half 0 [kAggSplit1, kAggSplit2),
// of column half 1 [kAggSplit2, JR).
template <int JR> constexpr int kAggSplit1 = JR - 2 * (JR / 3);
template <int JR> constexpr int kAggSplit2 = JR - JR / 3;

template <int DP, int DV, bool SUMF = false>
struct Plan {
    static constexpr int QB = kC * DP * 2;   // one Q or K chunk tile (bytes)
    static constexpr int kBudget = 227 * 1024 - 2048;
    // V tiles and S_prev are stored in 32-byte swizzle, as blocks of 16
    // columns: a V slot is followed by a constant ONES block [C x 16]
    // (columns 0-7 one, 8-15 zero) and S_prev by a z block [rows x 16]
    // (bf16 z | z - bf16(z)).  The MMAs that read V or S_prev then run with
    // N = DV + 16 and leave z, rowsum(P) and phiQ . z_prev in the 16 columns
    // after S or NUM: no separate narrow products (one tcgen05.mma costs
    // about the same for N = 16 as for N = 144 with these operands).
    static constexpr int NQ16 = DV + 16;
    static constexpr int VB = kC * NQ16 * 2;   // one V slot: DV / 16 blocks + ONES
    // The segment-sum form (SUMF; and DP = 256, both halves of a 256-feature
    // map at once, which runs only in that form) has no Q ring and no S_prev
    // buffer: its K and V rings take the space (three stages at D = Dv = 128
    // instead of two)
    static constexpr bool kSumOnly = DP > 128 || SUMF;
    // The segment-sum form at D = Dv = 64 issues one N = Dv + 16 product per K
    // step (else one N = Dv and one N = 16 product; its chunks are bound by
    // the issue of their products): V stays one 128-byte-swizzled 64-column
    // box (one TMA request per tile) and a shared ONES block in the same
    // layout is the operand's second 64-column block (its first 16 columns
    // read), reached through the descriptor's block stride
    static constexpr bool kOnesAgg = SUMF && DP == 64 && DV == 64;
    static constexpr int OB128 = kOnesAgg ? kC * 128 : 0;   // the shared ONES block
    // S_prev pieces along Dphi: one, or two 64-row halves when that is what
    // lets two-deep rings fit (each piece with its own z block)
    static constexpr int NSP = kSumOnly || (2 * (2 * QB + VB) + DP * NQ16 * 2 <= kBudget) ? 1 : 2;
    static constexpr int PR = DP / NSP;      // S_prev rows per piece
    static constexpr int SB = kSumOnly ? 0 : PR * NQ16 * 2;
    static constexpr int kFixed = SB + OB128;
    static constexpr int STAGE = (kSumOnly ? 1 : 2) * QB + VB;   // ring bytes per stage
    static constexpr int NS = (kFixed + 4 * STAGE <= kBudget)   ? 4
                              : (kFixed + 3 * STAGE <= kBudget) ? 3
                                                                : 2;
    static_assert(kFixed + 2 * STAGE <= kBudget, "no two-deep rings");
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + (kSumOnly ? 0 : NS * QB);
    static constexpr int V0 = K0 + NS * QB;
    static constexpr int ONES0 = V0 + NS * VB;   // segment-sum form at D = Dv = 64: the shared ONES block
    static constexpr int S0 = ONES0 + OB128;      // S_prev (and its z block)
    static constexpr int TILES = S0 + SB;
    static constexpr int SMEM = TILES + 1024 /* alignment */ + 1024 /* barriers */;
    // TMEM columns: state S | z; the regions R0, R1 (A, then NUM | DEN of
    // alternate chunks); the bf16 P.  Region stride: A (128 columns), then
    // NUM | DEN (DV + 16)
    static constexpr int RS = NQ16 > kC ? NQ16 : kC;
    static constexpr int T_S = 0, T_Z = DV;                // S | z
    static constexpr int T_R0 = DV == 128 ? 144 : DV + 64;  // regions R0, R1
    static constexpr int T_P = T_R0 + 2 * RS;               // the bf16 P
    // 32-column TMEM accesses at multiples of 32 use one x32 op, else two x16
    static constexpr bool ALN32 = T_R0 % 32 == 0 && RS % 32 == 0 && T_P % 32 == 0;
    // segment-sum form: the segment's S | z (one block of DV + 16 columns per
    // 128 feature rows) in one of two regions that alternate between items
    static constexpr int NRB = DP > 128 ? DP / 128 : 1;
    static constexpr int SUM_COL0 = kSumOnly ? 0 : T_R0;
    static constexpr int SUM_STRIDE = kSumOnly ? NRB * NQ16 : RS;
    static constexpr bool SUM_ALN32 = kSumOnly ? false : ALN32;
    static constexpr int TMEM_COLS = 512;
    static_assert(T_P + kC / 2 <= TMEM_COLS, "TMEM plan too large");
    static_assert(SUM_COL0 + 2 * SUM_STRIDE <= TMEM_COLS, "TMEM plan too large");
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
    static_assert(SMEM > 114 * 1024, "one CTA per SM: the kernel holds all 512 TMEM columns");
};

struct Geo {
    int BH, N, NC;   // heads, positions, chunks per head
    int L, nseg;     // chunks per segment, segments per head
    int n_items;     // items of this launch: B*H*(nseg-1) (aggregate form) or B*H*nseg
    int exp_rows;    // rows per head of the exported state S_out / z_out (>= DP)
};

struct Scratch {
    int *ticket;     // next item to hand out
    int *abort;      // raised by any CTA whose wait ran out
    float *preS;     // [BH, nseg, DP, DV]: segment sums, then their exclusive prefixes
    float *prez;     // [BH, nseg, DP]
    float *num_part; // [BH, N, DV] fp32: first feature half's NUM (split feature maps)
    float *den_part; // [BH, N]
    int pre_rows;    // feature rows per prefix slot (split feature maps: both halves' rows,
    int pre_off;     // this pass's from row pre_off); else DP and 0
    // Non-causal readout: nsum > 0 means preS / prez hold nsum per-segment sums
    // per head ([BH, nsum, DP, DV], [BH, nsum, DP]) that the readout adds up
    // itself (the CTAs of segment 0 also write the totals to exS / exz when
    // given); nsum = 0 means they hold the totals ([BH, DP, DV], [BH, DP]).
    int nsum;
    float *exS;
    float *exz;
};

// What the kernel applies to the Q and K tiles and how it finishes a chunk.
//   kModeElu       phi = elu + 1 on the tiles; out = NUM / DEN
//   kModeFeat      the tiles already hold phi(q), phi(k); out = NUM / DEN
//   kModeFeatPart  phi tiles of the first half of a feature map split in two:
//                  NUM, DEN (un-normalised) -> num_part, den_part
//   kModeFeatComb  the second half: out = (NUM + num_part) / (DEN + den_part)
// A feature map of Dphi = 2 x 128 thus runs as two passes whose sums over
// features add up exactly to the single-pass ones.
enum { kModeElu = 0, kModeFeat = 1, kModeFeatPart = 2, kModeFeatComb = 3 };

struct Ctl {
    volatile int *cta;     // shared abort word of this CTA
    volatile int *glob;    // per-launch abort word
    int *err;              // library error word
};

__device__ __forceinline__ void raise_abort(const Ctl &c)
{
    atomicExch(c.err, kErrTimeout);
    *c.cta = 1;
    *c.glob = 1;
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

// wait_bar for a lane that shares its warp with another waiting role: naps
// between polls so that the other lane keeps the warp's issue slots.
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

// Element (row r, 16 B chunk j) of a [kC x cols] 128B-swizzled tile.
__device__ __forceinline__ uint32_t tile_off(int r, int j)
{
    return (uint32_t)(j >> 3) * (kC * 128) + sw128_off(r, j & 7);
}

// elu + 1 in place on 16 B chunks [J0, J1) of row r of a [kC x cols] tile;
// rows marked `zero` (past the sequence end) become zero instead.
template <int J0, int J1>
__device__ __forceinline__ void phi_cols(uint32_t t, int r, bool zero)
{
    // (kept rolled: 16 warps of four roles share the SM's instruction caches,
    // and the fully unrolled phi loops cost more in fetch stalls than in loop
    // overhead: the long forward ran 13% faster rolled)
#pragma unroll 1
    for (int h = J0; h < J1; h += 8) {
        constexpr int kMax = 8;
        uint4 x[kMax];
#pragma unroll
        for (int j = 0; j < kMax; j++)
            if (h + j < J1) x[j] = lds128(t + tile_off(r, h + j));
#pragma unroll
        for (int j = 0; j < kMax; j++)
            if (h + j < J1) sts128(t + tile_off(r, h + j), zero ? make_uint4(0, 0, 0, 0) : phi_elu1_bf16x8(x[j]));
    }
}

// One S_prev row block: 32 fp32 state values -> bf16 at row r, columns
// [c0, c0 + 32) of an MN-major [PR x DV] piece in 32-byte swizzle (blocks of
// 16 columns, PR * 32 bytes apart).
template <int PR>
__device__ __forceinline__ void sprev_store32_sw32(uint32_t st, int r, int c0, const uint32_t (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int col = c0 + 8 * j;
        const uint32_t a = st + (uint32_t)(col >> 4) * (PR * 32) + sw32_off(r, (col >> 3) & 1);
        sts128(a, make_uint4(
                      pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]))));
    }
}

// 32 TMEM columns from a 16-aligned column address (one x32 access when the
// plan keeps it 32-aligned, else two x16).
template <bool A32>
__device__ __forceinline__ void tmem_ld32c(uint32_t taddr, uint32_t (&r)[32])
{
    if constexpr (A32)
        tmem_ld32_nowait(taddr, r);
    else
        tmem_ld32x2_nowait(taddr, r);
}
template <bool A32>
__device__ __forceinline__ void tmem_st32c(uint32_t taddr, const uint32_t (&r)[32])
{
    if constexpr (A32)
        tmem_st32_nowait(taddr, r);
    else
        tmem_st32x2_nowait(taddr, r);
}

// z (fp32) -> one row of ZP: columns 0-7 bf16(z), 8-15 bf16(z - bf16(z)).
__device__ __forceinline__ void zp_store(uint32_t zp, int r, float z)
{
    const float hi = __bfloat162float(__float2bfloat16_rn(z));
    const uint32_t h = pack_bf16x2(hi, hi), l = pack_bf16x2(z - hi, z - hi);
    sts128(zp + sw32_off(r, 0), make_uint4(h, h, h, h));
    sts128(zp + sw32_off(r, 1), make_uint4(l, l, l, l));
}

// ---------------------------------------------------------------- kernel

template <int DP, int DV, bool AGG, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
tc_causal_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 Geo g, Scratch sc,
                 __nv_bfloat16 *__restrict__ out, float *__restrict__ S_out,
                 float *__restrict__ z_out, int *err)
{
    using PL = Plan<DP, DV, AGG>;
    constexpr int NS = PL::NS, NSP = PL::NSP, PR = PL::PR;
    constexpr int HALF = DV / 2;   // state / NUM columns per TMEM warp
    constexpr bool kPhi = MODE == kModeElu;   // apply elu + 1 to the Q and K tiles in place
    static_assert(MODE != kModeFeatComb || HALF == 32, "the split feature map takes Dv = 64");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));   // generic view of `base`
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *q_full = bar, *q_ready = bar + 4, *q_empty = bar + 8;
    uint64_t *k_full = bar + 12, *k_ready = bar + 16, *k_empty = bar + 20;
    uint64_t *v_full = bar + 24, *v_empty = bar + 28;
    uint64_t *item_full = bar + 32, *item_empty = bar + 34;
    uint64_t *sp_ready = bar + 36;   // [2] S_prev piece written
    uint64_t *a_full = bar + 38, *a_free = bar + 39, *p_ready = bar + 40, *sp_free = bar + 41,
             *s_done = bar + 42, *num_full = bar + 43, *sloc_done = bar + 45, *drain = bar + 46;
    uint64_t *sloc_read = bar + 47;   // [2] aggregate form: the sums in region r have been read
    uint64_t *num_free = bar + 53;   // [2]: the epilogue has read NUM from region r
    uint64_t *out_ready = bar + 56;  // [NS]: the output tile of a chunk is in its V slot
    volatile int *item_slot = reinterpret_cast<volatile int *>(bar + 50);   // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 51);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(bar + 52);   // bar + 53, 54: num_free
    const Ctl ctl{abort_cta, sc.abort, err};

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // the segment-sum form is followed by the scan or the totals, launched as
    // its dependents (every block of this grid is resident by now)
    if constexpr (AGG) griddep_launch();

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_ready[i], kTmemWarps);
            mbar_init(&q_empty[i], 1);
            mbar_init(&k_full[i], 1);
            mbar_init(&k_ready[i], AGG && kPhi ? kPhiWarps + kTmemWarps : kPhiWarps);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], AGG ? kItemConsumers - 1 : kItemConsumers);   // no store lane in AGG
            mbar_init(&sp_ready[i], NSP == 1 ? kTmemWarps : kTmemWarps / 2);
        }
        mbar_init(a_full, 1);
        mbar_init(a_free, kTmemWarps);
        mbar_init(p_ready, kTmemWarps);
        mbar_init(sp_free, 1);
        mbar_init(s_done, 1);
        mbar_init(num_full, 1);
        mbar_init(&num_free[0], kTmemWarps);
        mbar_init(&num_free[1], kTmemWarps);
        for (int i = 0; i < NS; i++) mbar_init(&out_ready[i], kTmemWarps);
        mbar_init(&sloc_read[0], kTmemWarps);
        mbar_init(&sloc_read[1], kTmemWarps);
        mbar_init(sloc_done, 1);
        mbar_init(drain, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp < kTmemWarps && PL::kOnesAgg) {   // the shared ONES block: columns 0-7 one, the rest zero
        const uint32_t one = pack_bf16x2(1.f, 1.f);
        for (int i = threadIdx.x; i < kC * 8; i += kTmemWarps * 32) {
            const int r = i / 8, c = i % 8;
            sts128(base + PL::ONES0 + sw128_off(r, c), c == 0 ? make_uint4(one, one, one, one) : make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
    } else if (warp < kTmemWarps) {   // the ONES block after every V slot's DV / 16 blocks (never loaded over)
        const uint32_t one = pack_bf16x2(1.f, 1.f);
        for (int i = threadIdx.x; i < NS * kC; i += kTmemWarps * 32) {
            const int st = i / kC, r = i % kC;
            const uint32_t blk = base + PL::V0 + st * PL::VB + (DV / 16) * (kC * 32);
            sts128(blk + sw32_off(r, 0), make_uint4(one, one, one, one));
            sts128(blk + sw32_off(r, 1), make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kProducerWarp || warp == kKWarp || warp == kVWarp) {
        // ---------------------------------------- Q / K / V tile producers
        // The Q producer also hands out the items (the K producer in the
        // segment-sum form).  The segment-sum form streams a segment's K, V; the output form streams its Q, K, V (K
        // and V a second time: the two passes are too far apart for L2 to
        // keep them).
        if (lane == 0) {
            const int role = warp - kProducerWarp;   // 0 Q, 1 K, 2 V
            const CUtensorMap *tm = role == 0 ? &tm_q : role == 1 ? &tm_k : &tm_v;
            // boxes per tile, their width and stride: V of the output form in 16-column
            // boxes (32-byte swizzle); Q, K and the segment-sum form's V in 64-column
            // boxes (128-byte swizzle: fewer, longer rows per TMA request)
            constexpr bool kV32 = !AGG;
            const int nb = role == 2 ? (kV32 ? DV / 16 : DV / 64) : DP / 64;
            const int bw = role == 2 && kV32 ? 16 : 64;
            const int bs = role == 2 && kV32 ? kC * 32 : kC * 128;
            const int tb = role == 2 ? PL::VB : PL::QB;     // slot stride in the ring
            const int tx = role == 2 ? kC * DV * 2 : PL::QB;  // bytes one tile load brings (a fused V
                                                            // slot also holds the constant ONES block)
            unsigned char *ring = gbase + (role == 0 ? PL::Q0 : role == 1 ? PL::K0 : PL::V0);
            uint64_t *full = role == 0 ? q_full : role == 1 ? k_full : v_full;
            uint64_t *empty = role == 0 ? q_empty : role == 1 ? k_empty : v_empty;
            prefetch_tmap(tm);
            const uint64_t stream = policy_evict_first();
            uint32_t n = 0;
            bool ok = true;
            auto prefetch = [&](int head, int chunk) {
                for (int b = 0; b < nb; b++) tma_prefetch_3d(tm, b * bw, chunk * kC, head);
            };
            auto load = [&](int head, int chunk, uint64_t pol) {
                const int st = n % NS;
                if (n >= NS && !wait_bar(&empty[st], ((n / NS) - 1) & 1, ctl)) return false;
                mbar_arrive_expect_tx(&full[st], tx);
                for (int b = 0; b < nb; b++)
                    tma_load_3d_hint(ring + st * tb + b * bs, tm, &full[st], b * bw, chunk * kC, head, pol);
                n++;
                return true;
            };
            // Items: CTA b takes item b first, then tickets from the counter
            // (offset by the grid size).  The role that hands them out is one
            // whose loads pace it (Q here; K in the segment-sum form, which
            // reads no Q), so that it takes its next ticket only once the
            // current item's loads are all issued, never one an idle CTA
            // would have taken.
            const int item_role = AGG ? 1 : 0;
            for (int it = 0; ok; it++) {
                const int slot = it & 1;
                int item = -1;
                if (role == item_role) {
                    ok = it < 2 || wait_bar(&item_empty[slot], ((it >> 1) - 1) & 1, ctl);
                    // no new item once any CTA of this launch has given up a wait
                    // (with no more items than CTAs, no ticket and no shared abort word is
                    // read: the header need not be cleared for such a launch)
                    const bool dyn = g.n_items > (int)gridDim.x;
                    if (ok && !*abort_cta && (!dyn || !*ctl.glob)) {
                        item = it == 0 ? (int)blockIdx.x : dyn ? (int)gridDim.x + atomicAdd(sc.ticket, 1) : -1;
                        if (item >= g.n_items) item = -1;
                    }
                    item_slot[slot] = item;
                    mbar_arrive(&item_full[slot]);
                } else {
                    if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
                    item = item_slot[slot];
                    mbar_arrive(&item_empty[slot]);
                }
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                if (AGG && role == 0) continue;   // the aggregate form reads no Q
                for (int c = 0; c < nc && c < kPrefetch; c++) prefetch(h, c0 + c);
                for (int c = 0; c < nc && ok; c++) {
                    if (c + kPrefetch < nc) prefetch(h, c0 + c + kPrefetch);
                    ok = load(h, c0 + c, stream);
                }
            }
            // drain loads still in flight (only possible after an abort)
            for (uint32_t m = n > NS ? n - NS : 0; m < n; m++)
                mbar_wait(&full[m % NS], (m / NS) & 1, nullptr, 0);
        }
        if (!AGG && warp == kVWarp && lane == 1) {
            // ------------------------------------------ output tile stores
            prefetch_tmap(&tm_o);
            uint32_t nv = 0;        // V ring position
            uint32_t oc[4] = {0, 0, 0, 0};   // output tiles seen per V slot
            for (int it = 0;; it++) {
                const int slot = it & 1;
                if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
                const int item = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                for (int c = 0; c < nc; c++, nv++) {
                    const int st = nv % NS;
                    const bool ok = wait_bar_nap(&out_ready[st], oc[st] & 1, ctl);
                    oc[st]++;
                    if (ok && MODE != kModeFeatPart) {
                        const uint32_t src = base + PL::V0 + st * PL::VB;
#pragma unroll
                        for (int b = 0; b < DV / 64; b++)
                            tma_store_3d(&tm_o, src + b * kC * 128, b * 64, (c0 + c) * kC, h);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                    mbar_arrive(&v_empty[st]);
                }
            }
            bulk_wait_all();
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kC, 0, 0);
            // N = DV + 16: the z / denominator columns ride on every product with V or S_prev
            constexpr uint32_t id_qs = idesc_bf16(128, PL::NQ16, 0, 1);
            constexpr uint32_t id_kv = idesc_bf16(128, PL::NQ16, 1, 1);
            constexpr uint32_t lbo_v = kC * 32, lbo_s = PR * 32;   // 16-column block strides (32B swizzle)
            constexpr uint32_t lbo_kT = DP >= 128 ? kC * 128 : 0;   // DP = 64: rows 64-127 repeat 0-63
            const uint32_t s_addr = base + PL::S0;
            uint32_t nkv = 0;    // K / V ring loads consumed
            uint32_t nq = 0;     // Q ring loads consumed
            uint32_t ndone = 0;  // phase-C chunks whose MMA2 has been issued (global chunk index)
            uint32_t nfree[2] = {0, 0};   // num_free phases seen per region
            // region r = k % 2 is free once the epilogue of chunk k has read NUM
            auto wait_epi = [&](uint32_t k) {
                const int rr = k & 1;
                const uint32_t ph = k >> 1;
                if (nfree[rr] <= ph) {
                    wait_bar(&num_free[rr], ph & 1, ctl);
                    nfree[rr] = ph + 1;
                }
            };
            // MMA1(k): A = phiQ phiK^T into region k % 2
            auto mma1 = [&](uint32_t k, uint32_t qn, uint32_t kn) {
                if (k >= 2) wait_epi(k - 2);
                wait_bar(&q_ready[qn % NS], (qn / NS) & 1, ctl);
                wait_bar(&k_ready[kn % NS], (kn / NS) & 1, ctl);
                tc_fence_after();
                const uint32_t qa = base + PL::Q0 + (qn % NS) * PL::QB;
                const uint32_t ka = base + PL::K0 + (kn % NS) * PL::QB;
                const uint32_t dst = tmem + PL::T_R0 + (k & 1) * PL::RS;
                if (!*abort_cta) {
#pragma unroll
                    for (int kk = 0; kk < DP; kk += 16) {
                        const uint32_t off = (kk / 64) * (kC * 128) + (kk % 64) * 2;
                        mma_bf16_ss(dst, sw128_desc(qa + off, 16, 1024), sw128_desc(ka + off, 16, 1024),
                                    id_qk, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(a_full);
            };
            for (int it = 0;; it++) {
                const int slot = it & 1;
                if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
                const int item = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const int s = item / g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                if constexpr (AGG) {
                    // the segment's sums S_loc, z_loc into region it % 2 and its
                    // denominator slot, once the TMEM warps have read item it - 2's
                    const int rr = it & 1;
                    if (it >= 2) wait_bar(&sloc_read[rr], ((it >> 1) - 1) & 1, ctl);
                    const uint32_t dS = tmem + PL::SUM_COL0 + rr * PL::SUM_STRIDE;   // S | z of the segment
                    for (int c = 0; c < nc; c++) {
                        const int st = nkv % NS;
                        wait_bar(&k_ready[st], (nkv / NS) & 1, ctl);
                        wait_bar(&v_full[st], (nkv / NS) & 1, ctl);
                        tc_fence_after();
                        const uint32_t ka = base + PL::K0 + st * PL::QB;
                        const uint32_t va = base + PL::V0 + st * PL::VB;
                        if (!*abort_cta && PL::kOnesAgg) {
                            // S | z += phiK^T [V | ONES]: the shared ONES block is the second
                            // 64-column block of the operand, lbo bytes after this V slot
                            constexpr uint32_t id_kv = idesc_bf16(128, PL::NQ16, 1, 1);
                            const uint32_t lbo_ones = base + PL::ONES0 - va;
#pragma unroll
                            for (int k = 0; k < kC; k += 16)
                                mma_bf16_ss(dS, sw128_desc(ka + (k / 8) * 1024, lbo_kT, 1024),
                                            sw128_desc(va + (k / 8) * 1024, lbo_ones, 1024), id_kv,
                                            (c > 0 || k > 0) ? 1u : 0u);
                        } else if (!*abort_cta) {
                            // (V in 128-byte swizzle here; z from the slot's ONES block)
                            constexpr uint32_t id_s = idesc_bf16(128, DV, 1, 1);
                            constexpr uint32_t id_z = idesc_bf16(128, 16, 1, 1);
                            const uint32_t ones = va + DV * kC * 2;
#pragma unroll
                            for (int rb = 0; rb < PL::NRB; rb++) {   // 128 feature rows (two K boxes) each
                                const uint32_t kb = ka + rb * 2 * (kC * 128), d = dS + rb * PL::NQ16;
#pragma unroll
                                for (int k = 0; k < kC; k += 16)
                                    mma_bf16_ss(d, sw128_desc(kb + (k / 8) * 1024, lbo_kT, 1024),
                                                sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_s,
                                                (c > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                                for (int k = 0; k < kC; k += 16)
                                    mma_bf16_ss(d + DV, sw128_desc(kb + (k / 8) * 1024, lbo_kT, 1024),
                                                sw32_desc(ones + (k / 8) * 256, 256, 256), id_z,
                                                (c > 0 || k > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit(&k_empty[st]);
                        mma_commit(&v_empty[st]);
                        nkv++;
                    }
                    mma_commit(sloc_done);
                    continue;
                }
                const uint32_t G = ndone;   // global index of this item's first chunk
                // phase C: MMA1(G); then per chunk k: MMA3(k), MMA4(k), MMA1(k+1), MMA2(k)
                mma1(G, nq, nkv);
                for (int c = 0; c < nc; c++) {
                    const uint32_t k = G + c;
                    const int qs = nq % NS, st = nkv % NS;
                    const uint32_t qa = base + PL::Q0 + qs * PL::QB;
                    const uint32_t ka = base + PL::K0 + st * PL::QB;
                    const uint32_t va = base + PL::V0 + st * PL::VB;
                    const uint32_t rnum = tmem + PL::T_R0 + (k & 1) * PL::RS;   // NUM | DEN
                    // MMA3: NUM | DEN = phiQ [S_prev | z_prev] (A(k) has been read)
                    wait_bar(a_free, k & 1, ctl);
#pragma unroll
                    for (int pc = 0; pc < NSP; pc++) {
                        wait_bar(&sp_ready[pc], k & 1, ctl);
                        tc_fence_after();
                        if (!*abort_cta) {
#pragma unroll
                            for (int kk = 0; kk < PR; kk += 16) {
                                const int kq = pc * PR + kk;
                                mma_bf16_ss(rnum, sw128_desc(qa + (kq / 64) * (kC * 128) + (kq % 64) * 2, 16, 1024),
                                            sw32_desc(s_addr + (kk / 8) * 256, lbo_s, 256), id_qs,
                                            kq > 0 ? 1u : 0u);
                            }
                        }
                        if (pc + 1 < NSP) mma_commit(sp_free);
                    }
                    mma_commit(&q_empty[qs]);
                    // MMA4: S | z += phiK^T [V | ONES]
                    wait_bar(&v_full[st], (nkv / NS) & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kC; kk += 16)
                            mma_bf16_ss(tmem + PL::T_S, sw128_desc(ka + (kk / 8) * 1024, lbo_kT, 1024),
                                        sw32_desc(va + (kk / 8) * 256, lbo_v, 256), id_kv, 1u);
                    }
                    mma_commit(s_done);
                    mma_commit(&k_empty[st]);
                    // MMA1(k+1) into the other region
                    if (c + 1 < nc) mma1(k + 1, nq + 1, nkv + 1);
                    // MMA2: NUM | DEN += P [V | ONES]  (P in TMEM)
                    wait_bar(p_ready, k & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < kC; kk += 16)
                            mma_bf16_ts(rnum, tmem + PL::T_P + kk / 2, sw32_desc(va + (kk / 8) * 256, lbo_v, 256),
                                        id_qs, 1u);
                    }
                    mma_commit(num_full);
                    nq++;
                    nkv++;
                    ndone++;
                }
            }
            mma_commit(drain);   // every MMA issued above has completed
            mbar_wait(drain, 0, nullptr, 0);
        }
    } else if (warp >= kTmemWarps) {
        // ----------------------------------------------------- phi warps
        const int qd = warp - kTmemWarps;      // lane quadrant
        const int r = qd * 32 + lane;          // tile row
        constexpr int JR = DP / 8;             // 16 B chunks per row
        uint32_t nk = 0;
        // phi in place on row r of a ring tile; all loads issued before any math
        auto phi_tile = [&](uint64_t *full, uint64_t *ready, uint32_t ring, uint32_t &n, bool zero) {
            const int st = n % NS;
            wait_bar(&full[st], (n / NS) & 1, ctl);
            const uint32_t t = ring + st * PL::QB;
            if constexpr (kPhi) {   // (phi tiles arrive from HBM as they are; rows past N are zero-filled)
                // segment-sum form: the idle TMEM warps take the other two thirds of the columns
                phi_cols<0, AGG ? kAggSplit1<JR> : JR>(t, r, zero);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[st]);
            n++;
        };
        for (int it = 0;; it++) {
            const int slot = it & 1;
            if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
            const int item = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const int s = item / g.BH;
            const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
            // rows past the sequence end must add nothing to S, z
            for (int c = 0; c < nc; c++)
                phi_tile(k_full, k_ready, base + PL::K0, nk, r >= g.N - (c0 + c) * kC);
        }
    } else {
        // ----------------------------------------------------- TMEM warps
        const int qd = warp & 3, grp = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const bool srow = qd * 32 < DP;   // warp-uniform: this warp's rows hold state rows
        const int piece = NSP == 1 ? 0 : qd / 2;   // S_prev piece of this warp's rows
        // Warps of the second S_prev piece write it only once MMA3 has read the
        // first, and MMA3(c+1) also needs their a_free(c+1): so they write their
        // piece for chunk c + 1 after load_p(c + 1), between store_p(c + 1) and
        // the epilogue of c.
        const bool late = NSP == 2 && piece == 1;
        const int prow = r - piece * PR;           // row inside the piece
        const uint32_t s_addr = base + PL::S0;
        const uint32_t z_addr = s_addr + (DV / 16) * (PR * 32);   // the z block after S_prev's blocks
        uint32_t kg = 0;      // global index of the next chunk whose A is read
        uint32_t nkt = 0;     // K ring position (segment-sum form: this warp's share of phi(K))
        uint32_t nvr = 0;     // V ring position
        uint32_t nsp = 0;     // S_prev copies made (one per chunk)
        uint32_t nsd = 0;     // s_done phases consumed

        // S_prev piece + ZP rows <- the state in T_S, T_Z; arrives sp_ready.
        auto sprev_from_tmem = [&]() {
            if (NSP == 2 && piece == 1) {   // the buffer holds piece 0 until MMA3 has read it
                wait_bar(sp_free, nsp & 1, ctl);
            }
            tc_fence_after();
            if (srow) {
#pragma unroll 1
                for (int cb = 0; cb < HALF; cb += 32) {
                    uint32_t v[32];
                    tmem_ld32_nowait(tmem + lane_base + PL::T_S + grp * HALF + cb, v);
                    tmem_ld_wait();
                    sprev_store32_sw32<PR>(s_addr, prow, grp * HALF + cb, v);
                }
                if (grp == 0) {
                    uint32_t zv[16];
                    tmem_ld16_nowait(tmem + lane_base + PL::T_Z, zv);
                    tmem_ld_wait();
                    zp_store(z_addr, prow, __uint_as_float(zv[0]));
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && (NSP == 1 || srow)) mbar_arrive(&sp_ready[piece]);
            nsp++;
        };
        // phi(Q) in place on this thread's half row of the next Q tile
        uint32_t nqt = 0;
        auto phi_q = [&]() {
            const int st = nqt % NS;
            wait_bar(&q_full[st], (nqt / NS) & 1, ctl);
            const uint32_t t = base + PL::Q0 + st * PL::QB;
            if constexpr (kPhi) {
                constexpr int JH = DP / 16;   // 16 B chunks per half row
                constexpr int JB = JH > 4 ? 4 : JH;
#pragma unroll 1
                for (int j0 = 0; j0 < JH; j0 += JB) {
                    uint4 x[JB];
#pragma unroll
                    for (int j = 0; j < JB; j++) x[j] = lds128(t + tile_off(r, grp * JH + j0 + j));
#pragma unroll
                    for (int j = 0; j < JB; j++) sts128(t + tile_off(r, grp * JH + j0 + j), phi_elu1_bf16x8(x[j]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_ready[st]);
            nqt++;
        };
        // A(kg) from its region -> registers (masked, packed bf16 P), then a_free
        auto load_p = [&](uint32_t (&pk)[32]) {
            wait_bar(a_full, kg & 1, ctl);
            tc_fence_after();
            const uint32_t ra = tmem + lane_base + PL::T_R0 + (kg & 1) * PL::RS + grp * 64;
            uint32_t a0[32], a1[32];
            tmem_ld32c<PL::ALN32>(ra, a0);
            tmem_ld32c<PL::ALN32>(ra + 32, a1);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(a_free);
            const int cbase = grp * 64;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int col = cbase + 2 * i;
                pk[i] = pack_bf16x2(col <= r ? __uint_as_float(a0[2 * i]) : 0.f,
                                    col + 1 <= r ? __uint_as_float(a0[2 * i + 1]) : 0.f);
                pk[16 + i] = pack_bf16x2(col + 32 <= r ? __uint_as_float(a1[2 * i]) : 0.f,
                                         col + 33 <= r ? __uint_as_float(a1[2 * i + 1]) : 0.f);
            }
            kg++;
        };
        // P -> its TMEM slot (keys [64 grp, 64 grp + 64) -> columns [32 grp, 32 grp + 32))
        auto store_p = [&](const uint32_t (&pk)[32]) {
            tmem_st32c<PL::ALN32>(tmem + lane_base + PL::T_P + grp * 32, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready);
        };
        auto wait_sdone = [&]() {
            const bool ok = __all_sync(0xffffffffu, wait_bar(s_done, nsd & 1, ctl));
            nsd++;
            return ok;
        };

        for (int it = 0;; it++) {
            const int slot = it & 1;
            if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
            const int item = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const int s = item / g.BH, h = item % g.BH;
            const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
            const long long slot_id = (long long)h * g.nseg + s;   // this (head, segment) in scratch
            if constexpr (AGG) {
                if constexpr (kPhi) {
                    // their share of phi(K) on the segment's K tiles (the phi warps do the rest)
                    constexpr int JR = DP / 8;
                    for (int c = 0; c < nc; c++) {
                        const int st = nkt % NS;
                        wait_bar(&k_full[st], (nkt / NS) & 1, ctl);
                        const uint32_t t = base + PL::K0 + st * PL::QB;
                        const bool zero = r >= g.N - (c0 + c) * kC;
                        if (grp == 0)
                            phi_cols<kAggSplit1<JR>, kAggSplit2<JR>>(t, r, zero);
                        else
                            phi_cols<kAggSplit2<JR>, JR>(t, r, zero);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&k_ready[st]);
                        nkt++;
                    }
                }
                // the segment's sums (region it % 2 and its denominator slot) -> scratch
                const int rr = it & 1;
                wait_bar(sloc_done, it & 1, ctl);
                tc_fence_after();
                if (srow) {
#pragma unroll
                    for (int rb = 0; rb < PL::NRB; rb++) {   // feature rows r + 128 rb
                        const int row = r + 128 * rb;
                        const uint32_t src = tmem + lane_base + PL::SUM_COL0 + rr * PL::SUM_STRIDE + rb * PL::NQ16;
                        float4 *dst = reinterpret_cast<float4 *>(sc.preS + slot_id * DP * DV + (long long)row * DV +
                                                                 grp * HALF);
#pragma unroll
                        for (int cb = 0; cb < HALF; cb += 32) {
                            uint32_t l[32];
                            tmem_ld32c<PL::SUM_ALN32>(src + grp * HALF + cb, l);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 8; i++)
                                __stcg(dst + cb / 4 + i,
                                       make_float4(__uint_as_float(l[4 * i]), __uint_as_float(l[4 * i + 1]),
                                                   __uint_as_float(l[4 * i + 2]), __uint_as_float(l[4 * i + 3])));
                        }
                        if (grp == 0) {
                            uint32_t d[16];
                            // z of the segment: the columns after S in the block
                            tmem_ld16_nowait(src + DV, d);
                            tmem_ld_wait();
                            __stcg(sc.prez + slot_id * DP + row, __uint_as_float(d[0]));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sloc_read[rr]);
                continue;
            }
            const uint32_t G = kg;   // global index of chunk 0

            phi_q();   // phi(Q) of chunk 0 first: MMA1 of chunk 0 does not wait for phase B

            // ---- phase B: the state before this segment (the exclusive prefix of
            // the head's earlier segments; zero for the first) -> T_S, T_Z.  The
            // scan that writes the prefixes may still be running (this pass is its
            // dependent launch): wait for it here, after this warp's first phi(Q).
            griddep_wait();
            // (split feature maps: the prefix slots hold both halves' feature rows)
            const int prs = MODE >= kModeFeatPart ? sc.pre_rows : DP, pro = MODE >= kModeFeatPart ? sc.pre_off : 0;
            if (srow) {
                const float4 *src = reinterpret_cast<const float4 *>(sc.preS + slot_id * prs * DV +
                                                                     (long long)(pro + r) * DV + grp * HALF);
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float4 pv = s > 0 ? __ldcg(src + cb / 4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[4 * i] = __float_as_uint(pv.x);
                        v[4 * i + 1] = __float_as_uint(pv.y);
                        v[4 * i + 2] = __float_as_uint(pv.z);
                        v[4 * i + 3] = __float_as_uint(pv.w);
                    }
                    tmem_st32_nowait(tmem + lane_base + PL::T_S + grp * HALF + cb, v);
                }
                if (grp == 0) {
                    const float zprev = s > 0 ? __ldcg(sc.prez + slot_id * prs + pro + r) : 0.f;
                    uint32_t zw[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) zw[i] = i < 8 ? __float_as_uint(zprev) : 0u;
                    tmem_st16_nowait(tmem + lane_base + PL::T_Z, zw);
                }
            }
            tmem_st_wait();
            if (!late) sprev_from_tmem();   // S_prev, ZP for chunk 0, read back from T_S, T_Z

            // ---- phase C.  Prologue: P(G).  Then per chunk k = G + c, in the
            // order the tensor pipe completes their inputs: phi(Q(k+1)); S_prev
            // for k + 1 (after MMA4(k)); A(k+1) -> registers (after MMA1(k+1));
            // P(k+1) and the epilogue of k (after MMA2(k)).
            uint32_t pk[32];
            load_p(pk);
            store_p(pk);   // the P slot is free: the last MMA2 has completed
            if (late) sprev_from_tmem();
            for (int c = 0; c < nc; c++) {
                const uint32_t k = G + c;
                const int row0 = (c0 + c) * kC;
                const bool more = c + 1 < nc;
                bool sd = true;
                if constexpr (MODE == kModeFeatComb) {
                    // the first half's sums for this chunk's rows: into L2 now, read at the epilogue
                    if (row0 + r < g.N) {
                        const long long pr = (long long)h * g.N + row0 + r;
                        prefetch_l2(sc.num_part + pr * DV + grp * HALF);
                        if (grp == 0 && lane == 0) prefetch_l2(sc.den_part + pr);
                    }
                }
                if (more) {
                    phi_q();
                    wait_sdone();
                    if (!late) sprev_from_tmem();
                    load_p(pk);
                }
                const bool ok = __all_sync(0xffffffffu, wait_bar(num_full, k & 1, ctl));
                if (more) store_p(pk);
                if (more && late) sprev_from_tmem();
                tc_fence_after();
                const uint32_t rn = tmem + lane_base + PL::T_R0 + (k & 1) * PL::RS + grp * HALF;
                uint32_t d[16], n0[32], n1[32];
                tmem_ld16_nowait(tmem + lane_base + PL::T_R0 + (k & 1) * PL::RS + DV, d);   // DEN
                tmem_ld32c<PL::ALN32>(rn, n0);
                if constexpr (HALF == 64) tmem_ld32c<PL::ALN32>(rn + 32, n1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&num_free[k & 1]);
                {   // out(k) = NUM / (DEN[0] + DEN[8]) -> the V slot of chunk k (bf16, swizzled)
                    const int vs = nvr % NS;
                    const int pos = row0 + r;                 // this thread's position in the head
                    const long long prow = (long long)h * g.N + pos;
                    float den = __uint_as_float(d[0]) + __uint_as_float(d[8]);
                    if constexpr (MODE == kModeFeatPart) {
                        // first feature half: the un-normalised sums -> scratch
                        if (pos < g.N) {
                            float4 *dst = reinterpret_cast<float4 *>(sc.num_part + prow * DV + grp * HALF);
#pragma unroll
                            for (int i = 0; i < 8; i++)
                                __stcg(dst + i, make_float4(__uint_as_float(n0[4 * i]), __uint_as_float(n0[4 * i + 1]),
                                                            __uint_as_float(n0[4 * i + 2]),
                                                            __uint_as_float(n0[4 * i + 3])));
                            if constexpr (HALF == 64) {
#pragma unroll
                                for (int i = 0; i < 8; i++)
                                    __stcg(dst + 8 + i,
                                           make_float4(__uint_as_float(n1[4 * i]), __uint_as_float(n1[4 * i + 1]),
                                                       __uint_as_float(n1[4 * i + 2]), __uint_as_float(n1[4 * i + 3])));
                            }
                            if (grp == 0) __stcg(sc.den_part + prow, den);
                        }
                    } else {
                        if constexpr (MODE == kModeFeatComb) {
                            // second feature half: add the first half's sums (HALF = 32)
                            if (pos < g.N) {
                                const float4 *src = reinterpret_cast<const float4 *>(sc.num_part + prow * DV + grp * HALF);
#pragma unroll
                                for (int i = 0; i < 8; i++) {
                                    const float4 a = __ldcg(src + i);
                                    n0[4 * i] = __float_as_uint(__uint_as_float(n0[4 * i]) + a.x);
                                    n0[4 * i + 1] = __float_as_uint(__uint_as_float(n0[4 * i + 1]) + a.y);
                                    n0[4 * i + 2] = __float_as_uint(__uint_as_float(n0[4 * i + 2]) + a.z);
                                    n0[4 * i + 3] = __float_as_uint(__uint_as_float(n0[4 * i + 3]) + a.w);
                                }
                                den += __ldcg(sc.den_part + prow);
                            }
                        }
                        const float inv = 1.f / den;
                        const uint32_t vt = base + PL::V0 + vs * PL::VB + (grp * HALF / 64) * (kC * 128);
                        auto put = [&](const uint32_t(&v)[32], int j0) {
#pragma unroll
                            for (int j = 0; j < 4; j++)
                                sts128(vt + sw128_off(r, j0 + j),
                                       make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]) * inv,
                                                              __uint_as_float(v[8 * j + 1]) * inv),
                                                  pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv,
                                                              __uint_as_float(v[8 * j + 3]) * inv),
                                                  pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv,
                                                              __uint_as_float(v[8 * j + 5]) * inv),
                                                  pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv,
                                                              __uint_as_float(v[8 * j + 7]) * inv)));
                        };
                        // HALF = 64: this warp's half is one whole 64-column block;
                        // HALF = 32: half a block, starting at chunk 4 * (grp % 2)
                        put(n0, HALF == 64 ? 0 : 4 * grp);
                        if constexpr (HALF == 64) put(n1, 4);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&out_ready[vs]);
                    nvr++;
                }
                (void)ok;
                if (!more) sd = wait_sdone();   // the last chunk's state update
                // the head's final state after its last chunk
                if (!more && sd && s == g.nseg - 1 && srow && (S_out || z_out)) {
                    tc_fence_after();
#pragma unroll
                    for (int cb = 0; cb < HALF; cb += 32) {
                        uint32_t v[32];
                        tmem_ld32_nowait(tmem + lane_base + PL::T_S + grp * HALF + cb, v);
                        tmem_ld_wait();
                        if (S_out) {
                            float *dst = S_out + ((long long)h * g.exp_rows + r) * DV + grp * HALF + cb;
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(dst + i) =
                                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                        }
                    }
                    if (z_out && grp == 0) {
                        uint32_t zv[16];
                        tmem_ld16_nowait(tmem + lane_base + PL::T_Z, zv);
                        tmem_ld_wait();
                        z_out[(long long)h * g.exp_rows + r] = __uint_as_float(zv[0]);
                    }
                }
            }
            tc_fence_before();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// ------------------------------------------------ non-causal readout kernel
//
// The non-causal form (review page "Transformers are RNNs", proposed method
// b2: by associativity phi(K)^T V is formed once and reused by every query):
// the segment-sum form of the kernel above, run over every segment, gives the
// per-segment sums; nc_total_kernel adds them into S = phi(K)^T V and
// z = colsum phi(K) per head; this kernel reads them out for every query,
//   out = (phi(Q) S) / (phi(Q) z),
// one tcgen05 product per 128-position chunk (NUM = phiQ . S, DEN = phiQ . ZP)
// into one of two TMEM regions that alternate between chunks.
// Roles (10 warps): 8 math warps (phi(Q) in place; S, ZP per item; the
// epilogue), one producer warp (lane 0: Q tiles and items; lane 1: TMA stores
// of the output tiles from a staging ring), one MMA warp.

constexpr int kNcMath = 8;
constexpr int kNcProducer = kNcMath;          // warp 8
constexpr int kNcMma = kNcMath + 1;           // warp 9
constexpr int kNcThreads = (kNcMma + 1) * 32; // 320
constexpr int kNcItemConsumers = kNcMath + 2; // math warps, MMA thread, store lane

template <int DP, int DV>
struct NcPlan {
    static constexpr int QB = kC * DP * 2;
    static constexpr int OB = kC * DV * 2;
    // S in 32-byte swizzle (16-column blocks, DP * 32 bytes apart) followed by
    // the z block (bf16 z | z - bf16(z)): one N = DV + 16 product gives NUM | DEN
    static constexpr int NQ16 = DV + 16;
    static constexpr int SB = DP * NQ16 * 2;
    static constexpr int ZB = 0;
    static constexpr int NO = 2;
    // D = Dv = 64: two CTAs per SM (half the shared memory and TMEM each), so
    // that one CTA's per-chunk chain overlaps the other's; else one per SM
    static constexpr bool kTwo = DP == 64 && DV == 64;
    static constexpr int kBudget = kTwo ? 113 * 1024 - 2048 : 227 * 1024 - 2048;
    static constexpr int NQ0 = (kBudget - NO * OB - SB - ZB) / QB;
    static constexpr int NQ = NQ0 > 6 ? 6 : NQ0;   // Q ring depth: what fits, at most 6
    static_assert(NQ >= 2, "Q ring too shallow");
    static constexpr int Q0 = 0;
    static constexpr int O0 = Q0 + NQ * QB;
    static constexpr int S0 = O0 + NO * OB;
    static constexpr int Z0 = S0 + SB;
    static constexpr int TILES = Z0 + ZB;
    static constexpr int SMEM = TILES + 1024 + 1024;
    // TMEM: region r at column RS r holds NUM | DEN (DV + 16 columns)
    static constexpr int RS = NQ16 > kC ? NQ16 : kC;
    static constexpr bool ALN32 = RS % 32 == 0;
    static constexpr int TMEM_COLS = kTwo ? 256 : 512;
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
    static_assert(kTwo ? SMEM <= 113 * 1024 && 2 * RS <= TMEM_COLS
                       : SMEM > 114 * 1024, "CTAs per SM: shared memory and TMEM shares disagree");
};

template <int DP, int DV, bool PHI>
__global__ void __launch_bounds__(kNcThreads, NcPlan<DP, DV>::kTwo ? 2 : 1)
nc_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_o, Geo g,
              Scratch sc, int *err)
{
    using PL = NcPlan<DP, DV>;
    constexpr int NQ = PL::NQ, NO = PL::NO;
    constexpr int HALF = DV / 2;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));
    // barrier map: three Q-ring arrays of NQ, then fixed pairs and words
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *q_full = bar, *q_ready = bar + NQ, *q_empty = bar + 2 * NQ;
    uint64_t *num_full = bar + 3 * NQ, *num_free = num_full + 2;   // [2] per region
    uint64_t *out_ready = num_free + 2, *out_free = out_ready + NO;  // [NO]
    uint64_t *item_full = out_free + NO, *item_empty = item_full + 2;
    uint64_t *s_ready = item_empty + 2, *s_free = s_ready + 1, *drain = s_free + 1;
    volatile int *item_slot = reinterpret_cast<volatile int *>(drain + 1);   // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 2);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(drain + 3);
    static_assert((3 * NQ + 4 + 2 * NO + 4 + 3 + 3) * 8 <= 1024, "barrier map exceeds its 1 KB");
    const Ctl ctl{abort_cta, sc.abort, err};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NQ; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_ready[i], kNcMath);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&num_full[i], 1);
            mbar_init(&num_free[i], kNcMath);
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], kNcItemConsumers);
        }
        for (int i = 0; i < NO; i++) {
            mbar_init(&out_ready[i], kNcMath);
            mbar_init(&out_free[i], 1);
        }
        mbar_init(s_ready, kNcMath);
        mbar_init(s_free, 1);
        mbar_init(drain, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp == kNcMma) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // the item sequence, published by the Q producer
    auto next_item = [&](int it, bool producer) {
        const int slot = it & 1;
        if (producer) {
            const bool ok = it < 2 || wait_bar(&item_empty[slot], ((it >> 1) - 1) & 1, ctl);
            int item = -1;
            const bool dyn = g.n_items > (int)gridDim.x;   // (else no ticket or shared abort word is read)
            if (ok && !*abort_cta && (!dyn || !*ctl.glob)) {   // (not after another CTA gave up a wait)
                // item b for CTA b first, then tickets offset by the grid size
                item = it == 0 ? (int)blockIdx.x : dyn ? (int)gridDim.x + atomicAdd(sc.ticket, 1) : -1;
                if (item >= g.n_items) item = -1;
            }
            item_slot[slot] = item;
            mbar_arrive(&item_full[slot]);
            return item;
        }
        if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) return -1;
        const int item = item_slot[slot];
        __syncwarp(__activemask());
        return item;
    };

    if (warp == kNcProducer) {
        if (lane == 0) {
            // ---------------------------------------------- Q tile producer
            prefetch_tmap(&tm_q);
            const uint64_t stream = policy_evict_first();
            uint32_t n = 0;
            for (int it = 0;; it++) {
                const int item = next_item(it, true);
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                bool ok = true;
                for (int c = 0; c < nc && ok; c++) {
                    if (c + 1 < nc)
                        for (int b = 0; b < DP / 64; b++) tma_prefetch_3d(&tm_q, b * 64, (c0 + c + 1) * kC, h);
                    const int st = n % NQ;
                    if (n >= NQ && !wait_bar(&q_empty[st], ((n / NQ) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&q_full[st], PL::QB);
                    for (int b = 0; b < DP / 64; b++)
                        tma_load_3d_hint(gbase + PL::Q0 + st * PL::QB + b * kC * 128, &tm_q, &q_full[st], b * 64,
                                         (c0 + c) * kC, h, stream);
                    n++;
                }
            }
            for (uint32_t m = n > NQ ? n - NQ : 0; m < n; m++)
                mbar_wait(&q_full[m % NQ], (m / NQ) & 1, nullptr, 0);
        } else if (lane == 1) {
            // ------------------------------------------- output tile stores
            prefetch_tmap(&tm_o);
            uint32_t k = 0;
            for (int it = 0;; it++) {
                const int item = next_item(it, false);
                mbar_arrive(&item_empty[it & 1]);
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                for (int c = 0; c < nc; c++, k++) {
                    const int st = k % NO;
                    if (wait_bar(&out_ready[st], (k / NO) & 1, ctl)) {
                        const uint32_t src = base + PL::O0 + st * PL::OB;
                        for (int b = 0; b < DV / 64; b++)
                            tma_store_3d(&tm_o, src + b * kC * 128, b * 64, (c0 + c) * kC, h);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                    mbar_arrive(&out_free[st]);
                }
            }
            bulk_wait_all();
        }
    } else if (warp == kNcMma) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qs = idesc_bf16(128, PL::NQ16, 0, 1);
            const uint32_t s_addr = base + PL::S0;
            uint32_t k = 0, ni = 0;
            for (int it = 0;; it++) {
                const int item = next_item(it, false);
                mbar_arrive(&item_empty[it & 1]);
                if (item < 0) break;
                const int s = item / g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                wait_bar(s_ready, ni & 1, ctl);
                for (int c = 0; c < nc; c++, k++) {
                    const int st = k % NQ, rr = k & 1;
                    wait_bar(&q_ready[st], (k / NQ) & 1, ctl);
                    if (k >= 2) wait_bar(&num_free[rr], ((k >> 1) - 1) & 1, ctl);
                    tc_fence_after();
                    const uint32_t qa = base + PL::Q0 + st * PL::QB;
                    if (!*abort_cta) {
#pragma unroll
                        for (int kk = 0; kk < DP; kk += 16)
                            mma_bf16_ss(tmem + rr * PL::RS,
                                        sw128_desc(qa + (kk / 64) * (kC * 128) + (kk % 64) * 2, 16, 1024),
                                        sw32_desc(s_addr + (kk / 8) * 256, DP * 32, 256), id_qs, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&q_empty[st]);
                    mma_commit(&num_full[rr]);
                }
                mma_commit(s_free);   // S, ZP of this item have been read
                ni++;
            }
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, 0);
        }
    } else {
        // ----------------------------------------------------- math warps
        const int qd = warp & 3, grp = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const uint32_t s_addr = base + PL::S0;
        const uint32_t z_addr = s_addr + (DV / 16) * (DP * 32);   // the z block after S's blocks
        uint32_t k = 0, kq = 0, ni = 0;
        auto phi_q = [&]() {
            const int st = kq % NQ;
            wait_bar(&q_full[st], (kq / NQ) & 1, ctl);
            const uint32_t t = base + PL::Q0 + st * PL::QB;
            if constexpr (PHI) {
                constexpr int JH = DP / 16;
                uint4 x[JH];
#pragma unroll
                for (int j = 0; j < JH; j++) x[j] = lds128(t + tile_off(r, grp * JH + j));
#pragma unroll
                for (int j = 0; j < JH; j++) sts128(t + tile_off(r, grp * JH + j), phi_elu1_bf16x8(x[j]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_ready[st]);
            kq++;
        };
        for (int it = 0;; it++) {
            const int item = next_item(it, false);
            if (lane == 0) mbar_arrive(&item_empty[it & 1]);
            if (item < 0) break;
            const int s = item / g.BH, h = item % g.BH;
            const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
            // S (bf16) and ZP for this head, once the last item's products are done
            if (ni > 0) wait_bar(s_free, (ni - 1) & 1, ctl);
            const bool first_item = ni == 0;
            if (first_item) phi_q();   // phi(Q) of the first chunk does not wait for the sums
            griddep_wait();   // the totals kernel (or the segment-sum pass) has completed
            // the head's totals: read (nsum = 0), or added up from its segments' sums
            const int nsl = sc.nsum > 0 ? sc.nsum : 1;
            const bool exp_tot = sc.nsum > 0 && s == 0;   // this CTA exports the totals
            for (int row = r; row < DP; row += kC) {
                const float *src = sc.preS + (long long)h * nsl * DP * DV + (long long)row * DV + grp * HALF;
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    float4 acc[8];
#pragma unroll
                    for (int i = 0; i < 8; i++) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int t = 0; t < nsl; t++)
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const float4 x = __ldcg(reinterpret_cast<const float4 *>(src + (long long)t * DP * DV + cb) + i);
                            acc[i].x += x.x;
                            acc[i].y += x.y;
                            acc[i].z += x.z;
                            acc[i].w += x.w;
                        }
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        v[4 * i] = __float_as_uint(acc[i].x);
                        v[4 * i + 1] = __float_as_uint(acc[i].y);
                        v[4 * i + 2] = __float_as_uint(acc[i].z);
                        v[4 * i + 3] = __float_as_uint(acc[i].w);
                    }
                    if (exp_tot && sc.exS) {
                        float4 *dst = reinterpret_cast<float4 *>(sc.exS + ((long long)h * DP + row) * DV + grp * HALF + cb);
#pragma unroll
                        for (int i = 0; i < 8; i++) dst[i] = acc[i];
                    }
                    sprev_store32_sw32<DP>(s_addr, row, grp * HALF + cb, v);
                }
                if (grp == 0) {
                    float zt = 0.f;
                    for (int t = 0; t < nsl; t++) zt += __ldcg(sc.prez + ((long long)h * nsl + t) * DP + row);
                    if (exp_tot && sc.exz) sc.exz[(long long)h * DP + row] = zt;
                    zp_store(z_addr, row, zt);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_ready);
            ni++;
            if (!first_item) phi_q();
            for (int c = 0; c < nc; c++, k++) {
                if (c + 1 < nc) phi_q();
                // out = NUM / (DEN[0] + DEN[8]) for chunk k -> staging slot k % NO
                const int rr = k & 1, os = k % NO;
                wait_bar(&num_full[rr], (k >> 1) & 1, ctl);
                tc_fence_after();
                uint32_t d[16], n0[32], n1[32];
                const uint32_t rn = tmem + lane_base + rr * PL::RS + grp * HALF;
                tmem_ld16_nowait(tmem + lane_base + rr * PL::RS + DV, d);   // DEN
                tmem_ld32c<PL::ALN32>(rn, n0);
                if constexpr (HALF == 64) tmem_ld32c<PL::ALN32>(rn + 32, n1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&num_free[rr]);
                if (k >= NO) wait_bar(&out_free[os], ((k / NO) - 1) & 1, ctl);
                const float inv = 1.f / (__uint_as_float(d[0]) + __uint_as_float(d[8]));
                const uint32_t ot = base + PL::O0 + os * PL::OB + (grp * HALF / 64) * (kC * 128);
                auto put = [&](const uint32_t(&v)[32], int j0) {
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        sts128(ot + sw128_off(r, j0 + j),
                               make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]) * inv,
                                                      __uint_as_float(v[8 * j + 1]) * inv),
                                          pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv,
                                                      __uint_as_float(v[8 * j + 3]) * inv),
                                          pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv,
                                                      __uint_as_float(v[8 * j + 5]) * inv),
                                          pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv,
                                                      __uint_as_float(v[8 * j + 7]) * inv)));
                };
                put(n0, HALF == 64 ? 0 : 4 * grp);
                if constexpr (HALF == 64) put(n1, 4);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&out_ready[os]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kNcMma) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// Per head: the sums over all segments (preS [BH, nseg, szS], prez [BH,
// nseg, szz]) -> totals totS [BH, tot_rows * Dv] and totz [BH, tot_rows] at
// element offsets offS, offz (a feature map split in halves fills one half
// of the rows per call).
__global__ void nc_total_kernel(const float *__restrict__ preS, const float *__restrict__ prez, int nseg,
                                int szS, int szz, float *__restrict__ totS, float *__restrict__ totz,
                                int tot_szS, int tot_szz, int offS, int offz)
{
    griddep_launch();
    griddep_wait();   // the segment sums are complete
    const long long head = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const float *p;
    float *dst;
    int stride;
    if (e < szS) {
        p = preS + head * nseg * (long long)szS + e;
        stride = szS;
        dst = totS + head * tot_szS + offS + e;
    } else if (e < szS + szz) {
        p = prez + head * nseg * (long long)szz + (e - szS);
        stride = szz;
        dst = totz + head * tot_szz + offz + (e - szS);
    } else {
        return;
    }
    float t = 0.f;
    for (int s = 0; s < nseg; s++) t += p[(long long)s * stride];
    *dst = t;
}

// ------------------------------------------- random-feature map (PRF)
//
// phi(x) = exp(W x - |x|^2 / 2) / sqrt(m) for every row x of q and of k
// (positive random features; review page "Rethinking Attention with
// Performers", FAVOR+ positive random features), written to HBM as bf16
// [rows, m] so that the chunk kernels above take them as their phi tiles.
// U = X W^T runs on tcgen05 (M = 128 rows, N = m, K = D) with fp32
// accumulation; W (fp32) enters as two bf16 operands W_hi = bf16(W) and
// W_lo = bf16(W - W_hi) whose products add up in the same accumulator, so
// that W keeps about 16 significant bits.  |x|^2 comes from the X tile in
// shared memory; the exponent folds in the 1/sqrt(m) as -ln(m)/2.
// Roles (10 warps): 8 epilogue warps (lane quadrant w % 4, feature half
// w / 4), one producer warp (lane 0: X tiles; lane 1: TMA stores of the phi
// tiles), one MMA warp.  Tiles are striped over the CTAs: tile t of the
// 2 T tiles is q's tile t (t < T) or k's tile t - T.

template <int D, int M>
struct PrfPlan {
    static constexpr int XB = kC * D * 2;    // one X tile
    static constexpr int WB = M * D * 2;     // W_hi (then W_lo)
    static constexpr int OB = kC * M * 2;    // one phi tile
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int NO = (2 * WB + 2 * OB + 2 * XB <= kBudget) ? 2 : 1;
    static constexpr int NX0 = (kBudget - 2 * WB - NO * OB) / XB;
    static constexpr int NX = NX0 > 4 ? 4 : NX0;
    static_assert(NX >= 2, "X ring too shallow");
    static constexpr int X0 = 0;
    static constexpr int W0 = X0 + NX * XB;
    static constexpr int O0 = W0 + 2 * WB;
    static constexpr int TILES = O0 + NO * OB;
    static constexpr int SMEM = TILES + 1024 + 1024;
    static constexpr int TMEM_COLS = 2 * M;   // two accumulators
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
    static_assert(SMEM > 114 * 1024, "one CTA per SM");
    static_assert(D % 64 == 0 && M % 64 == 0 && M <= 256, "shape");
};

template <int D, int M>
__global__ void __launch_bounds__(kNcThreads, 1)
prf_phi_kernel(const __grid_constant__ CUtensorMap tm_xq, const __grid_constant__ CUtensorMap tm_xk,
               const __grid_constant__ CUtensorMap tm_pq, const __grid_constant__ CUtensorMap tm_pk,
               const float *__restrict__ W, int T, float log_scale, int normalize, int *err)
{
    using PL = PrfPlan<D, M>;
    constexpr int NX = PL::NX, NO = PL::NO;
    constexpr int MH = M / 2;   // features per epilogue warp
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *x_full = bar, *x_empty = bar + NX;
    uint64_t *acc_full = bar + 2 * NX, *acc_free = acc_full + 2;
    uint64_t *o_ready = acc_free + 2, *o_free = o_ready + NO, *drain = o_free + NO;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(drain + 2);
    static_assert((2 * NX + 4 + 2 * NO + 3) * 8 <= 1024, "barrier map exceeds its 1 KB");
    int dummy_glob = 0;   // tiles are independent: an abort stays inside this CTA
    const Ctl ctl{abort_cta, &dummy_glob, err};
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = 2 * T;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NX; i++) {
            mbar_init(&x_full[i], 1);
            mbar_init(&x_empty[i], kNcMath + 1);   // the epilogue warps (|x|^2) and the MMA commit
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_free[i], kNcMath);
        }
        for (int i = 0; i < NO; i++) {
            mbar_init(&o_ready[i], kNcMath);
            mbar_init(&o_free[i], 1);
        }
        mbar_init(drain, 1);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp < kNcMath) {
        // W -> W_hi, W_lo: K-major [M x D] operands, 128-byte swizzle, D / 64 blocks of M rows
        for (int row = threadIdx.x; row < M; row += kNcMath * 32) {
#pragma unroll
            for (int c = 0; c < D / 8; c++) {
                const float4 a = __ldg(reinterpret_cast<const float4 *>(W + (long long)row * D + 8 * c));
                const float4 b = __ldg(reinterpret_cast<const float4 *>(W + (long long)row * D + 8 * c + 4));
                const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                float hi[8], lo[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    hi[i] = __bfloat162float(__float2bfloat16_rn(w[i]));
                    lo[i] = w[i] - hi[i];
                }
                const uint32_t off = (uint32_t)(c / 8) * (M * 128) + sw128_off(row, c % 8);
                sts128(base + PL::W0 + off, make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                                       pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7])));
                sts128(base + PL::W0 + PL::WB + off,
                       make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]), pack_bf16x2(lo[4], lo[5]),
                                  pack_bf16x2(lo[6], lo[7])));
            }
        }
        fence_proxy_async_smem();
    }
    if (warp == kNcMma) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kNcProducer) {
        if (lane == 0) {
            // ---------------------------------------------- X tile producer
            prefetch_tmap(&tm_xq);
            prefetch_tmap(&tm_xk);
            const uint64_t stream = policy_evict_first();
            uint32_t n = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x, n++) {
                const int st = n % NX;
                if (n >= NX && !wait_bar(&x_empty[st], ((n / NX) - 1) & 1, ctl)) break;
                const CUtensorMap *tm = t < T ? &tm_xq : &tm_xk;
                const int row = (t < T ? t : t - T) * kC;
                mbar_arrive_expect_tx(&x_full[st], PL::XB);
                for (int b = 0; b < D / 64; b++)
                    tma_load_3d_hint(gbase + PL::X0 + st * PL::XB + b * kC * 128, tm, &x_full[st], b * 64, row, 0,
                                     stream);
            }
            for (uint32_t m = n > NX ? n - NX : 0; m < n; m++)
                mbar_wait(&x_full[m % NX], (m / NX) & 1, nullptr, 0);
        } else if (lane == 1) {
            // ------------------------------------------- phi tile stores
            prefetch_tmap(&tm_pq);
            prefetch_tmap(&tm_pk);
            uint32_t n = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x, n++) {
                const int os = n % NO;
                if (wait_bar(&o_ready[os], (n / NO) & 1, ctl)) {
                    const CUtensorMap *tm = t < T ? &tm_pq : &tm_pk;
                    const int row = (t < T ? t : t - T) * kC;
                    const uint32_t src = base + PL::O0 + os * PL::OB;
                    for (int b = 0; b < M / 64; b++) tma_store_3d(tm, src + b * kC * 128, b * 64, row, 0);
                    bulk_commit_group();
                    bulk_wait_read_all();
                }
                mbar_arrive(&o_free[os]);
            }
            bulk_wait_all();
        }
    } else if (warp == kNcMma) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id = idesc_bf16(128, M, 0, 0);
            const uint32_t w_hi = base + PL::W0, w_lo = base + PL::W0 + PL::WB;
            uint32_t n = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x, n++) {
                const int st = n % NX, a = n & 1;
                wait_bar(&x_full[st], (n / NX) & 1, ctl);
                if (n >= 2) wait_bar(&acc_free[a], ((n >> 1) - 1) & 1, ctl);
                tc_fence_after();
                const uint32_t xa = base + PL::X0 + st * PL::XB;
                if (!*abort_cta) {
#pragma unroll
                    for (int kk = 0; kk < D; kk += 16) {
                        const uint32_t ko = (kk / 64) * (kC * 128) + (kk % 64) * 2;
                        const uint32_t wo = (kk / 64) * (M * 128) + (kk % 64) * 2;
                        const uint64_t ad = sw128_desc(xa + ko, 16, 1024);
                        mma_bf16_ss(tmem + a * M, ad, sw128_desc(w_hi + wo, 16, 1024), id, kk > 0 ? 1u : 0u);
                        mma_bf16_ss(tmem + a * M, ad, sw128_desc(w_lo + wo, 16, 1024), id, 1u);
                    }
                }
                mma_commit(&x_empty[st]);
                mma_commit(&acc_full[a]);
            }
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, 0);
        }
    } else {
        // ------------------------------------------------- epilogue warps
        const int qd = warp & 3, grp = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        uint32_t n = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, n++) {
            const int st = n % NX, a = n & 1, os = n % NO;
            // |x|^2 of this thread's row
            wait_bar(&x_full[st], (n / NX) & 1, ctl);
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < D / 8; c++) {
                const uint4 w = lds128(base + PL::X0 + st * PL::XB + tile_off(r, c));
                const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float lo = __uint_as_float(u[i] << 16), hi = __uint_as_float(u[i] & 0xffff0000u);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&x_empty[st]);
            // PRF: exp(u - |x|^2/2 - ln(m)/2); NPRF (normalize): exp(u/|x| - 1/2 - ln(m)/2)
            const float uscale = normalize ? (ss > 0.f ? rsqrtf(ss) : 0.f) : 1.f;
            const float shift = normalize ? (ss > 0.f ? 0.5f : 0.f) + log_scale : 0.5f * ss + log_scale;
            wait_bar(&acc_full[a], (n >> 1) & 1, ctl);
            tc_fence_after();
            if (n >= NO) wait_bar(&o_free[os], ((n / NO) - 1) & 1, ctl);
            const uint32_t ot = base + PL::O0 + os * PL::OB;
#pragma unroll
            for (int cb = 0; cb < MH; cb += 32) {
                uint32_t v[32];
                tmem_ld32_nowait(tmem + lane_base + a * M + grp * MH + cb, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int col = grp * MH + cb + 8 * j;
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        w[i] = pack_bf16x2(__expf(__uint_as_float(v[8 * j + 2 * i]) * uscale - shift),
                                           __expf(__uint_as_float(v[8 * j + 2 * i + 1]) * uscale - shift));
                    sts128(ot + (uint32_t)(col >> 6) * (kC * 128) + sw128_off(r, (col & 63) >> 3),
                           make_uint4(w[0], w[1], w[2], w[3]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_free[a]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_ready[os]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kNcMma) {
        tc_fence_after();
        tmem_dealloc(tmem, PL::TMEM_COLS);
    }
}

// ------------------------------------------------ failure-detection self-test
//
// One thread waits, with the kernels' own bounded wait, for phase 0 of an
// mbarrier that expects one arrival which never comes; when the budget runs
// out the wait raises the error word (as in a real stall) and returns.
__global__ void wait_selftest_kernel(int *err, long long budget_cycles)
{
    __shared__ uint64_t bar;
    __shared__ int cta_abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        cta_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int glob = 0;
        const Ctl ctl{&cta_abort, &glob, err};
        const long long t0 = clock64();
        while (!mbar_try_wait(&bar, 0)) {
            if (clock64() - t0 > budget_cycles) {
                raise_abort(ctl);
                break;
            }
        }
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

// 3-D map over a [BH, N, cols] bf16 tensor whose rows are row_elems apart
// (cols, the default, or wider: one column block of a wider tensor); box =
// 64 columns x 128 rows x 1 head with 128-byte swizzle, or (sw = 32) 16
// columns x 128 rows with 32-byte swizzle; rows past N read as zero.
bool make_map(CUtensorMap *m, const void *base, long long BH, long long N, int cols, int row_elems = 0,
              int sw = 128)
{
    auto enc = get_encode();
    if (!enc) return false;
    if (row_elems <= 0) row_elems = cols;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)row_elems * 2, (cuuint64_t)N * row_elems * 2};
    cuuint32_t box[3] = {sw == 32 ? 16u : 64u, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
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

// Segments per head: enough (head, segment) items to give every SM one (one
// wave of the persistent grid), and no segmentation once B*H alone fills
// the GPU.  The output pass's time is about L chunk-times, the segment-sum
// pass adds about a third of that, so the forward scales with L.
Geo plan(long long BH, int N, int sms)
{
    Geo g;
    g.BH = (int)BH;
    g.N = N;
    g.NC = cdiv(N, kC);
    const int want = BH >= sms ? 1 : (int)(sms / BH);
    g.L = cdiv(g.NC, max(1, min(want, g.NC)));
    g.nseg = cdiv(g.NC, g.L);
    g.n_items = (int)(BH * g.nseg);
    g.exp_rows = 0;
    return g;
}

// Exclusive prefix over a head's segments of the segment sums, in place:
// afterwards slot (h, s) holds the sums over segments 0 .. s-1 (zero for
// s = 0).  The last segment's own sums are never computed or read.
__global__ void seg_scan_kernel(float *__restrict__ preS, float *__restrict__ prez, int nseg, int szS,
                                int szz)
{
    griddep_launch();
    griddep_wait();   // the segment sums are complete
    const long long head = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    float *p;
    int stride;
    if (e < szS) {
        p = preS + head * nseg * (long long)szS + e;
        stride = szS;
    } else if (e < szS + szz) {
        p = prez + head * nseg * (long long)szz + (e - szS);
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

size_t up256(size_t b) { return (b + 255) & ~(size_t)255; }

// Control words and, when segmented, the segment sums.  The 16-byte header
// holds the segment-sum pass's ticket (+0), the abort word (+4) and the
// output or readout pass's ticket (+8): one memset clears all three, so no
// stream operation sits between the passes.
template <int DP, int DV>
size_t seg_scratch_bytes(const Geo &g, bool every_segment)
{
    const bool seg = every_segment || g.nseg > 1;
    return up256(16 + (seg ? (size_t)g.BH * g.nseg * ((size_t)DP * DV + DP) * sizeof(float) : 0));
}

template <int DP, int DV>
Scratch carve(void *scratch, const Geo &g)
{
    unsigned char *b = (unsigned char *)scratch;
    Scratch sc;
    sc.ticket = (int *)b;   // (the second pass's ticket is at b + 8)
    sc.abort = (int *)(b + 4);
    sc.preS = (float *)(b + 16);
    sc.prez = sc.preS + (size_t)g.BH * g.nseg * DP * DV;
    sc.num_part = nullptr;
    sc.den_part = nullptr;
    sc.pre_rows = DP;
    sc.pre_off = 0;
    sc.nsum = 0;
    sc.exS = nullptr;
    sc.exz = nullptr;
    return sc;
}

template <int DP, int DV, int MODE>
cudaError_t set_smem()
{
    using PL = Plan<DP, DV>;
    cudaError_t e = set_max_smem_once<tc_causal_kernel<DP, DV, true, MODE == kModeElu ? kModeElu : kModeFeat>>(
        Plan<DP, DV, true>::SMEM);
    if (e != cudaSuccess) return e;
    return set_max_smem_once<tc_causal_kernel<DP, DV, false, MODE>>(PL::SMEM);
}

// The causal forward over prepared maps: when segmented, the segment-sum
// pass, the scan and then the output pass; else the output pass alone.
template <int DP, int DV, int MODE>
cudaError_t run_causal(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tv_agg, const CUtensorMap &to, Geo g, void *scratch, float *num_part,
                       float *den_part, void *out, float *S_out, float *z_out, int *err, cudaStream_t s)
{
    using PL = Plan<DP, DV>;
    constexpr int AMODE = MODE == kModeElu ? kModeElu : kModeFeat;
    const int sms = num_sms();
    Scratch sc = carve<DP, DV>(scratch, g);
    sc.num_part = num_part;
    sc.den_part = den_part;
    cudaError_t e;
    int launches = 0;
    if ((e = set_smem<DP, DV, MODE>()) != cudaSuccess) return e;
    // the header (tickets, abort word) is read only by launches with more items than CTAs
    if (g.n_items > sms && (e = cudaMemsetAsync(scratch, 0, 16, s)) != cudaSuccess) return e;
    if (g.nseg > 1) {
        // pass 1: the sums of every segment but the last of each head; then the scan
        Geo ga = g;
        ga.n_items = g.BH * (g.nseg - 1);
        tc_causal_kernel<DP, DV, true, AMODE><<<min(ga.n_items, sms), kThreads, Plan<DP, DV, true>::SMEM, s>>>(
            tq, tk, tv_agg, to, ga, sc, (__nv_bfloat16 *)out, nullptr, nullptr, err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int sz = DP * DV + DP;
        if ((e = launch_dependent(seg_scan_kernel, dim3(cdiv(sz, 256), (unsigned)g.BH), dim3(256), 0, s, sc.preS,
                                  sc.prez, g.nseg, DP * DV, DP)) != cudaSuccess)
            return e;
        launches += 2;
    }
    sc.ticket = (int *)((unsigned char *)scratch + 8);   // the output pass's own ticket
    // pass 2: the chunk recurrence of every segment from its prefix
    // (after the scan: a dependent launch, whose phase B waits for the scan)
    if (g.nseg > 1) {
        e = launch_dependent(tc_causal_kernel<DP, DV, false, MODE>, dim3(min(g.n_items, sms)), dim3(kThreads),
                             PL::SMEM, s, tq, tk, tv, to, g, sc, (__nv_bfloat16 *)out, S_out, z_out, err);
    } else {
        tc_causal_kernel<DP, DV, false, MODE><<<min(g.n_items, sms), kThreads, PL::SMEM, s>>>(
            tq, tk, tv, to, g, sc, (__nv_bfloat16 *)out, S_out, z_out, err);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    note_launches(launches + 1);
    return cudaSuccess;
}

// Non-causal, first half: the segment-sum form over every segment, then the
// per-head totals into rows [row_off, row_off + DP) of totS / totz, whose
// heads hold tot_rows feature rows.
template <int DP, int DV, int AMODE>
cudaError_t run_totals(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv_agg, const CUtensorMap &to,
                       Geo g, void *scratch, float *totS, float *totz, int tot_rows, int row_off, int *err,
                       cudaStream_t s, bool with_totals = true)
{
    using PL = Plan<DP, DV>;
    const int sms = num_sms();
    Scratch sc = carve<DP, DV>(scratch, g);
    cudaError_t e;
    if ((e = set_smem<DP, DV, AMODE>()) != cudaSuccess) return e;
    // the header (tickets, abort word) is read only by launches with more items than CTAs
    if (g.n_items > sms && (e = cudaMemsetAsync(scratch, 0, 16, s)) != cudaSuccess) return e;
    tc_causal_kernel<DP, DV, true, AMODE><<<min(g.n_items, sms), kThreads, Plan<DP, DV, true>::SMEM, s>>>(
        tq, tk, tv_agg, to, g, sc, nullptr, nullptr, nullptr, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!with_totals) {   // the readout adds the segment sums up itself
        note_launches(1);
        return cudaSuccess;
    }
    const int sz = DP * DV + DP;
    if ((e = launch_dependent(nc_total_kernel, dim3(cdiv(sz, 256), (unsigned)g.BH), dim3(256), 0, s,
                              (const float *)sc.preS, (const float *)sc.prez, g.nseg, DP * DV, DP, totS, totz,
                              tot_rows * DV, tot_rows, row_off * DV, row_off)) != cudaSuccess)
        return e;
    note_launches(2);
    return cudaSuccess;
}

// Non-causal, second half: out = phi(Q) S / phi(Q) z from the totals.
template <int DP, int DV, bool PHI>
cudaError_t run_readout(const CUtensorMap &tq, const CUtensorMap &to, Geo g, void *scratch, float *totS,
                        float *totz, int *err, cudaStream_t s, float *S_out = nullptr, float *z_out = nullptr)
{
    using NP = NcPlan<DP, DV>;
    Scratch sc = carve<DP, DV>(scratch, g);
    if (totS) {   // the totals kernel's output
        sc.preS = totS;
        sc.prez = totz;
    } else {      // the segment sums of the segment-sum pass, added up by the readout (which exports them)
        sc.nsum = g.nseg;
        sc.exS = S_out;
        sc.exz = z_out;
    }
    sc.ticket = (int *)((unsigned char *)scratch + 8);   // cleared with the header by run_totals
    // Items of the readout: its own segments (it needs only the per-head
    // totals); with two CTAs per SM, enough of them to give every CTA slot one
    int slots = num_sms();
    if constexpr (NP::kTwo) {
        slots *= 2;
        const int want = g.BH >= slots ? 1 : slots / g.BH;
        g.L = cdiv(g.NC, max(1, min(want, g.NC)));
        g.nseg = cdiv(g.NC, g.L);
        g.n_items = g.BH * g.nseg;
    }
    cudaError_t e;
    if ((e = set_max_smem_once<nc_out_kernel<DP, DV, PHI>>(NP::SMEM)) != cudaSuccess)
        return e;
    // (after the totals kernel: a dependent launch that waits for it before reading S, z)
    if ((e = launch_dependent(nc_out_kernel<DP, DV, PHI>, dim3(min(g.n_items, slots)), dim3(kNcThreads),
                              NP::SMEM, s, tq, to, g, sc, err)) != cudaSuccess)
        return e;
    note_launches(1);
    return cudaSuccess;
}

// Non-causal elu+1: with at most this many segments per head the readout reads
// and adds the segment sums itself (a few tens of KB per CTA from L2) instead
// of waiting for a totals kernel.
constexpr int kNcFoldSegs = 4;

cudaError_t export_totals(float *S_out, float *z_out, const float *totS, const float *totz, long long BH, int P,
                          int Dv, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    if (S_out) e = cudaMemcpyAsync(S_out, totS, (size_t)BH * P * Dv * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && z_out) e = cudaMemcpyAsync(z_out, totz, (size_t)BH * P * 4, cudaMemcpyDeviceToDevice, s);
    return e;
}

// ---- elu + 1 on q, k in the tile loads

template <int DP, int DV>
cudaError_t run_elu(const Problem &p, void *scratch, float *S_out, float *z_out, int *err, cudaStream_t s,
                    bool causal)
{
    // V: 32-byte swizzle for the output form (16-column blocks, each V slot followed
    // by its ONES block), 128-byte swizzle for the segment-sum form
    CUtensorMap tq, tk, tv, tva, to;
    if (!make_map(&tq, p.q, p.BH, p.N, p.D) || !make_map(&tk, p.k, p.BH, p.N, p.D) ||
        !make_map(&tv, p.v, p.BH, p.N, p.Dv, 0, 32) || !make_map(&tva, p.v, p.BH, p.N, p.Dv) ||
        !make_map(&to, p.out, p.BH, p.N, p.Dv))
        return cudaErrorInvalidValue;
    Geo g = plan(p.BH, p.N, num_sms());
    g.exp_rows = DP;
    if (causal)
        return run_causal<DP, DV, kModeElu>(tq, tk, tv, tva, to, g, scratch, nullptr, nullptr, p.out, S_out,
                                           z_out, err, s);
    float *totS = (float *)((unsigned char *)scratch + seg_scratch_bytes<DP, DV>(g, true));
    float *totz = totS + (size_t)g.BH * DP * DV;
    if (g.nseg <= kNcFoldSegs) {
        // few segments per head: the readout adds them up (no totals kernel)
        cudaError_t e = run_totals<DP, DV, kModeElu>(tq, tk, tva, to, g, scratch, totS, totz, DP, 0, err, s, false);
        if (e == cudaSuccess) e = run_readout<DP, DV, true>(tq, to, g, scratch, nullptr, nullptr, err, s, S_out, z_out);
        return e;
    }
    cudaError_t e = run_totals<DP, DV, kModeElu>(tq, tk, tva, to, g, scratch, totS, totz, DP, 0, err, s);
    if (e == cudaSuccess) e = run_readout<DP, DV, true>(tq, to, g, scratch, totS, totz, err, s);
    if (e == cudaSuccess) e = export_totals(S_out, z_out, totS, totz, g.BH, DP, DV, s);
    return e;
}

template <int DP, int DV>
size_t elu_scratch_bytes(const Geo &g, bool causal)
{
    if (causal) return seg_scratch_bytes<DP, DV>(g, false);
    return seg_scratch_bytes<DP, DV>(g, true) + (size_t)g.BH * ((size_t)DP * DV + DP) * sizeof(float);
}

// ---- random features: phi(q), phi(k) materialised in bf16, then the chunk
// kernels on those tiles; m = 256 as two feature halves of 128

struct PrfLayout {
    size_t phi_q, phi_k, part, half, tot, total;
};

PrfLayout prf_layout(const Problem &p, const Geo &g, bool causal)
{
    const size_t R = (size_t)p.BH * p.N;
    PrfLayout L;
    L.phi_q = 0;
    L.phi_k = up256(R * p.m * 2);
    L.part = L.phi_k + up256(R * p.m * 2);
    const size_t part = (causal && p.m == 256) ? up256(R * p.Dv * 4) + up256(R * 4) : 0;
    L.half = L.part + part;
    // (causal m = 256: one prefix slot holds both feature halves' rows)
    const size_t seg = causal && p.m == 256 ? seg_scratch_bytes<256, 64>(g, false)
                       : p.Dv == 64         ? seg_scratch_bytes<128, 64>(g, !causal)
                                            : seg_scratch_bytes<128, 128>(g, !causal);
    L.tot = L.half + seg;
    L.total = L.tot + (causal ? 0 : up256((size_t)g.BH * ((size_t)p.m * p.Dv + p.m) * 4));
    return L;
}

template <int M>
cudaError_t run_prf_phi(const Problem &p, void *phq, void *phk, int *err, cudaStream_t s)
{
    using PP = PrfPlan<64, M>;
    const long long R = p.BH * (long long)p.N;
    CUtensorMap xq, xk, pq, pk;
    if (!make_map(&xq, p.q, 1, R, 64) || !make_map(&xk, p.k, 1, R, 64) || !make_map(&pq, phq, 1, R, M) ||
        !make_map(&pk, phk, 1, R, M))
        return cudaErrorInvalidValue;
    const int T = (int)((R + kC - 1) / kC);
    cudaError_t e;
    if ((e = set_max_smem_once<prf_phi_kernel<64, M>>(PP::SMEM)) != cudaSuccess)
        return e;
    const float log_scale = (float)(0.5 * std::log((double)M));
    prf_phi_kernel<64, M><<<min(2 * T, num_sms()), kNcThreads, PP::SMEM, s>>>(xq, xk, pq, pk, p.W, T, log_scale,
                                                                             p.kind == PHI_NPRF ? 1 : 0, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(1);
    return cudaSuccess;
}

// Causal m = 256 over materialised phi tiles: one segment-sum pass over all
// 256 features (S as two 128-row blocks; V read once), one scan, then the
// output pass of the first 128-feature half (un-normalised sums to
// num_part, den_part) and that of the second (adds them and divides).  The
// prefix slots hold 256 feature rows; each output pass reads its half.
template <int DV>
cudaError_t run_causal_split(const CUtensorMap (&tq)[2], const CUtensorMap (&tk)[2], const CUtensorMap &tk_all,
                             const CUtensorMap &tv, const CUtensorMap &tv_agg, const CUtensorMap &to, Geo g,
                             void *scratch, float *num_part, float *den_part, void *out, float *S_out,
                             float *z_out, int *err, cudaStream_t s)
{
    using PA = Plan<256, DV>;
    using PL = Plan<128, DV>;
    const int sms = num_sms();
    Scratch sc = carve<256, DV>(scratch, g);
    sc.num_part = num_part;
    sc.den_part = den_part;
    cudaError_t e;
    int launches = 0;
    if ((e = set_max_smem_once<tc_causal_kernel<256, DV, true, kModeFeat>>(PA::SMEM)) != cudaSuccess ||
        (e = set_max_smem_once<tc_causal_kernel<128, DV, false, kModeFeatPart>>(PL::SMEM)) != cudaSuccess ||
        (e = set_max_smem_once<tc_causal_kernel<128, DV, false, kModeFeatComb>>(PL::SMEM)) != cudaSuccess)
        return e;
    // the 16-byte header: segment-sum ticket (+0), abort word (+4), the two
    // output passes' tickets (+8, +12)
    if ((e = cudaMemsetAsync(scratch, 0, 16, s)) != cudaSuccess) return e;
    if (g.nseg > 1) {
        Geo ga = g;
        ga.n_items = g.BH * (g.nseg - 1);
        tc_causal_kernel<256, DV, true, kModeFeat><<<min(ga.n_items, sms), kThreads, PA::SMEM, s>>>(
            tq[0], tk_all, tv_agg, to, ga, sc, (__nv_bfloat16 *)out, nullptr, nullptr, err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int sz = 256 * DV + 256;
        if ((e = launch_dependent(seg_scan_kernel, dim3(cdiv(sz, 256), (unsigned)g.BH), dim3(256), 0, s, sc.preS,
                                  sc.prez, g.nseg, 256 * DV, 256)) != cudaSuccess)
            return e;
        launches += 2;
    }
    sc.pre_rows = 256;
    sc.pre_off = 0;
    sc.ticket = (int *)((unsigned char *)scratch + 8);
    if (g.nseg > 1) {
        e = launch_dependent(tc_causal_kernel<128, DV, false, kModeFeatPart>, dim3(min(g.n_items, sms)),
                             dim3(kThreads), PL::SMEM, s, tq[0], tk[0], tv, to, g, sc, (__nv_bfloat16 *)out, S_out,
                             z_out, err);
    } else {
        tc_causal_kernel<128, DV, false, kModeFeatPart><<<min(g.n_items, sms), kThreads, PL::SMEM, s>>>(
            tq[0], tk[0], tv, to, g, sc, (__nv_bfloat16 *)out, S_out, z_out, err);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    sc.pre_off = 128;
    sc.ticket = (int *)((unsigned char *)scratch + 12);
    tc_causal_kernel<128, DV, false, kModeFeatComb><<<min(g.n_items, sms), kThreads, PL::SMEM, s>>>(
        tq[1], tk[1], tv, to, g, sc, (__nv_bfloat16 *)out, S_out ? S_out + 128 * DV : nullptr,
        z_out ? z_out + 128 : nullptr, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(launches + 2);
    return cudaSuccess;
}

template <int M, int DV>
cudaError_t run_prf(const Problem &p, void *scratch, float *S_out, float *z_out, int *err, cudaStream_t s,
                    bool causal)
{
    Geo g = plan(p.BH, p.N, num_sms());
    const PrfLayout L = prf_layout(p, g, causal);
    unsigned char *b = (unsigned char *)scratch;
    void *phq = b + L.phi_q, *phk = b + L.phi_k;
    cudaError_t e = run_prf_phi<M>(p, phq, phk, err, s);
    if (e != cudaSuccess) return e;
    // one map per 128-feature half of phi(q), phi(k)
    CUtensorMap tq[2], tk[2], tv, to;
    for (int f = 0; f < M / 128; f++)
        if (!make_map(&tq[f], (const __nv_bfloat16 *)phq + 128 * f, p.BH, p.N, 128, M) ||
            !make_map(&tk[f], (const __nv_bfloat16 *)phk + 128 * f, p.BH, p.N, 128, M))
            return cudaErrorInvalidValue;
    CUtensorMap tva;
    if (!make_map(&tv, p.v, p.BH, p.N, p.Dv, 0, 32) || !make_map(&tva, p.v, p.BH, p.N, p.Dv) ||
        !make_map(&to, p.out, p.BH, p.N, p.Dv))
        return cudaErrorInvalidValue;
    void *half = b + L.half;
    g.exp_rows = M;
    if (causal) {
        if constexpr (M == 128) {
            return run_causal<128, DV, kModeFeat>(tq[0], tk[0], tv, tva, to, g, half, nullptr, nullptr, p.out,
                                                  S_out, z_out, err, s);
        } else {
            float *num_part = (float *)(b + L.part);
            float *den_part = (float *)(b + L.part + up256((size_t)p.BH * p.N * DV * 4));
            CUtensorMap tk_all;
            if (!make_map(&tk_all, phk, p.BH, p.N, M, M)) return cudaErrorInvalidValue;
            return run_causal_split<DV>(tq, tk, tk_all, tv, tva, to, g, half, num_part, den_part, p.out, S_out,
                                        z_out, err, s);
        }
    }
    float *totS = (float *)(b + L.tot);
    float *totz = totS + (size_t)g.BH * M * DV;
    for (int f = 0; f < M / 128; f++)
        if ((e = run_totals<128, DV, kModeFeat>(tq[f], tk[f], tva, to, g, half, totS, totz, M, 128 * f, err, s)) !=
            cudaSuccess)
            return e;
    CUtensorMap tqa;
    if (!make_map(&tqa, phq, p.BH, p.N, M)) return cudaErrorInvalidValue;
    if ((e = run_readout<M, DV, false>(tqa, to, g, half, totS, totz, err, s)) != cudaSuccess) return e;
    return export_totals(S_out, z_out, totS, totz, g.BH, M, DV, s);
}

}  // namespace

cudaError_t wait_selftest(int budget_ms, int *err, cudaStream_t s)
{
    budget_ms = budget_ms < 1 ? 1 : budget_ms > 2000 ? 2000 : budget_ms;
    int dev = 0, khz = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0) khz = 2000000;
    wait_selftest_kernel<<<1, 32, 0, s>>>(err, (long long)budget_ms * khz);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) note_launches(1);
    return e;
}

bool tc_causal_supported(const Problem &p)
{
    return p.dtype == DT_BF16 && p.kind == PHI_ELU1 && (p.D == 64 || p.D == 128) &&
           (p.Dv == 64 || p.Dv == 128);
}

bool tc_prf_supported(const Problem &p)
{
    return p.dtype == DT_BF16 && (p.kind == PHI_PRF || p.kind == PHI_NPRF) && p.D == 64 &&
           ((p.m == 128 && (p.Dv == 64 || p.Dv == 128)) || (p.m == 256 && p.Dv == 64)) &&
           p.BH * (long long)p.N < (1LL << 31) - kC;
}

size_t tc_scratch_bytes(const Problem &p, bool causal)
{
    Geo g = plan(p.BH, p.N, num_sms());
    if (p.kind == PHI_PRF || p.kind == PHI_NPRF) return prf_layout(p, g, causal).total;
    if (p.D == 64 && p.Dv == 64) return elu_scratch_bytes<64, 64>(g, causal);
    if (p.D == 64 && p.Dv == 128) return elu_scratch_bytes<64, 128>(g, causal);
    if (p.D == 128 && p.Dv == 64) return elu_scratch_bytes<128, 64>(g, causal);
    return elu_scratch_bytes<128, 128>(g, causal);
}

cudaError_t tc_forward(const Problem &p, bool causal, void *scratch, float *S_out, float *z_out, int *err,
                       cudaStream_t s)
{
    if (p.kind == PHI_PRF || p.kind == PHI_NPRF) {
        if (p.m == 256) return run_prf<256, 64>(p, scratch, S_out, z_out, err, s, causal);
        if (p.Dv == 64) return run_prf<128, 64>(p, scratch, S_out, z_out, err, s, causal);
        return run_prf<128, 128>(p, scratch, S_out, z_out, err, s, causal);
    }
    if (p.D == 64 && p.Dv == 64) return run_elu<64, 64>(p, scratch, S_out, z_out, err, s, causal);
    if (p.D == 64 && p.Dv == 128) return run_elu<64, 128>(p, scratch, S_out, z_out, err, s, causal);
    if (p.D == 128 && p.Dv == 64) return run_elu<128, 64>(p, scratch, S_out, z_out, err, s, causal);
    return run_elu<128, 128>(p, scratch, S_out, z_out, err, s, causal);
}

}  // namespace la
