// tc_causal.cu -- chunked causal linear attention on the sm_103a tensor
// cores (tcgen05, TMEM accumulators, TMA loads), bf16 inputs, fp32 state,
// in ONE persistent kernel that reads q, k, v from HBM once.
//
// The method (review page "Transformers are RNNs", proposed method b2-b3,
// b5): with phi applied to q and k, out_i = phi(q_i)^T S_i / phi(q_i)^T z_i
// where S_i, z_i are cumulative sums over j <= i.  A sequence is cut into
// chunks of C = 128 positions; with S_prev, z_prev the sums before a chunk,
//   A    = tril(phi(Q_c) phi(K_c)^T)                      (j <= i)
//   out  = (A V_c + phi(Q_c) S_prev) / (rowsum(A) + phi(Q_c) z_prev)
//   S   += phi(K_c)^T V_c,   z += colsum(phi(K_c)).
//
// Work items.  Each head's chunks are grouped into segments of L chunks; an
// item is one (head, segment).  Items are numbered segment-major and handed
// out in that order from a global ticket counter, so an item's predecessor
// (same head, previous segment) is always taken by a CTA that is already
// running.  Per item a CTA runs
//   phase A  the segment's own sums  S_loc = phi(K)^T V,  z_loc = colsum phi(K)
//            (skipped for the last segment of a head, whose sums nobody needs);
//   phase B  waits for the predecessor's inclusive state (S, z after the
//            previous segment), publishes its own = that + (S_loc, z_loc),
//            and starts the chunk recurrence from the predecessor's state;
//   phase C  the chunk recurrence above over the segment, writing out.
// Phase C re-reads the K, V tiles that phase A loaded a few microseconds
// earlier; segments are short enough (L <= 8 chunks) for that re-read to be
// served by L2, so HBM sees q, k, v and out once.  This is the exclusive
// prefix over segments of the "RNN with two memories" view, chained through
// global memory with acquire/release flags.  With one segment per head
// (B*H >= the number of SMs) phases A and B reduce to zeroing the state.
//
// Warp roles (16 warps, 4 per SM sub-partition, so 128 registers):
//   warps 0-7   TMEM warps: the state copy S_prev / ZP for each chunk, the
//               masked scores P, the epilogue, phase B.  Warp w owns TMEM lane
//               quadrant w % 4 (rows 32 (w%4) ..) and column half w / 4.
//   warps 8-11  phi warps, one per lane quadrant (one tile row per thread):
//               phi(Q) written straight into TMEM as the A operand of the
//               Q-side products, phi(K) applied in place on the K tile.
//   warp 12     TMA producer of Q tiles and item scheduler.
//   warp 13     TMA producer of K tiles (freed after MMA4).
//   warp 14     TMA producer of V tiles (freed after MMA2).
//   warp 15     MMA issuer (one thread).
// The producers prefetch tiles two chunks ahead into L2, so the loads into
// shared memory (whose buffers free up only as the pipeline drains them)
// wait for L2 rather than HBM.
// Per chunk, all tcgen05.mma with fp32 accumulation in TMEM:
//   MMA1   A    = phiQ . phiK^T        M=C, N=C,  K=Dphi   (phiQ from TMEM)
//   MMA3   NUM  = phiQ . S_prev        M=C, N=Dv, K=Dphi   (S_prev bf16 in smem)
//   MMA3b  DEN  = phiQ . ZP            M=C, N=16, K=Dphi
//   MMA4   S   += phiK^T . V           M=Dphi, N=Dv, K=C
//   MMA4b  Z   += phiK^T . ONES        M=Dphi, N=16, K=C   (Z[:,0] = z)
//   MMA2   NUM += P . V                M=C, N=Dv, K=C      (P bf16 in TMEM)
//   MMA2b  DEN += P . ONES             M=C, N=16, K=C
// ONES is a constant [C x 16] tile (columns 0-7 = 1, 8-15 = 0) and ZP holds
// z_prev split into bf16 hi (columns 0-7) and lo (columns 8-15), so that
// out = NUM / (DEN[:,0] + DEN[:,8]).  phi never goes back to HBM.
//
// Every wait is bounded (clock64 budget).  On expiry the kernel sets the
// library's device error word, raises a per-launch abort word that every
// other CTA polls, and all roles run to the end without waiting.
#include <cuda.h>
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
constexpr int kMaxItemChunks = 8;     // L <= 8 keeps the phase-C re-read in L2

constexpr int kTmemWarps = 8;
constexpr int kPhiWarps = 4;
constexpr int kProducerWarp = kTmemWarps + kPhiWarps;   // 12: Q tiles, items
constexpr int kKWarp = kProducerWarp + 1;               // 13: K tiles
constexpr int kVWarp = kKWarp + 1;                      // 14: V tiles
constexpr int kMmaWarp = kVWarp + 1;                    // 15
constexpr int kThreads = (kMmaWarp + 1) * 32;           // 512
constexpr int kPrefetch = 3;                            // chunks of L2 prefetch ahead
constexpr int kItemConsumers = kTmemWarps + kPhiWarps + 3;

template <int DP, int DV>
struct Plan {
    static constexpr int QB = kC * DP * 2;   // one Q or K chunk tile (bytes)
    static constexpr int VB = kC * DV * 2;   // one V chunk tile
    static constexpr int SB = DP * DV * 2;   // S_prev, bf16
    static constexpr int ZB = DP * 32;       // ZP [DP x 16] bf16, 32-byte swizzle
    static constexpr int OB = kC * 32;       // ONES [C x 16]
    static constexpr int kFixed = SB + ZB + OB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int NS = (kFixed + QB + 4 * (QB + VB) <= kBudget)   ? 4
                              : (kFixed + QB + 3 * (QB + VB) <= kBudget) ? 3
                                                                          : 2;
    static constexpr int NQ = (kFixed + 2 * QB + NS * (QB + VB) <= kBudget) ? 2 : 1;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + NQ * QB;
    static constexpr int V0 = K0 + NS * QB;
    static constexpr int S0 = V0 + NS * VB;
    static constexpr int Z0 = S0 + SB;
    static constexpr int O0 = Z0 + ZB;
    static constexpr int TILES = O0 + OB;
    static constexpr int SMEM = TILES + 1024 /* alignment */ + 1024 /* barriers */;
    // TMEM columns
    static constexpr int T_S = 0, T_Z = DV, T_DEN = DV + 32, T_NUM = DV + 64, T_A = 2 * DV + 64,
                         T_Q = 2 * DV + 192;
    static constexpr int TMEM_COLS = 512;
    static_assert(T_Q + DP / 2 <= TMEM_COLS, "TMEM plan too large");
    static_assert(SMEM <= 227 * 1024, "shared memory plan too large");
};

struct Geo {
    int BH, N, NC;   // heads, positions, chunks per head
    int L, nseg;     // chunks per segment, segments per head
    int n_items;     // BH * nseg
};

struct Scratch {
    int *ticket;     // next item to hand out
    int *abort;      // raised by any CTA whose wait ran out
    int *flags;      // [BH * nseg]: 1 once the inclusive state of (head, seg) is published
    float *inclS;    // [BH * nseg, DP, DV]
    float *inclz;    // [BH * nseg, DP]
};

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

__device__ __forceinline__ uint32_t align1k(uint32_t a) { return (a + 1023u) & ~1023u; }

// Element (row r, 16 B chunk j) of a [kC x cols] 128B-swizzled tile.
__device__ __forceinline__ uint32_t tile_off(int r, int j)
{
    return (uint32_t)(j >> 3) * (kC * 128) + sw128_off(r, j & 7);
}

// One S_prev row block: 32 fp32 state values -> bf16 at row r, columns
// [c0, c0 + 32) of the MN-major [DP x DV] tile (DV / 64 blocks of DP rows).
template <int DP>
__device__ __forceinline__ void sprev_store32(uint32_t st, int r, int c0, const uint32_t (&v)[32])
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int col = c0 + 8 * j;
        const uint32_t a = st + (uint32_t)(col >> 6) * (DP * 128) + sw128_off(r, (col & 63) >> 3);
        sts128(a, make_uint4(
                      pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                      pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]))));
    }
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

template <int DP, int DV>
__global__ void __launch_bounds__(kThreads, 1)
tc_causal_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, Geo g, Scratch sc,
                 __nv_bfloat16 *__restrict__ out, float *__restrict__ S_out,
                 float *__restrict__ z_out, int *err)
{
    using PL = Plan<DP, DV>;
    constexpr int NS = PL::NS, NQ = PL::NQ;
    constexpr int HALF = DV / 2;   // state / NUM columns per TMEM warp
    extern __shared__ unsigned char smem_raw[];
    const uint32_t base = align1k(smem_u32(smem_raw));
    unsigned char *gbase = smem_raw + (base - smem_u32(smem_raw));   // generic view of `base`
    uint64_t *bar = reinterpret_cast<uint64_t *>(gbase + PL::TILES);
    uint64_t *k_full = bar, *k_ready = bar + 4, *k_empty = bar + 8;
    uint64_t *v_full = bar + 12, *v_empty = bar + 16;
    uint64_t *q_full = bar + 20, *q_empty = bar + 22;
    uint64_t *item_full = bar + 24, *item_empty = bar + 26;
    uint64_t *tq_full = bar + 28, *tq_free = bar + 29, *a_full = bar + 30, *p_ready = bar + 31,
             *sprev_ready = bar + 32, *s_done = bar + 33, *num_full = bar + 34,
             *num_free = bar + 35, *sloc_done = bar + 36, *drain = bar + 37,
             *chain_ok = bar + 38, *pub_ready = bar + 39;
    volatile int *item_slot = reinterpret_cast<volatile int *>(bar + 40);   // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 41);
    volatile int *abort_cta = reinterpret_cast<volatile int *>(bar + 42);
    const Ctl ctl{abort_cta, sc.abort, err};

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_ready[i], kPhiWarps);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NQ; i++) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], kPhiWarps);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], kItemConsumers);
        }
        mbar_init(tq_full, kPhiWarps);
        mbar_init(tq_free, 1);
        mbar_init(a_full, 1);
        mbar_init(p_ready, kTmemWarps);
        mbar_init(sprev_ready, kTmemWarps);
        mbar_init(s_done, 1);
        mbar_init(num_full, 1);
        mbar_init(num_free, kTmemWarps);
        mbar_init(sloc_done, 1);
        mbar_init(drain, 1);
        mbar_init(chain_ok, 1);
        mbar_init(pub_ready, kTmemWarps);
        *abort_cta = 0;
        fence_mbar_init();
    }
    if (warp < kTmemWarps) {   // the constant ONES tile
        const uint32_t one = pack_bf16x2(1.f, 1.f);
        const uint32_t ones = base + PL::O0;
        for (int r = threadIdx.x; r < kC; r += kTmemWarps * 32) {
            sts128(ones + sw32_off(r, 0), make_uint4(one, one, one, one));
            sts128(ones + sw32_off(r, 1), make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) tmem_alloc(tslot, PL::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kProducerWarp) {
        // ------------------------------------------ Q producer / scheduler
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            const uint64_t stream = policy_evict_first();
            uint32_t nq = 0;
            for (int it = 0;; it++) {
                const int slot = it & 1;
                bool ok = it < 2 || wait_bar(&item_empty[slot], ((it >> 1) - 1) & 1, ctl);
                int item = -1;
                if (ok && !*abort_cta) {
                    item = atomicAdd(sc.ticket, 1);
                    if (item >= g.n_items) item = -1;
                }
                item_slot[slot] = item;
                mbar_arrive(&item_full[slot]);
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                for (int c = 0; c < nc && c < kPrefetch; c++)
                    for (int b = 0; b < DP / 64; b++) tma_prefetch_3d(&tm_q, b * 64, (c0 + c) * kC, h);
                for (int c = 0; c < nc && ok; c++) {
                    if (c + kPrefetch < nc)
                        for (int b = 0; b < DP / 64; b++)
                            tma_prefetch_3d(&tm_q, b * 64, (c0 + c + kPrefetch) * kC, h);
                    const int st = nq % NQ;
                    if (nq >= NQ && !wait_bar(&q_empty[st], ((nq / NQ) - 1) & 1, ctl)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&q_full[st], PL::QB);
#pragma unroll
                    for (int b = 0; b < DP / 64; b++)
                        tma_load_3d_hint(gbase + PL::Q0 + st * PL::QB + b * kC * 128, &tm_q, &q_full[st],
                                         b * 64, (c0 + c) * kC, h, stream);
                    nq++;
                }
            }
            // drain loads still in flight (only possible after an abort)
            for (uint32_t n = nq > NQ ? nq - NQ : 0; n < nq; n++)
                mbar_wait(&q_full[n % NQ], (n / NQ) & 1, nullptr, 0);
        }
    } else if (warp == kKWarp || warp == kVWarp) {
        // ------------------------------------------- K or V tile producer
        if (lane == 0) {
            const bool isK = warp == kKWarp;
            const CUtensorMap *tm = isK ? &tm_k : &tm_v;
            const int nb = isK ? DP / 64 : DV / 64;   // 64-column boxes per tile
            const int tb = isK ? PL::QB : PL::VB;     // tile bytes
            unsigned char *ring = gbase + (isK ? PL::K0 : PL::V0);
            uint64_t *full = isK ? k_full : v_full, *empty = isK ? k_empty : v_empty;
            prefetch_tmap(tm);
            const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
            uint32_t n = 0;
            bool ok = true;
            auto prefetch = [&](int head, int chunk) {
                for (int b = 0; b < nb; b++) tma_prefetch_3d(tm, b * 64, chunk * kC, head);
            };
            auto load = [&](int head, int chunk, uint64_t pol) {
                const int st = n % NS;
                if (n >= NS && !wait_bar(&empty[st], ((n / NS) - 1) & 1, ctl)) return false;
                mbar_arrive_expect_tx(&full[st], tb);
                for (int b = 0; b < nb; b++)
                    tma_load_3d_hint(ring + st * tb + b * kC * 128, tm, &full[st], b * 64, chunk * kC,
                                     head, pol);
                n++;
                return true;
            };
            for (int it = 0; ok; it++) {
                const int slot = it & 1;
                if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
                const int item = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const int s = item / g.BH, h = item % g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                const bool hasA = s + 1 < g.nseg;
                // phase A streams the segment from HBM (kept in L2 for phase C);
                // phase C re-reads it (from L2 when phase A ran)
                for (int c = 0; c < nc && c < kPrefetch; c++) prefetch(h, c0 + c);
                if (hasA)
                    for (int c = 0; c < nc && ok; c++) {
                        if (c + kPrefetch < nc) prefetch(h, c0 + c + kPrefetch);
                        ok = load(h, c0 + c, keep);
                    }
                for (int c = 0; c < nc && ok; c++) {
                    if (!hasA && c + kPrefetch < nc) prefetch(h, c0 + c + kPrefetch);
                    ok = load(h, c0 + c, stream);
                }
            }
            for (uint32_t m = n > NS ? n - NS : 0; m < n; m++)
                mbar_wait(&full[m % NS], (m / NS) & 1, nullptr, 0);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t id_qs = idesc_bf16(128, DV, 0, 1);
            constexpr uint32_t id_q16 = idesc_bf16(128, 16, 0, 1);
            constexpr uint32_t id_kv = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t id_k16 = idesc_bf16(128, 16, 1, 1);
            constexpr uint32_t lbo_kT = DP == 128 ? kC * 128 : 0;   // DP = 64: rows 64-127 repeat 0-63
            const uint32_t s_addr = base + PL::S0, zp_addr = base + PL::Z0, ones = base + PL::O0;
            uint32_t nkv = 0, nchunk = 0, nfree = 0;
            for (int it = 0;; it++) {
                const int slot = it & 1;
                if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
                const int item = item_slot[slot];
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const int s = item / g.BH;
                const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
                const bool hasA = s + 1 < g.nseg;
                if (hasA) {
                    // phase A: S_loc -> T_NUM, z_loc -> T_DEN (the previous item's
                    // last epilogue must have read T_NUM first)
                    if (nchunk > 0) {
                        wait_bar(num_free, nfree & 1, ctl);
                        nfree++;
                    }
                    for (int c = 0; c < nc; c++) {
                        const int st = nkv % NS;
                        wait_bar(&k_ready[st], (nkv / NS) & 1, ctl);
                        wait_bar(&v_full[st], (nkv / NS) & 1, ctl);
                        tc_fence_after();
                        const uint32_t ka = base + PL::K0 + st * PL::QB;
                        const uint32_t va = base + PL::V0 + st * PL::VB;
                        if (!*abort_cta) {
#pragma unroll
                            for (int k = 0; k < kC; k += 16) {
                                const uint64_t ad = sw128_desc(ka + (k / 8) * 1024, lbo_kT, 1024);
                                const uint32_t acc = (c > 0 || k > 0) ? 1u : 0u;
                                mma_bf16_ss(tmem + PL::T_NUM, ad,
                                            sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_kv, acc);
                                mma_bf16_ss(tmem + PL::T_DEN, ad,
                                            sw32_desc(ones + (k / 8) * 256, 256, 256), id_k16, acc);
                            }
                        }
                        mma_commit(&k_empty[st]);
                        mma_commit(&v_empty[st]);
                        nkv++;
                    }
                    mma_commit(sloc_done);
                }
                for (int c = 0; c < nc; c++) {
                    const int st = nkv % NS;
                    const uint32_t ka = base + PL::K0 + st * PL::QB;
                    const uint32_t va = base + PL::V0 + st * PL::VB;
                    wait_bar(tq_full, nchunk & 1, ctl);
                    wait_bar(&k_ready[st], (nkv / NS) & 1, ctl);
                    if (nchunk > 0) wait_bar(num_full, (nchunk - 1) & 1, ctl);   // P of the last chunk read
                    tc_fence_after();
                    const bool live = !*abort_cta;
                    // MMA1: A = phiQ phiK^T
                    if (live) {
#pragma unroll
                        for (int k = 0; k < DP; k += 16)
                            mma_bf16_ts(tmem + PL::T_A, tmem + PL::T_Q + k / 2,
                                        sw128_desc(ka + (k / 64) * (kC * 128) + (k % 64) * 2, 16, 1024),
                                        id_qk, k > 0 ? 1u : 0u);
                    }
                    mma_commit(a_full);
                    // MMA3 / MMA3b: NUM = phiQ S_prev, DEN = phiQ ZP
                    wait_bar(sprev_ready, nchunk & 1, ctl);
                    if (nfree < nchunk) {   // the previous chunk's epilogue has read NUM
                        wait_bar(num_free, nfree & 1, ctl);
                        nfree++;
                    }
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int k = 0; k < DP; k += 16) {
                            mma_bf16_ts(tmem + PL::T_NUM, tmem + PL::T_Q + k / 2,
                                        sw128_desc(s_addr + (k / 8) * 1024, DP * 128, 1024), id_qs,
                                        k > 0 ? 1u : 0u);
                            mma_bf16_ts(tmem + PL::T_DEN, tmem + PL::T_Q + k / 2,
                                        sw32_desc(zp_addr + (k / 8) * 256, 256, 256), id_q16,
                                        k > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(tq_free);
                    // MMA4 / MMA4b: S += phiK^T V, Z += phiK^T ONES
                    wait_bar(&v_full[st], (nkv / NS) & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int k = 0; k < kC; k += 16) {
                            const uint64_t ad = sw128_desc(ka + (k / 8) * 1024, lbo_kT, 1024);
                            mma_bf16_ss(tmem + PL::T_S, ad,
                                        sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_kv, 1u);
                            mma_bf16_ss(tmem + PL::T_Z, ad, sw32_desc(ones + (k / 8) * 256, 256, 256),
                                        id_k16, 1u);
                        }
                    }
                    mma_commit(s_done);
                    mma_commit(&k_empty[st]);
                    // MMA2 / MMA2b: NUM += P V, DEN += P ONES  (P in TMEM)
                    wait_bar(p_ready, nchunk & 1, ctl);
                    tc_fence_after();
                    if (!*abort_cta) {
#pragma unroll
                        for (int k = 0; k < kC; k += 16) {
                            const uint32_t pa = tmem + PL::T_A + (k / 64) * 64 + (k % 64) / 2;
                            mma_bf16_ts(tmem + PL::T_NUM, pa,
                                        sw128_desc(va + (k / 8) * 1024, kC * 128, 1024), id_qs, 1u);
                            mma_bf16_ts(tmem + PL::T_DEN, pa, sw32_desc(ones + (k / 8) * 256, 256, 256),
                                        id_q16, 1u);
                        }
                    }
                    mma_commit(num_full);
                    mma_commit(&v_empty[st]);
                    nkv++;
                    nchunk++;
                }
            }
            mma_commit(drain);   // every MMA issued above has completed
            mbar_wait(drain, 0, nullptr, 0);
        }
    } else if (warp >= kTmemWarps) {
        // ----------------------------------------------------- phi warps
        const int qd = warp - kTmemWarps;      // lane quadrant
        const int r = qd * 32 + lane;          // tile row = TMEM lane
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        constexpr int JR = DP / 8;             // 16 B chunks per row
        uint32_t nkv = 0, nq = 0, nchunk = 0;
        // phi in place on the row of a K tile; all loads issued before any math
        auto phi_k = [&](int c_abs) {
            const int st = nkv % NS;
            wait_bar(&k_full[st], (nkv / NS) & 1, ctl);
            const bool zero = r >= g.N - c_abs * kC;   // rows past the sequence end add nothing
            const uint32_t t = base + PL::K0 + st * PL::QB;
#pragma unroll
            for (int h8 = 0; h8 < JR; h8 += 8) {
                uint4 x[8];
#pragma unroll
                for (int j = 0; j < 8; j++) x[j] = lds128(t + tile_off(r, h8 + j));
#pragma unroll
                for (int j = 0; j < 8; j++)
                    sts128(t + tile_off(r, h8 + j), zero ? make_uint4(0, 0, 0, 0) : phi_elu1_bf16x8(x[j]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&k_ready[st]);
            nkv++;
        };
        // phi(Q) of the chunk -> TMEM (A operand of MMA1 / MMA3), 64 values per step
        auto phi_q = [&]() {
            const int qs = nq % NQ;
            wait_bar(&q_full[qs], (nq / NQ) & 1, ctl);
            const uint32_t t = base + PL::Q0 + qs * PL::QB;
            uint4 x[JR];
#pragma unroll
            for (int j = 0; j < JR; j++) x[j] = lds128(t + tile_off(r, j));
            if (nchunk > 0) wait_bar(tq_free, (nchunk - 1) & 1, ctl);
            tc_fence_after();
#pragma unroll
            for (int b = 0; b < DP / 64; b++) {
                uint32_t w[32];
#pragma unroll
                for (int jj = 0; jj < 8; jj++) {
                    const uint4 y = phi_elu1_bf16x8(x[8 * b + jj]);
                    w[4 * jj] = y.x;
                    w[4 * jj + 1] = y.y;
                    w[4 * jj + 2] = y.z;
                    w[4 * jj + 3] = y.w;
                }
                tmem_st32_nowait(tmem + lane_base + PL::T_Q + 32 * b, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&q_empty[qs]);
                mbar_arrive(tq_full);
            }
            nq++;
            nchunk++;
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
            if (s + 1 < g.nseg)
                for (int c = 0; c < nc; c++) phi_k(c0 + c);
            // phi(K) only needs its TMA load, so it runs one chunk ahead; phi(Q)
            // also waits for the previous chunk's Q-side products (tq_free)
            if (nc > 0) phi_k(c0);
            for (int c = 0; c < nc; c++) {
                phi_q();
                if (c + 1 < nc) phi_k(c0 + c + 1);
            }
        }
    } else {
        // ----------------------------------------------------- TMEM warps
        const int qd = warp & 3, grp = warp >> 2;
        const int r = qd * 32 + lane;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const bool srow = qd * 32 < DP;   // warp-uniform: this warp's rows hold state rows
        const uint32_t s_addr = base + PL::S0, zp_addr = base + PL::Z0;
        uint32_t nchunk = 0, nA = 0, nchain = 0, npub = 0;
        for (int it = 0;; it++) {
            const int slot = it & 1;
            if (!wait_bar(&item_full[slot], (it >> 1) & 1, ctl)) break;
            const int item = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const int s = item / g.BH, h = item % g.BH;
            const int c0 = s * g.L, nc = min(g.L, g.NC - c0);
            const bool hasA = s + 1 < g.nseg;
            const long long pub = (long long)h * g.nseg + s;   // this item's state slot

            // ---- phase B: predecessor's state in, own inclusive state out
            if (hasA) {
                wait_bar(sloc_done, nA & 1, ctl);
                nA++;
                tc_fence_after();
            }
            if (s > 0) {   // one thread polls the predecessor's flag, the rest wait on chain_ok
                if (threadIdx.x == 0) {
                    const int *f = sc.flags + (pub - 1);
                    const long long t0 = clock64();
                    while (!*abort_cta && ld_acquire_gpu(f) == 0) {
                        if (*ctl.glob) {
                            *abort_cta = 1;
                            break;
                        }
                        if (clock64() - t0 > kWaitBudget) {
                            raise_abort(ctl);
                            break;
                        }
                        __nanosleep(64);
                    }
                    mbar_arrive(chain_ok);
                }
                wait_bar(chain_ok, nchain & 1, ctl);
                nchain++;
            }
            float zprev = 0.f;
            if (srow) {
                const float *prevS = s > 0 ? sc.inclS + (pub - 1) * DP * DV + (long long)r * DV : nullptr;
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    const int col = grp * HALF + cb;
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 x = prevS ? __ldcg(reinterpret_cast<const float4 *>(prevS + col + i))
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[i] = __float_as_uint(x.x);
                        v[i + 1] = __float_as_uint(x.y);
                        v[i + 2] = __float_as_uint(x.z);
                        v[i + 3] = __float_as_uint(x.w);
                    }
                    if (hasA) {   // publish prev + S_loc
                        uint32_t l[32];
                        tmem_ld32_nowait(tmem + lane_base + PL::T_NUM + col, l);
                        tmem_ld_wait();
                        float *dst = sc.inclS + pub * DP * DV + (long long)r * DV + col;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            __stcg(reinterpret_cast<float4 *>(dst + i),
                                   make_float4(__uint_as_float(v[i]) + __uint_as_float(l[i]),
                                               __uint_as_float(v[i + 1]) + __uint_as_float(l[i + 1]),
                                               __uint_as_float(v[i + 2]) + __uint_as_float(l[i + 2]),
                                               __uint_as_float(v[i + 3]) + __uint_as_float(l[i + 3])));
                    }
                    tmem_st32_nowait(tmem + lane_base + PL::T_S + col, v);
                    sprev_store32<DP>(s_addr, r, col, v);
                }
                zprev = s > 0 ? __ldcg(sc.inclz + (pub - 1) * DP + r) : 0.f;
                if (grp == 0) {
                    if (hasA) {
                        uint32_t d[16];
                        tmem_ld16_nowait(tmem + lane_base + PL::T_DEN, d);
                        tmem_ld_wait();
                        __stcg(sc.inclz + pub * DP + r, zprev + __uint_as_float(d[0]));
                    }
                    uint32_t zw[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) zw[i] = i < 8 ? __float_as_uint(zprev) : 0u;
                    tmem_st16_nowait(tmem + lane_base + PL::T_Z, zw);
                    zp_store(zp_addr, r, zprev);
                }
            }
            if (hasA) {   // every writer fences, then one thread raises the flag
                __threadfence();
                __syncwarp();
                if (lane == 0) mbar_arrive(pub_ready);
                if (threadIdx.x == 0 && wait_bar(pub_ready, npub & 1, ctl)) {
                    __threadfence();
                    st_release_gpu(sc.flags + pub, 1);
                }
                npub++;
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sprev_ready);

            // ---- phase C: the chunk recurrence.  Per chunk: P(c); then the
            // state copy for chunk c + 1 (needs only MMA4(c), which finishes
            // before MMA2(c)); then the epilogue of chunk c.
            for (int c = 0; c < nc; c++, nchunk++) {
                const int row0 = (c0 + c) * kC;
                // P = bf16(tril(A)): columns [64 grp, 64 grp + 64) of A -> the
                // first 32 columns of the same region
                wait_bar(a_full, nchunk & 1, ctl);
                tc_fence_after();
                {
                    uint32_t a0[32], a1[32], pk[32];
                    tmem_ld32_nowait(tmem + lane_base + PL::T_A + grp * 64, a0);
                    tmem_ld32_nowait(tmem + lane_base + PL::T_A + grp * 64 + 32, a1);
                    tmem_ld_wait();
                    const int cbase = grp * 64;
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int col = cbase + 2 * i;
                        pk[i] = pack_bf16x2(col <= r ? __uint_as_float(a0[2 * i]) : 0.f,
                                            col + 1 <= r ? __uint_as_float(a0[2 * i + 1]) : 0.f);
                        pk[16 + i] = pack_bf16x2(col + 32 <= r ? __uint_as_float(a1[2 * i]) : 0.f,
                                                 col + 33 <= r ? __uint_as_float(a1[2 * i + 1]) : 0.f);
                    }
                    tmem_st32_nowait(tmem + lane_base + PL::T_A + grp * 64, pk);
                    tmem_st_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_ready);
                if (c + 1 < nc) {   // S_prev, ZP <- state after this chunk
                    wait_bar(s_done, nchunk & 1, ctl);
                    tc_fence_after();
                    if (srow) {
#pragma unroll
                        for (int cb = 0; cb < HALF; cb += 32) {
                            uint32_t v[32];
                            tmem_ld32_nowait(tmem + lane_base + PL::T_S + grp * HALF + cb, v);
                            tmem_ld_wait();
                            sprev_store32<DP>(s_addr, r, grp * HALF + cb, v);
                        }
                        if (grp == 0) {
                            uint32_t zv[16];
                            tmem_ld16_nowait(tmem + lane_base + PL::T_Z, zv);
                            tmem_ld_wait();
                            zp_store(zp_addr, r, __uint_as_float(zv[0]));
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sprev_ready);
                }
                // out = NUM / (DEN[0] + DEN[8])
                const bool ok = wait_bar(num_full, nchunk & 1, ctl);
                tc_fence_after();
                uint32_t d[16], n0[32], n1[32];
                tmem_ld16_nowait(tmem + lane_base + PL::T_DEN, d);
                tmem_ld32_nowait(tmem + lane_base + PL::T_NUM + grp * HALF, n0);
                if constexpr (HALF == 64) tmem_ld32_nowait(tmem + lane_base + PL::T_NUM + grp * HALF + 32, n1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(num_free);
                if (ok && r < g.N - row0) {
                    const float inv = 1.f / (__uint_as_float(d[0]) + __uint_as_float(d[8]));
                    uint4 *orow = reinterpret_cast<uint4 *>(
                        out + ((long long)h * g.N + row0 + r) * DV + grp * HALF);
                    auto put = [&](const uint32_t(&v)[32], int j0) {
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            __stcs(orow + j0 + j,
                                   make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]) * inv,
                                                          __uint_as_float(v[8 * j + 1]) * inv),
                                              pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv,
                                                          __uint_as_float(v[8 * j + 3]) * inv),
                                              pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv,
                                                          __uint_as_float(v[8 * j + 5]) * inv),
                                              pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv,
                                                          __uint_as_float(v[8 * j + 7]) * inv)));
                    };
                    put(n0, 0);
                    if constexpr (HALF == 64) put(n1, 4);
                }
            }
            // the last chunk's state update; export after the head's last segment
            // (tcgen05.ld is warp-collective: the condition must be warp-uniform)
            const bool fin = __all_sync(0xffffffffu, wait_bar(s_done, (nchunk - 1) & 1, ctl));
            if (fin && s == g.nseg - 1 && srow && (S_out || z_out)) {
                tc_fence_after();
#pragma unroll
                for (int cb = 0; cb < HALF; cb += 32) {
                    uint32_t v[32];
                    tmem_ld32_nowait(tmem + lane_base + PL::T_S + grp * HALF + cb, v);
                    tmem_ld_wait();
                    if (S_out) {
                        float *dst = S_out + ((long long)h * DP + r) * DV + grp * HALF + cb;
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
                    z_out[(long long)h * DP + r] = __uint_as_float(zv[0]);
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

// Segment length L (chunks): the estimated makespan, in chunk-times, is
// waves * (L + [segmented] (L / 2 + 1)): phase C costs one chunk-time per
// chunk, phase A half of that (k, v only), and the chain about one more.
Geo plan(long long BH, int N, int sms)
{
    Geo g;
    g.BH = (int)BH;
    g.N = N;
    g.NC = cdiv(N, kC);
    int bestL = g.NC;   // one segment per head
    if (BH < sms) {
        double best = (double)((BH + sms - 1) / sms) * g.NC;
        for (int L = 1; L <= min(g.NC - 1, kMaxItemChunks); L++) {
            const int nseg = cdiv(g.NC, L);
            const long long waves = (BH * nseg + sms - 1) / sms;
            const double cost = (double)waves * (1.5 * L + 1.0);
            if (cost <= best) {
                best = cost;
                bestL = L;
            }
        }
    }
    g.L = bestL;
    g.nseg = cdiv(g.NC, g.L);
    g.n_items = (int)(BH * g.nseg);
    return g;
}

struct ScratchLayout {
    size_t flags, inclz, inclS, total, clear;
};

template <int DP, int DV>
ScratchLayout scratch_layout(const Geo &g)
{
    ScratchLayout L;
    const size_t n = (size_t)g.n_items;
    L.flags = 16;
    L.clear = L.flags + ((n * 4 + 15) & ~(size_t)15);
    L.inclz = L.clear;
    L.inclS = L.inclz + ((n * DP * 4 + 15) & ~(size_t)15);
    L.total = g.nseg > 1 ? L.inclS + n * DP * DV * 4 : L.clear;
    return L;
}

template <int DP, int DV>
cudaError_t run(const Problem &p, void *scratch, float *S_out, float *z_out, int *err,
                cudaStream_t s)
{
    using PL = Plan<DP, DV>;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, p.q, p.BH, p.N, p.D) || !make_map(&tk, p.k, p.BH, p.N, p.D) ||
        !make_map(&tv, p.v, p.BH, p.N, p.Dv))
        return cudaErrorInvalidValue;
    const int sms = num_sms();
    Geo g = plan(p.BH, p.N, sms);
    ScratchLayout L = scratch_layout<DP, DV>(g);
    unsigned char *b = (unsigned char *)scratch;
    Scratch sc;
    sc.ticket = (int *)b;
    sc.abort = (int *)(b + 4);
    sc.flags = (int *)(b + L.flags);
    sc.inclz = (float *)(b + L.inclz);
    sc.inclS = (float *)(b + L.inclS);
    cudaError_t e;
    if ((e = cudaMemsetAsync(scratch, 0, L.clear, s)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(tc_causal_kernel<DP, DV>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, PL::SMEM)) !=
        cudaSuccess)
        return e;
    const int grid = min(g.n_items, sms);
    tc_causal_kernel<DP, DV><<<grid, kThreads, PL::SMEM, s>>>(tq, tk, tv, g, sc,
                                                              (__nv_bfloat16 *)p.out, S_out, z_out, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    note_launches(1);
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
    Geo g = plan(p.BH, p.N, num_sms());
    if (p.D == 64 && p.Dv == 64) return scratch_layout<64, 64>(g).total;
    if (p.D == 64 && p.Dv == 128) return scratch_layout<64, 128>(g).total;
    if (p.D == 128 && p.Dv == 64) return scratch_layout<128, 64>(g).total;
    return scratch_layout<128, 128>(g).total;
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
