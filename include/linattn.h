/*
 * linattn.h -- C ABI of the B300 (sm_103a) kernelized linear-attention library.
 *
 * The method (review page "Transformers are RNNs: Fast Autoregressive
 * Transformers with Linear Attention", section "proposed method", bullets
 * 1-5): softmax attention is replaced by a kernel feature map phi, so that
 *
 *     out_i = phi(q_i)^T S_i / phi(q_i)^T z_i,
 *     S_i   = sum_{j<=i} phi(k_j) v_j^T      (Dphi x Dv),
 *     z_i   = sum_{j<=i} phi(k_j)            (Dphi),
 *
 * in the causal case (bullet 3: cumulative sums updated step by step); the
 * non-causal form uses the sums over all N positions (bullet 2: phi(K)^T V is
 * formed once and reused by every query).  The causal form is an RNN with
 * the two memories (S, z) (bullet 5), which la_step advances one token at a
 * time.  The sums include j = i.  No epsilon is added to the denominator.
 *
 * Feature maps:
 *   LA_PHI_ELU1  phi(x) = elu(x) + 1 (alpha = 1), elementwise; Dphi = D.
 *                ("main results", bullet 2: the elu-based feature map.)
 *   LA_PHI_PRF   positive random features, phi_r(x) = exp(w_r.x - |x|^2/2)/sqrt(m),
 *                r = 1..m, with W = [w_1..w_m] (m x D fp32) given by the
 *                caller; Dphi = m.  (Review page "Stable, Fast and Accurate:
 *                Kernelized Attention with Relative Positional Encoding",
 *                "proposed method", bullet 6, names PRF among the maps.)
 *
 * Conventions for every entry point:
 *  - Tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned (la_forward_host: q, k, v and out in HOST
 *    memory, the feature map's W on the device).  Heads are flattened as
 *    bh = b * H + h.
 *      q, k   [B, H, N, D]        v, out [B, H, N, Dv]     (dtype)
 *      S      [B, H, Dphi, Dv]    z      [B, H, Dphi]      (fp32)
 *      W      [m, D]                                       (fp32)
 *  - `dtype` is the type of q, k, v and out: LA_F32 or LA_BF16.  Arithmetic
 *    is fp32 (accumulators, state, feature map) in both cases.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously; nothing synchronises unless
 *    stated.  The device used is the current CUDA device of the calling thread.
 *  - Return value: LA_OK (0) or a negative la_status.  Argument errors are
 *    detected on the host before anything is enqueued and leave all outputs
 *    untouched.  LA_ERR_CUDA reports a failed launch or allocation
 *    (cudaGetLastError is consumed).  Nothing is thrown and nothing aborts.
 *  - Supported sizes: B, H, N >= 0 (a zero size is a no-op that returns
 *    LA_OK; la_forward_ex then writes zero states); D and Dv in
 *    {16, 32, 64, 128}; random-feature m in {16, 32, 64, 128, 256}, TRF
 *    m <= 128 (else LA_ERR_FEATURE); Dphi * Dv <= 32768.
 *  - Execution: bf16 inputs with elu+1 and D, Dv in {64, 128}, or with PRF or
 *    NPRF, D = 64 and (m = 128, Dv in {64, 128}) or (m = 256, Dv = 64), run on
 *    the tensor cores (tcgen05); causal PRF / NPRF with D = Dv = 64 form
 *    phi(q), phi(k) inside the chunk kernels, the other random-feature cases
 *    write them to scratch first; every other supported case (fp32, TRF,
 *    other sizes) runs on the CUDA cores.  All compute the same sums;
 *    rounding differs.
 *  - Scratch: la_forward may take stream-ordered scratch memory from a
 *    library-owned CUDA memory pool on the current device (per-segment
 *    states of the causal scan, partial sums of the non-causal pass, row
 *    norms and block partial sums of random features formed on chip, the
 *    phi(q), phi(k) tiles of the other random-feature cases); it is returned to the pool,
 *    in stream order, before the call returns.  la_shutdown() releases the
 *    pools.
 */
#ifndef LINATTN_H
#define LINATTN_H

#ifdef __cplusplus
extern "C" {
#endif

#define LA_VERSION 100

typedef enum {
    LA_F32 = 0,  /* float32 q, k, v, out */
    LA_BF16 = 1  /* bfloat16 q, k, v, out */
} la_dtype;

/* Feature maps (review page "Stable, Fast and Accurate: Kernelized Attention
 * with Relative Positional Encoding", proposed method: PRF, TRF, Sphere-PRF,
 * ORF and the normalised NPRF are supported maps; the page names them without
 * formulas, and these are the standard definitions).  Sphere-PRF and ORF are
 * LA_PHI_PRF with W drawn by la_random_features (LA_W_SPHERE, LA_W_ORTHOGONAL). */
typedef enum {
    LA_PHI_ELU1 = 0, /* elu(x) + 1                                        Dphi = D  */
    LA_PHI_PRF = 1,  /* exp(Wx - |x|^2/2) / sqrt(m)                       Dphi = m  */
    LA_PHI_NPRF = 2, /* PRF of x/|x|: exp(Wx/|x| - 1/2) / sqrt(m)         Dphi = m  */
    LA_PHI_TRF = 3   /* exp(|x|^2/2)/sqrt(m) [cos(Wx), sin(Wx)]           Dphi = 2m */
} la_feature_kind;

/* Feature-map descriptor.  Host memory, read during the call only.
 * kind: la_feature_kind.  m: the number of projections (rows of W; ignored
 * for ELU1): 16, 32, 64, 128 or 256 (TRF: at most 128).
 * W: DEVICE pointer to the m x D fp32 row-major projection (NULL for ELU1).
 * A NULL descriptor means ELU1.  TRF's features are not positive, so its
 * denominator can approach zero; PRF and NPRF keep it positive. */
typedef struct {
    int kind;
    int m;
    const float *W;
} la_feature_map;

typedef enum {
    LA_OK = 0,
    LA_ERR_NULL = -1,    /* a required pointer is NULL */
    LA_ERR_DIM = -2,     /* a size is negative or outside the supported set */
    LA_ERR_DTYPE = -3,   /* dtype is not LA_F32 / LA_BF16 */
    LA_ERR_FEATURE = -4, /* bad feature map (unknown kind, PRF without W, bad m) */
    LA_ERR_CUDA = -5,    /* a CUDA launch, allocation or query failed */
    LA_ERR_TIMEOUT = -6, /* a bounded device-side wait ran out (reported by la_check) */
    LA_ERR_ALIGN = -7,   /* a tensor pointer is not 16-byte aligned */
    LA_ERR_RANGE = -8    /* the tensor-core backward met a value outside fp16's
                            range (reported by la_check) */
} la_status;

/*
 * la_forward -- kernelized attention over whole sequences.
 *   causal != 0: out_i uses the prefix sums S_i, z_i (j <= i).
 *   causal == 0: out_i uses the full sums over j = 0..N-1.
 * q, k, v (inputs) and out (output) as in the conventions above; `out` must
 * not alias the inputs.
 */
int la_forward(const void *q, const void *k, const void *v, void *out,
               int B, int H, int N, int D, int Dv, int causal,
               const la_feature_map *fm, int dtype, void *stream);

/*
 * la_forward_ex -- la_forward that also exports the memories after the last
 * position: S_out [B, H, Dphi, Dv] = sum_j phi(k_j) v_j^T and
 * z_out [B, H, Dphi] = sum_j phi(k_j), fp32, device.  Either may be NULL.
 * These are the RNN state that la_step continues from (the state after a
 * prefix of the sequence is the checkpoint of the recurrence).
 */
int la_forward_ex(const void *q, const void *k, const void *v, void *out,
                  int B, int H, int N, int D, int Dv, int causal,
                  const la_feature_map *fm, int dtype, void *stream,
                  float *S_out, float *z_out);

/*
 * la_forward_host -- la_forward with q, k, v (inputs) and out (output) in
 * host memory, same layouts; the feature map's W stays in device memory.
 * The B*H heads are split into up to 16 groups of consecutive heads, which
 * flow through three stages on three streams: the host-to-device copy of
 * a group's q, k, v (a library stream), its forward (on `stream`) and the
 * device-to-host copy of its out (a second library stream).  So the copies
 * in both directions and the compute overlap, and a step costs about its
 * larger copy direction.  Device buffers for the whole problem come from
 * the library's stream-ordered pool and go back to it at the end.
 * Ordering: the first copy starts after the work queued on `stream` before
 * the call, and work queued on `stream` after the call starts after the last
 * copy has completed.  The host buffers must stay valid, and unmodified, until
 * then (synchronise `stream`).  Page-locked host buffers (cudaHostAlloc,
 * cudaHostRegister) give overlapped asynchronous copies; pageable ones give
 * the same results with the copies staged by the driver.  Each group's
 * segments are planned for that group alone, so outputs equal la_forward's
 * within the parity tolerances (not bit for bit).  Status codes as
 * la_forward; a host pointer the driver rejects gives LA_ERR_CUDA.
 */
int la_forward_host(const void *q, const void *k, const void *v, void *out,
                    int B, int H, int N, int D, int Dv, int causal,
                    const la_feature_map *fm, int dtype, void *stream);

/*
 * la_step -- one recurrent decode step for B*H independent heads ("proposed
 * method", bullet 5; "main results", bullet 3: the state is updated
 * incrementally).  In place on the fp32 memories:
 *     S += phi(k) v^T ;  z += phi(k) ;  out = phi(q)^T S / phi(q)^T z
 * (update first, then read out, matching the inclusive sums of la_forward).
 * S [B, H, Dphi, Dv] and z [B, H, Dphi] fp32 (in/out); q, k [B, H, D] and
 * v [B, H, Dv] (in), out [B, H, Dv] (out), all in `dtype`, device.  Calling
 * la_step N times from zero memories gives la_forward's causal outputs.
 */
int la_step(float *S, float *z, const void *q, const void *k, const void *v,
            void *out, int B, int H, int D, int Dv,
            const la_feature_map *fm, int dtype, void *stream);

/*
 * la_backward -- gradients of the forward ("proposed method", bullet 4: the
 * gradients of forward and backward propagation are computed in linear time,
 * with cumulative sums).  For L = sum over all elements of dout * out, where
 * out is la_forward(q, k, v, ..., causal, fm) with the same arguments:
 *     dq = dL/dq, dk = dL/dk, dv = dL/dv.
 * With g_i = phi(q_i), f_j = phi(k_j), den_i = g_i . z_i:
 *     dnum_i = dout_i / den_i,  dden_i = -(dout_i . out_i) / den_i,
 *     dL/dg_i = S_i dnum_i + z_i dden_i,
 *     dL/df_j = R_j v_j + r_j,  dL/dv_j = R_j^T f_j,
 *     R_j = sum_{i>=j} g_i dnum_i^T,  r_j = sum_{i>=j} g_i dden_i
 * (all positions instead of i >= j / j <= i when causal = 0), then through
 * phi to q and k (PRF: W is treated as a constant; no gradient for W).
 * q, k, dq, dk [B, H, N, D]; v, dout, dv [B, H, N, Dv]; all in `dtype`,
 * device, 16-byte aligned; dq, dk, dv are written, the rest read.  Same
 * feature maps, sizes and errors as la_forward, except that Dphi * Dv must
 * be at most 16384 (else LA_ERR_DIM).  bf16 elu+1 with D = Dv in {64, 128}
 * runs on the tensor cores with fp16 operands (dnum as an fp16 hi + lo pair,
 * per-chunk power-of-two scales; fp32 accumulation); a q, k or v entry of
 * magnitude >= 2^16 or not finite, scores phi(q).phi(k) or intra-chunk terms
 * that overflow fp16 after those scales, or a denominator below 1e-30, make
 * la_check report LA_ERR_RANGE (the results are then not to be used; the
 * fp32 path takes such inputs).  Every other case runs on the CUDA cores with fp32
 * arithmetic.  Takes stream-ordered scratch from the library's pool
 * (per-segment memories, and den, dden per position: 8 bytes per
 * position and head).  den and out are recomputed, not read.
 */
int la_backward(const void *q, const void *k, const void *v, const void *dout,
                void *dq, void *dk, void *dv, int B, int H, int N, int D, int Dv,
                int causal, const la_feature_map *fm, int dtype, void *stream);

/*
 * la_forward_rpe -- kernelized attention with relative positional encoding
 * (review page "Stable, Fast and Accurate: Kernelized Attention with
 * Relative Positional Encoding", proposed method: the RPE matrix is Toeplitz
 * - it depends only on i - j - and multiplies the kernelized attention):
 *   out_i = sum_{j in J(i)} c_{i-j} (phi(q_i).phi(k_j)) v_j
 *           / sum_{j in J(i)} c_{i-j} phi(q_i).phi(k_j),        c_t = exp(b_t)
 * with J(i) = {0..i} when causal, else all positions.  bias: DEVICE fp32
 * [H, 2N - 1], row h the log-weights b of head h (shared by every batch
 * row), b_t at index t + N - 1 for t = i - j.  Other arguments, layouts and
 * feature maps as la_forward.  The page multiplies by the Toeplitz matrix
 * with FFTs; this library evaluates the weighted form chunk against chunk
 * (O(N^2) work per head, on the tensor cores for bf16 elu+1 with D, Dv in
 * {64, 128}, else on the CUDA cores): see the source for the cost
 * comparison.  Allocates nothing; bounded waits report through la_check.
 */
int la_forward_rpe(const void *q, const void *k, const void *v, const float *bias, void *out,
                   int B, int H, int N, int D, int Dv, int causal,
                   const la_feature_map *fm, int dtype, void *stream);

/*
 * la_prefix_attention -- softmax attention read as an RNN, with its
 * many-to-many outputs (review page "Attention as an RNN", proposed method:
 * attention is a many-to-one RNN over the keys and values with a learned
 * query token q; its outputs after every prefix come from a parallel prefix
 * scan).  Per head, with s_i = q . k_i (no 1/sqrt(D) factor: scale q):
 *     out_k = sum_{i<=k} exp(s_i) v_i / sum_{i<=k} exp(s_i)     (k = 0..N-1)
 * The RNN state is (m, u, w): the largest score so far, sum exp(s_i - m) and
 * sum exp(s_i - m) v_i.  q [B, H, D]; k [B, H, N, D]; v, out [B, H, N, Dv]
 * in `dtype` (device); state_out (nullable, device fp32 [B, H, Dv + 2], laid
 * out as m, u, w_0..w_{Dv-1}) receives each head's state after position
 * N - 1 (for N = 0: the empty state m = -inf, u = 0, w = 0), which
 * la_prefix_step continues from.  D, Dv in {16, 32, 64, 128}.  One pass over
 * K and V (a single-pass scan with decoupled look-back across tiles of 256
 * positions); takes stream-ordered scratch from the library's pool.  Bounded
 * waits: a wait on another tile that runs out sets the error that la_check
 * reports as LA_ERR_TIMEOUT.
 */
int la_prefix_attention(const void *q, const void *k, const void *v, void *out,
                        float *state_out, int B, int H, int N, int D, int Dv,
                        int dtype, void *stream);

/*
 * la_prefix_step -- one token of the same RNN for B*H heads ("Attention as
 * an RNN": new tokens update the constant-size state): with s = q . k,
 *     m' = max(m, s),  u' = u e^(m - m') + e^(s - m'),
 *     w' = w e^(m - m') + e^(s - m') v,   out = w' / u'.
 * state [B, H, Dv + 2] fp32 (in/out, device); q, k [B, H, D], v, out
 * [B, H, Dv] in `dtype` (device).  Starting from the empty state and
 * stepping through a sequence gives la_prefix_attention's outputs.
 */
int la_prefix_step(float *state, const void *q, const void *k, const void *v, void *out,
                   int B, int H, int D, int Dv, int dtype, void *stream);

/*
 * la_random_features -- draw a projection W (m x D fp32, row-major) into
 * HOST memory `W`, deterministically from `seed` (a SplitMix64 counter
 * stream turned into N(0, 1) draws by the Box-Muller transform):
 *   LA_W_GAUSSIAN    every entry iid N(0, 1) (plain PRF / TRF / NPRF);
 *   LA_W_ORTHOGONAL  orthogonal random features: rows in blocks of D that are
 *                    orthogonal (Gram-Schmidt of a Gaussian D x D matrix),
 *                    each row rescaled to the norm of an independent
 *                    Gaussian D-vector (the last block keeps m mod D rows);
 *   LA_W_SPHERE      each row uniform on the sphere of radius sqrt(D)
 *                    (Sphere-PRF).
 * m, D >= 1.  Host-only: no device work.  Returns LA_ERR_NULL / LA_ERR_DIM /
 * LA_ERR_FEATURE (unknown w_kind) or LA_OK.
 */
typedef enum { LA_W_GAUSSIAN = 0, LA_W_ORTHOGONAL = 1, LA_W_SPHERE = 2 } la_w_kind;
int la_random_features(int w_kind, int m, int D, unsigned long long seed, float *W);

/* Human-readable name of a status code (static string, never NULL). */
const char *la_status_string(int status);

/*
 * la_check -- synchronise `stream` and report deferred device-side errors:
 * LA_ERR_TIMEOUT if a bounded wait inside a kernel of this library ran out
 * since the last la_check on this device, LA_ERR_RANGE if the tensor-core
 * backward met a value outside fp16's range (either flag is then cleared),
 * LA_ERR_CUDA if the stream reports an error, else LA_OK.
 */
int la_check(void *stream);

/*
 * la_selftest_timeout -- exercise the library's failure detection without
 * faulting the GPU: launches one small kernel on `stream` whose bounded
 * mbarrier wait (the same wait every tensor-core kernel uses) waits for a
 * phase that nothing completes.  After `budget_ms` milliseconds of SM clock
 * (clamped to 1..2000) the wait gives up, sets this device's error word and
 * the kernel returns normally, so the next la_check on the device returns
 * LA_ERR_TIMEOUT (and clears it) while the context stays usable.
 * Returns LA_OK once launched, LA_ERR_CUDA if the launch fails.
 */
int la_selftest_timeout(int budget_ms, void *stream);

/* Release the library's memory pools on every device it used.  Must not be
 * called while work from this library is still running. */
void la_shutdown(void);

/* LA_VERSION of the built library. */
int la_version(void);

/* Number of CUDA kernels this library has launched in this process (all
 * devices, all entry points).  Host-side counter; for accounting only. */
unsigned long long la_launch_count(void);

/*
 * la_forward_noncausal_noalloc -- the non-causal la_forward (causal = 0) for
 * callers that cannot allocate device memory: code running inside an
 * allocator or a memory-budgeted embedder, or real-time paths that forbid
 * cudaMalloc after start-up.  The method's pages have no counterpart; this
 * is a library convenience.
 *
 * Same arguments and layouts as la_forward with causal = 0; its results
 * agree with la_forward's within the same tolerances, not bit for bit,
 * because it always runs the CUDA-core non-causal kernels (fp32 arithmetic,
 * both passes), never the tensor-core path.  It is correspondingly slower:
 * about 17x on the B=8, H=8, N=4096, D=Dv=64 bf16 workload (914 us against
 * 55 us for la_forward).
 *
 * Steady-state calls allocate nothing: the scratch is a fixed device array
 * of LA_NOALLOC_SCRATCH_BYTES.  A problem needs B * H * Dphi * (Dv + 1) * 4
 * bytes of it; larger problems return LA_ERR_DIM before anything is
 * enqueued.  The FIRST call on each device is different: with CUDA's
 * default lazy module loading, the array (4 MiB) and the code of the
 * kernels it uses are loaded onto the device at that call, which is when
 * the library also looks up the array's device address
 * (cudaGetSymbolAddress, with that device current).  Make that first call
 * during start-up, outside any no-allocation context and before any stream
 * capture; from then on the device holds the array until the process exits.
 * All calls share the array, which keeps the last call's contents (each
 * call clears what it accumulates into); calls that overlap on the GPU
 * race, so serialise them.
 */
#define LA_NOALLOC_SCRATCH_BYTES (4u << 20)
int la_forward_noncausal_noalloc(const void *q, const void *k, const void *v, void *out,
                                 int B, int H, int N, int D, int Dv,
                                 const la_feature_map *fm, int dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
