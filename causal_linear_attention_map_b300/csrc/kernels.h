// kernels.h -- internal interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace la {

// Adds n to the library's launch counter (la_launch_count).
void note_launches(int n);

enum { DT_F32 = 0, DT_BF16 = 1 };
enum { PHI_ELU1 = 0, PHI_PRF = 1, PHI_NPRF = 2, PHI_TRF = 3 };

// One validated forward problem.  Pointers are device pointers.
struct Problem {
    const void *q, *k, *v;
    void *out;
    long long BH;  // B * H heads
    int N, D, Dv;
    int P;         // feature dimension: D (elu+1), m (PRF, NPRF) or 2m (TRF)
    int kind;      // PHI_*
    int m;
    const float *W;
    int dtype;     // DT_*
};

// CUDA-core (SIMT) chunked causal kernel, one CTA per head.  Any supported
// size; the fp32 path and the fallback for shapes the tensor-core kernel
// does not take.
cudaError_t simt_causal(const Problem &p, float *S_out, float *z_out, cudaStream_t s);

// Tensor-core (tcgen05) forward, causal or not, bf16:
//   elu + 1 with D, Dv in {64, 128} (tc_causal_supported), applied in the
//   tile loads;
//   random features with D = 64 and (m = 128, Dv in {64, 128}) or
//   (m = 256, Dv = 64) (tc_prf_supported): phi(q), phi(k) materialised in
//   bf16 scratch by a tcgen05 projection kernel, then the same chunk kernels.
// Scratch (tc_scratch_bytes): control words, segment sums, per-head totals
// (non-causal), phi tiles and partial sums (random features).  `err` is the
// device word that bounded waits set on timeout.
bool tc_causal_supported(const Problem &p);
bool tc_prf_supported(const Problem &p);
size_t tc_scratch_bytes(const Problem &p, bool causal);
cudaError_t tc_forward(const Problem &p, bool causal, void *scratch, float *S_out, float *z_out, int *err,
                       cudaStream_t s);

// Failure-detection self-test: one bounded wait that runs out after about
// budget_ms of SM clock and sets *err (see la_selftest_timeout).
cudaError_t wait_selftest(int budget_ms, int *err, cudaStream_t s);

// Non-causal: KV = phi(K)^T V and ksum = sum phi(k) reduced over N into
// fp32 scratch (KV [BH, P, Dv], ksum [BH, P]; zeroed here), then the readout.
size_t noncausal_scratch_bytes(const Problem &p);
cudaError_t noncausal(const Problem &p, void *scratch, float *S_out, float *z_out,
                      cudaStream_t s);

// Gradients dq, dk, dv of sum(dout * out) for the forward of the same
// arguments, any dtype and feature map with Dphi * Dv <= 16384
// (backward_supported): on the tensor cores for bf16 elu+1 with D = Dv in
// {64, 128} (backward_tc_supported, fp16 operands; an operand outside fp16's
// range sets the error word to 2), else on the CUDA cores (fp32 arithmetic).
// Scratch (backward_scratch_bytes): per-segment forward and reverse memories
// and per-position den, dden.
bool backward_supported(const Problem &p);
size_t backward_scratch_bytes(const Problem &p, bool causal);
cudaError_t backward(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal,
                     void *scratch, int *err, cudaStream_t s);
bool backward_tc_supported(const Problem &p);
size_t backward_tc_scratch_bytes(const Problem &p, bool causal);
cudaError_t backward_tc(const Problem &p, const void *dout, void *dq, void *dk, void *dv, bool causal,
                        void *scratch, int *err, cudaStream_t s);
// Exclusive prefix (mode 0), exclusive suffix (1) or total (2) over a head's
// segments of the per-segment memories st [BH, nseg, elems], in place.
cudaError_t backward_scan(float *st, long long BH, int nseg, int elems, int mode, cudaStream_t s);

// Softmax attention of one query token per head over every prefix (the
// many-to-many outputs of attention as an RNN), one pass with decoupled
// look-back over tiles; state (m, u, w) [BH, Dv + 2].  D, Dv <= 128.
size_t prefix_scratch_bytes(long long BH, int N, int Dv);
cudaError_t prefix_attention(const void *q, const void *k, const void *v, void *out, float *state_out,
                             long long BH, int N, int D, int Dv, int dtype, void *scratch, int *err,
                             cudaStream_t s);
cudaError_t prefix_empty_state(float *state, long long BH, int Dv, cudaStream_t s);
cudaError_t prefix_step(float *state, const void *q, const void *k, const void *v, void *out, long long BH,
                        int D, int Dv, int dtype, cudaStream_t s);

// Kernelized attention with a Toeplitz relative-position weight exp(b_{i-j}),
// b [H, 2N - 1] fp32 (device): the tensor-core kernel for bf16 elu+1 with D,
// Dv in {64, 128} (rpe_tc_supported), else a CUDA-core kernel.
bool rpe_tc_supported(const Problem &p);
cudaError_t rpe_tc_forward(const Problem &p, const float *bias, int H, bool causal, int *err, cudaStream_t s);
cudaError_t rpe_forward(const Problem &p, const float *bias, int H, bool causal, int *err, cudaStream_t s);

// One recurrent decode step for BH heads, in place on S [BH, P, Dv], z [BH, P].
cudaError_t step(float *S, float *z, const void *q, const void *k, const void *v, void *out,
                 long long BH, int D, int Dv, int P, int kind, int m, const float *W,
                 int dtype, cudaStream_t s);

}  // namespace la
