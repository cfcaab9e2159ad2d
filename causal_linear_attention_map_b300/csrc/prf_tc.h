// prf_tc.h -- the causal random-feature forward with the feature map formed
// in the chunk kernel (prf_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "kernels.h"

namespace la {

// Causal, bf16, PRF or NPRF with D = Dv = 64 and m in {128, 256}: phi(q),
// phi(k) are formed on chip by a tcgen05 projection and never reach HBM.
// Scratch (prf_fused_scratch_bytes): per-segment sums when a head is cut into
// segments, and the first feature block's un-normalised sums when m = 256.
// `err` is the device word that bounded waits set on timeout.
bool prf_fused_supported(const Problem &p, bool causal);
size_t prf_fused_scratch_bytes(const Problem &p);
cudaError_t prf_fused_forward(const Problem &p, void *scratch, float *S_out, float *z_out, int *err,
                              cudaStream_t s);

}  // namespace la
