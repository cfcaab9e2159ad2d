// noncausal_noalloc.cu -- la_forward_noncausal_noalloc: the non-causal
// forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine): code that
// runs under an allocator it must not re-enter, real-time paths that forbid
// allocation after start-up, and embedders whose device memory is budgeted
// up front.  This entry point serves them: it takes its scratch (the
// partial sums phi(K)^T V and sum phi(k)) from a fixed array in device
// global memory that the library declares below, so it allocates nothing.
//
// Facts a caller needs:
//  - The array holds LA_NOALLOC_SCRATCH_BYTES (4 MiB).  A problem needs
//    B * H * Dphi * (Dv + 1) * 4 bytes; larger ones are rejected with
//    LA_ERR_DIM before anything is enqueued.
//  - On host code the array's name is only a host-side stand-in, not a
//    device address.  Its device address is looked up once per device with
//    cudaGetSymbolAddress, with that device current, on the first call made
//    on that device.  With CUDA's default lazy module loading that first
//    call is also when this file's module (and with it the array) and the
//    non-causal kernels are loaded onto the device: make it during start-up,
//    outside any no-allocation context and before any stream capture.  From
//    then on the device holds the array until the process exits.
//  - Every call shares the one array and it keeps the last call's contents;
//    the accumulators are cleared on the stream at the start of each call.
//    Calls that overlap on the GPU (other streams, other threads) race on
//    the array: serialise them.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "linattn.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
int noalloc_scratch(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LA_OK;
}

bool a16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

}  // namespace

extern "C" int la_forward_noncausal_noalloc(const void *q, const void *k, const void *v,
                                            void *out, int B, int H, int N, int D, int Dv,
                                            const la_feature_map *fm, int dtype, void *stream)
{
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_DTYPE;
    const int kind = fm ? fm->kind : LA_PHI_ELU1;
    int m = 0;
    const float *W = nullptr;
    if (kind == LA_PHI_PRF || kind == LA_PHI_NPRF || kind == LA_PHI_TRF) {
        m = fm->m;
        if (m != 16 && m != 32 && m != 64 && m != 128 && m != 256) return LA_ERR_FEATURE;
        if (kind == LA_PHI_TRF && m > 128) return LA_ERR_FEATURE;
        if (!fm->W) return LA_ERR_FEATURE;
        if (!a16(fm->W)) return LA_ERR_ALIGN;
        W = fm->W;
    } else if (kind != LA_PHI_ELU1) {
        return LA_ERR_FEATURE;
    }
    if (B < 0 || H < 0 || N < 0 || !dim_ok(D) || !dim_ok(Dv)) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    const int P = kind == LA_PHI_ELU1 ? D : kind == LA_PHI_TRF ? 2 * m : m;
    if (BH * P * (long long)(Dv + 1) * 4 > (long long)LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_DIM;
    if (BH == 0 || N == 0) return LA_OK;
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    if (!a16(q) || !a16(k) || !a16(v) || !a16(out)) return LA_ERR_ALIGN;

    void *scratch = nullptr;
    int st = noalloc_scratch(&scratch);
    if (st != LA_OK) return st;

    la::Problem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.BH = BH;
    p.N = N;
    p.D = D;
    p.Dv = Dv;
    p.P = P;
    p.kind = kind;
    p.m = m;
    p.W = W;
    p.dtype = dtype;
    // la::noncausal clears the accumulators in the array, then runs the two passes.
    cudaError_t e = la::noncausal(p, scratch, nullptr, nullptr, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    return LA_OK;
}
