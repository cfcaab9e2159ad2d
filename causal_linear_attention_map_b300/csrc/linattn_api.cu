// linattn_api.cu -- the C ABI declared in include/linattn.h: argument
// validation on the host, kernel selection, and stream-ordered scratch from a
// library-owned CUDA memory pool per device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kernels.h"
#include "linattn.h"

namespace la {
std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace la

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCtx {
    bool pool_ready = false;
    cudaMemPool_t pool = nullptr;
    int *err_word = nullptr;   // device int: set by kernels whose bounded waits ran out
};

std::mutex g_mu;
DeviceCtx g_ctx[kMaxDevices];

// The per-device context of the current device (created on first use).
int get_ctx(DeviceCtx **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceCtx &c = g_ctx[dev];
    if (!c.pool_ready) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&c.pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_CUDA;
        }
        // keep freed blocks in the pool instead of returning them at every sync
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(c.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (cudaMalloc(&c.err_word, sizeof(int)) != cudaSuccess ||
            cudaMemset(c.err_word, 0, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            cudaMemPoolDestroy(c.pool);
            c.pool = nullptr;
            c.err_word = nullptr;
            return LA_ERR_CUDA;
        }
        c.pool_ready = true;
    }
    *out = &c;
    return LA_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool head_dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

bool prf_m_ok(int m) { return m == 16 || m == 32 || m == 64 || m == 128 || m == 256; }

// Shared checks of dtype, feature map and sizes; fills kind/m/W/P.
int check_common(int B, int H, int D, int Dv, const la_feature_map *fm, int dtype, int *kind,
                 int *m, const float **W, int *P)
{
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_DTYPE;
    *kind = fm ? fm->kind : LA_PHI_ELU1;
    *m = 0;
    *W = nullptr;
    if (*kind == LA_PHI_PRF) {
        if (!prf_m_ok(fm->m)) return LA_ERR_FEATURE;
        if (!fm->W) return LA_ERR_FEATURE;
        if (!aligned16(fm->W)) return LA_ERR_ALIGN;
        *m = fm->m;
        *W = fm->W;
    } else if (*kind != LA_PHI_ELU1) {
        return LA_ERR_FEATURE;
    }
    if (B < 0 || H < 0) return LA_ERR_DIM;
    if (!head_dim_ok(D) || !head_dim_ok(Dv)) return LA_ERR_DIM;
    *P = *kind == LA_PHI_PRF ? *m : D;
    if ((long long)*P * Dv > 32768) return LA_ERR_DIM;
    return LA_OK;
}

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return LA_OK;
    cudaGetLastError();
    return LA_ERR_CUDA;
}

int forward_impl(const void *q, const void *k, const void *v, void *out, int B, int H, int N,
                 int D, int Dv, int causal, const la_feature_map *fm, int dtype, void *stream,
                 float *S_out, float *z_out)
{
    int kind, m, P;
    const float *W;
    int st = check_common(B, H, D, Dv, fm, dtype, &kind, &m, &W, &P);
    if (st != LA_OK) return st;
    if (N < 0) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return LA_ERR_DIM;
    if (!aligned16(S_out) || !aligned16(z_out)) return LA_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    if (BH == 0) return LA_OK;
    if (N == 0) {   // empty sequence: nothing to compute, the memories are zero
        if (S_out && cudaMemsetAsync(S_out, 0, (size_t)BH * P * Dv * 4, s) != cudaSuccess)
            return cuda_status(cudaErrorUnknown);
        if (z_out && cudaMemsetAsync(z_out, 0, (size_t)BH * P * 4, s) != cudaSuccess)
            return cuda_status(cudaErrorUnknown);
        return LA_OK;
    }
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_ALIGN;

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

    DeviceCtx *ctx = nullptr;
    if ((st = get_ctx(&ctx)) != LA_OK) return st;

    const bool tc = la::tc_causal_supported(p) || la::tc_prf_supported(p);
    if (causal && !tc) return cuda_status(la::simt_causal(p, S_out, z_out, s));
    size_t bytes = tc ? la::tc_scratch_bytes(p, causal != 0) : la::noncausal_scratch_bytes(p);
    void *scratch = nullptr;
    if (bytes && cudaMallocFromPoolAsync(&scratch, bytes, ctx->pool, s) != cudaSuccess)
        return cuda_status(cudaErrorMemoryAllocation);
    cudaError_t e = tc ? la::tc_forward(p, causal != 0, scratch, S_out, z_out, ctx->err_word, s)
                       : la::noncausal(p, scratch, S_out, z_out, s);
    cudaError_t e2 = scratch ? cudaFreeAsync(scratch, s) : cudaSuccess;
    return cuda_status(e != cudaSuccess ? e : e2);
}

}  // namespace

extern "C" {

int la_forward(const void *q, const void *k, const void *v, void *out, int B, int H, int N, int D,
               int Dv, int causal, const la_feature_map *fm, int dtype, void *stream)
{
    return forward_impl(q, k, v, out, B, H, N, D, Dv, causal, fm, dtype, stream, nullptr,
                        nullptr);
}

int la_forward_ex(const void *q, const void *k, const void *v, void *out, int B, int H, int N,
                  int D, int Dv, int causal, const la_feature_map *fm, int dtype, void *stream,
                  float *S_out, float *z_out)
{
    return forward_impl(q, k, v, out, B, H, N, D, Dv, causal, fm, dtype, stream, S_out, z_out);
}

int la_step(float *S, float *z, const void *q, const void *k, const void *v, void *out, int B,
            int H, int D, int Dv, const la_feature_map *fm, int dtype, void *stream)
{
    int kind, m, P;
    const float *W;
    int st = check_common(B, H, D, Dv, fm, dtype, &kind, &m, &W, &P);
    if (st != LA_OK) return st;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return LA_ERR_DIM;
    if (BH == 0) return LA_OK;
    if (!S || !z || !q || !k || !v || !out) return LA_ERR_NULL;
    if (!aligned16(S) || !aligned16(z) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(out))
        return LA_ERR_ALIGN;
    return cuda_status(
        la::step(S, z, q, k, v, out, BH, D, Dv, P, kind, m, W, dtype, (cudaStream_t)stream));
}

const char *la_status_string(int status)
{
    switch (status) {
    case LA_OK: return "LA_OK: success";
    case LA_ERR_NULL: return "LA_ERR_NULL: a required pointer is NULL";
    case LA_ERR_DIM: return "LA_ERR_DIM: a size is negative or outside the supported set";
    case LA_ERR_DTYPE: return "LA_ERR_DTYPE: dtype must be LA_F32 or LA_BF16";
    case LA_ERR_FEATURE: return "LA_ERR_FEATURE: bad feature map (kind, W or m)";
    case LA_ERR_CUDA: return "LA_ERR_CUDA: a CUDA launch, allocation or query failed";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device-side wait ran out";
    case LA_ERR_ALIGN: return "LA_ERR_ALIGN: a tensor pointer is not 16-byte aligned";
    default: return "unknown linattn status";
    }
}

int la_check(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return cuda_status(cudaErrorUnknown);
    DeviceCtx *ctx = nullptr;
    int st = get_ctx(&ctx);
    if (st != LA_OK) return st;
    int flag = 0;
    if (cudaMemcpy(&flag, ctx->err_word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return cuda_status(cudaErrorUnknown);
    if (flag) {
        if (cudaMemset(ctx->err_word, 0, sizeof(int)) != cudaSuccess)
            return cuda_status(cudaErrorUnknown);
        return LA_ERR_TIMEOUT;
    }
    return LA_OK;
}

int la_selftest_timeout(int budget_ms, void *stream)
{
    DeviceCtx *ctx = nullptr;
    int st = get_ctx(&ctx);
    if (st != LA_OK) return st;
    return cuda_status(la::wait_selftest(budget_ms, ctx->err_word, (cudaStream_t)stream));
}

void la_shutdown(void)
{
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    for (int d = 0; d < kMaxDevices; d++) {
        DeviceCtx &c = g_ctx[d];
        if (!c.pool_ready) continue;
        cudaSetDevice(d);
        cudaDeviceSynchronize();
        cudaMemPoolDestroy(c.pool);
        cudaFree(c.err_word);
        c = DeviceCtx();
    }
    if (have_cur) cudaSetDevice(cur);
    cudaGetLastError();
}

int la_version(void) { return LA_VERSION; }

unsigned long long la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
