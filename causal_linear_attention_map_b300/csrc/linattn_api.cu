// linattn_api.cu -- the C ABI declared in include/linattn.h: argument
// validation on the host, kernel selection, and stream-ordered scratch from a
// library-owned CUDA memory pool per device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kernels.h"
#include "prf_tc.h"
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
    cudaStream_t h2d = nullptr, d2h = nullptr;   // la_forward_host copy streams (created on first use)
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
    if (*kind == LA_PHI_PRF || *kind == LA_PHI_NPRF || *kind == LA_PHI_TRF) {
        if (!prf_m_ok(fm->m) || (*kind == LA_PHI_TRF && fm->m > 128)) return LA_ERR_FEATURE;
        if (!fm->W) return LA_ERR_FEATURE;
        if (!aligned16(fm->W)) return LA_ERR_ALIGN;
        *m = fm->m;
        *W = fm->W;
    } else if (*kind != LA_PHI_ELU1) {
        return LA_ERR_FEATURE;
    }
    if (B < 0 || H < 0) return LA_ERR_DIM;
    if (!head_dim_ok(D) || !head_dim_ok(Dv)) return LA_ERR_DIM;
    *P = *kind == LA_PHI_ELU1 ? D : *kind == LA_PHI_TRF ? 2 * *m : *m;
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

    if (la::prf_fused_supported(p, causal != 0)) {
        // causal random features with the feature map formed on chip
        const size_t fb = la::prf_fused_scratch_bytes(p);
        void *scratch = nullptr;
        if (fb && cudaMallocFromPoolAsync(&scratch, fb, ctx->pool, s) != cudaSuccess)
            return cuda_status(cudaErrorMemoryAllocation);
        cudaError_t e = la::prf_fused_forward(p, scratch, S_out, z_out, ctx->err_word, s);
        cudaError_t e2 = scratch ? cudaFreeAsync(scratch, s) : cudaSuccess;
        return cuda_status(e != cudaSuccess ? e : e2);
    }
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

int backward_impl(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk,
                  void *dv, int B, int H, int N, int D, int Dv, int causal, const la_feature_map *fm,
                  int dtype, void *stream)
{
    int kind, m, P;
    const float *W;
    int st = check_common(B, H, D, Dv, fm, dtype, &kind, &m, &W, &P);
    if (st != LA_OK) return st;
    if (N < 0) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return LA_ERR_DIM;
    if ((long long)P * Dv > 16384) return LA_ERR_DIM;
    if (BH == 0 || N == 0) return LA_OK;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return LA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return LA_ERR_ALIGN;
    la::Problem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = nullptr;
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
    cudaStream_t s = (cudaStream_t)stream;
    void *scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, la::backward_scratch_bytes(p, causal != 0), ctx->pool, s) != cudaSuccess)
        return cuda_status(cudaErrorMemoryAllocation);
    cudaError_t e = la::backward(p, dout, dq, dk, dv, causal != 0, scratch, ctx->err_word, s);
    cudaError_t e2 = cudaFreeAsync(scratch, s);
    return cuda_status(e != cudaSuccess ? e : e2);
}

int prefix_impl(const void *q, const void *k, const void *v, void *out, float *state_out, int B, int H, int N,
                int D, int Dv, int dtype, void *stream)
{
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_DTYPE;
    if (B < 0 || H < 0 || N < 0 || !head_dim_ok(D) || !head_dim_ok(Dv)) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL || BH * (((long long)N + 255) / 256) > 0x7fffffffLL) return LA_ERR_DIM;
    if (!aligned16(state_out)) return LA_ERR_ALIGN;
    cudaStream_t s = (cudaStream_t)stream;
    if (BH == 0) return LA_OK;
    if (N == 0) {   // empty sequence: the empty state (m = -inf, u = 0, w = 0)
        if (!state_out) return LA_OK;
        return cuda_status(la::prefix_empty_state(state_out, BH, Dv, s));
    }
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_ALIGN;
    DeviceCtx *ctx = nullptr;
    int st = get_ctx(&ctx);
    if (st != LA_OK) return st;
    void *scratch = nullptr;
    if (cudaMallocFromPoolAsync(&scratch, la::prefix_scratch_bytes(BH, N, Dv), ctx->pool, s) != cudaSuccess)
        return cuda_status(cudaErrorMemoryAllocation);
    cudaError_t e = la::prefix_attention(q, k, v, out, state_out, BH, N, D, Dv, dtype, scratch, ctx->err_word, s);
    cudaError_t e2 = cudaFreeAsync(scratch, s);
    return cuda_status(e != cudaSuccess ? e : e2);
}

int rpe_impl(const void *q, const void *k, const void *v, const float *bias, void *out, int B, int H, int N, int D,
             int Dv, int causal, const la_feature_map *fm, int dtype, void *stream)
{
    int kind, m, P;
    const float *W;
    int st = check_common(B, H, D, Dv, fm, dtype, &kind, &m, &W, &P);
    if (st != LA_OK) return st;
    if (N < 0) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL || (long long)N * 2 > 0x7fffffffLL) return LA_ERR_DIM;
    if (BH == 0 || N == 0) return LA_OK;
    if (!q || !k || !v || !bias || !out) return LA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(bias)) return LA_ERR_ALIGN;
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
    return cuda_status(la::rpe_forward(p, bias, H, causal != 0, ctx->err_word, (cudaStream_t)stream));
}

// la_forward_host: at most kHostGroups head groups, each with at least
// kHostGroupBytes of inputs (a group's forward has a fixed cost of a few
// launches, so small problems take few groups)
constexpr int kHostGroups = 16;
constexpr size_t kHostGroupBytes = 16u << 20;

// The copy streams of la_forward_host on this device (created once).
int host_streams(DeviceCtx *c)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (c->h2d && c->d2h) return LA_OK;
    if (!c->h2d && cudaStreamCreateWithFlags(&c->h2d, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_status(cudaErrorUnknown);
    if (!c->d2h && cudaStreamCreateWithFlags(&c->d2h, cudaStreamNonBlocking) != cudaSuccess)
        return cuda_status(cudaErrorUnknown);
    return LA_OK;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

int forward_host_impl(const void *q, const void *k, const void *v, void *out, int B, int H, int N, int D,
                      int Dv, int causal, const la_feature_map *fm, int dtype, void *stream)
{
    int kind, m, P;
    const float *W;
    int st = check_common(B, H, D, Dv, fm, dtype, &kind, &m, &W, &P);
    if (st != LA_OK) return st;
    if (N < 0) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return LA_ERR_DIM;
    if (BH == 0 || N == 0) return LA_OK;   // nothing to copy or compute
    if (!q || !k || !v || !out) return LA_ERR_NULL;
    DeviceCtx *ctx = nullptr;
    if ((st = get_ctx(&ctx)) != LA_OK) return st;
    if ((st = host_streams(ctx)) != LA_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;

    const size_t es = dtype == LA_F32 ? 4 : 2;
    const size_t qh = (size_t)N * D * es, vh = (size_t)N * Dv * es;   // bytes per head
    const size_t oq = 0, ok = round256(BH * qh), ov = ok + round256(BH * qh), oo = ov + round256(BH * vh);
    const size_t total = oo + round256(BH * vh);
    const size_t in_bytes = BH * (2 * qh + vh);
    long long want = (long long)(in_bytes / kHostGroupBytes);
    want = want < 1 ? 1 : want > kHostGroups ? kHostGroups : want;
    const long long hg = (BH + want - 1) / want;   // heads per group
    const int G = (int)((BH + hg - 1) / hg);

    // events: the buffer is allocated; per group its inputs are in, its outputs are out
    cudaEvent_t ev[2 * kHostGroups + 2] = {};
    const int nev = 2 * G + 2;
    for (int i = 0; i < nev; i++)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; j++) cudaEventDestroy(ev[j]);
            return cuda_status(cudaErrorUnknown);
        }
    cudaEvent_t ev_alloc = ev[0], ev_done = ev[1], *ev_in = ev + 2, *ev_fw = ev + 2 + G;

    unsigned char *d = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync((void **)&d, total, ctx->pool, s);
    if (e == cudaSuccess) e = cudaEventRecord(ev_alloc, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->h2d, ev_alloc, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->d2h, ev_alloc, 0);
    for (int g = 0; g < G && e == cudaSuccess && st == LA_OK; g++) {
        const long long h0 = g * hg, nh = BH - h0 < hg ? BH - h0 : hg;
        const size_t bq = h0 * qh, bv = h0 * vh;
        e = cudaMemcpyAsync(d + oq + bq, (const unsigned char *)q + bq, nh * qh, cudaMemcpyHostToDevice, ctx->h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d + ok + bq, (const unsigned char *)k + bq, nh * qh, cudaMemcpyHostToDevice,
                                ctx->h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(d + ov + bv, (const unsigned char *)v + bv, nh * vh, cudaMemcpyHostToDevice,
                                ctx->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in[g], ctx->h2d);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_in[g], 0);
        if (e != cudaSuccess) break;
        // the group's heads as B = 1, H = nh (heads are contiguous in [B, H, N, .])
        st = forward_impl(d + oq + bq, d + ok + bq, d + ov + bv, d + oo + bv, 1, (int)nh, N, D, Dv, causal, fm,
                          dtype, stream, nullptr, nullptr);
        if (st != LA_OK) break;
        e = cudaEventRecord(ev_fw[g], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->d2h, ev_fw[g], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync((unsigned char *)out + bv, d + oo + bv, nh * vh, cudaMemcpyDeviceToHost, ctx->d2h);
    }
    // join both copy streams back into `stream` (also after a failure, so that
    // the buffer is released only once nothing uses it), then release it
    cudaError_t e2 = cudaEventRecord(ev_done, ctx->d2h);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev_done, 0);
    cudaEvent_t ev_in_done = ev_alloc;   // reused: the last host-to-device copy
    if (e2 == cudaSuccess) e2 = cudaEventRecord(ev_in_done, ctx->h2d);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev_in_done, 0);
    if (d && e2 == cudaSuccess) e2 = cudaFreeAsync(d, s);
    for (int i = 0; i < nev; i++) cudaEventDestroy(ev[i]);   // released once they have completed
    if (st != LA_OK) return st;
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

int la_forward_host(const void *q, const void *k, const void *v, void *out, int B, int H, int N, int D,
                    int Dv, int causal, const la_feature_map *fm, int dtype, void *stream)
{
    return forward_host_impl(q, k, v, out, B, H, N, D, Dv, causal, fm, dtype, stream);
}

int la_backward(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk, void *dv,
                int B, int H, int N, int D, int Dv, int causal, const la_feature_map *fm, int dtype,
                void *stream)
{
    return backward_impl(q, k, v, dout, dq, dk, dv, B, H, N, D, Dv, causal, fm, dtype, stream);
}

int la_prefix_attention(const void *q, const void *k, const void *v, void *out, float *state_out, int B, int H,
                        int N, int D, int Dv, int dtype, void *stream)
{
    return prefix_impl(q, k, v, out, state_out, B, H, N, D, Dv, dtype, stream);
}

int la_prefix_step(float *state, const void *q, const void *k, const void *v, void *out, int B, int H, int D,
                   int Dv, int dtype, void *stream)
{
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_DTYPE;
    if (B < 0 || H < 0 || !head_dim_ok(D) || !head_dim_ok(Dv)) return LA_ERR_DIM;
    const long long BH = (long long)B * H;
    if (BH > 0x7fffffffLL) return LA_ERR_DIM;
    if (BH == 0) return LA_OK;
    if (!state || !q || !k || !v || !out) return LA_ERR_NULL;
    if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return LA_ERR_ALIGN;
    return cuda_status(la::prefix_step(state, q, k, v, out, BH, D, Dv, dtype, (cudaStream_t)stream));
}

int la_forward_rpe(const void *q, const void *k, const void *v, const float *bias, void *out, int B, int H, int N,
                   int D, int Dv, int causal, const la_feature_map *fm, int dtype, void *stream)
{
    return rpe_impl(q, k, v, bias, out, B, H, N, D, Dv, causal, fm, dtype, stream);
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
    case LA_ERR_RANGE: return "LA_ERR_RANGE: an operand of the tensor-core backward is outside fp16's range";
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
        return flag == 2 ? LA_ERR_RANGE : LA_ERR_TIMEOUT;
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
        if (c.h2d) cudaStreamDestroy(c.h2d);
        if (c.d2h) cudaStreamDestroy(c.d2h);
        c = DeviceCtx();
    }
    if (have_cur) cudaSetDevice(cur);
    cudaGetLastError();
}

int la_version(void) { return LA_VERSION; }

unsigned long long la_launch_count(void) { return la::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
