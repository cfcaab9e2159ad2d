"""Python binding of liblinattn.so, the B300 kernelized linear-attention library.

Argument marshalling only: each function takes torch CUDA tensors, checks
that they are contiguous CUDA tensors of one dtype, and passes their device
pointers and sizes to the C entry point of the same name (``include/linattn.h``).
Every step of the computation runs in the library's CUDA kernels.  There is
no other implementation: if the library is not built, ``load()`` raises.

    out            = la_forward(q, k, v, causal=True, feature_map=None)
    out, S, z      = la_forward_ex(q, k, v, causal=True, feature_map=None)
    out            = la_step(S, z, q, k, v)           # S, z updated in place
    dq, dk, dv     = la_backward(q, k, v, dout)       # gradients of sum(dout * out)

Shapes: q, k [B, H, N, D]; v [B, H, N, Dv]; S [B, H, Dphi, Dv] fp32;
z [B, H, Dphi] fp32; decode q, k [B, H, D], v [B, H, Dv].
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblinattn.so")

LA_F32, LA_BF16 = 0, 1
LA_PHI_ELU1, LA_PHI_PRF, LA_PHI_NPRF, LA_PHI_TRF = 0, 1, 2, 3
LA_W_GAUSSIAN, LA_W_ORTHOGONAL, LA_W_SPHERE = 0, 1, 2
LA_OK = 0
LA_NOALLOC_SCRATCH_BYTES = 4 << 20   # the fixed scratch of la_forward_noncausal_noalloc
STATUS_NAMES = {0: "LA_OK", -1: "LA_ERR_NULL", -2: "LA_ERR_DIM", -3: "LA_ERR_DTYPE",
                -4: "LA_ERR_FEATURE", -5: "LA_ERR_CUDA", -6: "LA_ERR_TIMEOUT",
                -7: "LA_ERR_ALIGN", -8: "LA_ERR_RANGE"}
EXPORTED = ("la_forward", "la_forward_ex", "la_forward_host", "la_step", "la_backward",
            "la_prefix_attention", "la_prefix_step", "la_random_features", "la_forward_rpe",
            "la_status_string",
            "la_check", "la_shutdown", "la_version", "la_launch_count",
            "la_forward_noncausal_noalloc", "la_selftest_timeout")

_DT = {torch.float32: LA_F32, torch.bfloat16: LA_BF16}


class la_feature_map(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("m", ctypes.c_int), ("W", ctypes.c_void_p)]


class LinAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_KINDS = {"elu1": LA_PHI_ELU1, "prf": LA_PHI_PRF, "nprf": LA_PHI_NPRF, "trf": LA_PHI_TRF}


class FeatureMap:
    """phi: ``FeatureMap()`` is elu(x)+1; ``FeatureMap(kind, W)`` with an m x D
    fp32 CUDA tensor W is a random-feature map: "prf" exp(w_r.x - |x|^2/2)/sqrt(m),
    "nprf" the same of x/|x|, "trf" exp(|x|^2/2)/sqrt(m) [cos(Wx), sin(Wx)]
    (2m features).  Sphere-PRF and ORF are "prf" with W from la_random_features."""

    def __init__(self, kind: str = "elu1", W: torch.Tensor | None = None):
        if kind not in _KINDS:
            raise ValueError(kind)
        self.kind = kind
        self.W = W
        if kind != "elu1":
            if W is None or W.dtype != torch.float32 or not W.is_cuda or not W.is_contiguous():
                raise ValueError("random features need W as a contiguous fp32 CUDA tensor [m, D]")

    @property
    def m(self) -> int:
        return self.W.shape[0] if self.kind != "elu1" else 0

    def phi_dim(self, D: int) -> int:
        if self.kind == "elu1":
            return D
        return 2 * self.m if self.kind == "trf" else self.m

    def c_struct(self) -> la_feature_map:
        if self.kind != "elu1":
            return la_feature_map(_KINDS[self.kind], self.W.shape[0], self.W.data_ptr())
        return la_feature_map(LA_PHI_ELU1, 0, None)


def la_random_features(m: int, D: int, seed: int, kind: str = "gaussian") -> torch.Tensor:
    """W [m, D] fp32 (host) from la_random_features: kind "gaussian",
    "orthogonal" (ORF) or "sphere" (Sphere-PRF)."""
    codes = {"gaussian": LA_W_GAUSSIAN, "orthogonal": LA_W_ORTHOGONAL, "sphere": LA_W_SPHERE}
    W = torch.empty((m, D), dtype=torch.float32)
    _raise(load().la_random_features(codes[kind], m, D, seed, W.data_ptr()))
    return W


_lib = None


def load(path: str | None = None):
    """Load liblinattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build the CUDA library first "
                          "(python -m causal_linear_attention_map_b300.build)")
    lib = ctypes.CDLL(p)
    vp, i = ctypes.c_void_p, ctypes.c_int
    fm = ctypes.POINTER(la_feature_map)
    lib.la_forward.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, fm, i, vp]
    lib.la_forward.restype = i
    lib.la_forward_ex.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, fm, i, vp, vp, vp]
    lib.la_forward_ex.restype = i
    lib.la_forward_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, fm, i, vp]
    lib.la_forward_host.restype = i
    lib.la_step.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, fm, i, vp]
    lib.la_step.restype = i
    lib.la_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, fm, i, vp]
    lib.la_backward.restype = i
    lib.la_prefix_attention.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
    lib.la_prefix_attention.restype = i
    lib.la_prefix_step.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.la_prefix_step.restype = i
    lib.la_random_features.argtypes = [i, i, i, ctypes.c_ulonglong, vp]
    lib.la_random_features.restype = i
    lib.la_forward_rpe.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, fm, i, vp]
    lib.la_forward_rpe.restype = i
    lib.la_status_string.argtypes = [i]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_check.argtypes = [vp]
    lib.la_check.restype = i
    lib.la_selftest_timeout.argtypes = [i, vp]
    lib.la_selftest_timeout.restype = i
    lib.la_shutdown.argtypes = []
    lib.la_shutdown.restype = None
    lib.la_version.argtypes = []
    lib.la_version.restype = i
    lib.la_launch_count.argtypes = []
    lib.la_launch_count.restype = ctypes.c_ulonglong
    lib.la_forward_noncausal_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, fm, i, vp]
    lib.la_forward_noncausal_noalloc.restype = i
    if path is None:
        _lib = lib
    return lib


def la_status_string(status: int) -> str:
    return load().la_status_string(status).decode()


def _raise(st: int):
    if st != LA_OK:
        raise LinAttnError(st, la_status_string(st))


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_tensors(*ts):
    dt = ts[0].dtype
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.dtype != dt:
            raise ValueError("q, k, v, out must share one dtype")
    if dt not in _DT:
        raise ValueError(f"unsupported dtype {dt}")
    return _DT[dt]


def _check_host_tensors(*ts):
    dt = ts[0].dtype
    for t in ts:
        if t.is_cuda:
            raise ValueError("la_forward_host takes host (CPU) tensors")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.dtype != dt:
            raise ValueError("q, k, v, out must share one dtype")
    if dt not in _DT:
        raise ValueError(f"unsupported dtype {dt}")
    return _DT[dt]


def _fm(feature_map):
    fm = feature_map or FeatureMap()
    return fm, ctypes.byref(fm.c_struct())


def la_forward_ex(q, k, v, causal=True, feature_map: FeatureMap | None = None, out=None,
                  S_out=None, z_out=None, stream=None, return_state=True):
    """la_forward_ex: returns (out, S, z); S/z are allocated when not given."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N):
        raise ValueError("shape mismatch between q, k, v")
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=q.dtype, device=q.device)
    dt = _check_tensors(q, k, v, out)
    fm, fmp = _fm(feature_map)
    P = fm.phi_dim(D)
    if return_state:
        if S_out is None:
            S_out = torch.empty((B, H, P, Dv), dtype=torch.float32, device=q.device)
        if z_out is None:
            z_out = torch.empty((B, H, P), dtype=torch.float32, device=q.device)
    for t in (S_out, z_out):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda):
            raise ValueError("S_out / z_out must be contiguous fp32 CUDA tensors")
    st = load().la_forward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              B, H, N, D, Dv, int(bool(causal)), fmp, dt, _stream(stream),
                              S_out.data_ptr() if S_out is not None else None,
                              z_out.data_ptr() if z_out is not None else None)
    _raise(st)
    return out, S_out, z_out


def la_forward(q, k, v, causal=True, feature_map: FeatureMap | None = None, out=None,
               stream=None):
    """la_forward: kernelized attention over whole sequences -> out [B,H,N,Dv]."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N):
        raise ValueError("shape mismatch between q, k, v")
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=q.dtype, device=q.device)
    dt = _check_tensors(q, k, v, out)
    _, fmp = _fm(feature_map)
    st = load().la_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           B, H, N, D, Dv, int(bool(causal)), fmp, dt, _stream(stream))
    _raise(st)
    return out


def la_forward_host(q, k, v, causal=True, feature_map: FeatureMap | None = None, out=None,
                    stream=None):
    """la_forward_host: q, k, v and out in host memory (pinned for overlapped
    copies; ``out`` is allocated pinned when not given).  ``out`` holds the
    result once ``stream`` has been synchronised."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N):
        raise ValueError("shape mismatch between q, k, v")
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=q.dtype, pin_memory=True)
    dt = _check_host_tensors(q, k, v, out)
    _, fmp = _fm(feature_map)
    st = load().la_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                B, H, N, D, Dv, int(bool(causal)), fmp, dt, _stream(stream))
    _raise(st)
    return out


def la_step(S, z, q, k, v, feature_map: FeatureMap | None = None, out=None, stream=None):
    """la_step: one decode step; updates S [B,H,Dphi,Dv] and z [B,H,Dphi] in place."""
    B, H, D = q.shape
    Dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, Dv), dtype=q.dtype, device=q.device)
    dt = _check_tensors(q, k, v, out)
    for t in (S, z):
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("S and z must be contiguous fp32 CUDA tensors")
    _, fmp = _fm(feature_map)
    st = load().la_step(S.data_ptr(), z.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                        out.data_ptr(), B, H, D, Dv, fmp, dt, _stream(stream))
    _raise(st)
    return out


def la_backward(q, k, v, dout, causal=True, feature_map: FeatureMap | None = None, dq=None, dk=None,
                dv=None, stream=None):
    """la_backward: gradients (dq, dk, dv) of sum(dout * out) for out = la_forward(q, k, v)."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N) or dout.shape != v.shape:
        raise ValueError("shape mismatch between q, k, v, dout")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dt = _check_tensors(q, k, v, dout, dq, dk, dv)
    _, fmp = _fm(feature_map)
    st = load().la_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                            dk.data_ptr(), dv.data_ptr(), B, H, N, D, Dv, int(bool(causal)), fmp, dt,
                            _stream(stream))
    _raise(st)
    return dq, dk, dv


def la_forward_rpe(q, k, v, bias, causal=True, feature_map: FeatureMap | None = None, out=None, stream=None):
    """la_forward_rpe: kernelized attention with the Toeplitz weight exp(bias)
    (bias: fp32 CUDA [H, 2N-1], index t + N - 1 for t = i - j)."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N):
        raise ValueError("shape mismatch between q, k, v")
    if tuple(bias.shape) != (H, 2 * N - 1) or bias.dtype != torch.float32 or not bias.is_contiguous():
        raise ValueError("bias must be a contiguous fp32 [H, 2N - 1] tensor")
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=q.dtype, device=q.device)
    dt = _check_tensors(q, k, v, out)
    _, fmp = _fm(feature_map)
    st = load().la_forward_rpe(q.data_ptr(), k.data_ptr(), v.data_ptr(), bias.data_ptr(), out.data_ptr(),
                               B, H, N, D, Dv, int(bool(causal)), fmp, dt, _stream(stream))
    _raise(st)
    return out


def la_prefix_attention(q, k, v, out=None, state_out=None, return_state=False, stream=None):
    """la_prefix_attention: softmax attention of the query token q [B,H,D] over
    every prefix of k [B,H,N,D], v [B,H,N,Dv] -> out [B,H,N,Dv] (and the final
    state [B,H,Dv+2] = (m, u, w) when ``return_state`` or ``state_out``)."""
    B, H, N, D = k.shape
    Dv = v.shape[-1]
    if tuple(q.shape) != (B, H, D) or tuple(v.shape[:3]) != (B, H, N):
        raise ValueError("shape mismatch between q, k, v")
    if out is None:
        out = torch.empty((B, H, N, Dv), dtype=k.dtype, device=k.device)
    dt = _check_tensors(q, k, v, out)
    if return_state and state_out is None:
        state_out = torch.empty((B, H, Dv + 2), dtype=torch.float32, device=k.device)
    if state_out is not None and (state_out.dtype != torch.float32 or not state_out.is_contiguous()):
        raise ValueError("state_out must be a contiguous fp32 CUDA tensor")
    st = load().la_prefix_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    state_out.data_ptr() if state_out is not None else None,
                                    B, H, N, D, Dv, dt, _stream(stream))
    _raise(st)
    return (out, state_out) if state_out is not None else out


def la_prefix_step(state, q, k, v, out=None, stream=None):
    """la_prefix_step: one token of the prefix-attention RNN; state [B,H,Dv+2]
    fp32 is updated in place; q, k [B,H,D], v [B,H,Dv] -> out [B,H,Dv]."""
    B, H, D = q.shape
    Dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, Dv), dtype=q.dtype, device=q.device)
    dt = _check_tensors(q, k, v, out)
    if state.dtype != torch.float32 or not state.is_contiguous() or tuple(state.shape) != (B, H, Dv + 2):
        raise ValueError("state must be a contiguous fp32 [B, H, Dv + 2] CUDA tensor")
    st = load().la_prefix_step(state.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               B, H, D, Dv, dt, _stream(stream))
    _raise(st)
    return out


def la_check(stream=None) -> int:
    """Synchronise the stream and return deferred device errors as a status."""
    return load().la_check(_stream(stream))


def la_selftest_timeout(budget_ms: int = 50, stream=None) -> int:
    """Launch the failure-detection self-test: a bounded wait that nothing
    completes gives up after ~budget_ms; the next la_check returns
    LA_ERR_TIMEOUT.  Returns the launch status."""
    return load().la_selftest_timeout(int(budget_ms), _stream(stream))


def la_shutdown() -> None:
    load().la_shutdown()


def la_version() -> int:
    return load().la_version()


def la_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return load().la_launch_count()


def la_forward_noncausal_noalloc(q, k, v, out, feature_map: FeatureMap | None = None,
                                 stream=None):
    """Non-causal forward that allocates no device memory: ``out`` must be
    given (the caller owns every buffer); the library's scratch is a fixed
    device array shared by all calls (see include/linattn.h)."""
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or tuple(v.shape[:3]) != (B, H, N) or tuple(out.shape) != (B, H, N, Dv):
        raise ValueError("shape mismatch between q, k, v, out")
    dt = _check_tensors(q, k, v, out)
    _, fmp = _fm(feature_map)
    st = load().la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             out.data_ptr(), B, H, N, D, Dv, fmp, dt,
                                             _stream(stream))
    _raise(st)
    return out
