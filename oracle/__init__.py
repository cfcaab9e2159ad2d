"""The oracle for kernelized (linear) attention: fp64 CPU code in ``oracle.c``.

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's timed CPU baseline may import this module.  The product path
(the CUDA library and its binding) never imports, loads or calls it, and
this module imports nothing from the product.

Inputs are numpy arrays; they are widened to float64 exactly (bf16 and fp32
values are representable in fp64), so the oracle sees the same input values
as the GPU path.  Layouts: q, k [B, H, N, D]; v [B, H, N, Dv]; W [m, D].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

PHI_ELU1 = 0
PHI_PRF = 1
PHI_NPRF = 2
PHI_TRF = 3
_KINDS = {"elu1": PHI_ELU1, "prf": PHI_PRF, "nprf": PHI_NPRF, "trf": PHI_TRF}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (fp64, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` overrides it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.POINTER(ctypes.c_double)
    L = ctypes.c_long
    I = ctypes.c_int
    lib.oracle_causal.argtypes = [P, P, P, P, L, L, I, I, I, P, I, P, P]
    lib.oracle_noncausal.argtypes = [P, P, P, P, L, L, I, I, I, P, I]
    lib.oracle_step.argtypes = [P, P, P, P, P, P, L, I, I, I, P, I]
    lib.oracle_quadratic_rows.argtypes = [P, P, P, P, L, I, I, I, I, P, I,
                                          ctypes.POINTER(ctypes.c_long), L]
    lib.oracle_phi.argtypes = [P, I, I, P, I, P]
    lib.oracle_backward.argtypes = [P, P, P, P, P, P, P, L, L, I, I, I, I, P, I]
    lib.oracle_prefix_attention.argtypes = [P, P, P, P, L, L, I, I, P]
    lib.oracle_prefix_step.argtypes = [P, P, P, P, P, L, I, I]
    lib.oracle_rpe.argtypes = [P, P, P, P, P, L, L, I, I, I, I, I, P, I]
    lib.oracle_num_threads.restype = I
    return lib


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _fm(feature, W, D):
    kind = _KINDS[feature]
    if kind != PHI_ELU1:
        if W is None:
            raise ValueError("random features need W")
        W = _d(W)
        if W.ndim != 2 or W.shape[1] != D:
            raise ValueError("W must be [m, D]")
        return kind, W, W.shape[0]
    return kind, None, 0


def phi_dim(D, feature="elu1", m=0):
    kind = _KINDS[feature]
    if kind == PHI_ELU1:
        return D
    return 2 * m if kind == PHI_TRF else m


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()


def phi(x, feature="elu1", W=None, lib=None):
    """phi applied to each row of x [..., D] -> [..., Dphi]."""
    lib = lib or load()
    x = _d(x)
    D = x.shape[-1]
    kind, W, m = _fm(feature, W, D)
    P = phi_dim(D, feature, m)
    rows = x.reshape(-1, D)
    out = np.empty((rows.shape[0], P))
    for r in range(rows.shape[0]):
        lib.oracle_phi(_ptr(rows[r]), D, kind, _ptr(W), m, _ptr(out[r]))
    return out.reshape(x.shape[:-1] + (P,))


def forward(q, k, v, causal=True, feature="elu1", W=None, return_state=False, lib=None):
    """Causal (recurrence) or non-causal forward; q, k [B,H,N,D], v [B,H,N,Dv].

    Returns out [B,H,N,Dv] (float64), plus (S [B,H,Dphi,Dv], z [B,H,Dphi])
    after the last position when ``return_state`` (causal only).
    """
    lib = lib or load()
    q, k, v = _d(q), _d(k), _d(v)
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, N):
        raise ValueError("shape mismatch")
    kind, W, m = _fm(feature, W, D)
    P = phi_dim(D, feature, m)
    out = np.empty((B, H, N, Dv))
    if causal:
        S = np.empty((B, H, P, Dv)) if return_state else None
        z = np.empty((B, H, P)) if return_state else None
        lib.oracle_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, N, D, Dv,
                          kind, _ptr(W), m, _ptr(S), _ptr(z))
        return (out, S, z) if return_state else out
    if return_state:
        raise ValueError("return_state is for the causal form")
    lib.oracle_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, N, D, Dv,
                         kind, _ptr(W), m)
    return out


def backward(q, k, v, dout, causal=True, feature="elu1", W=None, lib=None):
    """Gradients (dq, dk, dv) of L = sum(dout * out) for the forward of the
    same arguments; q, k [B,H,N,D], v and dout [B,H,N,Dv]; float64 results."""
    lib = lib or load()
    q, k, v, dout = _d(q), _d(k), _d(v), _d(dout)
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, N) or dout.shape != v.shape:
        raise ValueError("shape mismatch")
    kind, W, m = _fm(feature, W, D)
    dq, dk, dv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
    lib.oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        B * H, N, D, Dv, int(causal), kind, _ptr(W), m)
    return dq, dk, dv


def rpe(q, k, v, b, causal=True, feature="elu1", W=None, lib=None):
    """Kernelized attention with a Toeplitz relative-position weight exp(b):
    q, k [B,H,N,D], v [B,H,N,Dv], b [H, 2N-1] (index t + N - 1 for t = i - j)
    -> out [B,H,N,Dv] (float64)."""
    lib = lib or load()
    q, k, v, b = _d(q), _d(k), _d(v), _d(b)
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, N) or b.shape != (H, 2 * N - 1):
        raise ValueError("shape mismatch")
    kind, W, m = _fm(feature, W, D)
    out = np.empty((B, H, N, Dv))
    lib.oracle_rpe(_ptr(q), _ptr(k), _ptr(v), _ptr(b), _ptr(out), B * H, N, H, D, Dv, int(causal),
                   kind, _ptr(W), m)
    return out


def prefix_attention(q, k, v, return_state=False, lib=None):
    """Softmax attention of one query token per head over every prefix, as an
    RNN: q [B,H,D], k [B,H,N,D], v [B,H,N,Dv] -> out [B,H,N,Dv] (float64),
    plus the final state [B,H,Dv+2] = (m, u, w) when ``return_state``."""
    lib = lib or load()
    q, k, v = _d(q), _d(k), _d(v)
    B, H, N, D = k.shape
    Dv = v.shape[-1]
    if q.shape != (B, H, D) or v.shape[:3] != (B, H, N):
        raise ValueError("shape mismatch")
    out = np.empty((B, H, N, Dv))
    st = np.empty((B, H, Dv + 2)) if return_state else None
    lib.oracle_prefix_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, N, D, Dv, _ptr(st))
    return (out, st) if return_state else out


def prefix_step(state, q, k, v, lib=None):
    """One RNN step of the prefix attention: state [B,H,Dv+2] (m, u, w),
    q, k [B,H,D], v [B,H,Dv] -> (out [B,H,Dv], new state); inputs unchanged."""
    lib = lib or load()
    st = _d(state).copy()
    q, k, v = _d(q), _d(k), _d(v)
    B, H, D = q.shape
    Dv = v.shape[-1]
    if st.shape != (B, H, Dv + 2):
        raise ValueError("state shape mismatch")
    out = np.empty((B, H, Dv))
    lib.oracle_prefix_step(_ptr(st), _ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, D, Dv)
    return out, st


def step(S, z, q, k, v, feature="elu1", W=None, lib=None):
    """One recurrent step; S [B,H,Dphi,Dv], z [B,H,Dphi], q,k [B,H,D], v [B,H,Dv].

    Returns (out [B,H,Dv], S_new, z_new); the inputs are not modified.
    """
    lib = lib or load()
    S, z = _d(S).copy(), _d(z).copy()
    q, k, v = _d(q), _d(k), _d(v)
    B, H, D = q.shape
    Dv = v.shape[-1]
    kind, W, m = _fm(feature, W, D)
    out = np.empty((B, H, Dv))
    lib.oracle_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, D, Dv,
                    kind, _ptr(W), m)
    return out, S, z


def step_inplace(S, z, q, k, v, feature="elu1", W=None, lib=None):
    """The same recurrent step as ``step``, applied to S, z in place.

    S [B,H,Dphi,Dv] and z [B,H,Dphi] must be C-contiguous float64 arrays (they
    are the memories carried from step to step, as in the RNN form); q, k, v
    as in ``step``.  Returns out [B,H,Dv].  Long decodes over many heads use
    this to avoid copying the memories at every step.
    """
    lib = lib or load()
    for a in (S, z):
        if a.dtype != np.float64 or not a.flags["C_CONTIGUOUS"]:
            raise ValueError("S and z must be C-contiguous float64")
    q, k, v = _d(q), _d(k), _d(v)
    B, H, D = q.shape
    Dv = v.shape[-1]
    kind, W, m = _fm(feature, W, D)
    if S.shape != (B, H, phi_dim(D, feature, m), Dv) or z.shape != S.shape[:3]:
        raise ValueError("memory shape mismatch")
    out = np.empty((B, H, Dv))
    lib.oracle_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), _ptr(out), B * H, D, Dv,
                    kind, _ptr(W), m)
    return out


def quadratic_rows(q, k, v, rows, causal=True, feature="elu1", W=None, lib=None):
    """Brute-force masked quadratic form for listed rows of one head.

    q, k [N, D]; v [N, Dv]; rows: iterable of positions -> [len(rows), Dv].
    """
    lib = lib or load()
    q, k, v = _d(q), _d(k), _d(v)
    N, D = q.shape
    Dv = v.shape[-1]
    kind, W, m = _fm(feature, W, D)
    rows = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int64)).astype(np.int_)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise ValueError("row out of range")
    out = np.empty((rows.size, Dv))
    lib.oracle_quadratic_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(out), N, D, Dv, int(causal),
                              kind, _ptr(W), m,
                              rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), rows.size)
    return out


def quadratic(q, k, v, causal=True, feature="elu1", W=None, lib=None):
    """Brute-force masked quadratic form for every row; q,k [B,H,N,D]."""
    q, k, v = _d(q), _d(k), _d(v)
    B, H, N, _ = q.shape
    out = np.empty(v.shape)
    for b in range(B):
        for h in range(H):
            out[b, h] = quadratic_rows(q[b, h], k[b, h], v[b, h], range(N), causal,
                                       feature, W, lib)
    return out
