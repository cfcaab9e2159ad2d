"""Pins for the oracle: checks against facts that the method and mathematics
fix, independent of the oracle's own code.

Each ``pin_*`` takes a loaded oracle library (ctypes handle) and raises
AssertionError when the oracle disagrees.  ``test_oracle_pins.py`` runs them
on the real oracle and, to show that they bite, on copies of the oracle with
planted mistakes.

Sources of truth (review page "Transformers are RNNs: Fast Autoregressive
Transformers with Linear Attention", section "proposed method" b1-b5, and
section "main results" b2 for the elu-based map; review page "Stable, Fast
and Accurate: Kernelized Attention with Relative Positional Encoding",
section "proposed method" b6, for positive random features):
  - brute force of the masked quadratic form in pure Python on tiny inputs;
  - exact rational arithmetic where phi(x) = x + 1 (all inputs > 0);
  - closed forms: equal keys give the running mean of V, constant V gives V;
  - special cases that reduce to library routines: with D = 1 and keys <= 0
    the elu+1 map gives causal softmax over the keys; with m = 1 the PRF map
    gives causal softmax over w.k - |k|^2/2; elu(x) + 1 from torch;
  - invariants: convex hull, last causal row = non-causal row, the recurrent
    step iterated N times = the forward pass, head and key/value
    permutations, linearity in V;
  - the PRF kernel's expectation E_w[phi(q).phi(k)] = exp(q.k).
Further feature maps the same page names (PRF, TRF, Sphere-PRF, ORF, NPRF;
readings: TRF = exp(|x|^2/2)/sqrt(m) [cos(Wx), sin(Wx)], NPRF = PRF of x/|x|):
  - TRF's expectation E_w[phi(q).phi(k)] = exp(q.k) (Gaussian W);
  - NPRF's expectation exp(q.k / (|q| |k|)), and its invariance to scaling
    each query and key by a positive factor;
  - their gradients by finite differences (below).
Gradients ("Transformers are RNNs", proposed method b4: linear-time
gradients of the same cumulative-sum form):
  - central finite differences of the forward oracle (itself pinned above);
  - torch autograd through the masked quadratic form written in torch;
  - closed forms: constant V gives zero gradients for q and k, and the
    gradients for v sum to the sum of the output cotangents.
Kernelized attention with a Toeplitz relative-position weight (review page
"Stable, Fast and Accurate: Kernelized Attention with RPE", proposed method:
the Toeplitz structure, multiplied through by FFT in O(n log n)):
  - the page's own algorithm, written with numpy's FFT: each Toeplitz
    matrix-vector product as a circulant convolution of length 2N;
  - b = 0 gives plain kernelized attention (the forward oracle); a constant
    added to b changes nothing; pure-Python brute force.
Softmax attention as an RNN over every prefix (review page "Attention as an
RNN", proposed method: many-to-one RNN cell, many-to-many outputs by a
parallel prefix scan, Hillis-Steele):
  - scipy softmax over each prefix (brute force with a library routine);
  - a pure-Python Hillis-Steele scan with the associative max-rescaling
    combine, an independent algorithm for the same outputs;
  - the last output is full softmax attention (torch); constant V gives V;
    the step iterated from the empty state gives the scan; scores of +-500.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import scipy.special
import torch

import oracle

RTOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol=RTOL, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    scale = max(np.max(np.abs(b)), 1e-300)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= rtol * scale + atol, f"{what}: max err {err:.3e} vs scale {scale:.3e}"


# ---------------------------------------------------------------- brute force

def _py_phi(x, feature, W):
    if feature == "elu1":
        return [xi + 1.0 if xi > 0 else math.exp(xi) for xi in x]
    m = len(W)
    sq = sum(xi * xi for xi in x)
    if feature == "nprf":
        n = math.sqrt(sq)
        x = [xi / n for xi in x]
        sq = 1.0
    u = [sum(w * xi for w, xi in zip(W[r], x)) for r in range(m)]
    if feature == "trf":
        a = math.exp(sq / 2) / math.sqrt(m)
        return [a * math.cos(t) for t in u] + [a * math.sin(t) for t in u]
    return [math.exp(t - sq / 2) / math.sqrt(m) for t in u]


def _py_attention(q, k, v, causal, feature, W):
    """sum_j (phi(q_i).phi(k_j)) v_j / sum_j phi(q_i).phi(k_j), pure Python."""
    N, Dv = len(q), len(v[0])
    fk = [_py_phi(kj, feature, W) for kj in k]
    out = []
    for i in range(N):
        fq = _py_phi(q[i], feature, W)
        J = range(i + 1) if causal else range(N)
        num = [0.0] * Dv
        den = 0.0
        for j in J:
            w = sum(a * b for a, b in zip(fq, fk[j]))
            den += w
            for c in range(Dv):
                num[c] += w * v[j][c]
        out.append([x / den for x in num])
    return out


def pin_pure_python_brute_force(lib):
    r = _rng(1)
    for (N, D, Dv, feature, m) in [(7, 3, 2, "elu1", 0), (9, 2, 5, "elu1", 0),
                                   (6, 3, 4, "prf", 5), (5, 1, 1, "elu1", 0),
                                   (6, 3, 2, "nprf", 4), (7, 2, 3, "trf", 6)]:
        q = r.normal(size=(1, 2, N, D))
        k = r.normal(size=(1, 2, N, D))
        v = r.normal(size=(1, 2, N, Dv))
        W = r.normal(size=(m, D)) if feature != "elu1" else None
        if feature == "trf":
            W = W * 0.3
        Wl = W.tolist() if W is not None else None
        for causal in (True, False):
            got = oracle.forward(q, k, v, causal=causal, feature=feature, W=W, lib=lib)
            for h in range(2):
                ref = _py_attention(q[0, h].tolist(), k[0, h].tolist(), v[0, h].tolist(),
                                    causal, feature, Wl)
                _close(got[0, h], ref, what=f"brute force {feature} causal={causal} N={N}")


def pin_exact_rational(lib):
    """All q, k > 0: phi(x) = x + 1 exactly, so the causal output is rational."""
    r = _rng(2)
    N, D, Dv = 8, 3, 2
    qi = r.integers(1, 17, size=(N, D))
    ki = r.integers(1, 17, size=(N, D))
    vi = r.integers(-16, 17, size=(N, Dv))
    q = [[Fraction(int(x), 8) for x in row] for row in qi]
    k = [[Fraction(int(x), 8) for x in row] for row in ki]
    v = [[Fraction(int(x), 4) for x in row] for row in vi]
    exact = []
    for i in range(N):
        num = [Fraction(0)] * Dv
        den = Fraction(0)
        for j in range(i + 1):
            w = sum((a + 1) * (b + 1) for a, b in zip(q[i], k[j]))
            den += w
            num = [n + w * vj for n, vj in zip(num, v[j])]
        exact.append([float(n / den) for n in num])
    to = lambda M: np.array([[float(x) for x in row] for row in M])[None, None]
    got = oracle.forward(to(q), to(k), to(v), causal=True, lib=lib)
    _close(got[0, 0], exact, rtol=1e-14, what="exact rational")


def pin_oracle_quadratic_vs_recurrence(lib):
    r = _rng(3)
    for (N, D, Dv, feature, m) in [(256, 1, 3, "elu1", 0), (200, 4, 4, "elu1", 0),
                                   (256, 16, 8, "elu1", 0), (128, 4, 6, "prf", 16),
                                   (96, 16, 16, "prf", 8)]:
        q = r.normal(size=(1, 2, N, D))
        k = r.normal(size=(1, 2, N, D))
        v = r.normal(size=(1, 2, N, Dv))
        W = r.normal(size=(m, D)) if feature == "prf" else None
        for causal in (True, False):
            a = oracle.forward(q, k, v, causal=causal, feature=feature, W=W, lib=lib)
            b = oracle.quadratic(q, k, v, causal=causal, feature=feature, W=W, lib=lib)
            _close(a, b, rtol=1e-11, what=f"quadratic vs recurrence {feature} {causal}")


# ------------------------------------------------------------- closed forms

def pin_equal_keys_running_mean(lib):
    r = _rng(4)
    N, D, Dv = 50, 6, 3
    q = r.normal(size=(1, 1, N, D))
    k = np.broadcast_to(r.normal(size=(D,)), (1, 1, N, D)).copy()
    v = r.normal(size=(1, 1, N, Dv))
    mean = np.cumsum(v[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    for feature, W in (("elu1", None), ("prf", r.normal(size=(7, D)))):
        got = oracle.forward(q, k, v, causal=True, feature=feature, W=W, lib=lib)
        _close(got[0, 0], mean, rtol=1e-12, what=f"running mean {feature}")
        got = oracle.forward(q, k, v, causal=False, feature=feature, W=W, lib=lib)
        _close(got[0, 0], np.broadcast_to(v[0, 0].mean(0), (N, Dv)), rtol=1e-12,
               what=f"mean {feature}")


def pin_constant_values(lib):
    r = _rng(5)
    N, D, Dv = 40, 5, 4
    q = r.normal(size=(2, 1, N, D))
    k = r.normal(size=(2, 1, N, D))
    c = r.normal(size=(Dv,))
    v = np.broadcast_to(c, (2, 1, N, Dv)).copy()
    for causal in (True, False):
        got = oracle.forward(q, k, v, causal=causal, lib=lib)
        _close(got, np.broadcast_to(c, got.shape), rtol=1e-13, what="constant v")


def pin_elu_is_torch_elu_plus_one(lib):
    x = np.linspace(-6, 6, 241)
    x = np.concatenate([x, [0.0, -0.0, 1e-300, -1e-300, 30.0, -30.0]])
    got = oracle.phi(x[:, None], "elu1", lib=lib)[:, 0]
    ref = torch.nn.functional.elu(torch.tensor(x, dtype=torch.float64), alpha=1.0).numpy() + 1
    _close(got, ref, rtol=1e-15, what="elu+1")


def pin_elu_d1_negative_keys_is_softmax(lib):
    """D = 1 and k <= 0: weights phi(q)exp(k_j), q cancels -> softmax over k."""
    r = _rng(6)
    N = 30
    q = r.normal(size=(1, 1, N, 1))
    k = -np.abs(r.normal(size=(1, 1, N, 1))) * 3
    v = r.normal(size=(1, 1, N, 3))
    got = oracle.forward(q, k, v, causal=True, lib=lib)[0, 0]
    ref = np.stack([scipy.special.softmax(k[0, 0, :i + 1, 0]) @ v[0, 0, :i + 1]
                    for i in range(N)])
    _close(got, ref, rtol=1e-13, what="softmax special case")


def pin_elu_d1_positive_keys_linear_weights(lib):
    """D = 1 and k > 0: weights proportional to k_j + 1."""
    r = _rng(7)
    N = 30
    q = r.normal(size=(1, 1, N, 1))
    k = np.abs(r.normal(size=(1, 1, N, 1))) + 0.01
    v = r.normal(size=(1, 1, N, 2))
    w = k[0, 0, :, 0] + 1
    ref = np.stack([np.average(v[0, 0, :i + 1], axis=0, weights=w[:i + 1]) for i in range(N)])
    got = oracle.forward(q, k, v, causal=True, lib=lib)[0, 0]
    _close(got, ref, rtol=1e-13, what="linear-weight special case")


def pin_prf_m1_is_softmax(lib):
    """m = 1: phi(q) cancels; weights exp(w.k_j - |k_j|^2/2) -> a softmax."""
    r = _rng(8)
    N, D = 25, 4
    W = r.normal(size=(1, D))
    q = r.normal(size=(1, 1, N, D))
    k = r.normal(size=(1, 1, N, D))
    v = r.normal(size=(1, 1, N, 3))
    logits = k[0, 0] @ W[0] - 0.5 * np.sum(k[0, 0] ** 2, axis=1)
    ref = np.stack([scipy.special.softmax(logits[:i + 1]) @ v[0, 0, :i + 1] for i in range(N)])
    got = oracle.forward(q, k, v, causal=True, feature="prf", W=W, lib=lib)[0, 0]
    _close(got, ref, rtol=1e-12, what="PRF m=1 softmax")
    got = oracle.forward(q, k, v, causal=False, feature="prf", W=W, lib=lib)[0, 0]
    _close(got, np.broadcast_to(ref[-1], got.shape), rtol=1e-12, what="PRF m=1 non-causal")


def pin_prf_kernel_expectation(lib):
    """E over w ~ N(0, I) of phi(q).phi(k) = exp(q.k) (standard PRF identity).

    With m = 2**16 features the sample mean is within a few standard errors.
    """
    r = _rng(9)
    D, m = 4, 1 << 16
    W = r.normal(size=(m, D))
    for _ in range(3):
        q = r.normal(size=D) * 0.4
        k = r.normal(size=D) * 0.4
        fq = oracle.phi(q[None], "prf", W, lib=lib)[0]
        fk = oracle.phi(k[None], "prf", W, lib=lib)[0]
        est = float(fq @ fk)
        # per-feature terms t_r = m * fq_r * fk_r have mean exp(q.k)
        t = m * fq * fk
        se = t.std() / math.sqrt(m)
        target = math.exp(float(q @ k))
        assert abs(est - target) < 5 * se + 1e-12, (est, target, se)
        assert np.all(fq > 0) and np.all(fk > 0)


def pin_trf_and_nprf_kernel_expectations(lib):
    """E over w ~ N(0, I): TRF gives exp(q.k) (the random Fourier features of
    the Gaussian kernel times exp(|q|^2/2 + |k|^2/2)), NPRF gives
    exp(q.k / (|q||k|)).  Checked to a few standard errors with m = 2**16."""
    r = _rng(30)
    D, m = 4, 1 << 16
    W = r.normal(size=(m, D))
    for _ in range(3):
        q = r.normal(size=D) * 0.4
        k = r.normal(size=D) * 0.4
        for feature, target in (("trf", math.exp(float(q @ k))),
                                ("nprf", math.exp(float(q @ k) / np.linalg.norm(q) / np.linalg.norm(k)))):
            fq = oracle.phi(q[None], feature, W, lib=lib)[0]
            fk = oracle.phi(k[None], feature, W, lib=lib)[0]
            t = fq * fk
            terms = m * (t[:m] + t[m:]) if feature == "trf" else m * t
            se = terms.std() / math.sqrt(m)
            assert abs(float(fq @ fk) - target) < 5 * se + 1e-12, (feature, float(fq @ fk), target, se)
        assert fq.shape == (2 * m,) or feature != "trf"


def pin_nprf_scale_invariance(lib):
    r = _rng(31)
    B, H, N, D, Dv = 1, 2, 30, 5, 3
    W = r.normal(size=(8, D))
    q, k, v = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv))
    cq = np.exp(r.normal(size=(B, H, N, 1)))
    ck = np.exp(r.normal(size=(B, H, N, 1)))
    for causal in (True, False):
        a = oracle.forward(q, k, v, causal=causal, feature="nprf", W=W, lib=lib)
        b = oracle.forward(q * cq, k * ck, v, causal=causal, feature="nprf", W=W, lib=lib)
        _close(a, b, rtol=1e-12, what=f"NPRF scale invariance causal={causal}")


# ------------------------------------------------------------- invariants

def pin_convex_hull(lib):
    r = _rng(10)
    N, D, Dv = 64, 8, 5
    q, k, v = (r.normal(size=(1, 2, N, x)) for x in (D, D, Dv))
    got = oracle.forward(q, k, v, causal=True, lib=lib)
    lo = np.minimum.accumulate(v, axis=2)
    hi = np.maximum.accumulate(v, axis=2)
    assert np.all(got >= lo - 1e-12) and np.all(got <= hi + 1e-12)


def pin_last_row_equals_noncausal(lib):
    r = _rng(11)
    N, D, Dv = 33, 7, 3
    q, k, v = (r.normal(size=(2, 1, N, x)) for x in (D, D, Dv))
    for feature, W in (("elu1", None), ("prf", r.normal(size=(9, D)))):
        c = oracle.forward(q, k, v, causal=True, feature=feature, W=W, lib=lib)
        n = oracle.forward(q, k, v, causal=False, feature=feature, W=W, lib=lib)
        _close(c[:, :, -1], n[:, :, -1], rtol=1e-13, what=f"last row {feature}")


def pin_step_iterated_equals_forward(lib):
    r = _rng(12)
    B, H, N, D, Dv = 2, 2, 20, 5, 3
    for feature, W in (("elu1", None), ("prf", r.normal(size=(6, D)))):
        P = oracle.phi_dim(D, feature, 0 if W is None else W.shape[0])
        q, k, v = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv))
        ref, Sref, zref = oracle.forward(q, k, v, causal=True, feature=feature, W=W,
                                         return_state=True, lib=lib)
        S = np.zeros((B, H, P, Dv))
        z = np.zeros((B, H, P))
        outs = []
        for i in range(N):
            o, S, z = oracle.step(S, z, q[:, :, i], k[:, :, i], v[:, :, i], feature, W, lib=lib)
            outs.append(o)
        _close(np.stack(outs, axis=2), ref, rtol=1e-12, what=f"step x N {feature}")
        _close(S, Sref, rtol=1e-12, what="final S")
        _close(z, zref, rtol=1e-12, what="final z")
        # resume: forward over the first N1 positions, then steps
        N1 = 7
        _, S1, z1 = oracle.forward(q[:, :, :N1], k[:, :, :N1], v[:, :, :N1], causal=True,
                                   feature=feature, W=W, return_state=True, lib=lib)
        for i in range(N1, N):
            o, S1, z1 = oracle.step(S1, z1, q[:, :, i], k[:, :, i], v[:, :, i], feature, W,
                                    lib=lib)
            _close(o, ref[:, :, i], rtol=1e-12, what="resume")
        # the in-place form carries the same memories through the same steps
        S2, z2 = np.zeros((B, H, P, Dv)), np.zeros((B, H, P))
        for i in range(N):
            o = oracle.step_inplace(S2, z2, q[:, :, i], k[:, :, i], v[:, :, i], feature, W,
                                    lib=lib)
            _close(o, ref[:, :, i], rtol=1e-12, what=f"in-place step {feature}")
        _close(S2, Sref, rtol=1e-12, what="in-place final S")
        _close(z2, zref, rtol=1e-12, what="in-place final z")


def pin_head_permutation(lib):
    r = _rng(13)
    N, D, Dv = 16, 4, 4
    q, k, v = (r.normal(size=(1, 5, N, x)) for x in (D, D, Dv))
    perm = r.permutation(5)
    a = oracle.forward(q, k, v, causal=True, lib=lib)
    b = oracle.forward(q[:, perm], k[:, perm], v[:, perm], causal=True, lib=lib)
    _close(b, a[:, perm], rtol=0.0, what="head permutation")


def pin_noncausal_key_permutation(lib):
    r = _rng(14)
    N, D, Dv = 31, 6, 2
    q, k, v = (r.normal(size=(1, 1, N, x)) for x in (D, D, Dv))
    perm = r.permutation(N)
    a = oracle.forward(q, k, v, causal=False, lib=lib)
    b = oracle.forward(q, k[:, :, perm], v[:, :, perm], causal=False, lib=lib)
    _close(a, b, rtol=1e-13, what="key permutation")


def pin_linear_in_v(lib):
    r = _rng(15)
    N, D, Dv = 24, 3, 4
    q, k, v1, v2 = (r.normal(size=(1, 1, N, x)) for x in (D, D, Dv, Dv))
    for causal in (True, False):
        a = oracle.forward(q, k, 2.0 * v1 - 3.0 * v2, causal=causal, lib=lib)
        b = 2.0 * oracle.forward(q, k, v1, causal=causal, lib=lib) \
            - 3.0 * oracle.forward(q, k, v2, causal=causal, lib=lib)
        _close(a, b, rtol=1e-12, what="linearity")


def _loss(q, k, v, dout, causal, feature, W, lib):
    return float(np.sum(dout * oracle.forward(q, k, v, causal=causal, feature=feature, W=W,
                                              lib=lib)))


def pin_backward_finite_differences(lib):
    r = _rng(16)
    B, H, N, D, Dv = 1, 2, 5, 3, 2
    h = 1e-5
    for feature, W in (("elu1", None), ("prf", r.normal(size=(4, D)) * 0.7),
                       ("nprf", r.normal(size=(4, D))), ("trf", r.normal(size=(6, D)) * 0.3)):
        for causal in (True, False):
            q, k, v, do = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv, Dv))
            if feature == "trf":   # small inputs keep the trigonometric denominator away from 0
                q, k = q * 0.3, k * 0.3
            got = oracle.backward(q, k, v, do, causal=causal, feature=feature, W=W, lib=lib)
            for t, (x, g) in enumerate(zip((q, k, v), got)):
                fd = np.empty_like(x)
                for idx in np.ndindex(x.shape):
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += h
                    xm[idx] -= h
                    args_p = [q, k, v]
                    args_m = [q, k, v]
                    args_p[t], args_m[t] = xp, xm
                    fd[idx] = (_loss(*args_p, do, causal, feature, W, lib)
                               - _loss(*args_m, do, causal, feature, W, lib)) / (2 * h)
                err = np.max(np.abs(g - fd)) / max(np.max(np.abs(fd)), 1e-30)
                assert err <= 1e-7, f"finite differences {feature} causal={causal} d{'qkv'[t]}: {err:.2e}"


def _torch_phi(x, feature, W):
    if feature == "elu1":
        return torch.nn.functional.elu(x) + 1.0
    m = W.shape[0]
    return torch.exp(x @ W.T - 0.5 * (x * x).sum(-1, keepdim=True)) / math.sqrt(m)


def pin_backward_torch_autograd_quadratic(lib):
    r = _rng(17)
    B, H, N, D, Dv = 2, 1, 9, 4, 3
    for feature in ("elu1", "prf"):
        Wn = r.normal(size=(6, D)) * 0.6 if feature == "prf" else None
        for causal in (True, False):
            q, k, v, do = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv, Dv))
            tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
            Wt = torch.tensor(Wn, dtype=torch.float64) if Wn is not None else None
            A = _torch_phi(tq, feature, Wt) @ _torch_phi(tk, feature, Wt).transpose(-1, -2)
            if causal:
                A = torch.tril(A)
            out = (A @ tv) / A.sum(-1, keepdim=True)
            (out * torch.tensor(do)).sum().backward()
            got = oracle.backward(q, k, v, do, causal=causal, feature=feature, W=Wn, lib=lib)
            for name, g, t in zip("qkv", got, (tq, tk, tv)):
                _close(g, t.grad.numpy(), rtol=1e-10, what=f"autograd {feature} causal={causal} d{name}")


def pin_backward_constant_values(lib):
    r = _rng(18)
    B, H, N, D, Dv = 1, 3, 11, 4, 3
    for feature, W in (("elu1", None), ("prf", r.normal(size=(5, D)))):
        for causal in (True, False):
            q, k = (r.normal(size=(B, H, N, D)) for _ in range(2))
            v = np.broadcast_to(r.normal(size=(1, 1, 1, Dv)), (B, H, N, Dv)).copy()
            do = r.normal(size=(B, H, N, Dv))
            dq, dk, dv = oracle.backward(q, k, v, do, causal=causal, feature=feature, W=W, lib=lib)
            scale = np.max(np.abs(do)) * np.max(np.abs(v))
            assert np.max(np.abs(dq)) <= 1e-12 * scale * N, f"constant V: dq != 0 ({feature})"
            assert np.max(np.abs(dk)) <= 1e-12 * scale * N, f"constant V: dk != 0 ({feature})"
            # each output is a convex combination of the values: sum_j d out_i / d v_j = I
            _close(dv.sum(axis=2), do.sum(axis=2), rtol=1e-12, what=f"sum of dv ({feature})")


def pin_prefix_softmax_brute_force(lib):
    r = _rng(20)
    B, H, N, D, Dv = 2, 2, 23, 5, 3
    q = r.normal(size=(B, H, D))
    k = r.normal(size=(B, H, N, D))
    v = r.normal(size=(B, H, N, Dv))
    got = oracle.prefix_attention(q, k, v, lib=lib)
    for b in range(B):
        for h in range(H):
            s_ = k[b, h] @ q[b, h]
            ref = np.stack([scipy.special.softmax(s_[:i + 1]) @ v[b, h, :i + 1] for i in range(N)])
            _close(got[b, h], ref, rtol=1e-13, what="prefix softmax")


def _hillis_steele(s_, v):
    """Inclusive scan of (m, u, w) with the combine (a, b) -> (max, rescaled
    sums), Hillis-Steele: log2(N) rounds, element i combines i - 2^d into i."""
    n = len(s_)
    st = [(s_[i], 1.0, list(v[i])) for i in range(n)]
    d = 1
    while d < n:
        nxt = list(st)
        for i in range(d, n):
            (ma, ua, wa), (mb, ub, wb) = st[i - d], st[i]
            m = max(ma, mb)
            ea, eb = math.exp(ma - m), math.exp(mb - m)
            nxt[i] = (m, ua * ea + ub * eb, [x * ea + y * eb for x, y in zip(wa, wb)])
        st = nxt
        d *= 2
    return [[x / u for x in w] for (_, u, w) in st]


def pin_prefix_hillis_steele(lib):
    r = _rng(21)
    for N in (1, 2, 7, 16, 33):
        q = r.normal(size=(1, 1, 4))
        k = r.normal(size=(1, 1, N, 4)) * 2.0
        v = r.normal(size=(1, 1, N, 3))
        got = oracle.prefix_attention(q, k, v, lib=lib)[0, 0]
        ref = _hillis_steele((k[0, 0] @ q[0, 0]).tolist(), v[0, 0].tolist())
        _close(got, ref, rtol=1e-13, what=f"Hillis-Steele N={N}")


def pin_prefix_last_row_full_softmax_and_constant_v(lib):
    r = _rng(22)
    B, H, N, D, Dv = 1, 3, 40, 6, 4
    q = r.normal(size=(B, H, D))
    k = r.normal(size=(B, H, N, D))
    v = r.normal(size=(B, H, N, Dv))
    got = oracle.prefix_attention(q, k, v, lib=lib)
    tq, tk, tv = (torch.tensor(a) for a in (q, k, v))
    full = torch.softmax(torch.einsum("bhd,bhnd->bhn", tq, tk), dim=-1)
    _close(got[:, :, -1], torch.einsum("bhn,bhnc->bhc", full, tv).numpy(), rtol=1e-13, what="last row")
    c = np.broadcast_to(r.normal(size=(1, 1, 1, Dv)), v.shape).copy()
    _close(oracle.prefix_attention(q, k, c, lib=lib), c, rtol=1e-14, what="constant v")


def pin_prefix_step_iterated_and_large_scores(lib):
    r = _rng(23)
    B, H, N, D, Dv = 2, 1, 17, 3, 2
    for scale in (1.0, 300.0):   # scores up to about +-500: exp(s) alone over/underflows
        q = r.normal(size=(B, H, D))
        k = r.normal(size=(B, H, N, D)) * scale
        v = r.normal(size=(B, H, N, Dv))
        ref, st_ref = oracle.prefix_attention(q, k, v, return_state=True, lib=lib)
        st = np.zeros((B, H, Dv + 2))
        st[..., 0] = -np.inf
        outs = []
        for i in range(N):
            o, st = oracle.prefix_step(st, q, k[:, :, i], v[:, :, i], lib=lib)
            outs.append(o)
        _close(np.stack(outs, axis=2), ref, rtol=1e-12, what=f"step x N scale={scale}")
        _close(st, st_ref, rtol=1e-12, what="final state")
        for b in range(B):
            s_ = k[b, 0] @ q[b, 0]
            want = np.stack([scipy.special.softmax(s_[:i + 1]) @ v[b, 0, :i + 1] for i in range(N)])
            _close(ref[b, 0], want, rtol=1e-12, what=f"large scores scale={scale}")


def _rpe_fft(q, k, v, b, causal, feature, W):
    """The page's FFT method for one head: for every feature a and value
    column c (and c = the denominator's column of ones), the sequence
    y_j = phi(k_j)_a v_j,c is convolved with the Toeplitz weights
    w_t = exp(b_t) (zero for t < 0 when causal) by FFT, and the results are
    read out with phi(q_i)."""
    N = q.shape[0]
    fq = oracle.phi(q, feature, W)
    fk = oracle.phi(k, feature, W)
    wt = np.exp(b)                              # index t + N - 1
    if causal:
        wt = np.where(np.arange(2 * N - 1) >= N - 1, wt, 0.0)
    L = 4 * N                                   # room for the full linear convolution
    Wf = np.fft.rfft(np.concatenate([wt, np.zeros(L - (2 * N - 1))]))
    vv = np.concatenate([v, np.ones((N, 1))], axis=1)
    num = np.zeros((N, vv.shape[1]))
    for a in range(fk.shape[1]):
        y = fk[:, a:a + 1] * vv                 # [N, Dv + 1]
        conv = np.fft.irfft(np.fft.rfft(y, n=L, axis=0) * Wf[:, None], n=L, axis=0)
        # (w * y)[n] with w shifted by N - 1: output i reads n = i + N - 1
        num += fq[:, a:a + 1] * conv[N - 1:2 * N - 1]
    return num[:, :-1] / num[:, -1:]


def pin_rpe_matches_the_fft_method(lib):
    r = _rng(40)
    B, H, N, D, Dv = 1, 2, 19, 3, 2
    q, k, v = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv))
    b = r.normal(size=(H, 2 * N - 1)) * 0.7
    for feature, W in (("elu1", None), ("prf", r.normal(size=(5, D)))):
        for causal in (True, False):
            got = oracle.rpe(q, k, v, b, causal=causal, feature=feature, W=W, lib=lib)
            for h in range(H):
                ref = _rpe_fft(q[0, h], k[0, h], v[0, h], b[h], causal, feature, W)
                _close(got[0, h], ref, rtol=1e-10, what=f"RPE vs FFT {feature} causal={causal}")


def pin_rpe_zero_bias_and_shift(lib):
    r = _rng(41)
    B, H, N, D, Dv = 2, 2, 25, 4, 3
    q, k, v = (r.normal(size=(B, H, N, x)) for x in (D, D, Dv))
    for causal in (True, False):
        got = oracle.rpe(q, k, v, np.zeros((H, 2 * N - 1)), causal=causal, lib=lib)
        _close(got, oracle.forward(q, k, v, causal=causal, lib=lib), rtol=1e-12, what="b = 0")
        b = r.normal(size=(H, 2 * N - 1))
        _close(oracle.rpe(q, k, v, b + 3.0, causal=causal, lib=lib),
               oracle.rpe(q, k, v, b, causal=causal, lib=lib), rtol=1e-12, what="b + const")


def pin_rpe_pure_python(lib):
    r = _rng(42)
    N, D, Dv = 8, 2, 2
    q, k, v = (r.normal(size=(1, 1, N, x)) for x in (D, D, Dv))
    b = r.normal(size=(1, 2 * N - 1))
    for causal in (True, False):
        got = oracle.rpe(q, k, v, b, causal=causal, lib=lib)[0, 0]
        fq = [_py_phi(x, "elu1", None) for x in q[0, 0].tolist()]
        fk = [_py_phi(x, "elu1", None) for x in k[0, 0].tolist()]
        for i in range(N):
            num, den = [0.0] * Dv, 0.0
            for j in range(i + 1 if causal else N):
                a = sum(x * y for x, y in zip(fq[i], fk[j])) * math.exp(b[0, i - j + N - 1])
                den += a
                num = [n_ + a * v[0, 0, j, c] for c, n_ in enumerate(num)]
            _close(got[i], [n_ / den for n_ in num], rtol=1e-12, what=f"RPE brute force {causal}")


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]
