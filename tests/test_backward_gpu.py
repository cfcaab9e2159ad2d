"""GPU parity of la_backward (dq, dk, dv) against the oracle's reverse-mode
recurrence, through the C ABI: small ragged cases over every path (causal or
not, elu+1 or random features, fp32 or bf16, head sizes 16-128, one segment
or many), and the benchmark's workloads at full size (all heads, or a fixed
sample of heads where the oracle would take too long)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_grad_close, np64

pytestmark = pytest.mark.gpu


def _check(la, w: wl.Workload, head_sample=None):
    q, k, v = wl.make_qkv(w)
    do = wl.make_dout(w)
    W = wl.make_W(w.m, w.D) if w.feature == "prf" else None
    fm = la.FeatureMap("prf", W.cuda()) if W is not None else None
    grads = la.la_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), causal=w.causal, feature_map=fm)
    torch.cuda.synchronize()
    BH = w.B * w.H
    heads = list(range(BH)) if head_sample is None else sorted(set(i % BH for i in head_sample))

    def pick(t, cols):
        return np64(t.reshape(BH, w.N, cols)[heads])[None]

    ref = oracle.backward(pick(q, w.D), pick(k, w.D), pick(v, w.Dv), pick(do, w.Dv), causal=w.causal,
                          feature=w.feature, W=W.double().numpy() if W is not None else None)
    floor = 1e-4 * float(do.abs().max()) * float(v.abs().max())
    errs = []
    for name, g, r, cols in zip(("dq", "dk", "dv"), grads, ref, (w.D, w.D, w.Dv)):
        errs.append(assert_grad_close(pick(g, cols), r, w.dtype, what=f"{w.name} {name}", floor=floor))
    return errs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,D,Dv,feature,m", [
    (1, 16, 16, "elu1", 0), (63, 32, 16, "elu1", 0), (65, 64, 64, "elu1", 0),
    (200, 128, 128, "elu1", 0), (1000 + 17, 64, 128, "elu1", 0), (300, 128, 64, "elu1", 0),
    (257, 64, 64, "prf", 128), (130, 64, 64, "prf", 256), (99, 32, 32, "prf", 64),
])
def test_backward_small(la, causal, dtype, N, D, Dv, feature, m):
    w = wl.small(B=2, H=2, N=N, D=D, Dv=Dv, causal=causal, feature=feature, m=m, dtype=dtype,
                 scaled=dtype == "bf16", seed=N * 5 + D + m)
    _check(la, w)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_many_segments(la, causal):
    """One head, a long sequence: many segments whose forward prefixes and
    reverse suffixes are chained by the scans."""
    w = wl.small(B=1, H=1, N=128 * 97 + 13, D=64, Dv=64, causal=causal, seed=404)
    _check(la, w)


def test_backward_image_3072(la):
    _check(la, wl.IMAGE_3072)


def test_backward_noncausal_4096(la):
    _check(la, wl.NONCAUSAL_4096)


def test_backward_long_65536_sampled_heads(la):
    _check(la, wl.LONG_65536, head_sample=[0, 7, 15])


def test_backward_prf_16384_sampled_heads(la):
    _check(la, wl.PRF_16384, head_sample=[0, 9])


def test_backward_tiny_f32(la):
    _check(la, wl.TINY_F32)


def test_backward_matches_finite_differences_of_the_gpu_forward(la):
    """dq, dk, dv against central differences of la_forward itself (fp32, a
    few entries): the two GPU entry points agree with each other."""
    w = wl.small(B=1, H=1, N=40, D=16, Dv=16, dtype="f32", scaled=False, seed=9)
    q, k, v = (t.cuda().double() for t in wl.make_qkv(w))
    do = wl.make_dout(w).cuda()
    dq, dk, dv = la.la_backward(q.float(), k.float(), v.float(), do, causal=True)
    h = 1e-2
    rng = np.random.default_rng(0)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.clone(), x.clone()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            lp = (la.la_forward(*(a.float() for a in args_p.values()), causal=True) * do).double().sum()
            lm = (la.la_forward(*(a.float() for a in args_m.values()), causal=True) * do).double().sum()
            fd = float((lp - lm) / (2 * h))
            assert abs(fd - float(g[idx])) <= 2e-3 * max(1.0, abs(fd)), (name, idx, fd, float(g[idx]))


# ---- the tensor-core path (bf16, elu+1, D = Dv in {64, 128}): fp16 operands,
# dnum as an fp16 hi + lo pair, per-chunk power-of-two scales

@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,D,B,H", [(2048 + 77, 64, 1, 2), (1000 + 17, 128, 2, 1), (128, 64, 1, 1),
                                     (129, 128, 1, 1), (4096, 128, 1, 3)])
def test_backward_tc_unscaled_inputs(la, causal, N, D, B, H):
    """Unscaled N(0, 1) q, k, v (|x| up to ~4.5): phi up to ~5.5, several
    segments per head; the same 2e-2 row-relative bar."""
    w = wl.small(B=B, H=H, N=N, D=D, Dv=D, causal=causal, dtype="bf16", scaled=False, seed=N + D + 31)
    _check(la, w)


def test_backward_tc_large_but_in_range_values(la):
    """One k entry of 2e4 and one v entry of -8e3 (phi and the memories well
    beyond the usual scale, inside fp16's range after the power-of-two
    scales): no flag, and the gradients still match."""
    w = wl.small(B=1, H=2, N=700, D=64, Dv=64, causal=True, dtype="bf16", scaled=False, seed=77)
    q, k, v = wl.make_qkv(w)
    do = wl.make_dout(w)
    q = (q.float() * 0.5).to(torch.bfloat16)
    k = k.clone()
    v = v.clone()
    k[0, 1, 5, 3] = 20000.0
    v[0, 0, 9, 7] = -8000.0
    assert la.la_check() == 0
    grads = la.la_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), causal=True)
    assert la.la_check() == 0
    ref = oracle.backward(np64(q), np64(k), np64(v), np64(do), causal=True)
    floor = 1e-4 * float(do.abs().max()) * float(v.abs().max())
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        assert_grad_close(np64(g.cpu()), r, "bf16", what=name, floor=floor)


def test_backward_tc_out_of_range_is_reported(la):
    """A v entry beyond fp16's range (1e5) cannot take the fp16 tensor-core
    path: la_check reports LA_ERR_RANGE once, then the flag is clear."""
    w = wl.small(B=1, H=1, N=300, D=64, Dv=64, causal=True, dtype="bf16", seed=5)
    q, k, v = wl.make_qkv(w)
    do = wl.make_dout(w)
    v = v.clone()
    v[0, 0, 17, 2] = 1.0e5
    assert la.la_check() == 0
    la.la_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), causal=True)
    assert la.la_check() == {v_: k_ for k_, v_ in la.STATUS_NAMES.items()}["LA_ERR_RANGE"]
    assert la.la_check() == 0
    # the same inputs in fp32 take the CUDA-core path, which has no such limit
    la.la_backward(q.float().cuda(), k.float().cuda(), v.float().cuda(), do.float().cuda(), causal=True)
    assert la.la_check() == 0
