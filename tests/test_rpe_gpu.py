"""GPU parity of kernelized attention with a Toeplitz relative-position
weight (la_forward_rpe) against the oracle (the definition written out,
itself pinned to the page's FFT method): the tensor-core kernel (bf16
elu+1, D, Dv in {64, 128}) causal and not, ragged lengths, and the CUDA-core
kernel for fp32 and the random-feature maps."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_close, np64

pytestmark = pytest.mark.gpu


def _check(la, w, feature="elu1", m=0, heads=None):
    q, k, v = wl.make_qkv(w)
    b = wl.make_rpe_bias(w)
    W = la.la_random_features(m, w.D, 5000) if feature != "elu1" else None
    fm = la.FeatureMap(feature, W.cuda()) if W is not None else None
    out = la.la_forward_rpe(q.cuda(), k.cuda(), v.cuda(), b.cuda(), causal=w.causal, feature_map=fm)
    torch.cuda.synchronize()
    BH = w.B * w.H
    heads = list(range(BH)) if heads is None else heads
    sub = lambda t, c: np64(t.reshape(BH, w.N, c)[heads])[None]
    bsub = np64(b)[[h % w.H for h in heads]]
    ref = oracle.rpe(sub(q, w.D), sub(k, w.D), sub(v, w.Dv), bsub, causal=w.causal, feature=feature,
                     W=W.double().numpy() if W is not None else None)
    got = np64(out.reshape(BH, w.N, w.Dv)[heads])[None]
    return assert_close(got, ref, w.dtype, what=f"rpe {w.name}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,D,Dv", [(1, 64, 64), (127, 64, 128), (128, 128, 64), (129, 128, 128),
                                    (1000, 64, 64), (4096 + 33, 128, 128)])
def test_rpe_tensor_cores(la, causal, N, D, Dv):
    w = wl.small(B=2, H=3, N=N, D=D, Dv=Dv, causal=causal, seed=N + D + Dv)
    e = _check(la, w)
    print(f"rpe tc causal={causal} N={N} D={D} Dv={Dv}: {e:.3e}")


def test_rpe_noncausal_4096_sampled_heads(la):
    w = wl.NONCAUSAL_4096
    _check(la, w, heads=[0, 21, 42, 63])


@pytest.mark.parametrize("feature,m,dtype", [("elu1", 0, "f32"), ("prf", 64, "bf16"), ("nprf", 32, "f32"),
                                             ("trf", 32, "f32")])
@pytest.mark.parametrize("causal", [True, False])
def test_rpe_cuda_cores(la, feature, m, dtype, causal):
    w = wl.small(B=1, H=2, N=300, D=32, Dv=16, causal=causal, dtype=dtype, scaled=True, seed=m + 1)
    _check(la, w, feature, m)


def test_rpe_zero_bias_is_plain_linear_attention(la):
    """b = 0: the same outputs as la_forward (both on the tensor cores)."""
    w = wl.small(B=1, H=4, N=2000, D=64, Dv=64, seed=4)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    for causal in (True, False):
        a = la.la_forward_rpe(q, k, v, torch.zeros((4, 2 * w.N - 1), device="cuda"), causal=causal)
        b = la.la_forward(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert_close(np64(a), np64(b), "bf16", what=f"b = 0, causal={causal}")
