"""GPU parity of the further feature maps the kernelized-attention page names
(NPRF, TRF; Sphere-PRF and ORF as PRF with W from la_random_features)
against the oracle: forward causal and non-causal on the CUDA cores and (NPRF,
bf16, D = 64) on the tensor cores, the decode step, and the backward."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_close, assert_grad_close, np64

pytestmark = pytest.mark.gpu


def _W(la, m, D, kind="gaussian", seed=5000, scale=1.0):
    return la.la_random_features(m, D, seed, kind) * scale


def _forward(la, w, W, feature):
    q, k, v = wl.make_qkv(w)
    fm = la.FeatureMap(feature, W.cuda())
    out = la.la_forward(q.cuda(), k.cuda(), v.cuda(), causal=w.causal, feature_map=fm)
    torch.cuda.synchronize()
    ref = oracle.forward(np64(q), np64(k), np64(v), causal=w.causal, feature=feature, W=W.double().numpy())
    return assert_close(np64(out), ref, w.dtype, what=f"{feature} {w.name}")


@pytest.mark.parametrize("feature", ["nprf", "trf"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype,N,D,Dv,m", [("f32", 77, 16, 16, 16), ("f32", 300, 32, 64, 64),
                                           ("bf16", 1000 + 9, 64, 64, 128), ("bf16", 129, 64, 128, 32)])
def test_cuda_core_maps(la, feature, causal, dtype, N, D, Dv, m):
    w = wl.small(B=2, H=2, N=N, D=D, Dv=Dv, causal=causal, dtype=dtype, scaled=True, seed=N + m)
    _forward(la, w, _W(la, m, D, scale=0.5 if feature == "trf" else 1.0), feature)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H,N,m,Dv", [(2, 128 * 21 + 77, 256, 64), (3, 128 * 13 + 5, 128, 128),
                                      (16, 4096, 128, 64)])
def test_nprf_tensor_cores(la, causal, H, N, m, Dv):
    """NPRF on the tensor-core path (the projection kernel normalises x): few
    heads and many segments, a ragged last chunk, every head and position."""
    w = wl.small(B=1, H=H, N=N, D=64, Dv=Dv, causal=causal, seed=N + 2 * m)
    _forward(la, w, _W(la, m, 64), "nprf")


@pytest.mark.parametrize("kind", ["orthogonal", "sphere"])
def test_orf_and_sphere_prf_on_tensor_cores(la, kind):
    """ORF and Sphere-PRF: the PRF map with W drawn orthogonally or on the
    sphere, through the tensor-core PRF path (bf16, D = 64, m = 256)."""
    w = wl.small(B=2, H=4, N=3000, D=64, Dv=64, seed=8)
    _forward(la, w, _W(la, 256, 64, kind), "prf")


@pytest.mark.parametrize("feature", ["nprf", "trf"])
def test_step_iterated_equals_forward(la, feature):
    w = wl.small(B=2, H=3, N=40, D=32, Dv=32, dtype="f32", scaled=True, seed=3)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    W = _W(la, 64, 32, scale=0.5 if feature == "trf" else 1.0)
    fm = la.FeatureMap(feature, W.cuda())
    P = fm.phi_dim(32)
    S = torch.zeros((2, 3, P, 32), device="cuda")
    z = torch.zeros((2, 3, P), device="cuda")
    outs = [la.la_step(S, z, q[:, :, i].contiguous(), k[:, :, i].contiguous(), v[:, :, i].contiguous(),
                       feature_map=fm) for i in range(w.N)]
    torch.cuda.synchronize()
    ref = oracle.forward(np64(q), np64(k), np64(v), causal=True, feature=feature, W=W.double().numpy())
    assert_close(np64(torch.stack(outs, dim=2)), ref, "f32", what=f"step {feature}")


@pytest.mark.parametrize("feature", ["nprf", "trf"])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_new_maps(la, feature, causal, dtype):
    w = wl.small(B=1, H=3, N=333, D=32, Dv=64, causal=causal, dtype=dtype, scaled=True, seed=12)
    q, k, v = wl.make_qkv(w)
    do = wl.make_dout(w)
    W = _W(la, 64, 32, scale=0.5 if feature == "trf" else 1.0)
    grads = la.la_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), causal=causal,
                           feature_map=la.FeatureMap(feature, W.cuda()))
    torch.cuda.synchronize()
    ref = oracle.backward(np64(q), np64(k), np64(v), np64(do), causal=causal, feature=feature,
                          W=W.double().numpy())
    floor = 1e-4 * float(do.abs().max()) * float(v.abs().max())
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        assert_grad_close(np64(g), r, dtype, what=f"{feature} {name}", floor=floor)
