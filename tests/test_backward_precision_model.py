"""The operand precision of the tensor-core backward, on the CPU.

A model of the chunked backward (chunks of 128 positions, the products the
kernel issues, exact sums) whose MMA operands are rounded the way the
kernel rounds them, compared with the fp64 oracle at the gradient bar
(row-relative 2e-2).  It shows why the kernel computes on fp16 operands
with dnum carried as an fp16 hi + lo pair in the dq pass: bf16 operands
miss dq by far more than the bar (the q and k gradients are small
differences: g_i . dg_i = 0), fp16 without the lo part is marginal, and the
kernel's arithmetic stays within a third of the bar.  Powers of two that the
kernel uses to keep fp16 in range are exact and left out of the model,
except the per-chunk scale of dnum, which keeps it out of fp16's subnormals.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

C = 128


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _f16(x):
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(x))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(x))


def _model_dq(q, k, v, dout, rnd, m_split):
    """dq of one causal head through the dq pass's products with operands
    rounded by `rnd`; M = [dnum | dden] scaled by the chunk's power of two and
    rounded once, or as hi + lo when `m_split`."""
    N, D = q.shape
    G, F, V = rnd(_phi(q)), rnd(_phi(k)), rnd(v)
    S, z = np.zeros((D, v.shape[1])), np.zeros(D)
    dq = np.zeros_like(q)

    def rnd_m(x, mu):
        h = rnd(x * mu)
        return (h + rnd(x * mu - h)) / mu if m_split else h / mu

    for c0 in range(0, N, C):
        sl = slice(c0, min(N, c0 + C))
        Gc, Fc, Vc = G[sl], F[sl], V[sl]
        P = rnd(np.tril(Gc @ Fc.T))
        Sr = rnd(S)
        zr = rnd(z) + rnd(z - rnd(z))                  # z as a hi + lo pair
        num = Gc @ Sr + P @ Vc
        den = Gc @ zr + P.sum(1)
        out = num / den[:, None]
        dnum = dout[sl] / den[:, None]
        dden = -(dout[sl] * out).sum(1) / den
        mu = 2.0 ** np.floor(np.log2(den.min()))
        M = np.concatenate([rnd_m(dnum, mu), (rnd(dden * mu) + rnd(dden * mu - rnd(dden * mu)))[:, None] / mu], 1)
        Vx = np.concatenate([Vc, np.ones((Vc.shape[0], 1))], 1)
        B = rnd(np.tril(M @ Vx.T) * mu) / mu
        SZ = np.concatenate([Sr, zr[:, None]], 1)
        dq[sl] = _dphi(q[sl]) * (B @ Fc + M @ SZ.T)
        S = S + Fc.T @ Vc
        z = z + Fc.sum(0)
    return dq


def _row_err(got, ref, floor):
    return float((np.abs(got - ref).max(-1) / np.maximum(np.abs(ref).max(-1), floor)).max())


@pytest.fixture(scope="module")
def case():
    w = wl.small(B=1, H=1, N=1024, D=64, Dv=64, causal=True, dtype="bf16", scaled=True, seed=1003)
    q, k, v = (t.double().numpy() for t in wl.make_qkv(w))
    do = wl.make_dout(w).double().numpy()
    rq, _, _ = oracle.backward(q, k, v, do, causal=True)
    floor = 1e-4 * np.abs(do).max() * np.abs(v).max()
    return q[0, 0], k[0, 0], v[0, 0], do[0, 0], rq[0, 0], floor


def test_model_is_exact_without_rounding(case):
    q, k, v, do, rq, floor = case
    assert _row_err(_model_dq(q, k, v, do, lambda x: np.asarray(x, np.float64), False), rq, floor) < 1e-9


def test_bf16_operands_miss_the_bar(case):
    q, k, v, do, rq, floor = case
    assert _row_err(_model_dq(q, k, v, do, _bf16, True), rq, floor) > 2e-2


def test_fp16_operands_with_split_dnum_are_within_a_third_of_the_bar(case):
    q, k, v, do, rq, floor = case
    e_split = _row_err(_model_dq(q, k, v, do, _f16, True), rq, floor)
    e_single = _row_err(_model_dq(q, k, v, do, _f16, False), rq, floor)
    assert e_split < 2e-2 / 3, e_split
    assert e_split < e_single, (e_split, e_single)
