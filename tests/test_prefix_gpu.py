"""GPU parity of softmax attention read as an RNN over every prefix
(la_prefix_attention, la_prefix_step) against the oracle's RNN cell, through
the C ABI: ragged tile counts, every head size, fp32 and bf16, scores far
apart (where a fixed shift would under- or overflow), the long workload's
keys and values over all 16 heads, the exported state, and steps that
continue from it."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_close, np64

pytestmark = pytest.mark.gpu


def _case(w, kscale=1.0):
    q = wl.make_prefix_q(w)
    _, k, v = wl.make_qkv(w)
    if kscale != 1.0:
        k = (k.float() * kscale).to(k.dtype)
    return q, k, v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,D,Dv", [(1, 16, 16), (255, 32, 64), (256, 64, 32), (257, 128, 128),
                                    (1000, 64, 64), (5000 + 3, 128, 16), (40000, 16, 128)])
def test_prefix_matches_oracle(la, dtype, N, D, Dv):
    w = wl.small(B=2, H=3, N=N, D=D, Dv=Dv, dtype=dtype, scaled=dtype == "bf16", seed=N + D * 3 + Dv)
    q, k, v = _case(w)
    out, st = la.la_prefix_attention(q.cuda(), k.cuda(), v.cuda(), return_state=True)
    torch.cuda.synchronize()
    ref, sref = oracle.prefix_attention(np64(q), np64(k), np64(v), return_state=True)
    assert_close(np64(out), ref, dtype, what=f"prefix N={N}")
    # the state: m exactly the largest score (up to fp32 rounding of s), then u and w
    # relative to it
    g = np64(st)
    assert np.max(np.abs(g[..., 0] - sref[..., 0])) <= 1e-3 * max(1.0, np.max(np.abs(sref[..., 0])))
    for sl, what in ((slice(1, 2), "u"), (slice(2, None), "w")):
        e = np.max(np.abs(g[..., sl] - sref[..., sl])) / np.max(np.abs(sref[..., sl]))
        assert e <= (1e-4 if dtype == "f32" else 2e-2), (what, e)


@pytest.mark.parametrize("kscale", [30.0, 300.0])
def test_prefix_scores_far_apart(la, kscale):
    """Scores spread over hundreds: every exponential is taken relative to a
    running maximum, so nothing over- or underflows."""
    w = wl.small(B=1, H=2, N=3000, D=32, Dv=32, dtype="f32", scaled=False, seed=77)
    q, k, v = _case(w, kscale)
    out = la.la_prefix_attention(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    ref = oracle.prefix_attention(np64(q), np64(k), np64(v))
    assert np.all(np.isfinite(np64(out)))
    # scores of this size magnify the fp32 rounding of s itself: compare where it is negligible
    assert_close(np64(out), ref, "bf16", what=f"kscale={kscale}")


def test_prefix_long_workload_all_heads(la):
    w = wl.LONG_65536
    q, k, v = _case(w)
    out = la.la_prefix_attention(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    ref = oracle.prefix_attention(np64(q), np64(k), np64(v))
    assert_close(np64(out), ref, "bf16", what="long workload")


def test_prefix_steps_continue_the_scan(la):
    """la_prefix_attention over N1 positions, then la_prefix_step through the
    next N2, equals la_prefix_attention over N1 + N2 (and the oracle)."""
    w = wl.small(B=2, H=4, N=700, D=64, Dv=64, dtype="f32", scaled=False, seed=5)
    q, k, v = (t.cuda() for t in _case(w))
    full = la.la_prefix_attention(q, k, v)
    N1 = 513
    _, st = la.la_prefix_attention(q, k[:, :, :N1].contiguous(), v[:, :, :N1].contiguous(),
                                   return_state=True)
    outs = []
    for i in range(N1, w.N):
        outs.append(la.la_prefix_step(st, q, k[:, :, i].contiguous(), v[:, :, i].contiguous()))
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=2)
    assert_close(np64(got), np64(full[:, :, N1:]), "f32", what="steps vs scan")
    ref = oracle.prefix_attention(np64(q), np64(k), np64(v))
    assert_close(np64(got), ref[:, :, N1:], "f32", what="steps vs oracle")


def test_prefix_empty_sequence_gives_the_empty_state(la):
    q = torch.zeros((1, 2, 16), device="cuda")
    k = torch.zeros((1, 2, 0, 16), device="cuda")
    v = torch.zeros((1, 2, 0, 32), device="cuda")
    st = torch.full((1, 2, 34), 7.0, device="cuda")
    la.la_prefix_attention(q, k, v, state_out=st)
    torch.cuda.synchronize()
    assert torch.all(torch.isinf(st[..., 0])) and torch.all(st[..., 0] < 0)
    assert torch.all(st[..., 1:] == 0)
    # the first step from it is the first value
    k1 = torch.randn((1, 2, 16), device="cuda")
    v1 = torch.randn((1, 2, 32), device="cuda")
    o = la.la_prefix_step(st, q, k1, v1)
    torch.cuda.synchronize()
    assert torch.allclose(o, v1, rtol=1e-6, atol=1e-6)


def test_prefix_repeated_calls_reuse_nothing(la):
    """Back-to-back calls of different sizes (the tile tickets and flags are
    reset by every call)."""
    for N, seed in ((3000, 1), (700, 2), (3000, 3)):
        w = wl.small(B=1, H=5, N=N, D=64, Dv=64, seed=seed)
        q, k, v = _case(w)
        out = la.la_prefix_attention(q.cuda(), k.cuda(), v.cuda())
        torch.cuda.synchronize()
        assert_close(np64(out), oracle.prefix_attention(np64(q), np64(k), np64(v)), "bf16", what=f"N={N}")
