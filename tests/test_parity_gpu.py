"""GPU parity: the CUDA library (through its C ABI) against the oracle, element
by element, on seeded inputs.  Small cases span several chunks and a ragged
tail; edge cases cover N = 1, N not a multiple of the chunk, one head, the
smallest and largest head sizes, and empty inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_close, assert_state_close, np64

pytestmark = pytest.mark.gpu


def _run(la, w: wl.Workload, export_state=False):
    q, k, v = wl.make_qkv(w)
    W = wl.make_W(w.m, w.D) if w.feature == "prf" else None
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    fm = la.FeatureMap("prf", W.cuda()) if W is not None else None
    if export_state:
        out, S, z = la.la_forward_ex(dq, dk, dv, causal=w.causal, feature_map=fm)
    else:
        out = la.la_forward(dq, dk, dv, causal=w.causal, feature_map=fm)
        S = z = None
    torch.cuda.synchronize()
    Wn = W.double().numpy() if W is not None else None
    res = oracle.forward(np64(q), np64(k), np64(v), causal=w.causal, feature=w.feature, W=Wn,
                         return_state=export_state and w.causal)
    return out, S, z, res


SMALL = [
    # (N, D, Dv, B, H, feature, m, dtype, causal)
    (64, 16, 16, 1, 1, "elu1", 0, "f32", True),
    (1, 64, 64, 1, 1, "elu1", 0, "bf16", True),
    (63, 64, 64, 1, 2, "elu1", 0, "bf16", True),
    (65, 64, 64, 2, 1, "elu1", 0, "bf16", True),
    (300, 64, 64, 1, 3, "elu1", 0, "bf16", True),
    (1000, 128, 128, 1, 2, "elu1", 0, "bf16", True),
    (257, 16, 32, 1, 2, "elu1", 0, "bf16", True),
    (129, 32, 16, 2, 1, "elu1", 0, "bf16", True),
    (333, 128, 64, 1, 1, "elu1", 0, "bf16", True),
    (200, 64, 128, 1, 1, "elu1", 0, "bf16", True),
    (500, 64, 64, 1, 2, "prf", 256, "bf16", True),
    (130, 32, 32, 1, 1, "prf", 16, "bf16", True),
    (300, 64, 64, 1, 1, "prf", 64, "f32", True),
    (300, 32, 64, 1, 2, "elu1", 0, "f32", True),
    (1, 16, 16, 1, 1, "elu1", 0, "f32", False),
    (100, 16, 16, 1, 1, "elu1", 0, "f32", False),
    (777, 64, 64, 2, 2, "elu1", 0, "bf16", False),
    (1025, 128, 128, 1, 1, "elu1", 0, "bf16", False),
    (300, 64, 64, 1, 2, "prf", 256, "bf16", False),
    (65, 32, 16, 1, 1, "prf", 32, "f32", False),
    # random features on the tensor cores (phi materialised, m = 256 as two halves)
    (1000, 64, 128, 1, 2, "prf", 128, "bf16", True),
    (700, 64, 64, 2, 1, "prf", 128, "bf16", False),
    (129, 64, 64, 1, 1, "prf", 256, "bf16", False),
    (1, 64, 64, 1, 1, "prf", 256, "bf16", True),
    # many heads (B*H >= the SM count): one segment per head, so no segment-sum
    # pass or scan, for both feature-map layouts of the causal random features
    (200, 64, 64, 2, 80, "prf", 256, "bf16", True),
    (150, 64, 128, 1, 160, "prf", 128, "bf16", True),
    # causal random features with phi formed in the chunk kernel (D = Dv = 64):
    # m = 128 with segments and a ragged tail, many heads with one segment
    # each, a head shorter than one chunk, and exactly one chunk
    (777, 64, 64, 1, 3, "prf", 128, "bf16", True),
    (300, 64, 64, 2, 80, "prf", 128, "bf16", True),
    (77, 64, 64, 1, 2, "prf", 256, "bf16", True),
    (128, 64, 64, 1, 1, "prf", 128, "bf16", True),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_forward_small(la, case):
    N, D, Dv, B, H, feature, m, dtype, causal = case
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, causal=causal, feature=feature, m=m, dtype=dtype,
                 scaled=dtype == "bf16", seed=N * 7 + D)
    out, S, z, res = _run(la, w, export_state=True)
    ref = res[0] if isinstance(res, tuple) else res
    assert_close(np64(out), ref, dtype, what=str(case))
    if causal:
        _, Sref, zref = res
        rt = 1e-5 if dtype == "f32" else 2e-2
        assert_state_close(np64(S), Sref, rt, what="S")
        assert_state_close(np64(z), zref, rt, what="z")


def test_tiny_f32_workload(la):
    w = wl.TINY_F32
    out, S, z, (ref, Sref, zref) = _run(la, w, export_state=True)
    assert_close(np64(out), ref, "f32", what=w.name)
    assert_state_close(np64(S), Sref, 1e-5, what="S")


def test_empty_and_zero_sizes(la):
    dev = "cuda"
    q = torch.zeros((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    v = torch.zeros((1, 2, 0, 64), dtype=torch.bfloat16, device=dev)
    out, S, z = la.la_forward_ex(q, q, v, causal=True)
    torch.cuda.synchronize()
    assert out.numel() == 0
    assert torch.count_nonzero(S).item() == 0 and torch.count_nonzero(z).item() == 0
    q = torch.zeros((0, 2, 5, 64), dtype=torch.bfloat16, device=dev)
    out = la.la_forward(q, q, q, causal=False)
    assert out.shape == (0, 2, 5, 64)


@pytest.mark.parametrize("feature,m,dtype", [("elu1", 0, "bf16"), ("prf", 64, "bf16"),
                                             ("elu1", 0, "f32")])
def test_step_matches_oracle_and_forward(la, feature, m, dtype):
    B, H, N, D, Dv = 2, 3, 40, 64, 32
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, feature=feature, m=m, dtype=dtype, seed=11)
    q, k, v = wl.make_qkv(w)
    W = wl.make_W(m, D) if feature == "prf" else None
    fm = la.FeatureMap("prf", W.cuda()) if W is not None else None
    P = m if feature == "prf" else D
    S = torch.zeros((B, H, P, Dv), dtype=torch.float32, device="cuda")
    z = torch.zeros((B, H, P), dtype=torch.float32, device="cuda")
    outs = []
    for i in range(N):
        o = la.la_step(S, z, q[:, :, i].cuda().contiguous(), k[:, :, i].cuda().contiguous(),
                       v[:, :, i].cuda().contiguous(), feature_map=fm)
        outs.append(o)
    got = torch.stack(outs, dim=2)
    torch.cuda.synchronize()
    Wn = W.double().numpy() if W is not None else None
    ref, Sref, zref = oracle.forward(np64(q), np64(k), np64(v), causal=True, feature=feature,
                                     W=Wn, return_state=True)
    assert_close(np64(got), ref, dtype, what="steps vs oracle forward")
    assert_state_close(np64(S), Sref, 1e-5, what="S after steps")
    assert_state_close(np64(z), zref, 1e-5, what="z after steps")


HOST_CASES = [
    # (N, D, Dv, B, H, feature, m, dtype, causal).  Groups take >= 16 MB of
    # inputs: 19 heads of 6.3 MB -> 7 groups of 3, 3, ..., 1 heads; 32 heads
    # of 1.6 MB -> 3 groups of 11, 11, 10; then single-group problems with
    # random features and on the CUDA-core path
    (8192 + 5, 128, 128, 1, 19, "elu1", 0, "bf16", True),
    (4096, 64, 64, 4, 8, "elu1", 0, "bf16", False),
    (1000, 64, 64, 1, 2, "prf", 256, "bf16", True),
    (300, 32, 32, 1, 3, "elu1", 0, "f32", True),
]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", HOST_CASES, ids=lambda c: "-".join(map(str, c)))
def test_forward_host_buffers(la, case, pinned):
    """la_forward_host: host q, k, v in and out, head groups pipelined
    through the copies and the forward; element-wise parity with the oracle
    (pageable buffers too, where the driver stages the copies)."""
    N, D, Dv, B, H, feature, m, dtype, causal = case
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, causal=causal, feature=feature, m=m, dtype=dtype,
                 scaled=dtype == "bf16", seed=N * 3 + D)
    q, k, v = wl.make_qkv(w)
    W = wl.make_W(m, D) if feature == "prf" else None
    fm = la.FeatureMap("prf", W.cuda()) if W is not None else None
    if pinned:
        hq, hk, hv = (t.pin_memory() for t in (q, k, v))
        hout = None
    else:
        hq, hk, hv = q, k, v
        hout = torch.full((B, H, N, Dv), float("nan"), dtype=q.dtype)
    out = la.la_forward_host(hq, hk, hv, causal=causal, feature_map=fm, out=hout)
    torch.cuda.synchronize()
    assert not out.is_cuda
    ref = oracle.forward(np64(q), np64(k), np64(v), causal=causal, feature=feature,
                         W=W.double().numpy() if W is not None else None)
    ref = ref[0] if isinstance(ref, tuple) else ref
    assert_close(np64(out), ref, dtype, what=f"host {case} pinned={pinned}")


def test_resume_forward_then_step(la):
    """forward_ex over N1 positions exports (S, z); steps continue from it."""
    B, H, N, N1, D, Dv = 1, 2, 300, 257, 64, 64
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, seed=12)
    q, k, v = wl.make_qkv(w)
    dq, dk, dv = (t.cuda() for t in (q, k, v))
    _, S, z = la.la_forward_ex(dq[:, :, :N1].contiguous(), dk[:, :, :N1].contiguous(),
                               dv[:, :, :N1].contiguous(), causal=True)
    outs = [la.la_step(S, z, dq[:, :, i].contiguous(), dk[:, :, i].contiguous(),
                       dv[:, :, i].contiguous()) for i in range(N1, N)]
    got = torch.stack(outs, dim=2)
    torch.cuda.synchronize()
    ref = oracle.forward(np64(q), np64(k), np64(v), causal=True)[:, :, N1:]
    assert_close(np64(got), ref, "bf16", what="resume")


def test_library_is_the_loaded_native_code(la):
    la.load()
    maps = open("/proc/self/maps").read()
    assert "liblinattn.so" in maps


def test_bounded_wait_timeout_is_reported_and_the_context_survives(la):
    """Failure detection without a GPU fault: a bounded wait that nothing
    completes gives up, the next la_check reports LA_ERR_TIMEOUT (once), and
    the library keeps working afterwards."""
    torch.cuda.synchronize()
    assert la.la_check() == la.LA_OK
    assert la.la_selftest_timeout(20) == la.LA_OK
    assert la.la_check() == -6
    assert la.la_check() == la.LA_OK
    w = wl.small(B=1, H=2, N=300, D=64, Dv=64, seed=77)
    out, _, _, ref = _run(la, w)
    assert_close(np64(out), ref, "bf16", what="after the self-test")
    assert la.la_check() == la.LA_OK
