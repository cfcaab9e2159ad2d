"""la_forward_noncausal_noalloc: the non-causal forward for callers that
cannot allocate device memory (allocator hooks, memory-budgeted embedders,
real-time paths).  Its scratch is a fixed device array shared by all calls.

Checked through the C ABI against the fp64 oracle (and la_forward,
causal = 0) on the same inputs, on two calls in a row with different
inputs, so that a stale accumulator left by the first call would show up in
the second.  This file is named to be collected last.
"""
import ctypes

import pytest
import torch

import oracle
import workloads as wl
from parity_util import assert_close, np64

pytestmark = pytest.mark.gpu


def _noalloc(la, q, k, v, out, fm_struct, dtype_code):
    B, H, N, D = q.shape
    Dv = v.shape[-1]
    lib = la.load()
    fmp = ctypes.byref(fm_struct) if fm_struct is not None else None
    return lib.la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            out.data_ptr(), B, H, N, D, Dv, fmp, dtype_code,
                                            torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape,dtype,feature,m", [
    ((2, 4, 777, 64, 64), "bf16", "elu1", 0),
    ((8, 8, 4096, 64, 64), "bf16", "elu1", 0),
    ((1, 3, 300, 32, 16), "f32", "elu1", 0),
    ((1, 2, 513, 64, 64), "bf16", "prf", 128),
])
def test_noalloc_matches_the_oracle_twice(la, shape, dtype, feature, m):
    B, H, N, D, Dv = shape
    W = wl.make_W(m, D).cuda() if feature == "prf" else None
    fm = la.FeatureMap("prf", W) if W is not None else la.FeatureMap()
    code = la.LA_F32 if dtype == "f32" else la.LA_BF16
    for call in range(2):
        w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, causal=False, feature=feature, m=m,
                     dtype=dtype, scaled=dtype == "bf16", seed=100 + call)
        q, k, v = (t.cuda() for t in wl.make_qkv(w))
        ref = la.la_forward(q, k, v, causal=False, feature_map=fm)
        out = torch.full_like(ref, float("nan"))
        st = _noalloc(la, q, k, v, out, fm.c_struct(), code)
        assert st == la.LA_OK, la.la_status_string(st)
        torch.cuda.synchronize()
        exact = oracle.forward(np64(q), np64(k), np64(v), causal=False, feature=feature,
                               W=W.double().cpu().numpy() if W is not None else None)
        assert_close(np64(out), exact, dtype, what=f"call {call} against the oracle")
        assert_close(np64(out), np64(ref), dtype, what=f"call {call} against la_forward")


def test_noalloc_accepts_the_largest_problem_that_fits(la):
    """B*H*Dphi*(Dv+1)*4 bytes: 63 heads x 128 x 129 x 4 = 4,161,024 B, the
    largest elu+1 D = Dv = 128 problem under the 4 MiB limit (64 heads is
    over it: the next test); results checked against the oracle and la_forward."""
    w = wl.small(B=1, H=63, N=300, D=128, Dv=128, causal=False, seed=77)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    assert 63 * 128 * 129 * 4 <= la.LA_NOALLOC_SCRATCH_BYTES < 64 * 128 * 129 * 4
    ref = la.la_forward(q, k, v, causal=False)
    out = torch.full_like(ref, float("nan"))
    st = _noalloc(la, q, k, v, out, la.FeatureMap().c_struct(), la.LA_BF16)
    assert st == la.LA_OK, la.la_status_string(st)
    torch.cuda.synchronize()
    assert_close(np64(out), oracle.forward(np64(q), np64(k), np64(v), causal=False), "bf16",
                 what="63 heads against the oracle")
    assert_close(np64(out), np64(ref), "bf16", what="63 heads against la_forward")


def test_noalloc_steady_state_calls_allocate_nothing(la):
    """After the first call on the device (which loads the array and the
    kernels), further calls leave the device's free memory and torch's
    allocator untouched."""
    w = wl.small(B=2, H=4, N=1000, D=64, Dv=64, causal=False, seed=5)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    out = torch.empty_like(v)
    fm = la.FeatureMap().c_struct()
    assert _noalloc(la, q, k, v, out, fm, la.LA_BF16) == la.LA_OK
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        assert _noalloc(la, q, k, v, out, fm, la.LA_BF16) == la.LA_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_allocated() == alloc0


def test_noalloc_rejects_problems_beyond_its_scratch(la):
    # B*H*Dphi*(Dv+1)*4 bytes: 64 heads x 128 x 129 x 4 = 4.2 MB > 4 MiB
    q = torch.zeros((4, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    st = _noalloc(la, q, q, q, out, la.FeatureMap().c_struct(), la.LA_BF16)
    assert st == -2, la.la_status_string(st)
    with pytest.raises(la.LinAttnError):
        la.la_forward_noncausal_noalloc(q, q, q, out)
