"""GPU results against closed forms the method fixes, with no oracle involved
("Transformers are RNNs", proposed method: each output row is an average of
the values with positive weights phi(q_i) . phi(k_j) over j <= i, or over
all j without the causal mask):
  - equal keys make every weight of a row the same, so out_i is the running
    mean of v_0 .. v_i (causal) or the mean of all values (non-causal);
  - a weighted average of equal vectors is that vector (constant values);
  - the last causal row averages over every key, as every non-causal row
    does, so the two forms agree there (two different kernels compute them).
Tolerances are the parity bars: fp32 1e-4 absolute; bf16 2e-2 of each
output row's largest magnitude."""
import numpy as np
import pytest
import torch

import workloads as wl
from parity_util import assert_close, np64

pytestmark = pytest.mark.gpu

# (B, H, N, D, Dv, feature, m, dtype): tensor-core shapes with several chunks,
# segments and a ragged tail, a random-feature case, and CUDA-core cases
CASES = [
    (1, 2, 128 * 23 + 45, 64, 64, "elu1", 0, "bf16"),
    (1, 3, 128 * 17 + 3, 128, 128, "elu1", 0, "bf16"),
    (2, 2, 128 * 9 + 100, 64, 64, "prf", 256, "bf16"),
    (1, 2, 1000, 64, 128, "prf", 128, "bf16"),
    (1, 2, 300, 32, 32, "elu1", 0, "f32"),
    (1, 1, 257, 16, 64, "prf", 32, "f32"),
]


def _fm(la, feature, m, D):
    return la.FeatureMap("prf", wl.make_W(m, D).cuda()) if feature == "prf" else None


def _ids(c):
    return "-".join(map(str, c))


@pytest.mark.parametrize("case", CASES, ids=_ids)
@pytest.mark.parametrize("causal", [True, False])
def test_equal_keys_give_the_mean_of_the_values(la, case, causal):
    B, H, N, D, Dv, feature, m, dtype = case
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, causal=causal, feature=feature, m=m, dtype=dtype, seed=N + D)
    q, k, v = wl.make_qkv(w)
    k = k[:, :, :1, :].expand(-1, -1, N, -1).contiguous()   # one key per head, repeated
    out = la.la_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, feature_map=_fm(la, feature, m, D))
    torch.cuda.synchronize()
    v64 = np64(v)
    if causal:
        ref = np.cumsum(v64, axis=2) / np.arange(1, N + 1, dtype=np.float64)[None, None, :, None]
    else:
        ref = np.broadcast_to(v64.mean(axis=2, keepdims=True), v64.shape)
    assert_close(np64(out), ref, dtype, what=f"equal keys {case} causal={causal}")


@pytest.mark.parametrize("case", CASES, ids=_ids)
@pytest.mark.parametrize("causal", [True, False])
def test_constant_values_come_back(la, case, causal):
    B, H, N, D, Dv, feature, m, dtype = case
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, causal=causal, feature=feature, m=m, dtype=dtype, seed=N + 2 * D)
    q, k, v = wl.make_qkv(w)
    v = v[:, :, :1, :].expand(-1, -1, N, -1).contiguous()   # one value vector per head, repeated
    out = la.la_forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, feature_map=_fm(la, feature, m, D))
    torch.cuda.synchronize()
    assert_close(np64(out), np.broadcast_to(np64(v), v.shape), dtype, what=f"constant values {case}")


@pytest.mark.parametrize("case", CASES[:4] + [(4, 8, 3072, 64, 64, "elu1", 0, "bf16")], ids=_ids)
def test_last_causal_row_is_the_noncausal_row(la, case):
    B, H, N, D, Dv, feature, m, dtype = case
    w = wl.small(B=B, H=H, N=N, D=D, Dv=Dv, feature=feature, m=m, dtype=dtype, seed=N + 3 * D)
    q, k, v = (t.cuda() for t in wl.make_qkv(w))
    fm = _fm(la, feature, m, D)
    oc = la.la_forward(q, k, v, causal=True, feature_map=fm)
    on = la.la_forward(q, k, v, causal=False, feature_map=fm)
    torch.cuda.synchronize()
    assert_close(np64(oc[:, :, -1, :]), np64(on[:, :, -1, :]), dtype, what=f"last row {case}")
