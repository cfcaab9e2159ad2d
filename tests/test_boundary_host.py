"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point that include/*.h declares, and rejects bad arguments on
the host with the documented status codes before touching the device."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from causal_linear_attention_map_b300 import build

    build.build()
    import causal_linear_attention_map_b300 as la

    return la.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(la_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("la_forward", "la_forward_ex", "la_step", "la_status_string", "la_check"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_binding_names_match(lib):
    import causal_linear_attention_map_b300 as la

    for name in declared_functions():
        assert hasattr(la, name), f"binding lacks {name}"


def test_status_strings(lib):
    import causal_linear_attention_map_b300 as la

    for code, name in la.STATUS_NAMES.items():
        assert la.la_status_string(code).startswith(name)
    assert "unknown" in la.la_status_string(12345)
    assert lib.la_version() == 100


FAKE = 0x10000000  # never dereferenced: every call below fails validation first


def _fwd(lib, B=1, H=1, N=8, D=64, Dv=64, causal=1, fm=None, dtype=1, ptrs=None, S=None, z=None):
    q, k, v, o = ptrs or (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288)
    import causal_linear_attention_map_b300 as la

    fmp = ctypes.byref(fm) if fm is not None else None
    return lib.la_forward_ex(q, k, v, o, B, H, N, D, Dv, causal, fmp, dtype, None, S, z)


def test_validation_codes(lib):
    import causal_linear_attention_map_b300 as la

    assert _fwd(lib, dtype=2) == -3
    assert _fwd(lib, dtype=-1) == -3
    assert _fwd(lib, D=48) == -2
    assert _fwd(lib, Dv=256) == -2
    assert _fwd(lib, D=8) == -2
    assert _fwd(lib, B=-1) == -2
    assert _fwd(lib, N=-5) == -2
    assert _fwd(lib, fm=la.la_feature_map(7, 0, None)) == -4
    assert _fwd(lib, fm=la.la_feature_map(1, 64, None)) == -4          # PRF without W
    assert _fwd(lib, fm=la.la_feature_map(1, 100, FAKE)) == -4         # bad m
    assert _fwd(lib, fm=la.la_feature_map(1, 64, FAKE + 4)) == -7      # unaligned W
    assert _fwd(lib, ptrs=(0, FAKE, FAKE, FAKE)) == -1
    assert _fwd(lib, ptrs=(FAKE, FAKE, FAKE, 0)) == -1
    assert _fwd(lib, ptrs=(FAKE + 2, FAKE, FAKE, FAKE)) == -7
    assert _fwd(lib, S=FAKE + 8) == -7
    # zero heads: a no-op that succeeds without touching the device
    assert _fwd(lib, B=0) == 0
    assert _fwd(lib, H=0, ptrs=(0, 0, 0, 0)) == 0


def test_step_validation_codes(lib):
    import causal_linear_attention_map_b300 as la

    p = [FAKE + 256 * i for i in range(6)]

    def st(*, B=2, H=2, D=64, Dv=64, fm=None, dtype=1, ptrs=p):
        fmp = ctypes.byref(fm) if fm is not None else None
        return lib.la_step(*ptrs, B, H, D, Dv, fmp, dtype, None)

    assert st(dtype=5) == -3
    assert st(D=12) == -2
    assert st(fm=la.la_feature_map(1, 0, FAKE)) == -4
    assert st(ptrs=[0] + p[1:]) == -1
    assert st(ptrs=p[:5] + [0]) == -1
    assert st(ptrs=[FAKE + 8] + p[1:]) == -7
    assert st(B=0) == 0


def test_host_forward_validation_codes(lib):
    """la_forward_host validates like la_forward before anything is enqueued
    (host pointers are not dereferenced on these paths)."""
    import causal_linear_attention_map_b300 as la

    p = (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288)

    def hf(*, B=1, H=1, N=8, D=64, Dv=64, fm=None, dtype=1, ptrs=p):
        fmp = ctypes.byref(fm) if fm is not None else None
        return lib.la_forward_host(*ptrs, B, H, N, D, Dv, 1, fmp, dtype, None)

    assert hf(dtype=3) == -3
    assert hf(D=48) == -2
    assert hf(N=-1) == -2
    assert hf(fm=la.la_feature_map(1, 64, None)) == -4
    assert hf(ptrs=(FAKE, 0, FAKE, FAKE)) == -1
    assert hf(ptrs=(FAKE, FAKE, FAKE, 0)) == -1
    # nothing to copy or compute: succeeds without touching the device
    assert hf(B=0) == 0
    assert hf(N=0, ptrs=(0, 0, 0, 0)) == 0


def test_noalloc_scratch_size_matches_the_header():
    import re

    import causal_linear_attention_map_b300 as la

    hdr = open(os.path.join(ROOT, "include", "linattn.h")).read()
    m = re.search(r"#define LA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m, "LA_NOALLOC_SCRATCH_BYTES not found in the header"
    assert la.LA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_backward_validation_codes(lib):
    """la_backward validates like la_forward before anything is enqueued; it
    also rejects Dphi * Dv above 16384."""
    import causal_linear_attention_map_b300 as la

    p = [FAKE + 256 * i for i in range(7)]

    def bw(*, B=1, H=2, N=8, D=64, Dv=64, fm=None, dtype=1, ptrs=p, causal=1):
        fmp = ctypes.byref(fm) if fm is not None else None
        return lib.la_backward(*ptrs, B, H, N, D, Dv, causal, fmp, dtype, None)

    assert bw(dtype=7) == -3
    assert bw(D=48) == -2
    assert bw(N=-1) == -2
    assert bw(fm=la.la_feature_map(1, 256, FAKE), Dv=128) == -2   # 256 x 128 > 16384
    assert bw(fm=la.la_feature_map(1, 64, None)) == -4
    for i in range(7):
        assert bw(ptrs=p[:i] + [0] + p[i + 1:]) == -1
    assert bw(ptrs=[FAKE + 8] + p[1:]) == -7
    assert bw(B=0) == 0
    assert bw(N=0, ptrs=[0] * 7) == 0


def test_prefix_validation_codes(lib):
    p = [FAKE + 256 * i for i in range(5)]

    def pa(*, B=1, H=2, N=8, D=64, Dv=64, dtype=1, ptrs=p):
        return lib.la_prefix_attention(*ptrs, B, H, N, D, Dv, dtype, None)

    assert pa(dtype=4) == -3
    assert pa(D=256) == -2
    assert pa(Dv=48) == -2
    assert pa(N=-1) == -2
    for i in range(4):
        assert pa(ptrs=p[:i] + [0] + p[i + 1:]) == -1
    assert pa(ptrs=p[:4] + [FAKE + 4]) == -7
    assert pa(B=0) == 0

    def ps(*, B=1, H=2, D=64, Dv=64, dtype=1, ptrs=p):
        return lib.la_prefix_step(*ptrs, B, H, D, Dv, dtype, None)

    assert ps(dtype=4) == -3
    assert ps(D=20) == -2
    for i in range(5):
        assert ps(ptrs=p[:i] + [0] + p[i + 1:]) == -1
    assert ps(H=0) == 0


def test_random_features_draws(lib):
    """la_random_features (host): deterministic by seed; Gaussian moments;
    ORF rows orthogonal within blocks of D with Gaussian-like norms; Sphere
    rows of norm sqrt(D); each gives valid positive random features for the
    softmax kernel (E[phi(q).phi(k)] = exp(q.k), through the oracle's map)."""
    import math

    import numpy as np

    import causal_linear_attention_map_b300 as la
    import oracle

    m, D = 4096, 16
    Wg = la.la_random_features(m, D, 11).numpy()
    assert np.array_equal(Wg, la.la_random_features(m, D, 11).numpy())
    assert not np.array_equal(Wg, la.la_random_features(m, D, 12).numpy())
    assert abs(Wg.mean()) < 0.02 and abs(Wg.var() - 1.0) < 0.03
    Wo = la.la_random_features(m + 5, D, 3, "orthogonal").numpy().astype(np.float64)
    for b0 in range(0, m + 5, D):
        blk = Wo[b0:b0 + D]
        G = blk @ blk.T
        nrm = np.sqrt(np.diag(G))
        off = G - np.diag(np.diag(G))
        assert np.max(np.abs(off)) <= 1e-5 * np.max(nrm) ** 2
    assert abs(np.mean(np.sum(Wo ** 2, axis=1)) - D) < 0.05 * D   # E|w|^2 = D, as for Gaussian rows
    Ws = la.la_random_features(m, D, 4, "sphere").numpy().astype(np.float64)
    assert np.allclose(np.linalg.norm(Ws, axis=1), math.sqrt(D), rtol=1e-6)
    r = np.random.default_rng(0)
    q, k = r.normal(size=D) * 0.3, r.normal(size=D) * 0.3
    for W in (Wg, Wo, Ws):
        W = W[: (m // D) * D].astype(np.float64)
        fq = oracle.phi(q[None], "prf", W)[0]
        fk = oracle.phi(k[None], "prf", W)[0]
        t = W.shape[0] * fq * fk
        assert abs(float(fq @ fk) - math.exp(float(q @ k))) < 5 * t.std() / math.sqrt(W.shape[0])
    st = lib.la_random_features(7, m, D, 1, ctypes.c_void_p(FAKE))
    assert st == -4
    assert lib.la_random_features(0, 0, D, 1, ctypes.c_void_p(FAKE)) == -2
    assert lib.la_random_features(0, m, D, 1, None) == -1
