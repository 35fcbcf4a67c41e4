"""The numpy oracle against a second, independent oracle: the same
definitions written as plain C loops (oracle/ragged_attention_ref.c), on tiny
cases (CPU only).  Indices must be identical, attention within 1e-12."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from oracle import build_c


@pytest.fixture(scope="module")
def C():
    try:
        path = build_c.build()
    except (RuntimeError, OSError) as e:
        pytest.skip(f"C oracle not built: {e}")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    lib.rra_oracle_pack_indices.argtypes = [P(ctypes.c_uint8), ctypes.c_int, ctypes.c_int, P(ctypes.c_int32),
                                            P(ctypes.c_int32), P(ctypes.c_int32)]
    lib.rra_oracle_attend.argtypes = [P(ctypes.c_double)] * 3 + [P(ctypes.c_int32), ctypes.c_int, ctypes.c_int,
                                                                 ctypes.c_int, ctypes.c_double, P(ctypes.c_double)]
    return lib


def _p(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _c_pack(C, keep):
    B, N = keep.shape
    keep = np.ascontiguousarray(keep, dtype=np.uint8)
    cu = np.zeros(B + 1, dtype=np.int32)
    dst = np.zeros(B * N, dtype=np.int32)
    src = np.full(B * N, -7, dtype=np.int32)
    C.rra_oracle_pack_indices(_p(keep, ctypes.c_uint8), B, N, _p(cu, ctypes.c_int32), _p(dst, ctypes.c_int32),
                              _p(src, ctypes.c_int32))
    return cu, dst, src[: cu[-1]]


def _c_attend(C, qp, kp, vp, cu, scale):
    T, H, d = qp.shape
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (qp, kp, vp))
    o = np.full((T, H, d), np.nan)
    cu32 = np.ascontiguousarray(cu, dtype=np.int32)
    C.rra_oracle_attend(_p(q, ctypes.c_double), _p(k, ctypes.c_double), _p(v, ctypes.c_double),
                        _p(cu32, ctypes.c_int32), len(cu) - 1, H, d, scale, _p(o, ctypes.c_double))
    return o


@pytest.mark.parametrize("seed", range(6))
def test_indices_identical(C, seed):
    rng = np.random.default_rng(100 + seed)
    B, N = int(rng.integers(1, 5)), int(rng.integers(1, 40))
    keep = (rng.random((B, N)) < rng.random()).astype(np.uint8)
    keep[rng.random(B) < 0.3] = 0                       # some images keep nothing
    for got, want in zip(_c_pack(C, keep), oracle.pack_indices(keep)):
        assert np.array_equal(got, np.asarray(want))


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("d", [8, 64])
def test_attention_within_1e12(C, seed, d):
    rng = np.random.default_rng(200 + seed)
    B, N, H = int(rng.integers(1, 4)), int(rng.integers(1, 33)), int(rng.integers(1, 4))
    keep = (rng.random((B, N)) < 0.6).astype(np.uint8)
    keep[:, 0] = 1
    q, k, v = (rng.standard_normal((B, N, H, d)) * 2.0 for _ in range(3))
    cu, dst, src = oracle.pack_indices(keep)
    qp, kp, vp = (oracle.pack_rows(x, src) for x in (q, k, v))
    scale = float(rng.uniform(0.05, 1.0))
    want = oracle.attend(qp, kp, vp, cu, scale)
    got = _c_attend(C, qp, kp, vp, cu, scale)
    assert np.all(np.isfinite(got))
    assert float(np.abs(got - want).max()) <= 1e-12
