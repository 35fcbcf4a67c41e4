"""Pins for the CPU oracle, checked against things other than itself.

Each pin below is a fact fixed by the pages or by mathematics:
  * brute force over every keep mask of tiny sizes (index work and copies);
  * padded torch SDPA in fp64 (an independent library routine): with no
    pruning it must equal the ragged result, and with a key-padding mask it
    must equal it at the kept rows -- the abstract's equivalence of the packed
    pipeline with padded SDPA;
  * closed forms: one kept token returns V; Q = 0 (or equal keys) returns the
    mean of the kept V rows; the two-token sigmoid form; exact evaluation of a
    tiny case in 50-digit decimal arithmetic;
  * invariants: permutation equivariance, convex hull, shift invariance of
    keys, linearity in V, NaN in pruned rows has no effect, large logits stay
    finite.
``test_pins_catch_planted_mistakes`` plants plausible mistakes in copies of
the oracle's attention and checks that every one of them trips a pin.
"""
from __future__ import annotations

import itertools
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from ragged_attention_token_gb300 import workloads as W

SCALE = 0.125


# ---------------------------------------------------------------- index work

def _enumerate(keep):
    """All kept (b, j) in batch order, token order: the packed order by definition."""
    B, N = keep.shape
    return [(b, j) for b in range(B) for j in range(N) if keep[b, j] != 0]


def test_indices_every_mask_single_image():
    for N in range(1, 11):
        for bits in range(2 ** N):
            keep = np.array([[(bits >> j) & 1 for j in range(N)]], dtype=np.uint8)
            cu, dst, src = oracle.pack_indices(keep)
            kept = [j for j in range(N) if (bits >> j) & 1]
            assert cu.tolist() == [0, len(kept)]
            assert src.tolist() == kept
            assert dst.tolist() == [kept.index(j) if j in kept else -1 for j in range(N)]


@pytest.mark.parametrize("B,N", [(2, 4), (3, 3), (2, 5)])
def test_indices_every_mask_small_batch(B, N):
    for bits in range(2 ** (B * N)):
        keep = np.array([(bits >> i) & 1 for i in range(B * N)], dtype=np.uint8).reshape(B, N)
        cu, dst, src = oracle.pack_indices(keep)
        kept = _enumerate(keep)
        assert src.tolist() == [b * N + j for b, j in kept]
        for t, (b, j) in enumerate(kept):
            assert dst[b * N + j] == t
            assert cu[b] <= t < cu[b + 1]
        assert sum(1 for x in dst if x >= 0) == len(kept)
        assert [cu[b + 1] - cu[b] for b in range(B)] == [int(keep[b].sum()) for b in range(B)]


def test_indices_invariants_on_workload_masks():
    for case in [W.make_tiny(), W.make_serving(4), W.make_batched(0.8), W.make_hires(0.5)]:
        keep = case.keep.numpy()
        B, N = keep.shape
        cu, dst, src = oracle.pack_indices(keep)
        assert cu[0] == 0 and np.all(np.diff(cu) >= 0)
        assert cu[B] == int((keep != 0).sum()) == len(src)
        flat = keep.reshape(-1) != 0
        assert np.all(dst[~flat] == -1)
        assert np.all(src[dst[flat]] == np.nonzero(flat)[0])
        assert np.all(np.diff(src) > 0)               # stable: original order
        for b in range(B):
            d = dst[b * N:(b + 1) * N]
            d = d[d >= 0]
            assert np.all(np.diff(d) == 1)
            assert len(d) == 0 or d[0] == cu[b]


def test_any_nonzero_byte_keeps():
    rng = np.random.default_rng(7)
    keep = rng.integers(0, 4, size=(3, 17)).astype(np.uint8) * 85   # 0, 85, 170, 255
    a = oracle.pack_indices(keep)
    b = oracle.pack_indices((keep != 0).astype(np.uint8))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------- copies (bits)

def test_pack_rows_is_a_bit_copy_of_kept_rows():
    rng = np.random.default_rng(3)
    B, N, H, d = 3, 9, 2, 4
    x = rng.integers(0, 2 ** 16, size=(B, N, H, d), dtype=np.uint16)  # NaN/Inf patterns included
    keep = (rng.random((B, N)) < 0.5).astype(np.uint8)
    _, _, src = oracle.pack_indices(keep)
    packed = oracle.pack_rows(x, src)
    expect = np.stack([x[b, j] for b, j in _enumerate(keep)]) if len(src) else np.zeros((0, H, d), np.uint16)
    assert packed.dtype == np.uint16
    assert np.array_equal(packed, expect)


def test_unpack_zero_fill_and_round_trip():
    rng = np.random.default_rng(4)
    B, N, H, d = 4, 11, 3, 8
    x = rng.standard_normal((B, N, H, d))
    keep = (rng.random((B, N)) < 0.4).astype(np.uint8)
    keep[2] = 0                                    # an image with nothing kept
    _, dst, src = oracle.pack_indices(keep)
    out = oracle.unpack(oracle.pack_rows(x, src), dst, B, N)
    assert np.array_equal(out, x * (keep[:, :, None, None] != 0))
    assert np.all(out[keep == 0] == 0.0) and not np.signbit(out[keep == 0]).any()


# ------------------------------------------------------------ attention pins

def _padded(case_like):
    keep, q, k, v = case_like
    return np.asarray(keep), np.asarray(q, np.float64), np.asarray(k, np.float64), np.asarray(v, np.float64)


def _ragged(attend_fn, keep, q, k, v, scale=SCALE):
    """Run the whole oracle path with a chosen attention implementation."""
    B, N = keep.shape
    cu, dst, src = oracle.pack_indices(keep)
    op = attend_fn(oracle.pack_rows(q, src), oracle.pack_rows(k, src), oracle.pack_rows(v, src), cu, scale)
    return oracle.unpack(op, dst, B, N)


def _sdpa(q, k, v, keep, scale=SCALE):
    """torch fp64 SDPA on the padded tensor, keys restricted by the mask."""
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3)
    mask = torch.from_numpy(keep != 0)[:, None, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


def _rand(B, N, H, d, seed, p_keep=0.6):
    rng = np.random.default_rng(seed)
    keep = (rng.random((B, N)) < p_keep).astype(np.uint8)
    keep[:, 0] = 1
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    return keep, q, k, v


def pin_dense_equals_sdpa(attend_fn):
    keep, q, k, v = _rand(3, 23, 2, 16, 11)
    keep[:] = 1
    got = _ragged(attend_fn, keep, q, k, v)
    ref = _sdpa(q, k, v, keep)
    return np.allclose(got, ref, rtol=0, atol=1e-12)


def pin_masked_equals_sdpa(attend_fn):
    keep, q, k, v = _rand(4, 29, 3, 16, 12)
    got = _ragged(attend_fn, keep, q, k, v)
    ref = _sdpa(q, k, v, keep)
    m = keep != 0
    return np.allclose(got[m], ref[m], rtol=0, atol=1e-12) and np.all(got[~m] == 0)


def pin_single_token_returns_v(attend_fn):
    keep, q, k, v = _rand(3, 13, 2, 8, 13)
    keep[:] = 0
    keep[:, 5] = 1
    got = _ragged(attend_fn, keep, q, k, v)
    return np.array_equal(got[:, 5], v[:, 5])


def pin_zero_query_gives_mean(attend_fn):
    keep, q, k, v = _rand(2, 17, 2, 8, 14)
    q[:] = 0.0
    got = _ragged(attend_fn, keep, q, k, v)
    ok = True
    for b in range(2):
        m = keep[b] != 0
        ok &= np.allclose(got[b, m], v[b, m].mean(axis=0)[None], rtol=0, atol=1e-13)
    return bool(ok)


def pin_two_tokens_closed_form(attend_fn):
    keep, q, k, v = _rand(1, 6, 1, 8, 15)
    keep[:] = 0
    keep[0, 1] = keep[0, 4] = 1
    got = _ragged(attend_fn, keep, q, k, v)
    ok = True
    for i in (1, 4):
        a = SCALE * float(q[0, i, 0] @ k[0, 1, 0])
        c = SCALE * float(q[0, i, 0] @ k[0, 4, 0])
        sig = 1.0 / (1.0 + math.exp(-(a - c)))
        want = sig * v[0, 1, 0] + (1.0 - sig) * v[0, 4, 0]
        ok &= np.allclose(got[0, i, 0], want, rtol=0, atol=1e-13)
    return bool(ok)


def pin_large_logits_stay_exact(attend_fn):
    # logits of order 1e4: exp overflows unless the row maximum is taken out;
    # the softmax then collapses to the argmax key.
    keep, q, k, v = _rand(2, 9, 1, 4, 16, p_keep=1.0)
    q *= 3000.0
    with np.errstate(all="ignore"):
        got = _ragged(attend_fn, keep, q, k, v)
    if not np.all(np.isfinite(got)):
        return False
    ok = True
    for b in range(2):
        s = q[b, :, 0] @ k[b, :, 0].T
        am = s.argmax(axis=1)
        top2 = np.sort(s, axis=1)[:, -2:]
        clear = (top2[:, 1] - top2[:, 0]) * SCALE > 50.0     # e^-50 below fp64 resolution of the rows
        ok &= np.allclose(got[b, clear, 0], v[b, am[clear], 0], rtol=0, atol=1e-12)
    return bool(ok)


def pin_exact_decimal_case(attend_fn):
    """B=2, N=3, H=1, d=2 with small integers, evaluated in 50-digit decimals."""
    getcontext().prec = 50
    keep = np.array([[1, 0, 1], [1, 1, 1]], dtype=np.uint8)
    q = np.array([[[[1, 2]], [[0, 1]], [[-1, 1]]], [[[2, 0]], [[1, -1]], [[0, 3]]]], dtype=np.float64)
    k = np.array([[[[0, 1]], [[5, 5]], [[2, -1]]], [[[1, 1]], [[-2, 0]], [[1, 2]]]], dtype=np.float64)
    v = np.array([[[[3, -1]], [[7, 7]], [[0, 2]]], [[[1, 0]], [[0, 1]], [[2, 2]]]], dtype=np.float64)
    scale = Fraction(1, 2)
    got = _ragged(attend_fn, keep, q, k, v, scale=0.5)
    ok = True
    for b in range(2):
        kept = [j for j in range(3) if keep[b, j]]
        for i in kept:
            logits = [scale * int(q[b, i, 0] @ k[b, j, 0]) for j in kept]
            w = [Decimal(l.numerator) / Decimal(l.denominator) for l in logits]
            e = [x.exp() for x in w]
            z = sum(e)
            for c in range(2):
                num = sum(e[n] * Decimal(int(v[b, j, 0, c])) for n, j in enumerate(kept))
                ok &= abs(float(num / z) - got[b, i, 0, c]) < 1e-14
        for j in range(3):
            if not keep[b, j]:
                ok &= bool(np.all(got[b, j] == 0))
    return bool(ok)


def pin_permutation_equivariance(attend_fn):
    keep, q, k, v = _rand(1, 21, 2, 8, 17, p_keep=1.0)
    perm = np.random.default_rng(0).permutation(21)
    a = _ragged(attend_fn, keep, q, k, v)
    b = _ragged(attend_fn, keep, q[:, perm], k[:, perm], v[:, perm])
    return np.allclose(a[:, perm], b, rtol=0, atol=1e-13)


def pin_nan_in_pruned_rows_ignored(attend_fn):
    keep, q, k, v = _rand(3, 19, 2, 8, 18, p_keep=0.5)
    a = _ragged(attend_fn, keep, q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for x in (q2, k2, v2):
        x[keep == 0] = np.nan
    b = _ragged(attend_fn, keep, q2, k2, v2)
    return np.array_equal(a, b)


PINS = [
    pin_dense_equals_sdpa,
    pin_masked_equals_sdpa,
    pin_single_token_returns_v,
    pin_zero_query_gives_mean,
    pin_two_tokens_closed_form,
    pin_large_logits_stay_exact,
    pin_exact_decimal_case,
    pin_permutation_equivariance,
    pin_nan_in_pruned_rows_ignored,
]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_attention_pin(pin):
    assert pin(oracle.attend)


def test_convex_hull_shift_and_linearity():
    keep, q, k, v = _rand(3, 31, 2, 16, 19)
    o = _ragged(oracle.attend, keep, q, k, v)
    m = keep != 0
    for b in range(3):
        vb = v[b, m[b]]
        assert np.all(o[b, m[b]] <= vb.max(axis=0) + 1e-12)
        assert np.all(o[b, m[b]] >= vb.min(axis=0) - 1e-12)
    c = np.random.default_rng(1).standard_normal((1, 1, 2, 16))
    o_shift = _ragged(oracle.attend, keep, q, k + c, v)
    assert np.allclose(o, o_shift, rtol=0, atol=1e-12)
    o_lin = _ragged(oracle.attend, keep, q, k, -2.5 * v)
    assert np.allclose(o_lin, -2.5 * o, rtol=0, atol=1e-12)


def test_equal_keys_give_mean():
    keep, q, k, v = _rand(2, 15, 1, 8, 20)
    k[:] = k[:, :1]
    o = _ragged(oracle.attend, keep, q, k, v)
    for b in range(2):
        m = keep[b] != 0
        assert np.allclose(o[b, m], v[b, m].mean(axis=0)[None], rtol=0, atol=1e-13)


def test_batch_permutation_permutes_output():
    keep, q, k, v = _rand(5, 13, 2, 8, 21)
    perm = np.array([3, 0, 4, 1, 2])
    a = _ragged(oracle.attend, keep, q, k, v)
    b = _ragged(oracle.attend, keep[perm], q[perm], k[perm], v[perm])
    assert np.array_equal(a[perm], b)


def test_empty_images_and_empty_batch():
    keep, q, k, v = _rand(3, 7, 2, 4, 22)
    keep[1] = 0
    out, cu, dst, src = oracle.pipeline(keep, q, k, v, SCALE)
    assert cu[2] == cu[1] and np.all(out[1] == 0) and np.all(np.isfinite(out))
    keep[:] = 0
    out, cu, dst, src = oracle.pipeline(keep, q, k, v, SCALE)
    assert len(src) == 0 and np.all(cu == 0) and np.all(out == 0)


def test_attend_row_matches_attend():
    keep, q, k, v = _rand(3, 25, 2, 8, 23)
    cu, dst, src = oracle.pack_indices(keep)
    qp, kp, vp = (oracle.pack_rows(x, src) for x in (q, k, v))
    full = oracle.attend(qp, kp, vp, cu, SCALE)
    for t in range(len(src)):
        for h in range(2):
            assert np.allclose(oracle.attend_row(qp, kp, vp, cu, SCALE, t, h), full[t, h], rtol=0, atol=1e-14)


def test_pipeline_on_workload_matches_sdpa():
    case = W.make_tiny()
    keep = case.keep.numpy()
    q, k, v = (x.double().numpy() for x in (case.q, case.k, case.v))
    out, *_ = oracle.pipeline(keep, q, k, v, SCALE)
    ref = _sdpa(q, k, v, keep)
    m = keep != 0
    assert np.allclose(out[m], ref[m], rtol=0, atol=1e-12)
    assert np.all(out[~m] == 0)


# ------------------------------------------------- planted mistakes must trip

def _mutant(kind):
    def attend(qp, kp, vp, cu, scale):
        qp, kp, vp = (np.asarray(x, np.float64) for x in (qp, kp, vp))
        T, H, d = qp.shape
        out = np.zeros((T, H, d))
        for b in range(len(cu) - 1):
            s0, s1 = int(cu[b]), int(cu[b + 1])
            if kind == "leak_next_image":
                s1k = min(s1 + 1, T)
            else:
                s1k = s1
            if s1 <= s0:
                continue
            for h in range(H):
                Q, K, V = qp[s0:s1, h], kp[s0:s1k, h], vp[s0:s1k, h]
                sc = 1.0 if kind == "no_scale" else scale
                S = sc * (Q @ K.T)
                if kind == "transposed":
                    S = sc * (K @ Q.T)
                if kind == "sign":
                    S = -S
                if kind != "no_max":
                    S = S - S.max(axis=1 if kind != "axis0" else 0, keepdims=True)
                P = np.exp(S)
                if kind != "no_norm":
                    P = P / P.sum(axis=1 if kind != "axis0" else 0, keepdims=True)
                out[s0:s1, h] = P @ (K if kind == "pk" else V)
                if kind == "first_row_only":
                    out[s0:s1, h] = (P @ V)[0]
        return out
    return attend


@pytest.mark.parametrize("kind", ["transposed", "axis0", "no_scale", "no_max", "sign",
                                  "no_norm", "pk", "leak_next_image", "first_row_only"])
def test_pins_catch_planted_mistakes(kind):
    bad = _mutant(kind)
    with np.errstate(all="ignore"):
        tripped = [p.__name__ for p in PINS if not p(bad)]
    assert tripped, f"planted mistake {kind!r} passed every pin"
