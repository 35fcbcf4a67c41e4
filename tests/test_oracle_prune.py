"""Pins of the oracle's device-side pruning step (CPU only).

``oracle.cls_scores`` (the class token's attention over its image's kept
tokens, averaged over heads) and ``oracle.topk_keep`` (keep the class token
and the top ceil(m*num/den) of the other kept tokens) are checked against
closed forms, invariants, brute force and the seeded workload generator's
own implementation of the same keep rule.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from ragged_attention_token_gb300 import workloads as W


def _packed(rng, B, N, H, d, p_keep=0.6, cls=True):
    keep = (rng.random((B, N)) < p_keep).astype(np.uint8)
    if cls:
        keep[:, 0] = 1
    q = rng.standard_normal((B, N, H, d))
    k = rng.standard_normal((B, N, H, d))
    cu, dst, src = oracle.pack_indices(keep)
    return keep, q, k, cu, src, oracle.pack_rows(q, src), oracle.pack_rows(k, src)


def test_scores_sum_to_one_and_vanish_at_pruned_positions():
    rng = np.random.default_rng(1)
    keep, q, k, cu, src, qp, kp = _packed(rng, 5, 23, 3, 8)
    s = oracle.cls_scores(qp, kp, cu, src, 23, 0.35)
    assert np.allclose(s.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(s[keep == 0] == 0) and np.all(s[keep != 0] > 0)


def test_zero_class_query_gives_uniform_scores():
    rng = np.random.default_rng(2)
    keep, q, k, cu, src, qp, kp = _packed(rng, 4, 17, 2, 4)
    for b in range(4):
        qp[cu[b]] = 0.0                               # the class token's query
    s = oracle.cls_scores(qp, kp, cu, src, 17, 0.5)
    n = keep.sum(axis=1)
    for b in range(4):
        assert np.allclose(s[b][keep[b] != 0], 1.0 / n[b], atol=1e-15)


def test_two_token_image_is_a_mean_of_sigmoids():
    # Keys {k0, k1}: the class token's weight on k1 is sigmoid(scale*q.(k1-k0)).
    rng = np.random.default_rng(3)
    H, d, scale = 4, 6, 0.7
    keep = np.zeros((1, 9), dtype=np.uint8)
    keep[0, [0, 5]] = 1
    q = rng.standard_normal((1, 9, H, d))
    k = rng.standard_normal((1, 9, H, d))
    cu, dst, src = oracle.pack_indices(keep)
    s = oracle.cls_scores(oracle.pack_rows(q, src), oracle.pack_rows(k, src), cu, src, 9, scale)
    sig = [1.0 / (1.0 + math.exp(-scale * float(q[0, 0, h] @ (k[0, 5, h] - k[0, 0, h])))) for h in range(H)]
    assert s[0, 5] == pytest.approx(sum(sig) / H, rel=1e-13)
    assert s[0, 0] == pytest.approx(1.0 - sum(sig) / H, rel=1e-13)


def test_one_token_and_empty_images():
    keep = np.zeros((3, 6), dtype=np.uint8)
    keep[1, 4] = 1                                    # a one-token image whose token is not at position 0
    q = np.ones((3, 6, 2, 4))
    k = np.ones((3, 6, 2, 4))
    cu, dst, src = oracle.pack_indices(keep)
    s = oracle.cls_scores(oracle.pack_rows(q, src), oracle.pack_rows(k, src), cu, src, 6, 0.125)
    want = np.zeros((3, 6))
    want[1, 4] = 1.0
    assert np.array_equal(s, want)


def test_scores_ignore_a_shift_common_to_all_keys_and_follow_permutations():
    rng = np.random.default_rng(4)
    keep, q, k, cu, src, qp, kp = _packed(rng, 3, 15, 2, 5)
    base = oracle.cls_scores(qp, kp, cu, src, 15, 0.4)
    shift = rng.standard_normal((1, 2, 5))
    assert np.allclose(oracle.cls_scores(qp, kp + shift, cu, src, 15, 0.4), base, atol=1e-12)
    # Swap two non-class kept tokens of image 0 (their key rows and positions).
    b = 0
    rows = list(range(int(cu[b]) + 1, int(cu[b + 1])))
    i, j = rows[0], rows[-1]
    kp2 = kp.copy()
    kp2[[i, j]] = kp2[[j, i]]
    s2 = oracle.cls_scores(qp, kp2, cu, src, 15, 0.4)
    pi, pj = int(src[i]) - b * 15, int(src[j]) - b * 15
    assert s2[b, pi] == pytest.approx(base[b, pj], rel=1e-12)
    assert s2[b, pj] == pytest.approx(base[b, pi], rel=1e-12)


def test_cls_weights_per_head_closed_forms():
    # Zero class query: every head's weights are uniform; two rows: sigmoid per head.
    rng = np.random.default_rng(6)
    keep, q, k, cu, src, qp, kp = _packed(rng, 3, 13, 3, 4)
    for b in range(3):
        qp[cu[b]] = 0.0
    w = oracle.cls_weights(qp, kp, cu, 0.5)
    for b in range(3):
        n = int(cu[b + 1] - cu[b])
        assert w[b].shape == (3, n)
        assert np.allclose(w[b], 1.0 / n, atol=1e-15)
    H, d, scale = 4, 6, 0.7
    keep = np.zeros((2, 9), dtype=np.uint8)
    keep[0, [2, 7]] = 1                                  # image 1 keeps nothing
    q = rng.standard_normal((2, 9, H, d))
    k = rng.standard_normal((2, 9, H, d))
    cu, dst, src = oracle.pack_indices(keep)
    w = oracle.cls_weights(oracle.pack_rows(q, src), oracle.pack_rows(k, src), cu, scale)
    for h in range(H):
        sig = 1.0 / (1.0 + math.exp(-scale * float(q[0, 2, h] @ (k[0, 7, h] - k[0, 2, h]))))
        assert w[0][h, 1] == pytest.approx(sig, rel=1e-13)
        assert w[0][h, 0] == pytest.approx(1.0 - sig, rel=1e-13)
    assert w[1].shape == (H, 0)


def test_cls_weights_rows_sum_to_one_and_their_mean_is_the_score():
    rng = np.random.default_rng(7)
    keep, q, k, cu, src, qp, kp = _packed(rng, 4, 21, 3, 8)
    w = oracle.cls_weights(qp, kp, cu, 0.3)
    s = oracle.cls_scores(qp, kp, cu, src, 21, 0.3)
    for b in range(4):
        assert np.allclose(w[b].sum(axis=1), 1.0, atol=1e-12)
        pos = src[cu[b]:cu[b + 1]] - b * 21
        assert np.allclose(w[b].mean(axis=0), s[b, pos], atol=1e-15)


def test_topk_counts_and_ties():
    keep = np.ones((4, 197), dtype=np.uint8)
    keep[1, 100:] = 0
    keep[2, 1:] = 0
    keep[3, :] = 0
    scores = np.ones((4, 197))                        # all equal: the lowest positions win
    out = oracle.topk_keep(scores, keep, 7, 10)
    assert out[0].sum() == 1 + math.ceil(196 * 7 / 10) == 139
    assert np.array_equal(np.nonzero(out[0])[0], np.arange(139))
    assert out[1].sum() == 1 + (99 * 7 + 9) // 10 and np.array_equal(np.nonzero(out[1])[0], np.arange(1 + 70))
    assert np.array_equal(np.nonzero(out[2])[0], [0])   # only the class token
    assert out[3].sum() == 0
    assert np.all(out <= keep)


def test_topk_is_the_best_subset_by_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(40):
        N = 9
        keep = (rng.random((1, N)) < 0.8).astype(np.uint8)
        keep[0, 0] = 1
        scores = rng.random((1, N))
        num, den = int(rng.integers(1, 5)), 4
        out = oracle.topk_keep(scores, keep, num, den)
        others = [j for j in range(1, N) if keep[0, j]]
        k = math.ceil(len(others) * num / den)
        best = max(itertools.combinations(others, k), key=lambda c: sum(scores[0, list(c)]))
        assert set(np.nonzero(out[0])[0]) == {0, *best}


def test_topk_nan_counts_as_minus_infinity():
    keep = np.ones((1, 6), dtype=np.uint8)
    scores = np.array([[0.0, np.nan, 0.2, np.nan, 0.1, 0.3]])
    out = oracle.topk_keep(scores, keep, 3, 5)        # m = 5, k = 3
    assert list(np.nonzero(out[0])[0]) == [0, 2, 4, 5]
    out = oracle.topk_keep(scores, keep, 4, 5)        # k = 4: the first NaN position
    assert list(np.nonzero(out[0])[0]) == [0, 1, 2, 4, 5]
    tie = np.array([[0.0, np.nan, -np.inf, 5.0]])     # NaN and -inf tie; the lower position wins
    assert list(np.nonzero(oracle.topk_keep(tie, np.ones((1, 4), np.uint8), 2, 3)[0])[0]) == [0, 1, 3]


def test_topk_reproduces_the_workload_generators_rule():
    # The progressive workload's generator applies the same keep rule with its
    # own code (torch stable sort); fed the generator's scores, topk_keep must
    # give its masks.
    B, N, seed = 6, 197, 77
    masks = W.progressive_masks(B, N, seed)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    scores = torch.rand((len(W.PROGRESSIVE_EVENTS), B, N), generator=g, dtype=torch.float32).double().numpy()
    keep = np.ones((B, N), dtype=np.uint8)
    for e, layer in enumerate(W.PROGRESSIVE_EVENTS):
        keep = oracle.topk_keep(scores[e], keep, 7, 10)
        assert np.array_equal(keep, masks[layer - 1].numpy()), f"layer {layer}"
