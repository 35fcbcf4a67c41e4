"""The seeded input generator: shapes, length mixes and determinism."""
import math

import torch

from ragged_attention_token_gb300 import workloads as W


def _check(case, B, N, H, dtype):
    assert case.keep.shape == (B, N) and case.keep.dtype == torch.uint8
    for x in (case.q, case.k, case.v):
        assert x.shape == (B, N, H, 64) and x.dtype == dtype and x.is_contiguous()
    assert bool((case.keep[:, 0] == 1).all())          # CLS kept


def test_tiny():
    c = W.make_tiny()
    _check(c, 2, 197, 3, torch.float16)
    for b, r in enumerate(c.meta["keep_rate"]):
        assert 0.2 <= r <= 1.0
        # Bernoulli(r) over 196 patches: well inside 6 sigma
        assert abs((c.lengths[b] - 1) - 196 * r) < 6 * math.sqrt(196 * r * (1 - r)) + 1


def test_serving_counts():
    for B in W.SERVING_BATCHES:
        c = W.make_serving(B)
        _check(c, B, 197, 6, torch.bfloat16)
        assert all(35 <= n <= 43 for n in c.lengths)


def test_batched_rates():
    for p in W.BATCHED_RATES:
        c = W.make_batched(p)
        _check(c, 64, 197, 12, torch.bfloat16)
        if p == 0.0:
            assert c.lengths == [197] * 64
        else:
            lo = 1 + round(196 * (1 - p) * 0.9) - 1
            hi = 1 + round(196 * (1 - p) * 1.1) + 1
            assert all(lo <= n <= hi for n in c.lengths)


def test_hires_rates():
    for p in W.HIRES_RATES:
        c = W.make_hires(p)
        _check(c, 32, 577, 12, torch.bfloat16)
        lo = 1 + round(576 * (1 - p) * 0.9) - 1
        hi = 1 + round(576 * (1 - p) * 1.1) + 1
        assert all(lo <= n <= hi for n in c.lengths)


def test_progressive_schedule():
    masks = W.progressive_masks()
    want = []
    n = 196
    for layer in range(1, 13):
        if layer in (4, 7, 10):
            n = math.ceil(0.7 * n)
        want.append(n + 1)
    assert want == [197] * 3 + [139] * 3 + [98] * 3 + [69] * 3
    for layer, m in enumerate(masks, start=1):
        assert m.shape == (256, 197)
        assert (m != 0).sum(dim=1).tolist() == [want[layer - 1]] * 256
        if layer > 1:                                      # pruned tokens stay pruned
            assert bool(((m != 0) <= (masks[layer - 2] != 0)).all())
    c = W.make_progressive_layer(5, masks)
    _check(c, 256, 197, 6, torch.bfloat16)


def test_progressive_keeps_top_scores():
    B, N = 4, 197
    masks = W.progressive_masks(B, N, seed=77)
    g = torch.Generator().manual_seed(77)
    scores = torch.rand((3, B, N), generator=g, dtype=torch.float32)
    before = masks[2]
    after = masks[3]
    for b in range(B):
        alive = [j for j in range(1, N) if before[b, j]]
        kept = [j for j in alive if after[b, j]]
        dropped = [j for j in alive if not after[b, j]]
        assert min(scores[0, b, kept]) >= max(scores[0, b, dropped])


def test_determinism():
    a, b = W.make_batched(0.5), W.make_batched(0.5)
    assert torch.equal(a.keep, b.keep)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert W.make_batched(0.5, seed=1).seed != a.seed
