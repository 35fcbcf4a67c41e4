"""The device-side pruning step against the oracle (needs a GPU).

rra_cls_scores (the class token's attention over each image's kept tokens,
head mean) within 1e-5 of the fp64 oracle; rra_topk_keep bit-exact against
the oracle's decision taken on the same fp32 scores (the integer decision is
made in the kernel's precision on both sides); and one pruning layer of the
progressive workload driven entirely by the device.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import SCALE
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCORE_ATOL = 1e-5


def _packed_on_device(case):
    B, N, H, d = case.B, case.N, case.H, case.d
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    cu = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    dst = torch.empty(B * N, dtype=torch.int32, device="cuda")
    src = torch.empty(B * N, dtype=torch.int32, device="cuda")
    qp, kp, vp = (torch.empty((B * N, H, d), dtype=case.dtype, device="cuda") for _ in range(3))
    rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp)
    return keep, cu, dst, src, qp, kp, vp


def _oracle_scores(case):
    keep = case.keep.numpy()
    cu, dst, src = oracle.pack_indices(keep)
    qp = oracle.pack_rows(case.q.double().numpy(), src)
    kp = oracle.pack_rows(case.k.double().numpy(), src)
    return oracle.cls_scores(qp, kp, cu, src, case.N, SCALE)


CASES = [
    ("tiny_fp16", lambda: W.make_tiny()),
    ("serving_B4", lambda: W.make_serving(4)),
    ("batched_p50", lambda: W.make_batched(0.5)),
    ("hires_p80", lambda: W.make_hires(0.8)),
    ("chain_L1_dense", lambda: W.make_progressive_chain(B=16)[1][0]),
    ("empty_images", lambda: W.make_custom(5, 64, 3, lengths=[0, 1, 64, 0, 17])),
    ("n1024", lambda: W.make_custom(2, 1024, 2, lengths=[1024, 700])),
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_cls_scores_match_oracle(name, make):
    case = make()
    keep, cu, dst, src, qp, kp, vp = _packed_on_device(case)
    scores = torch.full((case.B, case.N), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.cls_scores(qp, kp, cu, src, case.B, case.N, scores, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got = scores.cpu().double().numpy()
    ref = _oracle_scores(case)
    m = case.keep.numpy() != 0
    assert np.all(got[~m] == 0)
    err = float(np.abs(got - ref).max())
    assert err <= SCORE_ATOL, f"max-abs score error {err}"
    # each image with a kept token: scores sum to 1
    sums = got.sum(axis=1)
    have = m.any(axis=1)
    assert np.allclose(sums[have], 1.0, atol=1e-4)


@pytest.mark.parametrize("num,den", [(7, 10), (1, 2), (0, 1), (1, 1), (2, 3)])
def test_topk_keep_bit_exact_on_device_scores(num, den):
    case = W.make_batched(0.5)
    keep, cu, dst, src, qp, kp, vp = _packed_on_device(case)
    scores = torch.empty((case.B, case.N), dtype=torch.float32, device="cuda")
    rra.cls_scores(qp, kp, cu, src, case.B, case.N, scores, scale=SCALE)
    keep_new = torch.full_like(keep, 7)
    rra.topk_keep(scores, keep, num, den, keep_new)
    torch.cuda.synchronize()
    want = oracle.topk_keep(scores.cpu().double().numpy(), case.keep.numpy(), num, den)
    assert np.array_equal(keep_new.cpu().numpy(), want)


def test_topk_keep_ties_nan_and_the_longest_rows():
    g = torch.Generator().manual_seed(11)
    B, N = 6, 1024
    keep = (torch.rand((B, N), generator=g) < 0.7).to(torch.uint8)
    keep[0] = 1
    keep[1] = 0                                            # an image that keeps nothing
    keep[2, :5] = 0                                        # class token is position 5
    scores = torch.randint(0, 8, (B, N), generator=g).float()   # many ties
    scores[3, ::7] = float("nan")
    scores[4, ::5] = float("-inf")
    scores[4, 1::5] = float("nan")                         # NaN ties with -inf
    keep_d, scores_d = keep.cuda(), scores.cuda()
    keep_new = torch.full_like(keep_d, 7)
    rra.topk_keep(scores_d, keep_d, 7, 10, keep_new)
    torch.cuda.synchronize()
    want = oracle.topk_keep(scores.double().numpy(), keep.numpy(), 7, 10)
    assert np.array_equal(keep_new.cpu().numpy(), want)


def test_one_pruning_layer_driven_by_the_device():
    # Layer 3's packed Q/K give the class-token scores; the device keeps the
    # top 70% of the other tokens for layer 4 and re-packs layer 4's inputs;
    # layer 4's attention then matches the oracle on that mask.
    masks, cases = W.make_progressive_chain(B=16)
    c3, c4 = cases[2], cases[3]
    B, N, H, d = c3.B, c3.N, c3.H, c3.d
    keep3, cu3, dst3, src3, qp3, kp3, _ = _packed_on_device(c3)
    scores = torch.empty((B, N), dtype=torch.float32, device="cuda")
    rra.cls_scores(qp3, kp3, cu3, src3, B, N, scores, scale=SCALE)
    keep4 = torch.empty_like(keep3)
    rra.topk_keep(scores, keep3, 7, 10, keep4)
    # Layer 4's inputs arrive in layer 3's packed layout.
    q4, k4, v4 = (x.cuda() for x in (c4.q, c4.k, c4.v))
    prev = [torch.empty((B * N, H, d), dtype=c4.dtype, device="cuda") for _ in range(3)]
    t_idx = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (B + 1, B * N, B * N)]
    rra.pack(keep3, q4, k4, v4, *t_idx, *prev)
    cu4 = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    dst4 = torch.empty(B * N, dtype=torch.int32, device="cuda")
    src4 = torch.empty(B * N, dtype=torch.int32, device="cuda")
    packed4 = [torch.empty((B * N, H, d), dtype=c4.dtype, device="cuda") for _ in range(3)]
    rra.repack(keep4, dst3, *prev, cu4, dst4, src4, *packed4)
    o4 = torch.empty((B * N, H, d), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend(*packed4, cu4, B, N, o4, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    keep4_ref = oracle.topk_keep(scores.cpu().double().numpy(), c3.keep.numpy(), 7, 10)
    assert np.array_equal(keep4.cpu().numpy(), keep4_ref)
    cu_r, dst_r, src_r = oracle.pack_indices(keep4_ref)
    T = int(cu_r[-1])
    p64 = [oracle.pack_rows(x.double().numpy(), src_r) for x in (c4.q, c4.k, c4.v)]
    ref = oracle.attend(*p64, cu_r, SCALE)
    err = float(np.abs(o4[:T].cpu().double().numpy() - ref).max())
    assert err <= 2e-3, f"max-abs error {err}"
