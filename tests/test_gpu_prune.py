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


# --------------------------------------------------------------------------
# The class-token side output of the attention kernel and the one-launch
# decision taken from it.

def _stride(N):
    return (N + 15) // 16 * 16


def _check_cls(case, cls, cu_r):
    """Per-head weights of every image's first row within SCORE_ATOL of the oracle."""
    keep = case.keep.numpy()
    _, _, src_r = oracle.pack_indices(keep)
    qp = oracle.pack_rows(case.q.double().numpy(), src_r)
    kp = oracle.pack_rows(case.k.double().numpy(), src_r)
    ref = oracle.cls_weights(qp, kp, cu_r, SCALE)
    got = cls.cpu().double().numpy()
    for b, w in enumerate(ref):
        n = w.shape[1]
        if n == 0:
            continue
        err = float(np.abs(got[b, :, :n] - w).max())
        assert err <= SCORE_ATOL, f"image {b}: max-abs weight error {err}"


CLS_CASES = [
    ("tiny_fp16", lambda: W.make_tiny()),
    ("serving_B4", lambda: W.make_serving(4)),
    ("batched_p50", lambda: W.make_batched(0.5)),
    ("hires_p80", lambda: W.make_hires(0.8)),
    ("chain_L3", lambda: W.make_progressive_chain(B=16)[1][2]),
    ("empty_images", lambda: W.make_custom(5, 64, 3, lengths=[0, 1, 64, 0, 17])),
    ("n1024", lambda: W.make_custom(2, 1024, 2, lengths=[1024, 700])),
]


@pytest.mark.parametrize("name,make", CLS_CASES, ids=[c[0] for c in CLS_CASES])
def test_attend_cls_side_output_and_decision_match_oracle(name, make):
    case = make()
    B, N, H, d = case.B, case.N, case.H, case.d
    keep, cu, dst, src, qp, kp, vp = _packed_on_device(case)
    cu_r = cu.cpu().numpy()
    cls = torch.full((B, H, _stride(N)), float("nan"), dtype=torch.float32, device="cuda")
    o = torch.full((B * N, H, d), float("nan"), dtype=case.dtype, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend_cls(qp, kp, vp, cu, B, N, o, cls, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    _check_cls(case, cls, cu_r)
    # The attention output is the plain tcgen05 kernel's, bit for bit.
    o2 = torch.full_like(o, float("nan"))
    prev = rra.set_attend_kernel(rra.ATTEND_TCGEN05)
    try:
        rra.attend(qp, kp, vp, cu, B, N, o2, scale=SCALE)
    finally:
        rra.set_attend_kernel(prev)
    T = int(cu_r[-1])
    assert torch.equal(o[:T].view(torch.int16), o2[:T].view(torch.int16))
    # The decision: scores within SCORE_ATOL of the oracle's, keep bit-exact on them.
    keep_new = torch.full_like(keep, 7)
    scores = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    rra.topk_keep_cls(cls, cu, src, N, 7, 10, keep_new, scores=scores)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got = scores.cpu().double().numpy()
    err = float(np.abs(got - _oracle_scores(case)).max())
    assert err <= SCORE_ATOL, f"max-abs score error {err}"
    want = oracle.topk_keep(got, case.keep.numpy(), 7, 10)
    assert np.array_equal(keep_new.cpu().numpy(), want)


@pytest.mark.parametrize("num,den", [(7, 10), (0, 1), (1, 1), (2, 3)])
def test_topk_keep_cls_ties_and_nan(num, den):
    # Hand-made side outputs: many equal scores, NaN and -inf among them.
    g = torch.Generator().manual_seed(12)
    B, N, H = 5, 300, 3
    keep = (torch.rand((B, N), generator=g) < 0.8).to(torch.uint8)
    keep[:, 0] = 1
    keep[1] = 0
    keep[2, :7] = 0
    cu, dst, src = oracle.pack_indices(keep.numpy())
    stride = _stride(N)
    cls = torch.randint(0, 4, (B, H, stride), generator=g).float()
    cls[3, 0, ::7] = float("nan")
    cls[4, :, ::5] = float("-inf")
    keep_new = torch.full((B, N), 7, dtype=torch.uint8, device="cuda")
    scores = torch.empty((B, N), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.topk_keep_cls(cls.cuda(), torch.from_numpy(cu).cuda(), torch.from_numpy(src).cuda(), N, num, den,
                      keep_new, scores=scores)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    # The scores the kernel ranked: the head mean at the original positions.
    want_scores = np.zeros((B, N))
    for b in range(B):
        n = int(cu[b + 1] - cu[b])
        pos = src[cu[b]:cu[b + 1]] - b * N
        want_scores[b, pos] = cls[b, :, :n].double().sum(dim=0).numpy() * np.float32(1.0 / H)
    got_scores = scores.cpu().double().numpy()
    fin = np.isfinite(want_scores)
    assert np.allclose(got_scores[fin], want_scores[fin], rtol=1e-6, atol=0)
    assert np.array_equal(np.isnan(got_scores), np.isnan(want_scores))
    want = oracle.topk_keep(got_scores, keep.numpy(), num, den)
    assert np.array_equal(keep_new.cpu().numpy(), want)


def test_one_pruning_layer_from_the_side_output():
    # Layer 3's attention writes the class-token weights; one launch decides
    # layer 4's mask; layer 4 attends in place from layer 3's packed layout.
    masks, cases = W.make_progressive_chain(B=16)
    c3, c4 = cases[2], cases[3]
    B, N, H, d = c3.B, c3.N, c3.H, c3.d
    keep3, cu3, dst3, src3, qp3, kp3, vp3 = _packed_on_device(c3)
    o3 = torch.empty((B * N, H, d), dtype=c3.dtype, device="cuda")
    cls = torch.empty((B, H, _stride(N)), dtype=torch.float32, device="cuda")
    rra.attend_cls(qp3, kp3, vp3, cu3, B, N, o3, cls, scale=SCALE)
    keep4 = torch.empty_like(keep3)
    scores = torch.empty((B, N), dtype=torch.float32, device="cuda")
    rra.topk_keep_cls(cls, cu3, src3, N, 7, 10, keep4, scores=scores)
    q4, k4, v4 = (x.cuda() for x in (c4.q, c4.k, c4.v))
    prev = [torch.empty((B * N, H, d), dtype=c4.dtype, device="cuda") for _ in range(3)]
    t_idx = [torch.empty(n, dtype=torch.int32, device="cuda") for n in (B + 1, B * N, B * N)]
    rra.pack(keep3, q4, k4, v4, *t_idx, *prev)                # layer 4's inputs in layer 3's layout
    cu4, dst4, src4, rows4 = (torch.empty(n, dtype=torch.int32, device="cuda") for n in (B + 1, B * N, B * N, B * N))
    rra.pack_index(keep4, cu4, dst4, src4, rows4, dst_prev=dst3)
    o4 = torch.empty((B * N, H, d), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend_rows(*prev, rows4, cu4, B, N, o4, scale=SCALE)
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


def test_attend_rows_side_output_matches_oracle():
    # The side output from the in-place mode: layer 4 of the chain read from
    # layer 3's packed layout.
    masks, cases = W.make_progressive_chain(B=16)
    case = cases[3]
    B, N, H, d = case.B, case.N, case.H, case.d
    _, dst_prev_r, src_prev_r = oracle.pack_indices(masks[2].numpy())
    cu_r, dst_r, src_r = oracle.pack_indices(case.keep.numpy())
    src_in = []
    for x in (case.q, case.k, case.v):
        buf = torch.full((B * N, H, d), float("nan"), dtype=case.dtype)
        buf[: len(src_prev_r)] = x.reshape(B * N, H, d)[torch.from_numpy(src_prev_r).long()]
        src_in.append(buf.cuda())
    rows = torch.from_numpy(dst_prev_r[src_r].astype(np.int32)).cuda()
    cu = torch.from_numpy(cu_r).cuda()
    o = torch.empty((B * N, H, d), dtype=case.dtype, device="cuda")
    cls = torch.full((B, H, _stride(N)), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend_rows(*src_in, rows, cu, B, N, o, scale=SCALE, cls=cls)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    _check_cls(case, cls, cu_r)


def test_cls_output_argument_checks():
    case = W.make_tiny()
    B, N, H, d = case.B, case.N, case.H, case.d
    keep, cu, dst, src, qp, kp, vp = _packed_on_device(case)
    o32 = torch.empty((B * N, H, d), dtype=torch.float32, device="cuda")
    cls = torch.empty((B, H, _stride(N)), dtype=torch.float32, device="cuda")
    with pytest.raises(rra.RRAError):
        rra.attend_cls(qp, kp, vp, cu, B, N, o32, cls, scale=SCALE)      # out dtype != in dtype
    o = torch.empty((B * N, H, d), dtype=case.dtype, device="cuda")
    narrow = torch.empty((B, H, _stride(N) - 16), dtype=torch.float32, device="cuda")
    with pytest.raises(rra.RRAError):
        rra.attend_cls(qp, kp, vp, cu, B, N, o, narrow, scale=SCALE)     # stride below max_seqlen


PRUNE_CASES = [
    ("chain_L3", lambda: W.make_progressive_chain(B=16)[1][2], 7, 10),
    ("batched_p50_half", lambda: W.make_batched(0.5), 1, 2),
    ("empty_and_one_row", lambda: W.make_custom(6, 64, 3, lengths=[0, 1, 64, 0, 17, 2]), 7, 10),
    ("keep_none", lambda: W.make_custom(3, 50, 2, lengths=[50, 9, 1]), 0, 1),
    ("keep_all", lambda: W.make_custom(3, 50, 2, lengths=[50, 9, 1]), 1, 1),
    ("n1024", lambda: W.make_custom(2, 1024, 2, lengths=[1024, 700]), 2, 3),
]


@pytest.mark.parametrize("name,make,num,den", PRUNE_CASES, ids=[c[0] for c in PRUNE_CASES])
def test_prune_index_matches_oracle(name, make, num, den):
    """rra_prune_index: the decision of rra_topk_keep_cls and the indices of
    rra_pack_index(keep_new, dst_prev), in one launch."""
    case = make()
    B, N, H, d = case.B, case.N, case.H, case.d
    keep, cu, dst, src, qp, kp, vp = _packed_on_device(case)
    o = torch.empty((B * N, H, d), dtype=case.dtype, device="cuda")
    cls = torch.empty((B, H, _stride(N)), dtype=torch.float32, device="cuda")
    rra.attend_cls(qp, kp, vp, cu, B, N, o, cls, scale=SCALE)
    cu2, dst2, src2, rows2 = (torch.full((n,), -9, dtype=torch.int32, device="cuda")
                              for n in (B + 1, B * N, B * N, B * N))
    keep2 = torch.full_like(keep, 7)
    scores = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.prune_index(cls, cu, src, N, num, den, cu2, dst2, src2, rows2, keep_new=keep2, scores=scores)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got_scores = scores.cpu().double().numpy()
    assert float(np.abs(got_scores - _oracle_scores(case)).max()) <= SCORE_ATOL
    keep_ref = oracle.topk_keep(got_scores, case.keep.numpy(), num, den)
    assert np.array_equal(keep2.cpu().numpy(), keep_ref)
    cu_r, dst_r, src_r = oracle.pack_indices(keep_ref)
    _, dst_prev_r, _ = oracle.pack_indices(case.keep.numpy())
    T = int(cu_r[-1])
    assert np.array_equal(cu2.cpu().numpy(), cu_r)
    assert np.array_equal(dst2.cpu().numpy(), dst_r)
    assert np.array_equal(src2.cpu().numpy()[:T], src_r)
    assert np.array_equal(rows2.cpu().numpy()[:T], dst_prev_r[src_r])
    assert np.all(src2.cpu().numpy()[T:] == -9) and np.all(rows2.cpu().numpy()[T:] == -9)
    # The same as the two-launch form (decision, then the index pass).
    keep3 = torch.empty_like(keep)
    rra.topk_keep_cls(cls, cu, src, N, num, den, keep3)
    cu3, dst3, src3, rows3 = (torch.full((n,), -9, dtype=torch.int32, device="cuda")
                              for n in (B + 1, B * N, B * N, B * N))
    rra.pack_index(keep3, cu3, dst3, src3, rows3, dst_prev=dst)
    torch.cuda.synchronize()
    for a, b in ((keep2, keep3), (cu2, cu3), (dst2, dst3), (src2, src3), (rows2, rows3)):
        assert torch.equal(a, b)
