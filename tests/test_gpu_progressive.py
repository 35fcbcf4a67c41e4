"""Progressive token pruning as one chain of layers (needs a GPU).

Layer 1 packs its padded Q/K/V; every later layer receives its Q/K/V in the
previous layer's packed layout (as the projections of packed features would
produce them) and, at a pruning layer, re-packs them with rra_repack.  The
chain never builds a padded tensor until the final unpack.  Checked against
the oracle: indices and packed rows bit-exact, attention within the usual
bound, and a CUDA-graph replay of the whole chain bit-identical to the eager
run.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ATOL, SCALE, bits, out_tolerance
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KERNELS = [("tcgen05", rra.ATTEND_TCGEN05), ("mma_sync", rra.ATTEND_MMA_SYNC)]


@pytest.fixture(params=KERNELS, ids=[k[0] for k in KERNELS])
def kernel(request):
    prev = rra.set_attend_kernel(request.param[1])
    yield request.param[0]
    rra.set_attend_kernel(prev)


def _index_buffers(B, N):
    return (torch.full((B + 1,), -9, dtype=torch.int32, device="cuda"),
            torch.full((B * N,), -9, dtype=torch.int32, device="cuda"),
            torch.full((B * N,), -9, dtype=torch.int32, device="cuda"))


def _packed_buffers(B, N, H, d, dtype):
    return [torch.full((B * N, H, d), float("nan"), dtype=dtype, device="cuda") for _ in range(3)]


def _pack(keep, q, k, v):
    """rra_pack of padded q/k/v by `keep`: (cu, dst, src, [qp, kp, vp])."""
    B, N, H, d = q.shape
    cu, dst, src = _index_buffers(B, N)
    packed = _packed_buffers(B, N, H, d, q.dtype)
    rra.pack(keep, q, k, v, cu, dst, src, *packed)
    return cu, dst, src, packed


def test_repack_bit_exact_at_every_pruning_layer():
    masks, cases = W.make_progressive_chain(B=16)
    for layer in W.PROGRESSIVE_EVENTS:
        case = cases[layer - 1]
        B, N, H, d = case.B, case.N, case.H, case.d
        prev = masks[layer - 2].cuda()
        keep = case.keep.cuda()
        q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
        rra.get_device_error(clear=True)
        _, dst_prev, _, packed_prev = _pack(prev, q, k, v)     # the layer's inputs, previous packed layout
        cu, dst, src = _index_buffers(B, N)
        packed = _packed_buffers(B, N, H, d, case.dtype)
        rra.repack(keep, dst_prev, *packed_prev, cu, dst, src, *packed)
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        cu_r, dst_r, src_r = oracle.pack_indices(case.keep.numpy())
        T = int(cu_r[-1])
        assert np.array_equal(cu.cpu().numpy(), cu_r)
        assert np.array_equal(dst.cpu().numpy(), dst_r)
        assert np.array_equal(src.cpu().numpy()[:T], src_r)      # original positions, not previous rows
        for name, got, x in zip("qkv", packed, (case.q, case.k, case.v)):
            assert np.array_equal(bits(got)[:T], oracle.pack_rows(bits(x), src_r)), f"packed {name} differs"


def test_repack_flags_positions_pruned_before():
    masks, cases = W.make_progressive_chain(B=4)
    case = cases[3]
    B, N, H, d = case.B, case.N, case.H, case.d
    prev = masks[3].clone()                                  # the new mask itself ...
    drop = int(torch.nonzero(prev[1])[-1])
    prev[1, drop] = 0                                        # ... minus one position it keeps
    q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
    _, dst_prev, _, packed_prev = _pack(prev.cuda(), q, k, v)
    cu, dst, src = _index_buffers(B, N)
    packed = _packed_buffers(B, N, H, d, case.dtype)
    rra.get_device_error(clear=True)
    rra.repack(case.keep.cuda(), dst_prev, *packed_prev, cu, dst, src, *packed)
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_INDEX_RANGE
    cu_r, dst_r, src_r = oracle.pack_indices(case.keep.numpy())
    assert np.array_equal(cu.cpu().numpy(), cu_r)           # the indices are still the new mask's
    bad_row = int(dst_r[1 * N + drop])
    good = np.ones(int(cu_r[-1]), dtype=bool)
    good[bad_row] = False
    want = oracle.pack_rows(bits(case.q), src_r)
    assert np.array_equal(bits(packed[0])[: len(good)][good], want[good])


def test_pack_index_matches_oracle():
    """rra_pack_index: the indices of rra_pack and, per packed row, the row of the layer's input holding it."""
    masks, cases = W.make_progressive_chain(B=16)
    B, N = cases[0].B, cases[0].N
    for layer in (1,) + tuple(W.PROGRESSIVE_EVENTS):
        keep_np = masks[layer - 1].numpy()
        cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
        T = int(cu_r[-1])
        cu, dst, src = _index_buffers(B, N)
        rows = torch.full((B * N,), -9, dtype=torch.int32, device="cuda")
        dst_prev = None
        if layer == 1:
            rows_r = src_r                                    # padded input: the flat position
        else:
            _, dst_prev_r, _ = oracle.pack_indices(masks[layer - 2].numpy())
            rows_r = dst_prev_r[src_r]                         # the row in the previous packed layout
            dst_prev = torch.from_numpy(dst_prev_r).cuda()
        rra.get_device_error(clear=True)
        rra.pack_index(masks[layer - 1].cuda(), cu, dst, src, rows, dst_prev=dst_prev)
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        assert np.array_equal(cu.cpu().numpy(), cu_r)
        assert np.array_equal(dst.cpu().numpy(), dst_r)
        assert np.array_equal(src.cpu().numpy()[:T], src_r)
        got_rows = rows.cpu().numpy()
        assert np.array_equal(got_rows[:T], rows_r), f"layer {layer}: rows differ"
        assert np.all(got_rows[T:] == -9), "rows past T written"


def test_pack_index_flags_positions_pruned_before():
    masks, cases = W.make_progressive_chain(B=4)
    B, N = cases[0].B, cases[0].N
    prev = masks[3].clone()
    drop = int(torch.nonzero(prev[1])[-1])
    prev[1, drop] = 0
    _, dst_prev_r, _ = oracle.pack_indices(prev.numpy())
    cu_r, dst_r, src_r = oracle.pack_indices(masks[3].numpy())
    cu, dst, src = _index_buffers(B, N)
    rows = torch.full((B * N,), -9, dtype=torch.int32, device="cuda")
    rra.get_device_error(clear=True)
    rra.pack_index(masks[3].cuda(), cu, dst, src, rows, dst_prev=torch.from_numpy(dst_prev_r).cuda())
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_INDEX_RANGE
    T = int(cu_r[-1])
    want = dst_prev_r[src_r]
    assert np.array_equal(cu.cpu().numpy(), cu_r)
    got = rows.cpu().numpy()[:T]
    assert got[dst_r[1 * N + drop]] == -1
    assert np.array_equal(got, want)                       # want holds -1 there too


def _attend_rows_reference(case, src_r, cu_r):
    p64 = [oracle.pack_rows(x.double().numpy(), src_r) for x in (case.q, case.k, case.v)]
    return oracle.attend(*p64, cu_r, SCALE)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16], ids=["f32o", "bf16o", "f16o"])
@pytest.mark.parametrize("source", ["padded", "previous_packed"])
def test_attend_rows_matches_oracle(source, out_dtype, in_dtype):
    """rra_attend_rows at the first layer (rows of the padded input) and at a
    pruning layer (rows of the previous layer's packed buffers)."""
    masks, cases = W.make_progressive_chain(B=16)
    layer = W.PROGRESSIVE_EVENTS[0]
    case = cases[layer - 1]
    B, N, H, d = case.B, case.N, case.H, case.d
    qkv = [x.to(in_dtype) for x in (case.q, case.k, case.v)]
    keep_np = case.keep.numpy()
    cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
    T = int(cu_r[-1])
    ref_case = type("C", (), {})()
    ref_case.q, ref_case.k, ref_case.v = qkv
    o_ref = _attend_rows_reference(ref_case, src_r, cu_r)
    q, k, v = (x.cuda() for x in qkv)
    if source == "padded":
        src_in = (q.view(B * N, H, d), k.view(B * N, H, d), v.view(B * N, H, d))
        rows_r = src_r
    else:
        prev = masks[layer - 2].numpy()
        _, dst_prev_r, src_prev_r = oracle.pack_indices(prev)
        src_in = tuple(torch.full((B * N, H, d), float("nan"), dtype=in_dtype, device="cuda") for _ in range(3))
        Tp = len(src_prev_r)
        for buf, x in zip(src_in, (q, k, v)):
            buf[:Tp] = x.view(B * N, H, d)[torch.from_numpy(src_prev_r).long().cuda()]
        rows_r = dst_prev_r[src_r]
    rows = torch.from_numpy(rows_r.astype(np.int32)).cuda()
    cu = torch.from_numpy(cu_r).cuda()
    o = torch.full((B * N, H, d), float("nan"), dtype=out_dtype, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend_rows(*src_in, rows, cu, B, N, o, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got = o[:T].cpu()
    err = np.abs(got.double().numpy() - o_ref)
    tol = out_tolerance(o_ref, out_dtype)
    assert np.all(err <= tol), f"max-abs error {err.max():.3e}"
    assert torch.isnan(o[T:].float()).all(), "rows past T written"


def test_attend_rows_flags_a_row_out_of_range():
    masks, cases = W.make_progressive_chain(B=4)
    case = cases[0]
    B, N, H, d = case.B, case.N, case.H, case.d
    cu_r, dst_r, src_r = oracle.pack_indices(case.keep.numpy())
    rows_r = src_r.astype(np.int32).copy()
    rows_r[3] = B * N                                      # one past the last row
    q, k, v = (x.cuda().view(B * N, H, d) for x in (case.q, case.k, case.v))
    o = torch.empty((B * N, H, d), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.attend_rows(q, k, v, torch.from_numpy(rows_r).cuda(), torch.from_numpy(cu_r).cuda(), B, N, o, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_INDEX_RANGE
    assert torch.isfinite(o[: len(src_r)]).all()


def _run_chain(cases, inputs, bufs, B, N):
    """The chain after its inputs are in place: pack, attend, re-pack at pruning layers, final unpack."""
    first = cases[0]
    rra.pack(bufs["keep"][0], *inputs[0], *bufs["idx"][0], *bufs["packed"][0])
    for l in range(len(cases)):
        if l > 0:
            if bufs["event"][l]:
                rra.repack(bufs["keep"][l], bufs["idx"][l - 1][1], *inputs[l], *bufs["idx"][l], *bufs["packed"][l])
                packed = bufs["packed"][l]
            else:
                packed = inputs[l]
        else:
            packed = bufs["packed"][0]
        cu = bufs["idx"][l][0]
        rra.attend(*packed, cu, B, N, bufs["out"][l], scale=SCALE)
    last = len(cases) - 1
    rra.unpack(bufs["out"][last], bufs["idx"][last][1], B, N, bufs["final"])


def test_progressive_chain_matches_oracle_and_replays_in_a_graph(kernel):
    masks, cases = W.make_progressive_chain(B=16)
    B, N, H, d = cases[0].B, cases[0].N, cases[0].H, cases[0].d
    L = len(cases)
    # Layer l's inputs arrive in layer l-1's packed layout (layer 1: padded).
    inputs, idx_of = [], []
    for l, case in enumerate(cases):
        q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
        if l == 0:
            inputs.append((q, k, v))
        else:
            _, _, _, packed_prev = _pack(masks[l - 1].cuda(), q, k, v)
            inputs.append(tuple(packed_prev))
    event = [l > 0 and not torch.equal(masks[l], masks[l - 1]) for l in range(L)]
    # A layer without pruning reuses the previous layer's indices.
    idx = []
    for l in range(L):
        idx.append(_index_buffers(B, N) if (l == 0 or event[l]) else idx[l - 1])
    bufs = {
        "keep": [m.cuda() for m in masks],
        "event": event,
        "idx": idx,
        "packed": [_packed_buffers(B, N, H, d, torch.bfloat16) if (l == 0 or event[l]) else None for l in range(L)],
        "out": [torch.full((B * N, H, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(L)],
        "final": torch.full((B, N, H, d), float("nan"), dtype=torch.float32, device="cuda"),
    }
    rra.get_device_error(clear=True)
    _run_chain(cases, inputs, bufs, B, N)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    for l, case in enumerate(cases):
        keep_np = case.keep.numpy()
        cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
        T = int(cu_r[-1])
        p64 = [oracle.pack_rows(x.double().numpy(), src_r) for x in (case.q, case.k, case.v)]
        o_ref = oracle.attend(*p64, cu_r, SCALE)
        got = bufs["out"][l][:T].cpu().double().numpy()
        err = float(np.abs(got - o_ref).max())
        assert err <= ATOL, f"layer {l + 1}: max-abs error {err}"
        if l == L - 1:
            want = oracle.unpack(o_ref, dst_r, B, N)
            fin = bufs["final"].cpu().double().numpy()
            m = keep_np != 0
            assert np.all(fin[~m] == 0)
            assert float(np.abs(fin[m] - want[m]).max()) <= ATOL
    eager = [o.clone() for o in bufs["out"]] + [bufs["final"].clone()]
    # The whole chain as one CUDA graph, replayed: bit-identical results.
    for o in bufs["out"] + [bufs["final"]]:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _run_chain(cases, inputs, bufs, B, N)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, bufs["out"] + [bufs["final"]]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def _run_chain_in_place(cases, inputs, bufs, B, N):
    """The chain without packed copies: at the first layer and at every pruning
    layer an index pass (rra_pack_index) and attention reading the layer's
    input rows in place (rra_attend_rows); rra_attend elsewhere; final unpack."""
    for l in range(len(cases)):
        cu = bufs["idx"][l][0]
        if l == 0 or bufs["event"][l]:
            dst_prev = None if l == 0 else bufs["idx"][l - 1][1]
            src_in = tuple(x.view(-1, x.shape[-2], x.shape[-1]) for x in inputs[l])
            rra.pack_index(bufs["keep"][l], *bufs["idx"][l], bufs["rows"][l], dst_prev=dst_prev)
            rra.attend_rows(*src_in, bufs["rows"][l], cu, B, N, bufs["out"][l], scale=SCALE)
        else:
            rra.attend(*inputs[l], cu, B, N, bufs["out"][l], scale=SCALE)
    last = len(cases) - 1
    rra.unpack(bufs["out"][last], bufs["idx"][last][1], B, N, bufs["final"])


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32o", "bf16o"])
def test_progressive_chain_in_place_matches_oracle_and_replays_in_a_graph(out_dtype):
    masks, cases = W.make_progressive_chain(B=16)
    B, N, H, d = cases[0].B, cases[0].N, cases[0].H, cases[0].d
    L = len(cases)
    inputs = []
    for l, case in enumerate(cases):
        q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
        if l == 0:
            inputs.append((q, k, v))
        else:
            _, _, _, packed_prev = _pack(masks[l - 1].cuda(), q, k, v)
            inputs.append(tuple(packed_prev))
    event = [l > 0 and not torch.equal(masks[l], masks[l - 1]) for l in range(L)]
    idx = []
    for l in range(L):
        idx.append(_index_buffers(B, N) if (l == 0 or event[l]) else idx[l - 1])
    bufs = {
        "keep": [m.cuda() for m in masks],
        "event": event,
        "idx": idx,
        "rows": [torch.full((B * N,), -9, dtype=torch.int32, device="cuda") if (l == 0 or event[l]) else None
                 for l in range(L)],
        "out": [torch.full((B * N, H, d), float("nan"), dtype=out_dtype, device="cuda") for _ in range(L)],
        "final": torch.full((B, N, H, d), float("nan"), dtype=out_dtype, device="cuda"),
    }
    rra.get_device_error(clear=True)
    _run_chain_in_place(cases, inputs, bufs, B, N)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    for l, case in enumerate(cases):
        keep_np = case.keep.numpy()
        cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
        T = int(cu_r[-1])
        o_ref = _attend_rows_reference(case, src_r, cu_r)
        got = bufs["out"][l][:T].cpu().double().numpy()
        err = np.abs(got - o_ref)
        assert np.all(err <= out_tolerance(o_ref, out_dtype)), f"layer {l + 1}: max-abs error {err.max()}"
        if l == L - 1:
            want = oracle.unpack(o_ref, dst_r, B, N)
            fin = bufs["final"].cpu()
            m = keep_np != 0
            assert np.all(bits(fin)[~m] == 0)
            e = np.abs(fin.double().numpy()[m] - want[m])
            assert np.all(e <= out_tolerance(want[m], out_dtype))
    eager = [o.clone() for o in bufs["out"]] + [bufs["final"].clone()]
    for o in bufs["out"] + [bufs["final"]]:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _run_chain_in_place(cases, inputs, bufs, B, N)
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, bufs["out"] + [bufs["final"]]):
        assert np.array_equal(bits(a), bits(b))


def test_progressive_chain_with_device_decisions_matches_oracle():
    """The chain with every pruning decision made on the device: the layer
    before an event writes the class-token side output, one launch turns it
    into the next layer's mask and indices, and that layer attends in place.
    Each decision is checked bit-exact against the oracle's rule on the
    device's scores, each layer's attention against the oracle on the
    device's masks."""
    masks, cases = W.make_progressive_chain(B=16)
    B, N, H, d = cases[0].B, cases[0].N, cases[0].H, cases[0].d
    L = len(cases)
    events = set(l - 1 for l in W.PROGRESSIVE_EVENTS)        # 0-indexed layers whose input is pruned
    stride = (N + 15) // 16 * 16
    keep = cases[0].keep.cuda()
    cu, dst, src = _index_buffers(B, N)
    rows = torch.empty(B * N, dtype=torch.int32, device="cuda")
    rra.get_device_error(clear=True)
    rra.pack_index(keep, cu, dst, src, rows)
    keep_np = cases[0].keep.numpy()
    for l, case in enumerate(cases):
        # This layer's inputs arrive in the previous layer's packed layout (layer 1: padded).
        q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
        if l == 0:
            src_in = tuple(x.view(B * N, H, d) for x in (q, k, v))
        else:
            src_in = tuple(_pack(torch.from_numpy(prev_keep_np).cuda(), q, k, v)[3])
        o = torch.empty((B * N, H, d), dtype=torch.bfloat16, device="cuda")
        decide = (l + 1) in events
        cls = torch.empty((B, H, stride), dtype=torch.float32, device="cuda") if decide else None
        if l == 0 or l in events:
            rra.attend_rows(*src_in, rows, cu, B, N, o, scale=SCALE, cls=cls)
        elif decide:
            rra.attend_cls(*src_in, cu, B, N, o, cls, scale=SCALE)
        else:
            rra.attend(*src_in, cu, B, N, o, scale=SCALE)
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        # This layer against the oracle on the device's mask.
        cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
        T = int(cu_r[-1])
        assert np.array_equal(cu.cpu().numpy(), cu_r)
        p64 = [oracle.pack_rows(x.double().numpy(), src_r) for x in (case.q, case.k, case.v)]
        ref = oracle.attend(*p64, cu_r, SCALE)
        err = np.abs(o[:T].cpu().double().numpy() - ref)
        assert np.all(err <= out_tolerance(ref, torch.bfloat16)), f"layer {l + 1}: max-abs error {err.max()}"
        prev_keep_np = keep_np
        if decide:
            keep_new = torch.empty_like(keep)
            scores = torch.empty((B, N), dtype=torch.float32, device="cuda")
            cu2, dst2, src2 = _index_buffers(B, N)
            rows2 = torch.empty(B * N, dtype=torch.int32, device="cuda")
            rra.prune_index(cls, cu, src, N, 7, 10, cu2, dst2, src2, rows2, keep_new=keep_new, scores=scores)
            torch.cuda.synchronize()
            assert rra.get_device_error() == 0
            keep_np = keep_new.cpu().numpy()
            want = oracle.topk_keep(scores.cpu().double().numpy(), prev_keep_np, 7, 10)
            assert np.array_equal(keep_np, want), f"decision after layer {l + 1}"
            assert int(keep_np.sum()) == int(masks[l + 1].sum())   # the workload's counts
            cu, dst, src, rows = cu2, dst2, src2, rows2


def _sampled_rows_check(case, keep_np, o, n_samples=48, seed=0):
    """Sampled output rows of a layer's packed attention against oracle.attend_row."""
    cu_r, _, src_r = oracle.pack_indices(keep_np)
    T = int(cu_r[-1])
    rng = np.random.default_rng(seed)
    ts = rng.integers(0, T, n_samples)
    hs = rng.integers(0, case.H, n_samples)
    q64, k64, v64 = (x.double().numpy().reshape(case.B * case.N, case.H, case.d) for x in (case.q, case.k, case.v))
    got = o.float().cpu().double().numpy()
    for t, h in zip(ts, hs):
        b = int(np.searchsorted(cu_r, t, side="right")) - 1
        s0, s1 = int(cu_r[b]), int(cu_r[b + 1])
        rows = src_r[s0:s1]
        mini_cu = np.array([0, s1 - s0], dtype=np.int64)
        ref = oracle.attend_row(q64[rows], k64[rows], v64[rows], mini_cu, SCALE, int(t) - s0, int(h))
        err = np.abs(got[t, h] - ref)
        assert np.all(err <= out_tolerance(ref, o.dtype)), f"row {t} head {h}: max-abs error {err.max()}"


def test_progressive_chain_full_size_with_device_decisions():
    """The B=256 chain with device decisions in the launch sequence bench.py
    times (index pass, rows attention with the side output, decision + next
    indices in one launch): indices and decisions bit-exact against the oracle
    at every layer, class-token weights and sampled attention rows within
    tolerance, the final unpack's pruned rows +0."""
    masks, cases = W.make_progressive_chain(B=256)
    B, N, H, d = cases[0].B, cases[0].N, cases[0].H, cases[0].d
    L = len(cases)
    events = set(l - 1 for l in W.PROGRESSIVE_EVENTS)
    stride = (N + 15) // 16 * 16
    keep_np = cases[0].keep.numpy()
    cu, dst, src = _index_buffers(B, N)
    rows = torch.empty(B * N, dtype=torch.int32, device="cuda")
    rra.get_device_error(clear=True)
    rra.pack_index(cases[0].keep.cuda(), cu, dst, src, rows)
    prev_keep_np = None
    for l, case in enumerate(cases):
        q, k, v = (x.cuda() for x in (case.q, case.k, case.v))
        if l == 0:
            src_in = tuple(x.view(B * N, H, d) for x in (q, k, v))
        else:
            src_in = tuple(_pack(torch.from_numpy(prev_keep_np).cuda(), q, k, v)[3])
        o = torch.empty((B * N, H, d), dtype=torch.bfloat16, device="cuda")
        decide = (l + 1) in events
        cls = torch.full((B, H, stride), float("nan"), dtype=torch.float32, device="cuda") if decide else None
        if l == 0 or l in events:
            rra.attend_rows(*src_in, rows, cu, B, N, o, scale=SCALE, cls=cls)
        elif decide:
            rra.attend_cls(*src_in, cu, B, N, o, cls, scale=SCALE)
        else:
            rra.attend(*src_in, cu, B, N, o, scale=SCALE)
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        cu_r, dst_r, src_r = oracle.pack_indices(keep_np)
        T = int(cu_r[-1])
        assert np.array_equal(cu.cpu().numpy(), cu_r), f"layer {l + 1}: cu_seqlens"
        assert np.array_equal(dst.cpu().numpy(), dst_r), f"layer {l + 1}: dst_idx"
        assert np.array_equal(src.cpu().numpy()[:T], src_r), f"layer {l + 1}: src_idx"
        _sampled_rows_check(case, keep_np, o, seed=l)
        prev_keep_np = keep_np
        if decide:
            # Class-token weights of a few images against the oracle, per head.
            got_cls = cls.cpu().double().numpy()
            for b in (0, 77, 255):
                rows_b = src_r[cu_r[b]:cu_r[b + 1]]
                qb = case.q.double().numpy().reshape(B * N, H, d)[rows_b]
                kb = case.k.double().numpy().reshape(B * N, H, d)[rows_b]
                ref = oracle.cls_weights(qb, kb, np.array([0, len(rows_b)]), SCALE)[0]
                assert float(np.abs(got_cls[b, :, :len(rows_b)] - ref).max()) <= 1e-5
            keep_new = torch.empty((B, N), dtype=torch.uint8, device="cuda")
            scores = torch.empty((B, N), dtype=torch.float32, device="cuda")
            cu2, dst2, src2 = _index_buffers(B, N)
            rows2 = torch.empty(B * N, dtype=torch.int32, device="cuda")
            rra.prune_index(cls, cu, src, N, 7, 10, cu2, dst2, src2, rows2, keep_new=keep_new, scores=scores)
            torch.cuda.synchronize()
            assert rra.get_device_error() == 0
            keep_np = keep_new.cpu().numpy()
            assert np.array_equal(keep_np, oracle.topk_keep(scores.cpu().double().numpy(), prev_keep_np, 7, 10))
            _, dst_prev_r, _ = oracle.pack_indices(prev_keep_np)
            cu_n, _, src_n = oracle.pack_indices(keep_np)
            assert np.array_equal(rows2.cpu().numpy()[:int(cu_n[-1])], dst_prev_r[src_n])
            assert int(keep_np.sum()) == int(masks[l + 1].sum())
            cu, dst, src, rows = cu2, dst2, src2, rows2
    final = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    rra.unpack(o, dst, B, N, final)
    torch.cuda.synchronize()
    fin_bits = bits(final)
    assert np.all(fin_bits[keep_np == 0] == 0), "pruned positions are not +0"
    _, dst_r, _ = oracle.pack_indices(keep_np)
    kept = np.nonzero(keep_np.reshape(-1))[0][:64]
    assert np.array_equal(fin_bits.reshape(B * N, H, d)[kept], bits(o)[dst_r[kept]])
