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
from gpu_util import ATOL, SCALE, bits
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
