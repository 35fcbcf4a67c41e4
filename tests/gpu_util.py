"""Shared helpers for the GPU parity tests: run the oracle and the CUDA path
on the same seeded inputs and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from ragged_attention_token_gb300 import rra

SCALE = 0.125
# Max-abs bound on attention outputs for bf16/fp16 N(0,1) inputs, checked on
# the fp32-output mode.  A bf16/fp16-stored output is additionally allowed
# half an ulp of its own type at the oracle's magnitude (the final rounding).
ATOL = 2e-3

_ORACLE_CACHE: dict = {}


def bits(x: torch.Tensor) -> np.ndarray:
    x = x.contiguous().cpu()
    if x.element_size() == 2:
        return x.view(torch.int16).numpy()
    return x.view(torch.int32).numpy()


def oracle_result(case):
    """cu, dst, src, packed bits of q/k/v, packed fp64 O, padded fp64 out."""
    key = (case.name, case.seed, case.B, case.N, case.H, int(case.keep.sum()))
    if key in _ORACLE_CACHE:
        return _ORACLE_CACHE[key]
    keep = case.keep.numpy()
    cu, dst, src = oracle.pack_indices(keep)
    packed_bits = [oracle.pack_rows(bits(x), src) for x in (case.q, case.k, case.v)]
    p64 = [oracle.pack_rows(x.double().numpy(), src) for x in (case.q, case.k, case.v)]
    o = oracle.attend(*p64, cu, SCALE)
    out = oracle.unpack(o, dst, case.B, case.N)
    res = dict(cu=cu, dst=dst, src=src, packed_bits=packed_bits, o=o, out=out)
    if len(_ORACLE_CACHE) > 8:
        _ORACLE_CACHE.clear()
    _ORACLE_CACHE[key] = res
    return res


def out_tolerance(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.full(ref.shape, ATOL)
    explicit = 7 if dtype == torch.bfloat16 else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -60)))
    return ATOL + 2.0 ** (e - explicit - 1)


def pair_tolerance(ref: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """The same rule for two stored GPU results: each may sit half an output ulp
    from the exact value on its own side, so together they may differ by one ulp."""
    if dtype == torch.float32:
        return np.full(ref.shape, ATOL)
    explicit = 7 if dtype == torch.bfloat16 else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -60)))
    return ATOL + 2.0 ** (e - explicit)


def to_device(case, device="cuda"):
    return (case.keep.to(device), case.q.to(device), case.k.to(device), case.v.to(device))


def run_pipeline(case, out_dtype=None, poison=True):
    """rra_pipeline on `case`; returns CPU copies of out and the workspace sections."""
    keep, q, k, v = to_device(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    out_dtype = out_dtype or case.dtype
    out = torch.empty((B, N, H, d), dtype=out_dtype, device="cuda")
    ws = rra.alloc_workspace(B, N, H, d, case.dtype)
    if poison:
        out.view(torch.uint8).fill_(0xFF)        # NaN everywhere: unwritten rows show up
        ws.fill_(0xFF)
    rra.pipeline(keep, q, k, v, out, ws, scale=SCALE)
    torch.cuda.synchronize()
    err = rra.get_device_error()
    cu, dst, src, qp, kp, vp = rra.workspace_views(ws, B, N, H, d, case.dtype)
    return dict(out=out.cpu(), cu=cu.cpu().numpy(), dst=dst.cpu().numpy(), src=src.cpu().numpy(),
                qp=qp.cpu(), kp=kp.cpu(), vp=vp.cpu(), err=err)


def check_indices(got, ref):
    T = int(ref["cu"][-1])
    assert np.array_equal(got["cu"], ref["cu"]), "cu_seqlens differ"
    assert np.array_equal(got["dst"], ref["dst"]), "dst_idx differ"
    assert np.array_equal(got["src"][:T], ref["src"]), "src_idx differ"


def check_indices_and_packing(got, ref):
    check_indices(got, ref)
    T = int(ref["cu"][-1])
    for name, g, r in zip(("q", "k", "v"), (got["qp"], got["kp"], got["vp"]), ref["packed_bits"]):
        assert np.array_equal(bits(g)[:T], r), f"packed {name} differs"


def run_pack(case):
    """rra_pack alone (row copy + indices + zero fill); CPU copies of its outputs."""
    keep, q, k, v = to_device(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    cu = torch.full((B + 1,), -9, dtype=torch.int32, device="cuda")
    dst = torch.full((B * N,), -9, dtype=torch.int32, device="cuda")
    src = torch.full((B * N,), -9, dtype=torch.int32, device="cuda")
    qp, kp, vp = (torch.full((B * N, H, d), float("nan"), dtype=case.dtype, device="cuda") for _ in range(3))
    out = torch.full((B, N, H, d), float("nan"), dtype=case.dtype, device="cuda")
    rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp, out_zero_fill=out)
    torch.cuda.synchronize()
    return dict(cu=cu.cpu().numpy(), dst=dst.cpu().numpy(), src=src.cpu().numpy(), qp=qp.cpu(), kp=kp.cpu(),
                vp=vp.cpu(), out=out.cpu())


def check_output(out: torch.Tensor, keep: np.ndarray, ref_out: np.ndarray):
    """Pruned positions +0 bit-exact; kept positions within tolerance. Returns max-abs error."""
    m = keep != 0
    ob = bits(out)
    assert np.all(ob[~m] == 0), "pruned positions are not +0"
    got = out.double().numpy()
    err = np.abs(got[m] - ref_out[m])
    tol = out_tolerance(ref_out[m], out.dtype)
    assert np.all(np.isfinite(got[m])), "non-finite output at a kept position"
    bad = err > tol
    assert not bad.any(), f"max-abs err {err.max():.3e} over tolerance at {int(bad.sum())} elements"
    return float(err.max()) if err.size else 0.0


def packed_inputs(case):
    """Oracle result plus device packed Q/K/V (rows past T poisoned with NaN) and cu_seqlens."""
    ref = oracle_result(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    cap = B * N
    qp, kp, vp = (torch.empty((cap, H, d), dtype=case.dtype, device="cuda") for _ in range(3))
    for t, r in zip((qp, kp, vp), ref["packed_bits"]):
        t.view(torch.uint8).fill_(0xFF)
        t[: len(ref["src"])].view(torch.int16).copy_(torch.from_numpy(r))
    cu = torch.from_numpy(ref["cu"]).to("cuda")
    return ref, qp, kp, vp, cu
