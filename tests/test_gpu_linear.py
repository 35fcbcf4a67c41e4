"""rra_linear_packed (tcgen05 GEMM over the packed rows) against the oracle (needs a GPU).

Rows t < T = cu_seqlens[B] within 1e-3 of the fp64 product (fp32
accumulation over K <= 768 of N(0,1) x N(0,1/K) terms), plus half an output
ulp when stored as bf16/fp16; rows t >= T untouched; a cu_seqlens[B] past
the buffer is reported and nothing is written.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from ragged_attention_token_gb300 import rra

pytestmark = pytest.mark.gpu

ATOL = 1e-3


def _inputs(cap, K, N, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((cap, K), generator=g).to(dtype)
    w = (torch.randn((N, K), generator=g) / np.sqrt(K)).to(dtype)
    bias = torch.randn((N,), generator=g)
    return a, w, bias


def _cu(T, B=2):
    cut = T // 3
    return torch.tensor([0, cut, T][: B + 1] if B == 2 else [0, T], dtype=torch.int32)


@pytest.mark.parametrize("K,N", [(384, 1152), (768, 2304), (384, 384), (64, 128)])
@pytest.mark.parametrize("T", [1, 127, 128, 129, 500])
def test_linear_packed_matches_oracle(K, N, T):
    cap = 512
    a, w, bias = _inputs(cap, K, N, seed=K * 7 + N + T)
    c = torch.full((cap, N), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.linear_packed(a.cuda(), w.cuda(), _cu(T).cuda(), 2, c, bias=bias.cuda())
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got = c.cpu().double().numpy()
    ref = oracle.linear_packed(a.double().numpy(), w.double().numpy(), bias.double().numpy(), T)
    err = float(np.abs(got[:T] - ref).max())
    assert err <= ATOL, f"max-abs error {err}"
    assert np.all(np.isnan(got[T:])), "rows past T were written"


@pytest.mark.parametrize("dtype,out", [(torch.bfloat16, torch.bfloat16), (torch.float16, torch.float16),
                                       (torch.float16, torch.float32)])
def test_linear_packed_dtypes_and_no_bias(dtype, out):
    cap, K, N, T = 300, 384, 384, 257
    a, w, _ = _inputs(cap, K, N, seed=5, dtype=dtype)
    c = torch.zeros((cap, N), dtype=out, device="cuda")
    rra.linear_packed(a.cuda(), w.cuda(), _cu(T, B=1).cuda(), 1, c)
    torch.cuda.synchronize()
    ref = oracle.linear_packed(a.double().numpy(), w.double().numpy(), None, T)
    got = c.cpu().double().numpy()
    if out == torch.float32:
        tol = np.full(ref.shape, ATOL)
    else:
        explicit = 7 if out == torch.bfloat16 else 10
        e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -60)))
        tol = ATOL + 2.0 ** (e - explicit - 1)
    assert np.all(np.abs(got[:T] - ref) <= tol)
    assert np.all(got[T:] == 0)


def test_linear_packed_empty_and_bad_count():
    cap, K, N = 256, 64, 128
    a, w, bias = _inputs(cap, K, N, seed=3)
    c = torch.full((cap, N), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.linear_packed(a.cuda(), w.cuda(), torch.tensor([0, 0], dtype=torch.int32, device="cuda"), 1, c)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0 and bool(torch.isnan(c).all())     # T = 0: nothing written
    rra.linear_packed(a.cuda(), w.cuda(), torch.tensor([0, cap + 1], dtype=torch.int32, device="cuda"), 1, c)
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_INDEX_RANGE
    assert bool(torch.isnan(c).all())


@pytest.mark.parametrize("K,N", [(768, 2304), (384, 1152)])
@pytest.mark.parametrize("T", [2569, 12608])
def test_linear_packed_full_size(K, N, T):
    """The sizes the benchmark times: cap = 12608 rows (B=64 x N=197), T kept rows
    at 80% pruning (2569) and dense (12608); several waves of output tiles."""
    cap = 12608
    a, w, bias = _inputs(cap, K, N, seed=K + N + T)
    c = torch.full((cap, N), float("nan"), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    rra.linear_packed(a.cuda(), w.cuda(), torch.tensor([0, T], dtype=torch.int32).cuda(), 1, c, bias=bias.cuda())
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    got = c.cpu().double().numpy()
    ref = oracle.linear_packed(a.double().numpy(), w.double().numpy(), bias.double().numpy(), T)
    err = float(np.abs(got[:T] - ref).max())
    assert err <= ATOL, f"max-abs error {err}"
    assert np.all(np.isnan(got[T:])), "rows past T were written"
