"""rra_pipeline_static: the pipeline for callers that cannot allocate.

Some callers may not call cudaMalloc at all: a plugin running inside a host
that owns every byte of device memory, code running inside someone else's
capture region, or a real-time loop that cannot pay for an allocation's
implicit synchronisation.  They cannot hand rra_pipeline a workspace, so
the library keeps one static device array for them.  These tests call that
entry point through the C ABI and check it against the CPU oracle (and
against rra_pipeline, which uses a caller workspace) on the same inputs:
twice in a row on one workload, and a large workload followed at once by a
small one, so that later calls run on scratch still holding an earlier
call's contents.  They also check which workloads fit in the array.

The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import SCALE, bits, check_output, oracle_result, pair_tolerance
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _call(L, keep, q, k, v, out):
    B, N, H, d = q.shape
    return L.rra_pipeline_static(keep.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), B, N, H, d,
                                 ctypes.c_float(SCALE), rra.dtype_code(q.dtype), out.data_ptr(),
                                 rra.dtype_code(out.dtype), torch.cuda.current_stream().cuda_stream)


def _run_static(L, case, out_dtype):
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    assert _call(L, keep, q, k, v, out) == rra.RRA_OK
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    return out.cpu()


@pytest.mark.parametrize("make", [lambda: W.make_serving(4), lambda: W.make_batched(0.8),
                                  lambda: W.make_tiny()], ids=["serving_B4", "batched_p80", "tiny"])
def test_static_scratch_matches_oracle_and_workspace_pipeline(make):
    L = rra.lib()
    case = make()
    ref = oracle_result(case)
    keep_np = case.keep.numpy()
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    for out_dtype in (case.dtype, torch.float32):
        want, _ = rra.run_pipeline(keep, q, k, v, scale=SCALE, out_dtype=out_dtype)
        want = want.cpu()
        for _ in range(2):                      # two calls in a row share the scratch
            got = _run_static(L, case, out_dtype)
            check_output(got, keep_np, ref["out"])          # against the oracle
            g, w = got.double().numpy(), want.double().numpy()
            assert np.all(np.abs(g - w) <= pair_tolerance(w, out_dtype)), float(np.abs(g - w).max())


def test_static_scratch_large_then_small_call():
    """A call right after a larger one reads only what it wrote itself."""
    L = rra.lib()
    big, small = W.make_batched(0.8), W.make_tiny()
    _run_static(L, big, big.dtype)
    for out_dtype in (small.dtype, torch.float32):
        got = _run_static(L, small, out_dtype)
        check_output(got, small.keep.numpy(), oracle_result(small)["out"])
        _run_static(L, big, torch.float32)


@pytest.mark.parametrize("name,B,N,H,fits", [
    ("tiny", 2, 197, 3, True), ("serving_B4", 4, 197, 6, True), ("batched_B64", 64, 197, 12, True),
    ("hires_B32", 32, 577, 12, False), ("progressive_B256", 256, 197, 6, False)])
def test_static_scratch_fit_per_workload(name, B, N, H, fits):
    assert (rra.workspace_bytes(B, N, H, 64, torch.bfloat16) <= 64 * 1024 * 1024) == fits


def test_static_scratch_rejects_sizes_over_its_maximum():
    L = rra.lib()
    B, N, H = 256, 197, 12
    assert rra.workspace_bytes(B, N, H, 64, torch.bfloat16) > 64 * 1024 * 1024
    x = torch.empty((16,), dtype=torch.bfloat16, device="cuda")       # never touched
    keep = torch.empty((16,), dtype=torch.uint8, device="cuda")
    st = L.rra_pipeline_static(keep.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), B, N, H, 64,
                               ctypes.c_float(SCALE), rra.RRA_BF16, x.data_ptr(), rra.RRA_BF16, None)
    assert st == rra.RRA_ERR_UNSUPPORTED
    assert b"64 MiB" in L.rra_last_error_message()
