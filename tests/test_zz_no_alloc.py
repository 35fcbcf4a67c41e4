"""rra_pipeline_static: the pipeline for callers that cannot allocate.

Some callers may not call cudaMalloc at all: a plugin running inside a host
that owns every byte of device memory, code running inside someone else's
capture region, or a real-time loop that cannot pay for an allocation's
implicit synchronisation.  They cannot hand rra_pipeline a workspace, so
the library keeps one static device array for them.  This test calls that
entry point through the C ABI and checks it against rra_pipeline (which
uses a caller workspace) on the same inputs, twice in a row, so the second
call also runs on scratch that still holds the first call's contents.

The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import SCALE, bits, pair_tolerance
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _call(L, keep, q, k, v, out):
    B, N, H, d = q.shape
    return L.rra_pipeline_static(keep.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), B, N, H, d,
                                 ctypes.c_float(SCALE), rra.dtype_code(q.dtype), out.data_ptr(),
                                 rra.dtype_code(out.dtype), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("make", [lambda: W.make_serving(4), lambda: W.make_batched(0.8),
                                  lambda: W.make_tiny()], ids=["serving_B4", "batched_p80", "tiny"])
def test_static_scratch_matches_workspace_pipeline(make):
    L = rra.lib()
    case = make()
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    for out_dtype in (case.dtype, torch.float32):
        ref, _ = rra.run_pipeline(keep, q, k, v, scale=SCALE, out_dtype=out_dtype)
        for _ in range(2):                      # two calls in a row share the scratch
            out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
            assert _call(L, keep, q, k, v, out) == rra.RRA_OK
            torch.cuda.synchronize()
            assert rra.get_device_error() == 0
            m = case.keep.numpy() != 0
            got, want = out.cpu(), ref.cpu()
            assert np.all(bits(got)[~m] == 0)
            g, w = got.double().numpy(), want.double().numpy()
            assert np.all(np.abs(g - w) <= pair_tolerance(w, out_dtype)), float(np.abs(g - w).max())


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
