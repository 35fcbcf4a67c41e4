"""rra_pipeline_mapped (inputs and output in pinned host memory, no copies)
against the CPU oracle (needs a GPU).

The kernels read the keep mask and the kept Q/K/V rows over the CPU-GPU
link and write the padded output into host memory.  Bit-exact: cu_seqlens,
pack indices and packed Q/K/V in the device workspace, and the +0 rows at
pruned positions.  Attention outputs: the same bound as the device-resident
pipeline (max-abs 2e-3 plus half an output ulp for a bf16/fp16 store).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import SCALE, check_indices_and_packing, check_output, oracle_result
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KERNELS = [("tcgen05", rra.ATTEND_TCGEN05), ("tcgen05_latency", rra.ATTEND_TCGEN05_LATENCY),
           ("mma_sync", rra.ATTEND_MMA_SYNC), ("auto", rra.ATTEND_AUTO)]

CASES = [
    ("tiny", lambda: W.make_tiny()),
    ("serving_B1", lambda: W.make_serving(1)),
    ("serving_B4", lambda: W.make_serving(4)),
    ("batched_p80", lambda: W.make_batched(0.8)),
    ("hires_p90", lambda: W.make_hires(0.9)),
]


@pytest.fixture(params=KERNELS, ids=[k[0] for k in KERNELS])
def kernel(request):
    prev = rra.set_attend_kernel(request.param[1])
    yield request.param[0]
    rra.set_attend_kernel(prev)


def _pinned(case, out_dtype=None):
    keep_h, q_h, k_h, v_h = (x.contiguous().pin_memory() for x in (case.keep, case.q, case.k, case.v))
    out_h = torch.empty(case.q.shape, dtype=out_dtype or case.dtype).pin_memory()
    out_h.view(torch.uint8).fill_(0xFF)          # NaN everywhere: unwritten rows show up
    return keep_h, q_h, k_h, v_h, out_h


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_mapped_pipeline_matches_oracle(name, make, kernel):
    case = make()
    B, N, H, d = case.B, case.N, case.H, case.d
    keep_h, q_h, k_h, v_h, out_h = _pinned(case)
    ws = rra.alloc_workspace(B, N, H, d, case.dtype)
    ws.fill_(0xFF)
    rra.get_device_error(clear=True)
    rra.pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, ws, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    ref = oracle_result(case)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one_launch = kernel != "mma_sync" and B * H * ((N + 127) // 128) <= sms
    if not one_launch:
        # pack + attend: the workspace holds the indices and the packed rows
        cu, dst, src, qp, kp, vp = rra.workspace_views(ws, B, N, H, d, case.dtype)
        got = dict(cu=cu.cpu().numpy(), dst=dst.cpu().numpy(), src=src.cpu().numpy(), qp=qp.cpu(), kp=kp.cpu(),
                   vp=vp.cpu())
        check_indices_and_packing(got, ref)
    else:
        # the one-launch kernel (serving sizes) scans the mask itself and leaves the workspace alone
        assert bool((ws == 0xFF).all())
    check_output(out_h, case.keep.numpy(), ref["out"])


def test_mapped_pipeline_fp32_output_and_repeat(kernel):
    case = W.make_serving(2)
    keep_h, q_h, k_h, v_h, out_h = _pinned(case, torch.float32)
    ws = rra.alloc_workspace(case.B, case.N, case.H, case.d, case.dtype)
    rra.pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, ws, scale=SCALE)
    torch.cuda.synchronize()
    first = out_h.clone()
    err = check_output(first, case.keep.numpy(), oracle_result(case)["out"])
    assert err <= 2e-3
    out_h.view(torch.uint8).fill_(0xFF)
    rra.pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, ws, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int32), first.view(torch.int32))


@pytest.mark.parametrize("kid", [rra.ATTEND_MMA_SYNC, rra.ATTEND_TCGEN05], ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("make", [lambda: W.make_serving(4), lambda: W.make_batched(0.5)], ids=["serving_B4",
                                                                                            "batched_p50"])
def test_mapped_pipeline_matches_device_pipeline_bitwise(kid, make):
    # The same arithmetic on the same bits: host-resident buffers change
    # where the bytes live (and, for the one-launch kernel, cp.async copies
    # replace the TMA gathers), not one result bit.  The device-resident
    # reference runs the kernel the mapped path takes: the fused tcgen05
    # kernel at serving sizes, else pack + the mma.sync attention.
    case = make()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    one_launch = kid != rra.ATTEND_MMA_SYNC and case.B * case.H * ((case.N + 127) // 128) <= sms
    prev = rra.set_attend_kernel(rra.ATTEND_TCGEN05 if one_launch else rra.ATTEND_MMA_SYNC)
    try:
        keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
        direct, _ = rra.run_pipeline(keep, q, k, v, scale=SCALE)
        rra.set_attend_kernel(kid)
        keep_h, q_h, k_h, v_h, out_h = _pinned(case)
        ws = rra.alloc_workspace(case.B, case.N, case.H, case.d, case.dtype)
        rra.pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, ws, scale=SCALE)
        torch.cuda.synchronize()
        assert torch.equal(out_h.view(torch.int16), direct.cpu().view(torch.int16))
    finally:
        rra.set_attend_kernel(prev)


def test_mapped_pipeline_rejects_unmapped_buffers():
    case = W.make_tiny()
    B, N, H, d = case.B, case.N, case.H, case.d
    keep_h, q_h, k_h, v_h, out_h = _pinned(case)
    ws = rra.alloc_workspace(B, N, H, d, case.dtype)
    n0 = rra.launch_count()
    pageable = case.q.clone()                                  # ordinary (pageable) host memory
    with pytest.raises(rra.RRAError) as e:
        rra.pipeline_mapped(keep_h, pageable, k_h, v_h, out_h, ws, scale=SCALE)
    assert e.value.status == rra.RRA_ERR_INVALID_ARG and "q_h" in str(e.value)
    ws_host = torch.empty(ws.numel(), dtype=ws.dtype).pin_memory()
    with pytest.raises(rra.RRAError) as e:
        rra._check(rra.lib().rra_pipeline_mapped(keep_h.data_ptr(), q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                                                 B, N, H, d, SCALE, rra.dtype_code(case.dtype), out_h.data_ptr(),
                                                 rra.dtype_code(case.dtype), ws_host.data_ptr(),
                                                 ws_host.numel() * ws_host.element_size(), None))
    assert e.value.status == rra.RRA_ERR_INVALID_ARG and "workspace" in str(e.value)
    q_dev = case.q.cuda()                                      # device memory is not host memory
    with pytest.raises(rra.RRAError) as e:
        rra._check(rra.lib().rra_pipeline_mapped(keep_h.data_ptr(), q_dev.data_ptr(), k_h.data_ptr(),
                                                 v_h.data_ptr(), B, N, H, d, SCALE, rra.dtype_code(case.dtype),
                                                 out_h.data_ptr(), rra.dtype_code(case.dtype), ws.data_ptr(),
                                                 ws.numel() * ws.element_size(), None))
    assert e.value.status == rra.RRA_ERR_INVALID_ARG
    assert rra.launch_count() == n0                            # nothing was enqueued
    assert np.all(out_h.view(torch.uint8).numpy() == 0xFF)
