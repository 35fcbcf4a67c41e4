"""Device-side error reporting (needs a GPU).

Per-call error words: launches enqueued by a thread that bound its own
device word (rra_bind_error_word) record into that word only, so two calls
on two streams, one of them with inconsistent cu_seqlens, report separately;
a plan records into the word bound when it was created.  The bounded-wait
failure path: with rra_set_wait_limit set to a few hundred cycles the
tcgen05 kernel's first waits give up, the launch records
RRA_DEVERR_WAIT_TIMEOUT and returns, and the next normal call is correct.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_util import ATOL, SCALE, check_output, oracle_result, packed_inputs
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

KERNELS = [("tcgen05", rra.ATTEND_TCGEN05), ("mma_sync", rra.ATTEND_MMA_SYNC),
           ("tcgen05_latency", rra.ATTEND_TCGEN05_LATENCY)]


@pytest.fixture(params=KERNELS, ids=[k[0] for k in KERNELS])
def kernel(request):
    prev = rra.set_attend_kernel(request.param[1])
    yield request.param[0]
    rra.set_attend_kernel(prev)


def _word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_error_words_are_per_call(kernel):
    case = W.make_serving(4)
    ref, qp, kp, vp, cu = packed_inputs(case)
    B, N = case.B, case.N
    T = len(ref["src"])
    bad = cu.clone()
    bad[2] = bad[1] - 1                       # image 1 gets a negative length
    wa, wb = _word(), _word()
    oa = torch.zeros_like(qp, dtype=torch.float32)
    ob = torch.full_like(qp, float("nan"), dtype=torch.float32)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    rra.get_device_error(clear=True)
    torch.cuda.synchronize()
    try:
        rra.bind_error_word(wa)
        rra.attend(qp, kp, vp, bad, B, N, oa, scale=SCALE, stream=s1)
        rra.bind_error_word(wb)
        rra.attend(qp, kp, vp, cu, B, N, ob, scale=SCALE, stream=s2)
    finally:
        rra.bind_error_word(None)
    torch.cuda.synchronize()
    assert rra.read_error_word(wa) == rra.DEVERR_SEQ_NEGATIVE
    assert rra.read_error_word(wb) == 0
    assert rra.get_device_error() == 0            # the device's own word saw nothing
    err = float(np.abs(ob[:T].cpu().double().numpy() - ref["o"]).max())
    assert err <= ATOL, err


def test_bound_word_rejects_misaligned_pointer():
    w = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert rra.lib().rra_bind_error_word(w.data_ptr() + 2) == rra.RRA_ERR_MISALIGNED
    rra.bind_error_word(None)


def _serving_launch(path, case):
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    B, N, H, d = case.B, case.N, case.H, case.d
    out = torch.full((B, N, H, d), float("nan"), dtype=torch.float32, device="cuda")
    if path == "pipeline":
        ws = rra.alloc_workspace(B, N, H, d, case.dtype)
        return out, lambda: rra.pipeline(keep, q, k, v, out, ws, scale=SCALE)
    ref, qp, kp, vp, cu = packed_inputs(case)
    src = torch.from_numpy(np.asarray(ref["src"], dtype=np.int32)).cuda()
    out.zero_()
    return out, lambda: rra.attend(qp, kp, vp, cu, B, N, out, scale=SCALE, src_idx=src, N=N)


@pytest.mark.parametrize("tc", [rra.ATTEND_TCGEN05, rra.ATTEND_TCGEN05_LATENCY], ids=["tcgen05", "tcgen05_latency"])
@pytest.mark.parametrize("path", ["attend", "pipeline"])
def test_wait_timeout_is_recorded_and_the_next_call_is_correct(path, tc):
    prev = rra.set_attend_kernel(tc)
    try:
        case = W.make_serving(1)
        ref = oracle_result(case)
        out, launch = _serving_launch(path, case)
        rra.get_device_error(clear=True)
        old = rra.set_wait_limit(300)
        try:
            launch()
            torch.cuda.synchronize()
        finally:
            rra.set_wait_limit(old)
        assert rra.get_device_error(clear=True) == rra.DEVERR_WAIT_TIMEOUT
        out2, launch2 = _serving_launch(path, case)
        launch2()
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        check_output(out2.cpu(), case.keep.numpy(), ref["out"])
    finally:
        rra.set_attend_kernel(prev)


@pytest.mark.parametrize("tc", [rra.ATTEND_TCGEN05, rra.ATTEND_TCGEN05_LATENCY], ids=["tcgen05", "tcgen05_latency"])
def test_plan_records_into_the_word_bound_at_creation(tc):
    prev = rra.set_attend_kernel(tc)
    case = W.make_serving(2)
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    B, N, H, d = case.B, case.N, case.H, case.d
    out = torch.empty((B, N, H, d), dtype=case.dtype, device="cuda")
    ws = rra.alloc_workspace(B, N, H, d, case.dtype)
    wc = _word()
    rra.get_device_error(clear=True)
    try:
        rra.bind_error_word(wc)
        old = rra.set_wait_limit(300)           # the plan's launches give up at once
        try:
            plan = rra.Plan(keep, q, k, v, out, ws, scale=SCALE)
        finally:
            rra.set_wait_limit(old)
            rra.bind_error_word(None)
        torch.cuda.synchronize()
        assert rra.read_error_word(wc) == rra.DEVERR_WAIT_TIMEOUT   # the warm-up run
        plan.launch()
        torch.cuda.synchronize()
        assert rra.read_error_word(wc) == rra.DEVERR_WAIT_TIMEOUT   # the captured graph
        assert rra.get_device_error() == 0
        plan.close()
        good = rra.Plan(keep, q, k, v, out, ws, scale=SCALE)
        good.launch()
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        check_output(out.cpu(), case.keep.numpy(), oracle_result(case)["out"])
        good.close()
    finally:
        rra.set_attend_kernel(prev)
