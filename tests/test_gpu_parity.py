"""CUDA path vs the CPU oracle on the same seeded inputs (needs a GPU).

Bit-exact: cu_seqlens, dst_idx, src_idx, packed Q/K/V, pruned output rows
(+0), a one-token image's output (= its V), unpack, NaN-poisoned pruned rows,
repeat runs and batch permutations.  Attention outputs: max-abs <= 2e-3 in
fp32-output mode, plus half an output ulp when stored as bf16/fp16.
Every workload runs at its full size in the pipeline's own launch
configuration; the oracle is cheap enough to compute every output.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (ATOL, SCALE, bits, check_indices, check_indices_and_packing, check_output, oracle_result,
                      packed_inputs, run_pack, run_pipeline)
from ragged_attention_token_gb300 import rra
from ragged_attention_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu

_PROGRESSIVE_MASKS = None


def _progressive(layer):
    global _PROGRESSIVE_MASKS
    if _PROGRESSIVE_MASKS is None:
        _PROGRESSIVE_MASKS = W.progressive_masks()
    return W.make_progressive_layer(layer, _PROGRESSIVE_MASKS)


CASES = (
    [("tiny", lambda: W.make_tiny())]
    + [(f"serving_B{B}", (lambda B=B: W.make_serving(B))) for B in W.SERVING_BATCHES]
    + [(f"batched_p{int(p * 100)}", (lambda p=p: W.make_batched(p))) for p in W.BATCHED_RATES]
    + [(f"hires_p{int(p * 100)}", (lambda p=p: W.make_hires(p))) for p in W.HIRES_RATES]
    + [(f"progressive_L{L}", (lambda L=L: _progressive(L))) for L in range(1, 13)]
)


KERNELS = [("tcgen05", rra.ATTEND_TCGEN05), ("mma_sync", rra.ATTEND_MMA_SYNC),
           ("tcgen05_latency", rra.ATTEND_TCGEN05_LATENCY)]
DEFAULT_KERNEL = rra.ATTEND_AUTO


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    rra.lib()
    rra.get_device_error(clear=True)
    yield
    rra.set_attend_kernel(DEFAULT_KERNEL)


@pytest.fixture(params=KERNELS, ids=[k[0] for k in KERNELS])
def kernel(request):
    prev = rra.set_attend_kernel(request.param[1])
    yield request.param[0]
    rra.set_attend_kernel(prev)


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_pipeline_full_size(name, make, kernel):
    case = make()
    ref = oracle_result(case)
    keep = case.keep.numpy()
    for out_dtype in (case.dtype, torch.float32):
        got = run_pipeline(case, out_dtype)
        assert got["err"] == 0
        err = check_output(got["out"], keep, ref["out"])
        if out_dtype == torch.float32:
            assert err <= ATOL
        print(f"{kernel} {name} out={out_dtype} max_abs_err={err:.3e}")


def _edge_cases():
    C = W.make_custom
    return [
        ("B1_one_token", lambda: C(1, 197, 6, [1])),
        ("empty_images", lambda: C(3, 197, 6, [0, 5, 0])),
        ("all_empty", lambda: C(2, 50, 3, [0, 0])),
        ("N1", lambda: C(3, 1, 4, [1, 0, 1])),
        ("N63_all", lambda: C(2, 63, 3, [63, 63])),
        ("N64_all", lambda: C(2, 64, 3, [64, 64])),
        ("N65_all", lambda: C(2, 65, 3, [65, 65])),
        ("N127_mixed", lambda: C(3, 127, 2, [127, 64, 1])),
        ("N128_all", lambda: C(1, 128, 2, [128])),
        ("N129_mixed", lambda: C(2, 129, 2, [129, 65])),
        ("N1024_max", lambda: C(2, 1024, 2, [1024, 777])),
        ("no_cls_random", lambda: C(5, 197, 3, [20, 197, 0, 100, 1], cls=False)),
        ("bernoulli_half", lambda: C(7, 300, 3, None, random_mask=True)),
        ("large_logits_x8", lambda: C(4, 197, 6, [197, 100, 39, 2], value_scale=8.0)),
        ("fp16_ragged", lambda: C(4, 197, 3, [197, 60, 7, 1], dtype=torch.float16)),
        ("fp16_large_logits", lambda: C(2, 577, 2, [577, 300], dtype=torch.float16, value_scale=4.0)),
        ("H1", lambda: C(9, 97, 1, [97, 1, 2, 3, 50, 0, 64, 65, 96])),
    ]


EDGE = _edge_cases()


@pytest.mark.parametrize("name,make", EDGE, ids=[e[0] for e in EDGE])
def test_pipeline_edge_cases(name, make, kernel):
    case = make()
    ref = oracle_result(case)
    keep = case.keep.numpy()
    for out_dtype in (case.dtype, torch.float32):
        got = run_pipeline(case, out_dtype)
        assert got["err"] == 0
        check_output(got["out"], keep, ref["out"])


def test_single_token_returns_v_bit_exact(kernel):
    case = W.make_custom(4, 197, 6, [1, 1, 1, 1])
    got = run_pipeline(case)
    m = case.keep.numpy() != 0
    assert np.array_equal(bits(got["out"])[m], bits(case.v)[m])
    got32 = run_pipeline(case, torch.float32)
    assert np.array_equal(got32["out"].numpy()[m], case.v.float().numpy()[m])


def test_nan_in_pruned_rows_changes_nothing(kernel):
    case = W.make_batched(0.8)
    clean = run_pipeline(case)
    pruned = (case.keep == 0)[:, :, None, None]
    for x in (case.q, case.k, case.v):
        x.masked_fill_(pruned, float("nan"))
    dirty = run_pipeline(case)
    assert np.array_equal(bits(clean["out"]), bits(dirty["out"]))


def test_repeat_runs_and_batch_permutation_bit_exact(kernel):
    case = W.make_batched(0.5)
    a = run_pipeline(case)
    b = run_pipeline(case)
    diff = bits(a["out"]) != bits(b["out"])
    assert not diff.any(), (
        f"{int(diff.sum())} elements in {int(diff.any(axis=3).sum())} rows differ between two runs, "
        f"max |diff| {float((a['out'].double() - b['out'].double()).abs().max())}, "
        f"first rows (b, n, h): {np.argwhere(diff.any(axis=3))[:8].tolist()}")
    perm = torch.randperm(case.B, generator=torch.Generator().manual_seed(5))
    case2 = W.Case(case.name + "_perm", case.B, case.N, case.H, case.d, case.dtype, case.keep[perm].clone(),
                   case.q[perm].clone(), case.k[perm].clone(), case.v[perm].clone(), case.seed)
    c = run_pipeline(case2)
    assert np.array_equal(bits(a["out"])[perm.numpy()], bits(c["out"]))


def _packed_inputs(case):
    return packed_inputs(case)


@pytest.mark.parametrize("make", [lambda: W.make_tiny(), lambda: W.make_hires(0.5)], ids=["tiny", "hires_p50"])
def test_attend_packed_output_and_unpack(make, kernel):
    case = make()
    ref, qp, kp, vp, cu = _packed_inputs(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    T = len(ref["src"])
    o = torch.full((B * N, H, d), float("nan"), dtype=torch.float32, device="cuda")
    rra.attend(qp, kp, vp, cu, B, N, o, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    err = np.abs(o[:T].cpu().double().numpy() - ref["o"]).max()
    assert err <= ATOL
    assert torch.isnan(o[T:]).all()                       # rows >= T untouched
    # unpack is a bit copy of the packed rows plus +0 at pruned positions
    ob = o.to(case.dtype)
    dst = torch.from_numpy(ref["dst"]).to("cuda")
    out = torch.full((B, N, H, d), float("nan"), dtype=case.dtype, device="cuda")
    rra.unpack(ob, dst, B, N, out)
    torch.cuda.synchronize()
    assert rra.get_device_error() == 0
    want = oracle.unpack(bits(ob), ref["dst"], B, N)
    assert np.array_equal(bits(out), want)


def test_pack_standalone_leaves_rows_beyond_T():
    case = W.make_serving(2)
    ref = oracle_result(case)
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    B, N, H, d = case.B, case.N, case.H, case.d
    cu = torch.empty(B + 1, dtype=torch.int32, device="cuda")
    dst = torch.empty(B * N, dtype=torch.int32, device="cuda")
    src = torch.full((B * N,), -7, dtype=torch.int32, device="cuda")
    qp, kp, vp = (torch.empty((B * N, H, d), dtype=case.dtype, device="cuda") for _ in range(3))
    rra.pack(keep, q, k, v, cu, dst, src, qp, kp, vp)
    torch.cuda.synchronize()
    T = len(ref["src"])
    assert np.array_equal(cu.cpu().numpy(), ref["cu"])
    assert np.array_equal(dst.cpu().numpy(), ref["dst"])
    assert np.array_equal(src.cpu().numpy()[:T], ref["src"])
    assert (src[T:] == -7).all()                          # beyond T untouched


def test_mask_values_any_nonzero_keeps():
    case = W.make_serving(4)
    ref = oracle_result(case)
    mult = torch.randint(1, 256, case.keep.shape, generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    case.keep = (case.keep.to(torch.int32) * mult).to(torch.uint8)
    assert ((case.keep != 0).numpy() == (ref["dst"].reshape(case.B, case.N) >= 0)).all()
    got = run_pipeline(case)
    check_output(got["out"], case.keep.numpy(), ref["out"])


@pytest.mark.parametrize("name,make", CASES + EDGE, ids=[c[0] for c in CASES + EDGE])
def test_pack_bit_exact(name, make):
    """rra_pack: indices, packed rows and the zero fill are bit copies of the oracle's."""
    case = make()
    ref = oracle_result(case)
    got = run_pack(case)
    check_indices_and_packing(got, ref)
    T = int(ref["cu"][-1])
    assert (torch.from_numpy(got["src"][T:]) == -9).all()          # rows >= T untouched
    m = case.keep.numpy() != 0
    assert np.all(bits(got["out"])[~m] == 0)                        # pruned rows +0
    assert np.all(np.isnan(got["out"].float().numpy()[m]))          # kept rows untouched


def test_device_error_codes(kernel):
    case = W.make_serving(2)
    ref, qp, kp, vp, cu = _packed_inputs(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    o = torch.zeros((B * N, H, d), dtype=torch.float32, device="cuda")
    rra.get_device_error(clear=True)
    n0 = int(ref["cu"][1])
    rra.attend(qp, kp, vp, cu, B, n0 - 1, o, scale=SCALE)      # max_seqlen below a real length
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_SEQ_TOO_LONG
    assert rra.get_device_error() == 0
    bad = torch.tensor([0, 10, 5], dtype=torch.int32, device="cuda")
    rra.attend(qp, kp, vp, bad, B, N, o, scale=SCALE)
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_SEQ_NEGATIVE
    src = torch.full((B * N,), B * N + 5, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, N, H, d), dtype=torch.float32, device="cuda")
    rra.attend(qp, kp, vp, cu, B, N, out, scale=SCALE, src_idx=src, N=N)
    torch.cuda.synchronize()
    assert rra.get_device_error(clear=True) == rra.DEVERR_INDEX_RANGE
    assert (out == 0).all()
    got = run_pipeline(case)                                    # a later good call reports nothing
    assert got["err"] == 0


def test_graph_plan_and_host_pipeline_match_direct():
    case = W.make_serving(4)
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    B, N, H, d = case.B, case.N, case.H, case.d
    direct, _ = rra.run_pipeline(keep, q, k, v, scale=SCALE)
    out = torch.empty_like(q)
    ws = rra.alloc_workspace(B, N, H, d, case.dtype)
    n0 = rra.launch_count()
    rra.pipeline(keep, q, k, v, out, ws, scale=SCALE)
    per_call = rra.launch_count() - n0
    assert per_call in (1, 2)
    plan = rra.Plan(keep, q, k, v, out, ws, scale=SCALE)
    out.zero_()
    n0 = rra.launch_count()
    plan.launch()
    plan.launch()
    torch.cuda.synchronize()
    assert rra.launch_count() - n0 == 2 * per_call
    assert torch.equal(out.view(torch.int16), direct.view(torch.int16))
    samples = plan.time_host(2, 5)
    assert all(s > 0 for s in samples)
    plan.close()
    keep_h, q_h, k_h, v_h = (x.pin_memory() for x in (case.keep, case.q, case.k, case.v))
    out_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    bufs = [torch.empty_like(x) for x in (keep, q, k, v)]
    out_d = torch.empty_like(q)
    rra.pipeline_host(keep_h, q_h, k_h, v_h, out_h, *bufs, out_d, ws, scale=SCALE)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), direct.cpu().view(torch.int16))


GRAPH_CASES = [("serving_B4", lambda: W.make_serving(4)), ("batched_p80", lambda: W.make_batched(0.8)),
               ("tiny", lambda: W.make_tiny()), ("hires_p90", lambda: W.make_hires(0.9))]


@pytest.mark.parametrize("name,make", GRAPH_CASES, ids=[c[0] for c in GRAPH_CASES])
def test_graph_plan_matches_oracle(name, make, kernel):
    """rra_plan_launch (the captured graph) against the oracle, over repeated replays
    on a poisoned output."""
    case = make()
    ref = oracle_result(case)
    keep_np = case.keep.numpy()
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    B, N, H, d = case.B, case.N, case.H, case.d
    for out_dtype in (case.dtype, torch.float32):
        out = torch.empty((B, N, H, d), dtype=out_dtype, device="cuda")
        ws = rra.alloc_workspace(B, N, H, d, case.dtype)
        plan = rra.Plan(keep, q, k, v, out, ws, scale=SCALE)
        try:
            for _ in range(2):
                out.view(torch.uint8).fill_(0xFF)
                plan.launch()
                torch.cuda.synchronize()
                assert rra.get_device_error() == 0
                check_output(out.cpu(), keep_np, ref["out"])
        finally:
            plan.close()


@pytest.mark.parametrize("make", [lambda: W.make_serving(1), lambda: W.make_serving(4),
                                  lambda: W.make_batched(0.8)], ids=["serving_B1", "serving_B4", "batched_p80"])
def test_attend_wait_matches_oracle(make, kernel):
    """rra_attend_wait's result, read right after it returns, against the oracle:
    packed fp32 output and the padded scatter."""
    case = make()
    ref, qp, kp, vp, cu = _packed_inputs(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    T = len(ref["src"])
    src = torch.from_numpy(ref["src"]).to("cuda")
    side = torch.cuda.Stream()
    o = torch.full((B * N, H, d), float("nan"), dtype=torch.float32, device="cuda")
    o_pad = torch.zeros((B, N, H, d), dtype=case.dtype, device="cuda")
    torch.cuda.synchronize()
    rra.attend_wait(qp, kp, vp, cu, B, N, o, scale=SCALE)
    with torch.cuda.stream(side):
        got = o[:T].clone()
    side.synchronize()
    err = float(np.abs(got.cpu().double().numpy() - ref["o"]).max())
    assert err <= ATOL, err
    rra.attend_wait(qp, kp, vp, cu, B, N, o_pad, scale=SCALE, src_idx=src, N=N)
    with torch.cuda.stream(side):
        got_pad = o_pad.clone()
    side.synchronize()
    check_output(got_pad.cpu(), case.keep.numpy(), ref["out"])


GATHER_CASES = GRAPH_CASES + [("no_cls_random", lambda: W.make_custom(5, 197, 3, [20, 197, 0, 100, 1], cls=False)),
                               ("N1024_max", lambda: W.make_custom(2, 1024, 2, [1024, 777]))]


@pytest.mark.parametrize("name,make", GATHER_CASES, ids=[c[0] for c in GATHER_CASES])
def test_attend_gather_matches_oracle(name, make):
    """rra_attend_gather (rows src_idx of the padded tensors in, padded output
    out) against the oracle; pruned positions are left as they were."""
    case = make()
    ref = oracle_result(case)
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    cu = torch.from_numpy(ref["cu"]).cuda()
    src = torch.from_numpy(np.asarray(ref["src"], dtype=np.int32)).cuda()
    for out_dtype in (case.dtype, torch.float32):
        out = torch.zeros(q.shape, dtype=out_dtype, device="cuda")
        rra.attend_gather(q, k, v, cu, src, out, scale=SCALE)
        torch.cuda.synchronize()
        assert rra.get_device_error() == 0
        check_output(out.cpu(), case.keep.numpy(), ref["out"])


def test_host_timed_helpers():
    case = W.make_serving(1)
    ref, qp, kp, vp, cu = _packed_inputs(case)
    o = torch.empty_like(qp)
    s = rra.time_attend_host(qp, kp, vp, cu, case.B, case.N, o, warmup=5, reps=20)
    assert len(s) == 20 and all(x > 0 for x in s)
    torch.cuda.synchronize()
    T = len(ref["src"])
    err = np.abs(o[:T].cpu().double().numpy() - ref["o"]).max()
    assert err <= ATOL + 2 ** -8
    z = rra.time_null_host(5, 20)
    assert len(z) == 20 and all(x > 0 for x in z)


@pytest.mark.parametrize("make", [lambda: W.make_serving(4), lambda: W.make_batched(0.8)], ids=["serving_B4",
                                                                                             "batched_p80"])
def test_attend_wait_returns_complete_output(make, kernel):
    # rra_attend_wait returns only once the output is complete: read it right
    # away (a copy on another stream, no sync in between) and compare with
    # rra_attend + sync, bit for bit, over repeated calls (fresh tickets).
    case = make()
    ref, qp, kp, vp, cu = _packed_inputs(case)
    B, N, H, d = case.B, case.N, case.H, case.d
    T = len(ref["src"])
    src = torch.from_numpy(ref["src"]).to("cuda")
    want_packed = torch.empty((B * N, H, d), dtype=torch.float32, device="cuda")
    rra.attend(qp, kp, vp, cu, B, N, want_packed, scale=SCALE)
    want_pad = torch.zeros((B, N, H, d), dtype=case.dtype, device="cuda")
    rra.attend(qp, kp, vp, cu, B, N, want_pad, scale=SCALE, src_idx=src, N=N)
    torch.cuda.synchronize()
    err = np.abs(want_packed[:T].cpu().double().numpy() - ref["o"]).max()
    assert err <= ATOL
    side = torch.cuda.Stream()
    n0 = rra.launch_count()
    for _ in range(3):
        o = torch.full((B * N, H, d), float("nan"), dtype=torch.float32, device="cuda")
        o_pad = torch.zeros((B, N, H, d), dtype=case.dtype, device="cuda")
        torch.cuda.synchronize()
        rra.attend_wait(qp, kp, vp, cu, B, N, o, scale=SCALE)
        with torch.cuda.stream(side):
            got = o[:T].clone()
        side.synchronize()
        assert torch.equal(got.view(torch.int32), want_packed[:T].view(torch.int32))
        rra.attend_wait(qp, kp, vp, cu, B, N, o_pad, scale=SCALE, src_idx=src, N=N)
        with torch.cuda.stream(side):
            got_pad = o_pad.clone()
        side.synchronize()
        assert torch.equal(got_pad.view(torch.int16), want_pad.view(torch.int16))
    assert rra.launch_count() - n0 == 6
    s = rra.time_attend_wait_host(qp, kp, vp, cu, B, N, o, warmup=3, reps=10)
    assert len(s) == 10 and all(x > 0 for x in s)


def test_attend_wait_device_count_form():
    # The same test in a fresh process with the device-word form of the
    # completion signal forced (the host-word form is the default where the
    # device has native atomics on host memory).
    import os
    import subprocess
    import sys
    env = dict(os.environ, RRA_WAIT_DEVICE_COUNT="1")
    here = os.path.dirname(os.path.abspath(__file__))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(here, "test_gpu_parity.py"), "-k", "attend_wait_returns_complete_output"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


def test_launch_count_counts_kernels(kernel):
    case = W.make_tiny()
    keep, q, k, v = (x.cuda() for x in (case.keep, case.q, case.k, case.v))
    n0 = rra.launch_count()
    rra.run_pipeline(keep, q, k, v)
    assert rra.launch_count() - n0 == (2 if kernel == "mma_sync" else 1)   # fused single launch vs pack + attend


def test_attend_kernel_selector():
    prev = rra.set_attend_kernel(rra.ATTEND_MMA_SYNC)
    assert prev == DEFAULT_KERNEL
    assert rra.set_attend_kernel(rra.ATTEND_AUTO) == rra.ATTEND_MMA_SYNC
    with pytest.raises(ValueError):
        rra.set_attend_kernel(7)
    rra.set_attend_kernel(prev)


@pytest.mark.parametrize("make", [lambda: W.make_serving(4), lambda: W.make_tiny(), lambda: W.make_batched(0.8),
                                  lambda: W.make_serving(32, seed=4321)],
                         ids=["serving", "tiny", "large", "serving_B32"])
def test_auto_kernel_matches_explicit(make):
    """AUTO with N <= 256: the pipeline runs the small-grid tcgen05 kernel
    while B*H*ceil(N/128) units are at most four per SM, rra_attend the
    mma.sync one while they are at most two per SM; beyond, the
    warp-specialised kernel -- bit for bit."""
    case = make()
    units = case.B * case.H * ((case.N + 127) // 128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    small_pipe = units <= 4 * sms and case.N <= 256
    small = units <= 2 * sms and case.N <= 256
    expect = rra.ATTEND_TCGEN05_LATENCY if small_pipe else rra.ATTEND_TCGEN05
    outs = {}
    for k in (rra.ATTEND_AUTO, expect):
        prev = rra.set_attend_kernel(k)
        outs[k] = run_pipeline(case)["out"]
        rra.set_attend_kernel(prev)
    a, b = outs.values()
    assert np.array_equal(bits(a), bits(b))
    check_output(a, case.keep.numpy(), oracle_result(case)["out"])
    ref, qp, kp, vp, cu = _packed_inputs(case)
    B, N = case.B, case.N
    res = {}
    for k in (rra.ATTEND_AUTO, rra.ATTEND_MMA_SYNC if small else rra.ATTEND_TCGEN05):
        prev = rra.set_attend_kernel(k)
        o = torch.zeros((B * N, case.H, case.d), dtype=torch.float32, device="cuda")
        rra.attend(qp, kp, vp, cu, B, N, o, scale=SCALE)
        torch.cuda.synchronize()
        res[k] = o.cpu()
        rra.set_attend_kernel(prev)
    a, b = res.values()
    assert torch.equal(a, b)


def test_fused_pipeline_leaves_workspace_alone():
    """The one-launch pipeline writes only `out`; the packed path fills the workspace."""
    case = W.make_batched(0.8)
    prev = rra.set_attend_kernel(rra.ATTEND_TCGEN05)
    try:
        got = run_pipeline(case)
        assert np.all(got["cu"] == -1) and np.all(got["src"] == -1)   # 0xFF poison untouched
    finally:
        rra.set_attend_kernel(prev)
    prev = rra.set_attend_kernel(rra.ATTEND_MMA_SYNC)
    try:
        got = run_pipeline(case)
        check_indices_and_packing(got, oracle_result(case))
    finally:
        rra.set_attend_kernel(prev)
