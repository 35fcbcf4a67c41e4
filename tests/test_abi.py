"""The C-ABI library loads and exports every symbol include/rra.h declares.

CPU only: the calls below fail host-side argument checks before any CUDA
call is made, so no GPU is needed.
"""
import ctypes
import subprocess

import pytest

from ragged_attention_token_gb300 import build, rra


@pytest.fixture(scope="module")
def L():
    if not build.up_to_date():
        build.build()
    return rra.lib()


def test_header_declares_the_boundary():
    syms = rra.header_symbols()
    for name in ("rra_pack", "rra_attend", "rra_unpack", "rra_pipeline", "rra_plan_create",
                 "rra_plan_launch", "rra_plan_destroy", "rra_workspace_bytes", "rra_get_device_error"):
        assert name in syms
    assert set(syms) == set(rra._SIGNATURES), "binding and header disagree"


def test_every_declared_symbol_is_exported(L):
    for name in rra.header_symbols():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", rra.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(rra.header_symbols()), exported ^ set(rra.header_symbols())


def test_workspace_layout(L):
    B, N, H, d = 3, 197, 6, 64
    n = L.rra_workspace_bytes(B, N, H, d, rra.RRA_BF16)
    off = (ctypes.c_size_t * 6)()
    assert L.rra_workspace_offsets(B, N, H, d, rra.RRA_BF16, off) == rra.RRA_OK
    off = list(off)
    assert off[0] == 0 and all(o % 256 == 0 for o in off)
    assert off[1] >= (B + 1) * 4 and off[2] - off[1] >= B * N * 4 and off[3] - off[2] >= B * N * 4
    packed = B * N * H * d * 2
    assert off[4] - off[3] >= packed and off[5] - off[4] >= packed and n - off[5] >= packed
    assert L.rra_workspace_bytes(B, N, H, 32, rra.RRA_BF16) == 0
    assert L.rra_workspace_bytes(B, 2000, H, d, rra.RRA_BF16) == 0
    assert L.rra_workspace_bytes(B, N, H, d, rra.RRA_F32) == 0     # fp32 inputs unsupported


def _attend(L, **kw):
    a = dict(qp=0x1000, kp=0x2000, vp=0x3000, cu=0x4000, B=2, S=197, H=6, d=64, scale=0.125,
             ind=rra.RRA_BF16, o=0x5000, outd=rra.RRA_BF16, src=None, N=197, stream=None)
    a.update(kw)
    return L.rra_attend(a["qp"], a["kp"], a["vp"], a["cu"], a["B"], a["S"], a["H"], a["d"], a["scale"],
                        a["ind"], a["o"], a["outd"], a["src"], a["N"], a["stream"])


def test_host_side_errors(L):
    assert _attend(L, d=32) == rra.RRA_ERR_UNSUPPORTED
    assert _attend(L, S=1025) == rra.RRA_ERR_UNSUPPORTED
    assert _attend(L, B=0) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, H=0) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, qp=None) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, cu=None) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, kp=0x2008) == rra.RRA_ERR_MISALIGNED
    assert _attend(L, o=0x5004) == rra.RRA_ERR_MISALIGNED
    assert b"not 16-byte aligned" in L.rra_last_error_message()
    assert _attend(L, ind=rra.RRA_F32) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, outd=7) == rra.RRA_ERR_INVALID_ARG
    assert _attend(L, scale=float("nan")) == rra.RRA_ERR_INVALID_ARG
    st = L.rra_pipeline(0x100, 0x1000, 0x2000, 0x3000, 2, 197, 6, 64, 0.125, rra.RRA_BF16, 0x5000,
                        rra.RRA_BF16, 0x6000, 16, None)
    assert st == rra.RRA_ERR_INVALID_ARG and b"workspace" in L.rra_last_error_message()
    st = L.rra_pack(None, 2, 197, 6, 64, rra.RRA_BF16, 0x1000, 0x2000, 0x3000, 0x100, 0x200, 0x300,
                    0x1000, 0x2000, 0x3000, None, rra.RRA_BF16, None)
    assert st == rra.RRA_ERR_INVALID_ARG
    st = L.rra_unpack(0x1000, 0x100, 2, 197, 6, 64, rra.RRA_BF16, 0x1001, None)
    assert st == rra.RRA_ERR_MISALIGNED
    plan = ctypes.c_void_p()
    st = L.rra_plan_create(0x100, 0x1000, 0x2000, 0x3000, 2, 197, 6, 48, 0.125, rra.RRA_BF16, 0x5000,
                           rra.RRA_BF16, 0x6000, 1 << 30, ctypes.byref(plan))
    assert st == rra.RRA_ERR_UNSUPPORTED and not plan.value
    assert L.rra_plan_launch(None, None) == rra.RRA_ERR_INVALID_ARG
    L.rra_plan_destroy(None)
    buf = (ctypes.c_double * 1)()
    assert L.rra_time_null_host(None, 0, 0, buf) == rra.RRA_ERR_INVALID_ARG


def test_status_strings(L):
    for s, name in enumerate(["RRA_OK", "RRA_ERR_INVALID_ARG", "RRA_ERR_UNSUPPORTED", "RRA_ERR_MISALIGNED",
                              "RRA_ERR_CUDA", "RRA_ERR_DEVICE"]):
        assert L.rra_status_string(s).decode() == name


def test_host_side_errors_of_the_later_entry_points(L):
    # rra_repack: shape, null, alignment and overlap checks, all before any CUDA call.
    def repack(**kw):
        a = dict(keep=0x100, dst=0x200, B=2, N=197, H=6, d=64, dt=rra.RRA_BF16, qp=0x10000, kp=0x20000,
                 vp=0x30000, cu=0x300, di=0x400, si=0x500, q2=0x1000000, k2=0x2000000, v2=0x3000000)
        a.update(kw)
        return L.rra_repack(a["keep"], a["dst"], a["B"], a["N"], a["H"], a["d"], a["dt"], a["qp"], a["kp"],
                            a["vp"], a["cu"], a["di"], a["si"], a["q2"], a["k2"], a["v2"], None)
    assert repack(d=32) == rra.RRA_ERR_UNSUPPORTED
    assert repack(keep=None) == rra.RRA_ERR_INVALID_ARG
    assert repack(dst=None) == rra.RRA_ERR_INVALID_ARG
    assert repack(si=None) == rra.RRA_ERR_INVALID_ARG
    assert repack(kp=0x20008) == rra.RRA_ERR_MISALIGNED
    assert repack(dt=rra.RRA_F32) == rra.RRA_ERR_INVALID_ARG
    assert repack(q2=0x10000 + 256) == rra.RRA_ERR_INVALID_ARG            # new rows overlap the previous ones
    assert b"overlap" in L.rra_last_error_message()
    # rra_attend_wait takes rra_attend's checks first.
    def wait(**kw):
        a = dict(qp=0x1000, kp=0x2000, vp=0x3000, cu=0x4000, B=2, S=197, H=6, d=64, scale=0.125,
                 ind=rra.RRA_BF16, o=0x5000, outd=rra.RRA_BF16)
        a.update(kw)
        return L.rra_attend_wait(a["qp"], a["kp"], a["vp"], a["cu"], a["B"], a["S"], a["H"], a["d"], a["scale"],
                                 a["ind"], a["o"], a["outd"], None, 0, None)
    assert wait(d=32) == rra.RRA_ERR_UNSUPPORTED
    assert wait(qp=None) == rra.RRA_ERR_INVALID_ARG
    assert wait(o=0x5004) == rra.RRA_ERR_MISALIGNED
    assert wait(scale=float("inf")) == rra.RRA_ERR_INVALID_ARG
    buf = (ctypes.c_double * 1)()
    assert L.rra_time_attend_wait_host(0x1000, 0x2000, 0x3000, 0x4000, 2, 197, 6, 64, 0.125, rra.RRA_BF16,
                                       0x5000, rra.RRA_BF16, None, 0, None, 0, 0, buf) == rra.RRA_ERR_INVALID_ARG
    # rra_pipeline_mapped: a null host buffer is refused by name.
    st = L.rra_pipeline_mapped(None, 0x1000, 0x2000, 0x3000, 2, 197, 6, 64, 0.125, rra.RRA_BF16, 0x5000,
                               rra.RRA_BF16, 0x6000, 1 << 30, None)
    assert st == rra.RRA_ERR_INVALID_ARG and b"keep_h" in L.rra_last_error_message()


def test_host_side_errors_of_the_next_step_entry_points(L):
    # rra_cls_scores / rra_topk_keep
    st = L.rra_cls_scores(0x1000, 0x2000, 0x300, 0x400, 2, 197, 6, 32, 0.125, rra.RRA_BF16, 0x5000, None)
    assert st == rra.RRA_ERR_UNSUPPORTED
    st = L.rra_cls_scores(0x1000, 0x2000, None, 0x400, 2, 197, 6, 64, 0.125, rra.RRA_BF16, 0x5000, None)
    assert st == rra.RRA_ERR_INVALID_ARG
    st = L.rra_cls_scores(0x1008, 0x2000, 0x300, 0x400, 2, 197, 6, 64, 0.125, rra.RRA_BF16, 0x5000, None)
    assert st == rra.RRA_ERR_MISALIGNED
    assert L.rra_topk_keep(0x1000, 0x2000, 2, 197, 8, 7, 0x9000, None) == rra.RRA_ERR_INVALID_ARG   # num > den
    assert L.rra_topk_keep(0x1000, 0x2000, 2, 197, 1, 0, 0x9000, None) == rra.RRA_ERR_INVALID_ARG   # den = 0
    assert L.rra_topk_keep(0x1000, 0x2000, 2, 197, 7, 10, 0x2010, None) == rra.RRA_ERR_INVALID_ARG  # overlap
    assert b"overlap" in L.rra_last_error_message()
    assert L.rra_topk_keep(None, 0x2000, 2, 197, 7, 10, 0x9000, None) == rra.RRA_ERR_INVALID_ARG
    # rra_linear_packed: K a multiple of 64, N a multiple of 128, alignment, null counts.
    def lin(**kw):
        a = dict(a=0x10000, w=0x20000, bias=None, cu=0x300, B=1, cap=512, K=384, N=1152,
                 ind=rra.RRA_BF16, c=0x40000, outd=rra.RRA_F32)
        a.update(kw)
        return L.rra_linear_packed(a["a"], a["w"], a["bias"], a["cu"], a["B"], a["cap"], a["K"], a["N"],
                                   a["ind"], a["c"], a["outd"], None)
    assert lin(K=96) == rra.RRA_ERR_UNSUPPORTED
    assert lin(N=192) == rra.RRA_ERR_UNSUPPORTED
    assert lin(cu=None) == rra.RRA_ERR_INVALID_ARG
    assert lin(cap=0) == rra.RRA_ERR_INVALID_ARG
    assert lin(a=0x10008) == rra.RRA_ERR_MISALIGNED
    assert lin(bias=0x50004) == rra.RRA_ERR_MISALIGNED
    assert lin(ind=rra.RRA_F32) == rra.RRA_ERR_INVALID_ARG


def test_host_side_errors_of_the_chain_and_pruning_entry_points(L):
    # rra_pack_index: shape, nulls, aliasing of the previous and new dst.
    assert L.rra_pack_index(None, None, 2, 197, 0x300, 0x400, 0x500, None, None) == rra.RRA_ERR_INVALID_ARG
    assert L.rra_pack_index(0x100, None, 2, 197, None, 0x400, 0x500, None, None) == rra.RRA_ERR_INVALID_ARG
    assert L.rra_pack_index(0x100, None, 0, 197, 0x300, 0x400, 0x500, None, None) == rra.RRA_ERR_INVALID_ARG
    assert L.rra_pack_index(0x100, None, 2, 1025, 0x300, 0x400, 0x500, None, None) == rra.RRA_ERR_UNSUPPORTED
    assert L.rra_pack_index(0x100, 0x400, 2, 197, 0x300, 0x400, 0x500, 0x600, None) == rra.RRA_ERR_INVALID_ARG

    # rra_attend_rows: rra_attend's checks, then rows, src_rows and the side output's.
    def rows(**kw):
        a = dict(q=0x10000, k=0x20000, v=0x30000, src_rows=394, rows=0x600, cu=0x300, B=2, S=197, H=6, d=64,
                 scale=0.125, ind=rra.RRA_BF16, o=0x40000, outd=rra.RRA_BF16, cls=None, stride=0)
        a.update(kw)
        return L.rra_attend_rows(a["q"], a["k"], a["v"], a["src_rows"], a["rows"], a["cu"], a["B"], a["S"],
                                 a["H"], a["d"], a["scale"], a["ind"], a["o"], a["outd"], a["cls"], a["stride"],
                                 None)
    assert rows(d=32) == rra.RRA_ERR_UNSUPPORTED
    assert rows(rows=None) == rra.RRA_ERR_INVALID_ARG
    assert rows(src_rows=0) == rra.RRA_ERR_INVALID_ARG
    assert rows(q=0x10008) == rra.RRA_ERR_MISALIGNED
    assert rows(cls=0x50000, stride=210) == rra.RRA_ERR_INVALID_ARG          # not a multiple of 4
    assert rows(cls=0x50000, stride=204) == rra.RRA_ERR_INVALID_ARG          # below max_seqlen rounded up to 16
    assert rows(cls=0x50004, stride=208) == rra.RRA_ERR_MISALIGNED
    assert rows(cls=0x50000, stride=208, outd=rra.RRA_F32) == rra.RRA_ERR_UNSUPPORTED

    # rra_attend_cls: the side output is required.
    def cls(**kw):
        a = dict(qp=0x10000, kp=0x20000, vp=0x30000, cu=0x300, B=2, S=197, H=6, d=64, scale=0.125,
                 ind=rra.RRA_BF16, o=0x40000, outd=rra.RRA_BF16, cls=0x50000, stride=208)
        a.update(kw)
        return L.rra_attend_cls(a["qp"], a["kp"], a["vp"], a["cu"], a["B"], a["S"], a["H"], a["d"], a["scale"],
                                a["ind"], a["o"], a["outd"], a["cls"], a["stride"], None)
    assert cls(cls=None) == rra.RRA_ERR_INVALID_ARG
    assert cls(outd=rra.RRA_F16) == rra.RRA_ERR_UNSUPPORTED
    assert cls(stride=192) == rra.RRA_ERR_INVALID_ARG
    assert cls(cu=None) == rra.RRA_ERR_INVALID_ARG

    # rra_topk_keep_cls / rra_prune_index: fraction, stride, nulls, aliasing.
    assert L.rra_topk_keep_cls(0x50000, 208, 0x300, 0x400, 2, 197, 6, 8, 7, 0x9000, None, None) == \
        rra.RRA_ERR_INVALID_ARG                                             # num > den
    assert L.rra_topk_keep_cls(0x50000, 100, 0x300, 0x400, 2, 197, 6, 7, 10, 0x9000, None, None) == \
        rra.RRA_ERR_INVALID_ARG                                             # stride < N
    assert L.rra_topk_keep_cls(0x50000, 208, None, 0x400, 2, 197, 6, 7, 10, 0x9000, None, None) == \
        rra.RRA_ERR_INVALID_ARG

    def prune(**kw):
        a = dict(cls=0x50000, stride=208, cu_prev=0x300, src_prev=0x400, B=2, N=197, H=6, num=7, den=10,
                 cu=0x700, dst=0x800, src=0x900, rows=0xa00)
        a.update(kw)
        return L.rra_prune_index(a["cls"], a["stride"], a["cu_prev"], a["src_prev"], a["B"], a["N"], a["H"],
                                 a["num"], a["den"], a["cu"], a["dst"], a["src"], a["rows"], None, None, None)
    assert prune(rows=None) == rra.RRA_ERR_INVALID_ARG
    assert prune(cu=0x300) == rra.RRA_ERR_INVALID_ARG                     # new indices alias the previous
    assert b"alias" in L.rra_last_error_message()
    assert prune(den=0) == rra.RRA_ERR_INVALID_ARG
    assert prune(stride=150) == rra.RRA_ERR_INVALID_ARG
    assert prune(N=2000) == rra.RRA_ERR_UNSUPPORTED
