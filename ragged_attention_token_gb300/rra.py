"""ctypes binding of librra (include/rra.h), with the same names.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (torch provides device memory and
streams); sizes and dtypes are read from them and passed as plain integers.
Loading fails loudly when librra.so is missing -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "librra.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG_DIR), "include", "rra.h")

RRA_OK, RRA_ERR_INVALID_ARG, RRA_ERR_UNSUPPORTED, RRA_ERR_MISALIGNED, RRA_ERR_CUDA, RRA_ERR_DEVICE = range(6)
RRA_F16, RRA_BF16, RRA_F32 = 0, 1, 2
ATTEND_TCGEN05, ATTEND_MMA_SYNC, ATTEND_AUTO, ATTEND_TCGEN05_LATENCY = 0, 1, 2, 3
DEVERR_NONE, DEVERR_SEQ_TOO_LONG, DEVERR_SEQ_NEGATIVE, DEVERR_INDEX_RANGE, DEVERR_WAIT_TIMEOUT = range(5)

_DTYPE = {torch.float16: RRA_F16, torch.bfloat16: RRA_BF16, torch.float32: RRA_F32}

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
_dp = ctypes.POINTER(ctypes.c_double)

_SIGNATURES = {
    "rra_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "rra_workspace_offsets": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(_sz)]),
    "rra_pack": (_i, [_vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp]),
    "rra_attend": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i, _vp]),
    "rra_repack": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rra_cls_scores": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "rra_linear_packed": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "rra_topk_keep": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "rra_attend_gather": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "rra_pack_index": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "rra_attend_rows": (_i, [_vp, _vp, _vp, ctypes.c_longlong, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i,
                             _vp]),
    "rra_attend_cls": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i, _vp]),
    "rra_topk_keep_cls": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp]),
    "rra_prune_index": (_i, [_vp, _i, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rra_unpack": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "rra_pipeline": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp]),
    "rra_pipeline_static": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "rra_pipeline_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i,
                               _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "rra_pipeline_mapped": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz, _vp]),
    "rra_plan_create": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _sz,
                             ctypes.POINTER(_vp)]),
    "rra_plan_launch": (_i, [_vp, _vp]),
    "rra_plan_destroy": (None, [_vp]),
    "rra_get_device_error": (_i, [ctypes.POINTER(ctypes.c_int32), _i]),
    "rra_time_attend_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i, _vp,
                                  _i, _i, _dp]),
    "rra_time_attend_wait_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i, _vp,
                                       _i, _i, _dp]),
    "rra_attend_wait": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _i, _vp, _i, _vp]),
    "rra_time_plan_host": (_i, [_vp, _vp, _i, _i, _dp]),
    "rra_time_null_host": (_i, [_vp, _i, _i, _dp]),
    "rra_set_attend_kernel": (_i, [_i]),
    "rra_bind_error_word": (_i, [_vp]),
    "rra_read_error_word": (_i, [_vp, ctypes.POINTER(ctypes.c_int32), _i]),
    "rra_set_wait_limit": (ctypes.c_longlong, [ctypes.c_longlong]),
    "rra_status_string": (ctypes.c_char_p, [_i]),
    "rra_last_error_message": (ctypes.c_char_p, []),
    "rra_launch_count": (ctypes.c_uint64, []),
}

_LIB = None


class RRAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def header_symbols(path: str = HEADER_PATH) -> list[str]:
    """Every function the C header declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"RRA_API\s+[\w\s\*]*?\b(rra_\w+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """Load librra.so once (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m ragged_attention_token_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int) -> None:
    if status != RRA_OK:
        L = lib()
        raise RRAError(status, f"{L.rra_status_string(status).decode()}: "
                               f"{L.rra_last_error_message().decode()}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def dtype_code(dt: torch.dtype) -> int:
    return _DTYPE[dt]


def workspace_bytes(B: int, N: int, H: int, d: int, dtype: torch.dtype) -> int:
    return int(lib().rra_workspace_bytes(B, N, H, d, _DTYPE[dtype]))


def workspace_offsets(B: int, N: int, H: int, d: int, dtype: torch.dtype) -> list[int]:
    arr = (_sz * 6)()
    _check(lib().rra_workspace_offsets(B, N, H, d, _DTYPE[dtype], arr))
    return list(arr)


def workspace_views(ws: torch.Tensor, B: int, N: int, H: int, d: int, dtype: torch.dtype):
    """(cu_seqlens, dst_idx, src_idx, qp, kp, vp) views into a pipeline workspace."""
    off = workspace_offsets(B, N, H, d, dtype)
    es = torch.empty((), dtype=dtype).element_size()
    cap = B * N
    cu = ws[off[0]:off[0] + 4 * (B + 1)].view(torch.int32)
    dst = ws[off[1]:off[1] + 4 * cap].view(torch.int32)
    src = ws[off[2]:off[2] + 4 * cap].view(torch.int32)
    packed = [ws[o:o + cap * H * d * es].view(dtype).view(cap, H, d) for o in off[3:6]]
    return (cu, dst, src, *packed)


def pack(keep, q, k, v, cu_seqlens, dst_idx, src_idx, qp=None, kp=None, vp=None, out_zero_fill=None,
         stream=None):
    """rra_pack; with qp = kp = vp = None only the indices and the zero fill are produced."""
    B, N, H, d = q.shape
    out_dt = _DTYPE[out_zero_fill.dtype] if out_zero_fill is not None else RRA_F32
    _check(lib().rra_pack(_ptr(keep), B, N, H, d, _DTYPE[q.dtype], _ptr(q), _ptr(k), _ptr(v),
                          _ptr(cu_seqlens), _ptr(dst_idx), _ptr(src_idx), _ptr(qp), _ptr(kp), _ptr(vp),
                          _ptr(out_zero_fill), out_dt, _stream(stream)))


def repack(keep_new, dst_prev, qp_prev, kp_prev, vp_prev, cu_seqlens, dst_idx, src_idx, qp, kp, vp, stream=None):
    """rra_repack: the next layer's packed rows from the previous layer's packed rows."""
    B, N = keep_new.shape
    H, d = qp_prev.shape[-2], qp_prev.shape[-1]
    _check(lib().rra_repack(_ptr(keep_new), _ptr(dst_prev), B, N, H, d, _DTYPE[qp_prev.dtype], _ptr(qp_prev),
                            _ptr(kp_prev), _ptr(vp_prev), _ptr(cu_seqlens), _ptr(dst_idx), _ptr(src_idx),
                            _ptr(qp), _ptr(kp), _ptr(vp), _stream(stream)))


def linear_packed(a, w, cu_seqlens, B: int, c, bias=None, stream=None):
    """rra_linear_packed: c[t] = a[t] @ w.T (+ bias) for the T = cu_seqlens[B] packed rows."""
    cap, K = a.shape
    N = w.shape[0]
    if bias is not None and bias.dtype != torch.float32:
        raise ValueError("bias must be float32")
    _check(lib().rra_linear_packed(_ptr(a), _ptr(w), _ptr(bias), _ptr(cu_seqlens), B, cap, K, N, _DTYPE[a.dtype],
                                   _ptr(c), _DTYPE[c.dtype], _stream(stream)))


def cls_scores(qp, kp, cu_seqlens, src_idx, B: int, N: int, scores, scale: float = 0.125, stream=None):
    """rra_cls_scores: the class token's attention over each image's kept tokens, head mean, [B, N] fp32."""
    H, d = qp.shape[-2], qp.shape[-1]
    if scores.dtype != torch.float32:
        raise ValueError("scores must be float32")
    _check(lib().rra_cls_scores(_ptr(qp), _ptr(kp), _ptr(cu_seqlens), _ptr(src_idx), B, N, H, d, float(scale),
                                _DTYPE[qp.dtype], _ptr(scores), _stream(stream)))


def topk_keep(scores, keep_prev, keep_num: int, keep_den: int, keep_new, stream=None):
    """rra_topk_keep: the class token plus the top ceil(m*num/den) other kept tokens by score."""
    B, N = keep_prev.shape
    _check(lib().rra_topk_keep(_ptr(scores), _ptr(keep_prev), B, N, int(keep_num), int(keep_den), _ptr(keep_new),
                               _stream(stream)))


def attend(qp, kp, vp, cu_seqlens, B: int, max_seqlen: int, o, scale: float = 0.125,
           src_idx=None, N: int = 0, stream=None):
    H, d = qp.shape[-2], qp.shape[-1]
    _check(lib().rra_attend(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(cu_seqlens), B, max_seqlen, H, d,
                            float(scale), _DTYPE[qp.dtype], _ptr(o), _DTYPE[o.dtype], _ptr(src_idx), N,
                            _stream(stream)))


def attend_wait(qp, kp, vp, cu_seqlens, B: int, max_seqlen: int, o, scale: float = 0.125,
                src_idx=None, N: int = 0, stream=None):
    """rra_attend_wait: rra_attend, returning once `o` is complete (polls a host completion word)."""
    H, d = qp.shape[-2], qp.shape[-1]
    _check(lib().rra_attend_wait(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(cu_seqlens), B, max_seqlen, H, d,
                                 float(scale), _DTYPE[qp.dtype], _ptr(o), _DTYPE[o.dtype], _ptr(src_idx), N,
                                 _stream(stream)))


def attend_gather(q, k, v, cu_seqlens, src_idx, out, scale: float = 0.125, stream=None):
    """rra_attend_gather: attention reading rows src_idx of padded q/k/v, writing padded out."""
    B, N, H, d = q.shape
    _check(lib().rra_attend_gather(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(src_idx), B, N, H, d,
                                   float(scale), _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], _stream(stream)))


def pack_index(keep, cu_seqlens, dst_idx, src_idx, rows=None, dst_prev=None, stream=None):
    """rra_pack_index: cu_seqlens/dst_idx/src_idx of `keep` and (optionally) the input row of each packed row."""
    B, N = keep.shape
    _check(lib().rra_pack_index(_ptr(keep), _ptr(dst_prev), B, N, _ptr(cu_seqlens), _ptr(dst_idx), _ptr(src_idx),
                                _ptr(rows), _stream(stream)))


def attend_rows(q, k, v, rows, cu_seqlens, B: int, max_seqlen: int, o, scale: float = 0.125, cls=None,
                stream=None):
    """rra_attend_rows: packed attention whose row t is read from row rows[t] of q/k/v [src_rows, H, d];
    `cls` ([B, H, stride] float32) receives the class-token side output when given."""
    H, d = q.shape[-2], q.shape[-1]
    src_rows = q.numel() // (H * d)
    stride = cls.shape[-1] if cls is not None else 0
    _check(lib().rra_attend_rows(_ptr(q), _ptr(k), _ptr(v), src_rows, _ptr(rows), _ptr(cu_seqlens), B, max_seqlen,
                                 H, d, float(scale), _DTYPE[q.dtype], _ptr(o), _DTYPE[o.dtype], _ptr(cls), stride,
                                 _stream(stream)))


def attend_cls(qp, kp, vp, cu_seqlens, B: int, max_seqlen: int, o, cls, scale: float = 0.125, stream=None):
    """rra_attend_cls: packed attention plus the class-token weights cls [B, H, stride] (float32)."""
    H, d = qp.shape[-2], qp.shape[-1]
    _check(lib().rra_attend_cls(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(cu_seqlens), B, max_seqlen, H, d, float(scale),
                                _DTYPE[qp.dtype], _ptr(o), _DTYPE[o.dtype], _ptr(cls), cls.shape[-1],
                                _stream(stream)))


def topk_keep_cls(cls, cu_seqlens, src_idx, N: int, keep_num: int, keep_den: int, keep_new, scores=None,
                  stream=None):
    """rra_topk_keep_cls: the keep decision [B, N] from the class-token side output cls [B, H, stride]."""
    B, H, stride = cls.shape
    _check(lib().rra_topk_keep_cls(_ptr(cls), stride, _ptr(cu_seqlens), _ptr(src_idx), B, N, H, keep_num, keep_den,
                                   _ptr(keep_new), _ptr(scores), _stream(stream)))


def prune_index(cls, cu_prev, src_prev, N: int, keep_num: int, keep_den: int, cu_seqlens, dst_idx, src_idx, rows,
                keep_new=None, scores=None, stream=None):
    """rra_prune_index: the keep decision from cls [B, H, stride] and the next layer's indices in one launch."""
    B, H, stride = cls.shape
    _check(lib().rra_prune_index(_ptr(cls), stride, _ptr(cu_prev), _ptr(src_prev), B, N, H, keep_num, keep_den,
                                 _ptr(cu_seqlens), _ptr(dst_idx), _ptr(src_idx), _ptr(rows), _ptr(keep_new),
                                 _ptr(scores), _stream(stream)))


def unpack(op, dst_idx, B: int, N: int, out, stream=None):
    H, d = op.shape[-2], op.shape[-1]
    _check(lib().rra_unpack(_ptr(op), _ptr(dst_idx), B, N, H, d, _DTYPE[op.dtype], _ptr(out),
                            _stream(stream)))


def pipeline(keep, q, k, v, out, workspace, scale: float = 0.125, stream=None):
    B, N, H, d = q.shape
    _check(lib().rra_pipeline(_ptr(keep), _ptr(q), _ptr(k), _ptr(v), B, N, H, d, float(scale),
                              _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], _ptr(workspace),
                              _nbytes(workspace), _stream(stream)))


def pipeline_static(keep, q, k, v, out, scale: float = 0.125, stream=None):
    """rra_pipeline_static: the pipeline with the library's static scratch (no workspace)."""
    B, N, H, d = q.shape
    _check(lib().rra_pipeline_static(_ptr(keep), _ptr(q), _ptr(k), _ptr(v), B, N, H, d, float(scale),
                                     _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], _stream(stream)))


def pipeline_host(keep_h, q_h, k_h, v_h, out_h, keep_d, q_d, k_d, v_d, out_d, workspace,
                  scale: float = 0.125, stream=None):
    """Host-buffer pipeline: H2D copies, pipeline, D2H copy, all enqueued on `stream`."""
    for t in (keep_h, q_h, k_h, v_h, out_h):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors (pinned for async copies)")
    B, N, H, d = q_h.shape
    _check(lib().rra_pipeline_host(keep_h.data_ptr(), q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                                   B, N, H, d, float(scale), _DTYPE[q_h.dtype], out_h.data_ptr(),
                                   _DTYPE[out_h.dtype], _ptr(keep_d), _ptr(q_d), _ptr(k_d), _ptr(v_d),
                                   _ptr(out_d), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def pipeline_mapped(keep_h, q_h, k_h, v_h, out_h, workspace, scale: float = 0.125, stream=None):
    """rra_pipeline_mapped: the kernels read the kept rows from, and write the output into, pinned host memory."""
    for t in (keep_h, q_h, k_h, v_h, out_h):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors in pinned memory")
    B, N, H, d = q_h.shape
    _check(lib().rra_pipeline_mapped(keep_h.data_ptr(), q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                                     B, N, H, d, float(scale), _DTYPE[q_h.dtype], out_h.data_ptr(),
                                     _DTYPE[out_h.dtype], _ptr(workspace), _nbytes(workspace),
                                     _stream(stream)))


class Plan:
    """A CUDA graph of one pipeline call on fixed buffers (rra_plan_*)."""

    def __init__(self, keep, q, k, v, out, workspace, scale: float = 0.125):
        B, N, H, d = q.shape
        self._h = _vp()
        self._keepalive = (keep, q, k, v, out, workspace)
        _check(lib().rra_plan_create(_ptr(keep), _ptr(q), _ptr(k), _ptr(v), B, N, H, d, float(scale),
                                     _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], _ptr(workspace),
                                     _nbytes(workspace), ctypes.byref(self._h)))

    def launch(self, stream=None):
        _check(lib().rra_plan_launch(self._h, _stream(stream)))

    def time_host(self, warmup: int, reps: int, stream=None) -> list[float]:
        buf = (ctypes.c_double * reps)()
        _check(lib().rra_time_plan_host(self._h, _stream(stream), warmup, reps, buf))
        return list(buf)

    def close(self):
        if self._h:
            lib().rra_plan_destroy(self._h)
            self._h = _vp()
            self._keepalive = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def get_device_error(clear: bool = True) -> int:
    code = ctypes.c_int32(0)
    st = lib().rra_get_device_error(ctypes.byref(code), 1 if clear else 0)
    if st not in (RRA_OK, RRA_ERR_DEVICE):
        _check(st)
    return int(code.value)


def bind_error_word(word=None) -> None:
    """rra_bind_error_word: this thread's launches record device errors into `word`
    (an int32 CUDA tensor of one element), or into the device's own word (None)."""
    if word is not None and (word.dtype != torch.int32 or word.numel() < 1):
        raise ValueError("expected an int32 CUDA tensor")
    _check(lib().rra_bind_error_word(_ptr(word)))


def read_error_word(word, clear: bool = True) -> int:
    """rra_read_error_word: the code in a bound error word (0: none), zeroed if clear."""
    code = ctypes.c_int32(0)
    st = lib().rra_read_error_word(_ptr(word), ctypes.byref(code), 1 if clear else 0)
    if st not in (RRA_OK, RRA_ERR_DEVICE):
        _check(st)
    return int(code.value)


def set_wait_limit(cycles: int) -> int:
    """rra_set_wait_limit: bound (clock cycles) on one on-chip wait; 0 = default. Returns the previous."""
    return int(lib().rra_set_wait_limit(int(cycles)))


def time_attend_host(qp, kp, vp, cu_seqlens, B: int, max_seqlen: int, o, warmup: int, reps: int,
                     scale: float = 0.125, src_idx=None, N: int = 0, stream=None) -> list[float]:
    H, d = qp.shape[-2], qp.shape[-1]
    buf = (ctypes.c_double * reps)()
    _check(lib().rra_time_attend_host(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(cu_seqlens), B, max_seqlen, H, d,
                                      float(scale), _DTYPE[qp.dtype], _ptr(o), _DTYPE[o.dtype],
                                      _ptr(src_idx), N, _stream(stream), warmup, reps, buf))
    return list(buf)


def time_attend_wait_host(qp, kp, vp, cu_seqlens, B: int, max_seqlen: int, o, warmup: int, reps: int,
                          scale: float = 0.125, src_idx=None, N: int = 0, stream=None) -> list[float]:
    """Host-timed µs of rra_attend_wait calls (each returns with its output complete)."""
    H, d = qp.shape[-2], qp.shape[-1]
    buf = (ctypes.c_double * reps)()
    _check(lib().rra_time_attend_wait_host(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(cu_seqlens), B, max_seqlen, H, d,
                                           float(scale), _DTYPE[qp.dtype], _ptr(o), _DTYPE[o.dtype],
                                           _ptr(src_idx), N, _stream(stream), warmup, reps, buf))
    return list(buf)


def time_null_host(warmup: int, reps: int, stream=None) -> list[float]:
    """Host-timed {empty kernel launch + sync}: the platform's dispatch floor."""
    buf = (ctypes.c_double * reps)()
    _check(lib().rra_time_null_host(_stream(stream), warmup, reps, buf))
    return list(buf)


def set_attend_kernel(kernel: int) -> int:
    """Select the attention kernel (ATTEND_TCGEN05, ATTEND_MMA_SYNC, ATTEND_TCGEN05_LATENCY or ATTEND_AUTO); returns the previous one."""
    prev = int(lib().rra_set_attend_kernel(int(kernel)))
    if prev < 0:
        raise ValueError(f"unknown attention kernel {kernel}")
    return prev


def launch_count() -> int:
    return int(lib().rra_launch_count())


# ------------------------------------------------------------- conveniences

def alloc_workspace(B: int, N: int, H: int, d: int, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    n = workspace_bytes(B, N, H, d, dtype)
    if n == 0:
        raise RRAError(RRA_ERR_INVALID_ARG, "unsupported sizes for a workspace")
    return torch.empty(n, dtype=torch.uint8, device=device)


def run_pipeline(keep, q, k, v, scale: float = 0.125, out_dtype=None, stream=None):
    """Allocate output + workspace with torch and run rra_pipeline once."""
    B, N, H, d = q.shape
    out = torch.empty((B, N, H, d), dtype=out_dtype or q.dtype, device=q.device)
    ws = alloc_workspace(B, N, H, d, q.dtype, q.device)
    pipeline(keep, q, k, v, out, ws, scale=scale, stream=stream)
    return out, ws
