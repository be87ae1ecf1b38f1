"""GB300-native (sm_103a) MLA paged decode: a thin Python binding over the
C ABI in ``include/mla_decode.h``.

The three calls of one decode step of a Multi-head Latent Attention layer:

    o, lse = attend(q, kv, pages, indptr, scale, kv_scale, num_splits, split_tokens)
    latent, lse_merged = merge(o, lse)
    out = value_gate(latent, w_uv, gate, lengths, qlen)

This module only marshals arguments: it checks dtypes / shapes, allocates
outputs with torch (device memory), passes raw pointers and the current CUDA
stream to the native library, and turns error codes into exceptions.  Every
step of the computation runs in the library's CUDA kernels; there is no
fallback.  If the library has not been built (``build()``), every call
raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

D_QK, D_LATENT, D_V = 576, 512, 128
MLA_OK, MLA_ERR_INVALID, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA = 0, -1, -2, -3
ATTEND_CAUSAL, ATTEND_Q_FP8 = 1, 2
DEV_BAD_PAGE, DEV_BAD_INDPTR, DEV_TIMEOUT, DEV_BAD_PLAN = 1, 2, 4, 8
STATIC_SCRATCH_BYTES = 32 << 20   # MLA_STATIC_SCRATCH_BYTES: the partials buffer of decode_step_static

__all__ = ["Prepared", "attend", "merge", "value_gate", "merge_value_gate", "decode_step", "decode_step_static",
           "STATIC_SCRATCH_BYTES", "choose_splits", "plan_units", "debug_gather",
           "debug_wait_timeout", "debug_attend_mma",
           "kv_append", "device_status", "build", "library", "MlaError"]


class MlaError(RuntimeError):
    """A non-zero status from the native library."""

    def __init__(self, status: int, where: str, detail: str):
        super().__init__("%s failed: %s (%d)%s" % (where, _status_name(status), status,
                                                  ": " + detail if detail else ""))
        self.status = status


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (sm_103a) and return its path."""
    return _build.build(force=force, verbose=verbose)


def library() -> ctypes.CDLL:
    """The loaded native library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("mla_decode_paged_gb300: native library %s is missing; run "
                           "mla_decode_paged_gb300.build() first (no CPU fallback exists)" % path)
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.mla_decode_attend.argtypes = [vp, i64, vp, i64, vp, i64, vp, i32, i32, i32, f32, f32, i32, i32,
                                      vp, vp, vp]
    lib.mla_decode_attend_ex.argtypes = [vp, i64, vp, i64, vp, i64, vp, i32, i32, i32, f32, f32, i32, i32,
                                         vp, vp, ctypes.c_uint, vp]
    lib.mla_decode_attend_paged.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i32, i32, i32, i32, f32, f32,
                                            i32, i32, vp, vp, ctypes.c_uint, vp]
    lib.mla_decode_attend_planned.argtypes = [vp, i64, vp, i64, vp, i64, vp, vp, i32, i32, i32, i32, f32, f32,
                                              f32, i32, i32, vp, vp, ctypes.c_uint, vp, i64, vp]
    lib.mla_debug_attend_mma.argtypes = [vp, i64, vp, i64, vp, i64, vp, i32, i32, i32, f32, f32, i32, i32, vp, vp,
                                         vp]
    lib.mla_plan_units.argtypes = [i32, i32, i32, vp, i32, i32, vp, i64, ctypes.POINTER(ctypes.c_int)]
    lib.mla_plan_units.restype = i64
    lib.mla_plan_units_ex.argtypes = [i32, i32, i32, vp, i32, i32, i32, vp, i64, ctypes.POINTER(ctypes.c_int)]
    lib.mla_plan_units_ex.restype = i64
    lib.mla_merge_splits.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.mla_value_gate.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp]
    lib.mla_merge_value_gate.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp]
    lib.mla_choose_splits.argtypes = [i32, i32, i32, i32, i64, vp, i32, ctypes.POINTER(ctypes.c_int)]
    lib.mla_debug_gather.argtypes = [vp, i64, vp, i64, vp, i32, i64, vp, vp]
    lib.mla_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.mla_debug_wait_timeout.argtypes = [vp]
    lib.mla_kv_append.argtypes = [vp, i64, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.mla_decode_step_static.argtypes = [vp, i64, vp, i64, vp, i64, vp, i32, i32, i32, f32, f32, i32, i32,
                                           vp, i64, vp, vp, vp, vp, vp, vp, vp]
    for name in ("mla_decode_attend", "mla_decode_attend_ex", "mla_decode_attend_paged", "mla_decode_attend_planned", "mla_merge_splits", "mla_value_gate", "mla_merge_value_gate", "mla_debug_gather",
                 "mla_device_status", "mla_choose_splits", "mla_kv_append", "mla_debug_wait_timeout",
                 "mla_decode_step_static", "mla_debug_attend_mma"):
        getattr(lib, name).restype = ctypes.c_int
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_last_error.restype = ctypes.c_char_p
    lib.mla_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _status_name(status: int) -> str:
    try:
        return library().mla_status_string(status).decode()
    except Exception:  # pragma: no cover - only when the library is absent
        return "status"


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MlaError(status, where, library().mla_last_error().decode())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None) -> int:
    if stream is None:
        if _raw_stream is not None:   # the current stream's handle without building a Stream object
            return int(_raw_stream(torch.cuda.current_device() if device is None else device))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class Prepared:
    """A validated call with its arguments marshalled once: calling it
    launches on ``stream`` (default: the current stream of the tensors'
    device) with no further checks.  The tensors it was prepared from must
    stay alive with their shapes and addresses (as for a captured CUDA
    graph); their contents may change between calls.  ``outputs`` holds what
    the plain call returns."""

    def __init__(self, fn, args, where, device, outputs, keep):
        self._fn, self._args, self._where, self._device = fn, args, where, device
        self.outputs, self._keep = outputs, keep

    def __call__(self, stream=None):
        st = self._fn(*self._args, ctypes.c_void_p(_stream(stream, self._device)))
        if st != MLA_OK:
            _check(st, self._where)
        return self.outputs


def _marshal(fn, args):
    """Arguments converted to their ctypes types once (None and ctypes
    instances as they are)."""
    return [a if a is None or isinstance(a, ctypes._SimpleCData) else t(a) for t, a in zip(fn.argtypes, args)]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _same_device(dev, **named):
    """Every given tensor lives on the CUDA device ``dev``: a host pointer or
    another device's pointer handed to a kernel would fault."""
    _need(dev.type == "cuda", "tensors must be CUDA tensors (got %s)" % dev)
    for name, t in named.items():
        if t is not None:
            _need(t.device == dev, "%s is on %s, expected %s" % (name, t.device, dev))


def _buffer(t, name, dtype, shape):
    """A caller-supplied output: exactly this dtype and shape, contiguous
    (the kernels write every element of that extent)."""
    _need(t.dtype == dtype and tuple(t.shape) == tuple(shape) and t.is_contiguous(),
          "%s must be a contiguous %s tensor of shape %s" % (name, dtype, list(shape)))


def _as_u8(kv: torch.Tensor) -> torch.Tensor:
    if kv.dtype == torch.float8_e4m3fn:
        kv = kv.view(torch.uint8)
    _need(kv.dtype == torch.uint8, "kv must be uint8 codes or float8_e4m3fn")
    return kv


def attend(q, kv, pages, indptr, scale, kv_scale, num_splits, split_tokens, *, heads=None, qlen=1,
           o=None, lse=None, causal=False, page_size=1, last_page_len=None, q_scale=1.0, plan=None, stream=None,
           prepare=False):
    """Split-KV attention: returns ``(o [num_splits, S, heads, 512] bf16,
    lse [num_splits, S, heads] f32)``.

    ``q``: bf16 ``[S, H_pad, 576]`` whose rows may be strided (a padded query:
    ``heads`` < H_pad reads only the first ``heads``); ``kv``: ``[pool, 576]``
    fp8 codes; ``pages``/``indptr``: int32; S = (len(indptr) - 1) * qlen.
    ``causal``: row tq of a request sees only its first L - qlen + tq + 1
    tokens (``mla_decode_attend_ex`` with ``MLA_ATTEND_CAUSAL``).
    ``page_size`` > 1: block tables (``pages`` = block indices, ``indptr``
    counts blocks, ``last_page_len`` int32 [R] rows used in each request's
    last block; ``mla_decode_attend_paged``).
    A ``q`` of dtype float8_e4m3fn / uint8 is an fp8 query (codes); its
    ``q_scale`` multiplies the softmax scale (``MLA_ATTEND_Q_FP8``).
    ``plan``: a device int32 work plan from :func:`plan_units` for the same
    lengths and shape (``mla_decode_attend_planned``): its splits replace
    the ``split_tokens`` rule; the merged result is the same up to rounding.
    ``prepare=True`` validates and marshals once and returns a
    :class:`Prepared` call (launch it with ``call(stream)``) instead of
    launching.
    """
    kv = _as_u8(kv)
    heads = q.shape[1] if heads is None else heads
    R = indptr.numel() - 1
    S = R * qlen
    q8 = q.dtype in (torch.float8_e4m3fn, torch.uint8)
    if q.dtype == torch.float8_e4m3fn:
        q = q.view(torch.uint8)
    _need((q8 or q.dtype == torch.bfloat16) and q.dim() == 3 and q.shape[2] == D_QK,
          "q must be bf16 or fp8 e4m3 [S, H, 576]")
    _need(q.stride(2) == 1 and q.stride(1) == D_QK, "q rows must have contiguous [H, 576] heads")
    _need(q.shape[0] == S and heads <= q.shape[1], "q shape does not match indptr / qlen / heads")
    _need(kv.dim() == 2 and kv.shape[1] == D_QK and kv.is_contiguous(), "kv must be contiguous [pool, 576]")
    _need(pages.dtype == torch.int32 and indptr.dtype == torch.int32, "pages / indptr must be int32")
    _need(pages.is_contiguous() and indptr.is_contiguous(), "pages / indptr must be contiguous")
    _same_device(q.device, kv=kv, pages=pages, indptr=indptr, o=o, lse=lse, plan=plan,
                 last_page_len=last_page_len if page_size > 1 else None)
    if o is None:
        o = torch.empty((num_splits, S, heads, D_LATENT), dtype=torch.bfloat16, device=q.device)
    else:
        _buffer(o, "o", torch.bfloat16, (num_splits, S, heads, D_LATENT))
    if lse is None:
        lse = torch.empty((num_splits, S, heads), dtype=torch.float32, device=q.device)
    else:
        _buffer(lse, "lse", torch.float32, (num_splits, S, heads))
    if page_size > 1:
        _need(last_page_len is not None and last_page_len.dtype == torch.int32 and last_page_len.numel() == R
              and last_page_len.is_contiguous(), "page_size > 1 needs last_page_len int32 [R]")
    if plan is not None:
        _need(plan.dtype == torch.int32 and plan.dim() == 1 and plan.is_contiguous(),
              "plan must be a contiguous int32 device tensor")
    args = (_ptr(q), q.stride(0), _ptr(kv), kv.shape[0], _ptr(pages), pages.numel(), _ptr(indptr),
            _ptr(last_page_len) if page_size > 1 else None, int(page_size), R, qlen,
            heads, float(scale), float(kv_scale), float(q_scale), int(num_splits), int(split_tokens), _ptr(o),
            _ptr(lse), (ATTEND_CAUSAL if causal else 0) | (ATTEND_Q_FP8 if q8 else 0), _ptr(plan),
            0 if plan is None else plan.numel())
    lib = library()
    if prepare:
        # marshal once: ctypes converts each argument on every call otherwise
        conv = _marshal(lib.mla_decode_attend_planned, args)
        return Prepared(lib.mla_decode_attend_planned, conv, "mla_decode_attend", q.device.index, (o, lse),
                        (q, kv, pages, indptr, last_page_len, plan))
    st = lib.mla_decode_attend_planned(*args, ctypes.c_void_p(_stream(stream, q.device.index)))
    _check(st, "mla_decode_attend")
    return o, lse


def debug_attend_mma(q, kv, pages, indptr, scale, kv_scale, num_splits, split_tokens, *, heads=None, qlen=1,
                     o=None, lse=None, stream=None):
    """The same partials as :func:`attend` (page size 1, bf16 query, no
    options) from the library's second attend kernel, the warp-MMA one that
    the tests run as a cross-check (``mla_debug_attend_mma``)."""
    kv = _as_u8(kv)
    heads = q.shape[1] if heads is None else heads
    R = indptr.numel() - 1
    S = R * qlen
    _need(q.dtype == torch.bfloat16 and q.dim() == 3 and q.shape[2] == D_QK and q.stride(2) == 1
          and q.stride(1) == D_QK, "q must be bf16 [S, H, 576] with contiguous [H, 576] heads")
    _need(q.shape[0] == S and heads <= q.shape[1], "q shape does not match indptr / qlen / heads")
    _need(kv.dim() == 2 and kv.shape[1] == D_QK and kv.is_contiguous(), "kv must be contiguous [pool, 576]")
    _need(pages.dtype == torch.int32 and indptr.dtype == torch.int32 and pages.is_contiguous()
          and indptr.is_contiguous(), "pages / indptr must be contiguous int32")
    _same_device(q.device, kv=kv, pages=pages, indptr=indptr, o=o, lse=lse)
    if o is None:
        o = torch.empty((num_splits, S, heads, D_LATENT), dtype=torch.bfloat16, device=q.device)
    else:
        _buffer(o, "o", torch.bfloat16, (num_splits, S, heads, D_LATENT))
    if lse is None:
        lse = torch.empty((num_splits, S, heads), dtype=torch.float32, device=q.device)
    else:
        _buffer(lse, "lse", torch.float32, (num_splits, S, heads))
    st = library().mla_debug_attend_mma(_ptr(q), q.stride(0), _ptr(kv), kv.shape[0], _ptr(pages), pages.numel(),
                                        _ptr(indptr), R, qlen, heads, float(scale), float(kv_scale), int(num_splits),
                                        int(split_tokens), _ptr(o), _ptr(lse),
                                        ctypes.c_void_p(_stream(stream, q.device.index)))
    _check(st, "mla_debug_attend_mma")
    return o, lse


def merge(o, lse, *, latent=None, lse_out=None, want_lse=True, stream=None):
    """LSE merge: returns ``(latent [S, heads, 512] bf16, lse [S, heads] f32 or None)``."""
    _need(o.dtype == torch.bfloat16 and o.dim() == 4 and o.shape[3] == D_LATENT and o.is_contiguous(),
          "o must be contiguous bf16 [splits, S, heads, 512]")
    _need(lse.dtype == torch.float32 and lse.shape == o.shape[:3] and lse.is_contiguous(),
          "lse must be contiguous f32 [splits, S, heads]")
    ns, S, H = o.shape[:3]
    _same_device(o.device, lse=lse, latent=latent, lse_out=lse_out)
    if latent is None:
        latent = torch.empty((S, H, D_LATENT), dtype=torch.bfloat16, device=o.device)
    else:
        _buffer(latent, "latent", torch.bfloat16, (S, H, D_LATENT))
    if lse_out is None and want_lse:
        lse_out = torch.empty((S, H), dtype=torch.float32, device=o.device)
    elif lse_out is not None:
        _buffer(lse_out, "lse_out", torch.float32, (S, H))
    st = library().mla_merge_splits(_ptr(o), _ptr(lse), ns, S, H, _ptr(latent), _ptr(lse_out),
                                    ctypes.c_void_p(_stream(stream, o.device.index)))
    _check(st, "mla_merge_splits")
    return latent, lse_out


def value_gate(latent, w_uv, gate, lengths, qlen=1, *, out=None, stream=None):
    """W_UV + sigmoid gate: returns ``out [S, heads*128] bf16``."""
    _need(latent.dtype == torch.bfloat16 and latent.dim() == 3 and latent.shape[2] == D_LATENT
          and latent.is_contiguous(), "latent must be contiguous bf16 [S, heads, 512]")
    S, H = latent.shape[:2]
    _need(w_uv.dtype == torch.bfloat16 and tuple(w_uv.shape) == (H, D_V, D_LATENT) and w_uv.is_contiguous(),
          "w_uv must be contiguous bf16 [heads, 128, 512]")
    _need(gate.dtype == torch.bfloat16 and tuple(gate.shape) == (S, H * D_V) and gate.is_contiguous(),
          "gate must be contiguous bf16 [S, heads*128]")
    _need(lengths.dtype == torch.int32 and lengths.numel() * qlen == S and lengths.is_contiguous(),
          "lengths must be contiguous int32 [S / qlen]")
    _same_device(latent.device, w_uv=w_uv, gate=gate, lengths=lengths, out=out)
    if out is None:
        out = torch.empty((S, H * D_V), dtype=torch.bfloat16, device=latent.device)
    else:
        _buffer(out, "out", torch.bfloat16, (S, H * D_V))
    st = library().mla_value_gate(_ptr(latent), _ptr(w_uv), _ptr(gate), _ptr(lengths), lengths.numel(), qlen,
                                  H, _ptr(out), ctypes.c_void_p(_stream(stream, latent.device.index)))
    _check(st, "mla_value_gate")
    return out


def merge_value_gate(o, lse, w_uv, gate, lengths, qlen=1, *, out=None, latent=None, lse_out=None,
                     stream=None, prepare=False):
    """Merge + W_UV + gate in one call (one launch for small batches):
    returns ``out [S, heads*128] bf16``.  ``latent`` (allocated if not given)
    receives the merged latent, ``lse_out`` (optional) the merged LSE.
    ``prepare=True``: a :class:`Prepared` call instead (see :func:`attend`)."""
    _need(o.dtype == torch.bfloat16 and o.dim() == 4 and o.shape[3] == D_LATENT and o.is_contiguous(),
          "o must be contiguous bf16 [splits, S, heads, 512]")
    _need(lse.dtype == torch.float32 and lse.shape == o.shape[:3] and lse.is_contiguous(),
          "lse must be contiguous f32 [splits, S, heads]")
    ns, S, H = o.shape[:3]
    _need(w_uv.dtype == torch.bfloat16 and tuple(w_uv.shape) == (H, D_V, D_LATENT) and w_uv.is_contiguous(),
          "w_uv must be contiguous bf16 [heads, 128, 512]")
    _need(gate.dtype == torch.bfloat16 and tuple(gate.shape) == (S, H * D_V) and gate.is_contiguous(),
          "gate must be contiguous bf16 [S, heads*128]")
    _need(lengths.dtype == torch.int32 and lengths.numel() * qlen == S and lengths.is_contiguous(),
          "lengths must be contiguous int32 [S / qlen]")
    _same_device(o.device, lse=lse, w_uv=w_uv, gate=gate, lengths=lengths, out=out, latent=latent, lse_out=lse_out)
    if latent is not None:
        _buffer(latent, "latent", torch.bfloat16, (S, H, D_LATENT))
    if lse_out is not None:
        _buffer(lse_out, "lse_out", torch.float32, (S, H))
    if out is None:
        out = torch.empty((S, H * D_V), dtype=torch.bfloat16, device=o.device)
    else:
        _buffer(out, "out", torch.bfloat16, (S, H * D_V))
    if latent is None:
        latent = torch.empty((S, H, D_LATENT), dtype=torch.bfloat16, device=o.device)
    args = (_ptr(o), _ptr(lse), ns, _ptr(w_uv), _ptr(gate), _ptr(lengths), lengths.numel(), qlen, H, _ptr(out),
            _ptr(latent), _ptr(lse_out))
    lib = library()
    if prepare:
        conv = _marshal(lib.mla_merge_value_gate, args)
        return Prepared(lib.mla_merge_value_gate, conv, "mla_merge_value_gate", o.device.index, out,
                        (o, lse, w_uv, gate, lengths, out, latent, lse_out))
    st = lib.mla_merge_value_gate(*args, ctypes.c_void_p(_stream(stream, o.device.index)))
    _check(st, "mla_merge_value_gate")
    return out


def choose_splits(num_requests, qlen, heads, max_len=0, total_len=0, sm_count=0, lengths=None):
    """Host-side split plan: returns ``(num_splits, split_tokens)``.
    ``lengths`` (host-known per-request lengths, any int sequence or CPU
    tensor) makes the plan exact; otherwise ``max_len`` / ``total_len``
    estimate it."""
    st = ctypes.c_int(0)
    host = None
    if lengths is not None:
        host = torch.as_tensor(lengths, dtype=torch.int32, device="cpu").contiguous()
        num_requests = host.numel()
    ns = library().mla_choose_splits(int(num_requests), int(qlen), int(heads), int(max_len), int(total_len),
                                     None if host is None else ctypes.c_void_p(host.data_ptr()),
                                     int(sm_count), ctypes.byref(st))
    if ns < 1:
        _check(ns, "choose_splits")
    return int(ns), int(st.value)


def plan_units(lengths, qlen, heads, num_splits, sm_count=0, min_splits=1):
    """Balanced host work plan for :func:`attend` (``mla_plan_units_ex``):
    the requests cut into at most ``num_splits`` splits (and, where their
    tiles allow, at least ``min_splits``) so that each of ``sm_count`` CTAs
    (0: the current device's SMs) gets about the same number of tiles.
    Returns ``(plan, splits_used)``: a CPU int32 tensor (copy it to the
    device and pass it as ``attend(..., plan=)``) and the most splits any
    request got (the smallest ``num_splits`` the partial buffers need)."""
    host = torch.as_tensor(lengths, dtype=torch.int32, device="cpu").contiguous()
    lib = library()
    used = ctypes.c_int(0)
    args = (host.numel(), int(qlen), int(heads), ctypes.c_void_p(host.data_ptr()), int(min_splits),
            int(num_splits), int(sm_count))
    n = lib.mla_plan_units_ex(*args, None, 0, ctypes.byref(used))
    if n < 0:
        _check(int(n), "mla_plan_units_ex")
    plan = torch.empty(n, dtype=torch.int32)
    n2 = lib.mla_plan_units_ex(*args, ctypes.c_void_p(plan.data_ptr()), n, ctypes.byref(used))
    if n2 < 0:
        _check(int(n2), "mla_plan_units_ex")
    return plan, int(used.value)


def debug_gather(kv, pages, indptr, total_rows=None, stream=None):
    """Every request's KV rows in request order ([sum L, 576] uint8), gathered
    by the attend kernels' own row addressing."""
    kv = _as_u8(kv)
    _need(kv.dim() == 2 and kv.shape[1] == D_QK and kv.is_contiguous(), "kv must be contiguous [pool, 576]")
    _need(pages.dtype == torch.int32 and indptr.dtype == torch.int32 and pages.is_contiguous()
          and indptr.is_contiguous(), "pages / indptr must be contiguous int32")
    _same_device(kv.device, pages=pages, indptr=indptr)
    if total_rows is None:
        total_rows = int(indptr[-1].item())
    out = torch.empty((total_rows, D_QK), dtype=torch.uint8, device=kv.device)
    st = library().mla_debug_gather(_ptr(kv), kv.shape[0], _ptr(pages), pages.numel(), _ptr(indptr),
                                    indptr.numel() - 1, total_rows, _ptr(out),
                                    ctypes.c_void_p(_stream(stream, kv.device.index)))
    _check(st, "mla_debug_gather")
    return out


def kv_append(kv, kv_c, k_pe, slots, k_scale, *, stream=None):
    """Write new tokens into the fp8 cache in place: ``kv[slots[i]] =
    e4m3((kv_c[i] ++ k_pe[i]) / k_scale)`` (negative slots skipped).

    ``kv``: uint8 / float8_e4m3fn ``[pool, 576]``; ``kv_c``: bf16 ``[T, 512]``
    and ``k_pe``: bf16 ``[T, 64]`` (rows may be strided); ``slots``: int64
    ``[T]``.  Returns ``kv``.
    """
    kvu = _as_u8(kv)
    _need(kvu.dim() == 2 and kvu.shape[1] == D_QK and kvu.is_contiguous(), "kv must be contiguous [pool, 576]")
    _need(kv_c.dtype == torch.bfloat16 and kv_c.dim() == 2 and kv_c.shape[1] == D_LATENT and kv_c.stride(1) == 1,
          "kv_c must be bf16 [T, 512] with contiguous rows")
    _need(k_pe.dtype == torch.bfloat16 and k_pe.dim() == 2 and k_pe.shape[1] == D_QK - D_LATENT and k_pe.stride(1) == 1,
          "k_pe must be bf16 [T, 64] with contiguous rows")
    T = kv_c.shape[0]
    _need(k_pe.shape[0] == T and slots.dtype == torch.int64 and slots.numel() == T and slots.is_contiguous(),
          "slots must be contiguous int64 [T] matching kv_c / k_pe")
    _same_device(kvu.device, kv_c=kv_c, k_pe=k_pe, slots=slots)
    st = library().mla_kv_append(_ptr(kv_c), kv_c.stride(0), _ptr(k_pe), k_pe.stride(0), _ptr(slots), T,
                                 float(k_scale), _ptr(kvu), kvu.shape[0],
                                 ctypes.c_void_p(_stream(stream, kvu.device.index)))
    _check(st, "mla_kv_append")
    return kv


def debug_wait_timeout(stream=None):
    """Test hook: enqueue a kernel whose bounded wait runs out (about 2 s);
    it sets DEV_TIMEOUT, which :func:`device_status` then reports."""
    _check(library().mla_debug_wait_timeout(ctypes.c_void_p(_stream(stream))), "mla_debug_wait_timeout")


def device_status(stream=None) -> int:
    """Synchronise the stream, return and clear the device status bits
    (DEV_BAD_PAGE, DEV_BAD_INDPTR, DEV_TIMEOUT, DEV_BAD_PLAN)."""
    flags = ctypes.c_uint(0)
    _check(library().mla_device_status(ctypes.c_void_p(_stream(stream)), ctypes.byref(flags)),
           "mla_device_status")
    return int(flags.value)


def decode_step(q, kv, pages, indptr, scale, kv_scale, w_uv, gate, lengths, *, heads=None, qlen=1,
                num_splits=None, split_tokens=None, max_len=None, total_len=0, causal=False, page_size=1,
                last_page_len=None, q_scale=1.0, plan=None, stream=None):
    """The whole step (attend, then the merge with value/gate through
    :func:`merge_value_gate`: one launch for small batches); returns
    ``(out, latent, lse)``.  Without a split plan one is chosen from
    ``max_len`` (host-known longest request).  ``causal``, ``page_size``,
    ``last_page_len``, ``q_scale`` and ``plan`` as in :func:`attend`."""
    heads = q.shape[1] if heads is None else heads
    if num_splits is None or split_tokens is None:
        if max_len is None:
            raise ValueError("give num_splits and split_tokens, or max_len for the split plan")
        num_splits, split_tokens = choose_splits(indptr.numel() - 1, qlen, heads, max_len, total_len)
    o, lse = attend(q, kv, pages, indptr, scale, kv_scale, num_splits, split_tokens, heads=heads,
                    qlen=qlen, causal=causal, page_size=page_size, last_page_len=last_page_len,
                    q_scale=q_scale, plan=plan, stream=stream)
    lse_m = torch.empty(lse.shape[1:], dtype=torch.float32, device=lse.device)
    latent = torch.empty(o.shape[1:], dtype=torch.bfloat16, device=o.device)
    out = merge_value_gate(o, lse, w_uv, gate, lengths, qlen, latent=latent, lse_out=lse_m, stream=stream)
    return out, latent, lse_m


def decode_step_static(q, kv, pages, indptr, scale, kv_scale, w_uv, gate, lengths, num_splits, split_tokens, *,
                       heads=None, qlen=1, plan=None, out=None, latent=None, lse_out=None, stream=None):
    """The whole step through ``mla_decode_step_static``: the split partials
    live in the library's own 32 MiB device buffer, so the native call
    allocates nothing (for callers that cannot allocate device memory while
    they run; see the header).  Returns ``(out, latent, lse_out)``; the
    outputs are allocated here with torch unless given.  Calls on one
    device share the buffer: keep them ordered on one stream.  The first
    call on a device looks up the buffer's address, so make it before any
    stream capture.  Raises :class:`MlaError` (MLA_ERR_UNSUPPORTED) when the
    partials, ``num_splits * S * heads * 1028`` bytes, do not fit."""
    kv = _as_u8(kv)
    heads = q.shape[1] if heads is None else heads
    R = indptr.numel() - 1
    S = R * qlen
    _need(q.dtype == torch.bfloat16 and q.dim() == 3 and q.shape[2] == D_QK and q.stride(2) == 1
          and q.stride(1) == D_QK, "q must be bf16 [S, H, 576] with contiguous [H, 576] heads")
    _need(q.shape[0] == S and heads <= q.shape[1], "q shape does not match indptr / qlen / heads")
    _need(kv.dim() == 2 and kv.shape[1] == D_QK and kv.is_contiguous(), "kv must be contiguous [pool, 576]")
    _need(pages.dtype == torch.int32 and indptr.dtype == torch.int32 and pages.is_contiguous()
          and indptr.is_contiguous(), "pages / indptr must be contiguous int32")
    _need(w_uv.dtype == torch.bfloat16 and tuple(w_uv.shape) == (heads, D_V, D_LATENT) and w_uv.is_contiguous(),
          "w_uv must be contiguous bf16 [heads, 128, 512]")
    _need(gate.dtype == torch.bfloat16 and tuple(gate.shape) == (S, heads * D_V) and gate.is_contiguous(),
          "gate must be contiguous bf16 [S, heads*128]")
    _need(lengths.dtype == torch.int32 and lengths.numel() == R and lengths.is_contiguous(),
          "lengths must be contiguous int32 [R]")
    if plan is not None:
        _need(plan.dtype == torch.int32 and plan.dim() == 1 and plan.is_contiguous(),
              "plan must be a contiguous int32 device tensor")
    _same_device(q.device, kv=kv, pages=pages, indptr=indptr, w_uv=w_uv, gate=gate, lengths=lengths, plan=plan,
                 out=out, latent=latent, lse_out=lse_out)
    if out is None:
        out = torch.empty((S, heads * D_V), dtype=torch.bfloat16, device=q.device)
    else:
        _buffer(out, "out", torch.bfloat16, (S, heads * D_V))
    if latent is None:
        latent = torch.empty((S, heads, D_LATENT), dtype=torch.bfloat16, device=q.device)
    else:
        _buffer(latent, "latent", torch.bfloat16, (S, heads, D_LATENT))
    if lse_out is not None:
        _buffer(lse_out, "lse_out", torch.float32, (S, heads))
    st = library().mla_decode_step_static(
        _ptr(q), q.stride(0), _ptr(kv), kv.shape[0], _ptr(pages), pages.numel(), _ptr(indptr), R, qlen, heads,
        float(scale), float(kv_scale), int(num_splits), int(split_tokens), _ptr(plan),
        0 if plan is None else plan.numel(), _ptr(w_uv), _ptr(gate), _ptr(lengths), _ptr(out), _ptr(latent),
        _ptr(lse_out), ctypes.c_void_p(_stream(stream, q.device.index)))
    _check(st, "mla_decode_step_static")
    return out, latent, lse_out
