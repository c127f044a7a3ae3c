"""Zigzag context-parallel causal attention on GB300 (sm_103a).

Thin Python layer over the C ABI of ``libcpattn.so`` (``include/cpattn.h``):
it checks tensors, owns the workspace buffer and passes device pointers and
the current CUDA stream down.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.

Functions keep the names of the C entry points:

* :func:`cp_zigzag_index`, :func:`cp_zigzag_gather`, :func:`cp_zigzag_scatter`
* :func:`cp_attn_fwd`, :func:`cp_lse_merge`, :func:`cp_attn_bwd`
* :func:`cp_attn_fwd_gqa`, :func:`cp_attn_bwd_gqa` -- grouped KV heads
* :func:`cp_workspace_status`, :func:`cp_set_wait_limit`, :func:`cp_plan_pairs`,
  :func:`cp_plan_unit_lists`
* :func:`attention_host` -- end-to-end call on host (pinned) tensors.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _binding as _b
from ._binding import CP_BF16, CP_F32, CpError  # noqa: F401

__all__ = ["cp_zigzag_index", "cp_zigzag_gather", "cp_zigzag_scatter", "cp_attn_fwd",
           "cp_attn_fwd_noalloc", "cp_attn_fwd_gqa", "cp_attn_bwd_gqa",
           "cp_lse_merge", "cp_attn_bwd", "cp_workspace_status", "cp_set_wait_limit",
           "cp_plan_pairs", "cp_plan_unit_lists", "cp_profile_begin", "cp_profile_end", "Workspace",
           "attention_host", "CpError"]


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CP_BF16
    if t.dtype == torch.float32:
        return CP_F32
    raise CpError(3, "dtype %s not supported (bf16 or fp32)" % t.dtype)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise CpError(1, "tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise CpError(1, "tensors must be contiguous")


class Workspace:
    """A growable device byte buffer (256-byte aligned) reused across calls on
    one stream."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else None
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=device)
        return self.buf

    def ptr(self):
        p = self.buf.data_ptr()
        return (p + 255) // 256 * 256

    def nbytes(self):
        return self.buf.numel() - (self.ptr() - self.buf.data_ptr())


_default_ws = {}


def _ws(ws: Optional[Workspace], device, nbytes: int, key: str) -> Workspace:
    if ws is None:
        ws = _default_ws.setdefault((key, str(device)), Workspace(device))
    ws.get(nbytes, device)
    return ws


# ---------------------------------------------------------------------------
def cp_zigzag_index(cu_seqlens: Sequence[int], prefix_len: int, P: int, device=None):
    """Zigzag gather table ``fwd_idx`` and inverse ``inv_idx`` (int32).  On the
    host when ``device`` is None, else copied to that device on its current
    stream."""
    cu = _b.cu_array(cu_seqlens)
    n = len(cu_seqlens) - 1
    text = sum(int(cu_seqlens[i + 1]) - int(cu_seqlens[i]) - prefix_len for i in range(n))
    text = max(text, 0)
    if device is None:
        fwd = torch.empty(text, dtype=torch.int32)
        inv = torch.empty(text, dtype=torch.int32)
        _b.check(_b.lib().cp_zigzag_index(cu, n, prefix_len, P, _ptr(fwd), _ptr(inv), 0, None))
    else:
        fwd = torch.empty(text, dtype=torch.int32, device=device)
        inv = torch.empty(text, dtype=torch.int32, device=device)
        _b.check(_b.lib().cp_zigzag_index(cu, n, prefix_len, P, _ptr(fwd), _ptr(inv), 1,
                                          _stream(fwd.device)))
    return fwd, inv


def cp_zigzag_gather(src: torch.Tensor, idx: torch.Tensor, out: Optional[torch.Tensor] = None):
    """``out[k] = src[idx[k]]`` along dim 0 (rows of ``src[0].nbytes`` bytes)."""
    _need_cuda(src, idx, out)
    if out is None:
        out = torch.empty((idx.numel(),) + tuple(src.shape[1:]), dtype=src.dtype,
                          device=src.device)
    row = src[0].numel() * src.element_size() if src.dim() > 1 else src.element_size()
    _b.check(_b.lib().cp_zigzag_gather(_ptr(src), _ptr(out), row, _ptr(idx), idx.numel(),
                                       _stream(src.device)))
    return out


def cp_zigzag_scatter(src: torch.Tensor, idx: torch.Tensor, out: torch.Tensor):
    """``out[idx[k]] = src[k]`` along dim 0."""
    _need_cuda(src, idx, out)
    row = src[0].numel() * src.element_size() if src.dim() > 1 else src.element_size()
    _b.check(_b.lib().cp_zigzag_scatter(_ptr(src), _ptr(out), row, _ptr(idx), idx.numel(),
                                        _stream(src.device)))
    return out


def cp_attn_fwd(q, k, v, cu_seqlens, P: int, prefix_len: int, softmax_scale: float,
                out=None, lse=None, workspace: Optional[Workspace] = None,
                residual: bool = False, out_lo=None):
    """Context-parallel causal attention forward; returns ``(out, lse)`` with
    out ``[T,H,d]`` (q's dtype) and lse ``[H,T]`` fp32 (natural log).  With
    ``residual=True`` (bf16 only) it returns ``(out, lse, out_lo)``, where
    out_lo holds the bf16 rounding remainder of out, for :func:`cp_attn_bwd`.
    ``k``/``v`` with fewer heads than ``q`` go to :func:`cp_attn_fwd_gqa`."""
    return _attn_fwd(q, k, v, cu_seqlens, P, prefix_len, softmax_scale, out, lse, workspace,
                     residual, out_lo, k.shape[1] != q.shape[1])


def cp_attn_fwd_gqa(q, k, v, cu_seqlens, P: int, prefix_len: int, softmax_scale: float,
                    out=None, lse=None, workspace: Optional[Workspace] = None,
                    residual: bool = False, out_lo=None):
    """:func:`cp_attn_fwd` with grouped KV heads: ``k``/``v`` are
    ``[T,H_kv,d]`` and query head h reads KV head ``h // (H / H_kv)``."""
    return _attn_fwd(q, k, v, cu_seqlens, P, prefix_len, softmax_scale, out, lse, workspace,
                     residual, out_lo, True)


def _attn_fwd(q, k, v, cu_seqlens, P, prefix_len, softmax_scale, out, lse, workspace, residual,
              out_lo, gqa):
    _need_cuda(q, k, v, out, lse, out_lo)
    T, H, d = q.shape
    Hkv = k.shape[1]
    dt = _dt(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if residual and out_lo is None and dt == CP_BF16:
        out_lo = torch.empty_like(q)
    cu = _b.cu_array(cu_seqlens)
    n = len(cu_seqlens) - 1
    L = _b.lib()
    if gqa:
        nbytes = L.cp_attn_fwd_workspace_size_gqa(dt, T, H, Hkv, d, cu, n, P, prefix_len,
                                                  float(softmax_scale))

        def run(ws_ptr, ws_bytes):
            return L.cp_attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), dt, T, H, Hkv, d, cu, n, P,
                                     prefix_len, float(softmax_scale), _ptr(out), _ptr(lse),
                                     _ptr(out_lo), ws_ptr, ws_bytes, _stream(q.device))
    else:
        nbytes = L.cp_attn_fwd_workspace_size(dt, T, H, d, cu, n, P, prefix_len,
                                              float(softmax_scale))

        def run(ws_ptr, ws_bytes):
            return L.cp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), dt, T, H, d, cu, n, P, prefix_len,
                                 float(softmax_scale), _ptr(out), _ptr(lse), _ptr(out_lo),
                                 ws_ptr, ws_bytes, _stream(q.device))
    if nbytes == 0:  # invalid arguments: let the library name the problem
        _b.check(run(None, 0))
    ws = _ws(workspace, q.device, nbytes, "fwd")
    _b.check(run(ctypes.c_void_p(ws.ptr()), ws.nbytes()))
    if residual:
        return out, lse, out_lo
    return out, lse


def cp_attn_fwd_noalloc(q, k, v, cu_seqlens, P: int, prefix_len: int, softmax_scale: float,
                        out=None, lse=None, out_lo=None):
    """The forward for callers that cannot allocate device memory (their
    memory is owned by another allocator, or fixed up front): same result as
    :func:`cp_attn_fwd`, but the library's fixed 64 MiB scratch replaces the
    workspace.  Outputs may be passed in (``out``, ``lse``, ``out_lo``) so the
    call allocates nothing; the first call on a device must precede any
    stream capture; calls that overlap on the GPU race on the shared scratch.
    ``cp_workspace_status()`` (no workspace) reports a device wait that gave up."""
    _need_cuda(q, k, v, out, lse, out_lo)
    T, H, d = q.shape
    dt = _dt(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    cu = _b.cu_array(cu_seqlens)
    _b.check(_b.lib().cp_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), dt, T, H, d, cu,
                                          len(cu_seqlens) - 1, P, prefix_len,
                                          float(softmax_scale), _ptr(out), _ptr(lse),
                                          _ptr(out_lo), _stream(q.device)))
    return out, lse


def cp_lse_merge(part_out: torch.Tensor, part_lse: torch.Tensor, out_dtype=torch.float32,
                 out=None, lse=None):
    """Merge ``part_out [n,rows,H,d]`` / ``part_lse [n,H,rows]`` (fp32) into
    ``(out [rows,H,d], lse [H,rows])`` by log-sum-exp (outputs may be passed in)."""
    _need_cuda(part_out, part_lse, out, lse)
    n, rows, H, d = part_out.shape
    if out is None:
        out = torch.empty((rows, H, d), dtype=out_dtype, device=part_out.device)
    if lse is None:
        lse = torch.empty((H, rows), dtype=torch.float32, device=part_out.device)
    _b.check(_b.lib().cp_lse_merge(n, _ptr(part_out), _ptr(part_lse), rows, H, d, _ptr(out),
                                   _dt(out), _ptr(lse), _stream(part_out.device)))
    return out, lse


def cp_attn_bwd(q, k, v, out, lse, dout, cu_seqlens, P: int, prefix_len: int,
                softmax_scale: float, per_rank_prefix: bool = False,
                workspace: Optional[Workspace] = None, grads=None, out_lo=None):
    """Backward; returns ``(dq, dk, dv)`` fp32 (dq ``[T,H,d]``, dk/dv shaped
    like k) and, with ``per_rank_prefix``, the per-rank prefix gradients
    ``[2, P+1, n*prefix_len, H_kv, d]`` (slot P: prefix queries' own term).
    ``out_lo``: the remainder returned by ``cp_attn_fwd(..., residual=True)``.
    ``k``/``v`` with fewer heads than ``q`` go to :func:`cp_attn_bwd_gqa`."""
    return _attn_bwd(q, k, v, out, lse, dout, cu_seqlens, P, prefix_len, softmax_scale,
                     per_rank_prefix, workspace, grads, out_lo, k.shape[1] != q.shape[1])


def cp_attn_bwd_gqa(q, k, v, out, lse, dout, cu_seqlens, P: int, prefix_len: int,
                    softmax_scale: float, per_rank_prefix: bool = False,
                    workspace: Optional[Workspace] = None, grads=None, out_lo=None):
    """:func:`cp_attn_bwd` with grouped KV heads: dk/dv ``[T,H_kv,d]`` sum the
    contributions of each KV head's query heads."""
    return _attn_bwd(q, k, v, out, lse, dout, cu_seqlens, P, prefix_len, softmax_scale,
                     per_rank_prefix, workspace, grads, out_lo, True)


def _attn_bwd(q, k, v, out, lse, dout, cu_seqlens, P, prefix_len, softmax_scale,
              per_rank_prefix, workspace, grads, out_lo, gqa):
    _need_cuda(q, k, v, out, lse, dout, out_lo)
    T, H, d = q.shape
    Hkv = k.shape[1]
    dt = _dt(q)
    if grads is None:
        grads = (torch.empty((T, H, d), dtype=torch.float32, device=q.device),
                 torch.empty((T, Hkv, d), dtype=torch.float32, device=q.device),
                 torch.empty((T, Hkv, d), dtype=torch.float32, device=q.device))
    dq, dk, dv = grads
    n = len(cu_seqlens) - 1
    pgrad = None
    if per_rank_prefix:
        pgrad = torch.empty((2, P + 1, n * prefix_len, Hkv, d), dtype=torch.float32,
                            device=q.device)
    cu = _b.cu_array(cu_seqlens)
    L = _b.lib()
    if gqa:
        nbytes = L.cp_attn_bwd_workspace_size_gqa(dt, T, H, Hkv, d, cu, n, P, prefix_len,
                                                  float(softmax_scale))

        def run(ws_ptr, ws_bytes):
            return L.cp_attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(out_lo),
                                     _ptr(lse), _ptr(dout), dt, T, H, Hkv, d, cu, n, P,
                                     prefix_len, float(softmax_scale), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(pgrad), ws_ptr, ws_bytes, _stream(q.device))
    else:
        nbytes = L.cp_attn_bwd_workspace_size(dt, T, H, d, cu, n, P, prefix_len,
                                              float(softmax_scale))

        def run(ws_ptr, ws_bytes):
            return L.cp_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(out_lo), _ptr(lse),
                                 _ptr(dout), dt, T, H, d, cu, n, P, prefix_len,
                                 float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(pgrad),
                                 ws_ptr, ws_bytes, _stream(q.device))
    if nbytes == 0:  # invalid arguments: let the library name the problem
        _b.check(run(None, 0))
    ws = _ws(workspace, q.device, nbytes, "bwd")
    _b.check(run(ctypes.c_void_p(ws.ptr()), ws.nbytes()))
    if per_rank_prefix:
        return dq, dk, dv, pgrad
    return dq, dk, dv


def cp_workspace_status(workspace: Optional[Workspace] = None, device=None) -> int:
    """Synchronise the current stream; 0, the CP_ERR_TIMEOUT status, or (in
    the bounds-checked build, see ``_binding.bounds_checked``) CP_ERR_BOUNDS.  With
    no workspace it reads the status of :func:`cp_attn_fwd_noalloc`'s fixed
    scratch on ``device`` (default: the current device)."""
    if workspace is None:
        dev = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        with torch.cuda.device(dev):
            return _b.lib().cp_workspace_status(None, _stream(dev))
    st = _b.lib().cp_workspace_status(ctypes.c_void_p(workspace.ptr()),
                                      _stream(workspace.buf.device))
    return st


def default_workspace(kind: str, device) -> Workspace:
    return _default_ws[(kind, str(torch.device(device)))]


def cp_set_wait_limit(rounds: int):
    _b.lib().cp_set_wait_limit(int(rounds))


PROFILE_KINDS = ("zigzag_index", "zigzag_gather", "tc_fwd_step", "bwd_preprocess",
                 "tc_bwd_step", "prefix_reduce", "simt_fwd_step", "simt_bwd_step")


def cp_profile_begin():
    """Start recording CUDA events around every kernel the library launches."""
    _b.lib().cp_profile_begin()


def cp_profile_end():
    """Stop recording; returns {kind: (total_ms, launches)}."""
    ms = (ctypes.c_double * 8)()
    n = (ctypes.c_int64 * 8)()
    _b.check(_b.lib().cp_profile_end(ms, n))
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(PROFILE_KINDS)}


def cp_plan_pairs(cu_seqlens, prefix_len: int, P: int):
    """Host-only: visible pairs and items per ring step of both work lists."""
    arrs = [(ctypes.c_int64 * P)() for _ in range(4)]
    cu = _b.cu_array(cu_seqlens)
    _b.check(_b.lib().cp_plan_pairs(cu, len(cu_seqlens) - 1, prefix_len, P, *arrs))
    return tuple([int(x) for x in a] for a in arrs)


def cp_plan_unit_lists(cu_seqlens, prefix_len: int, P: int, H: int, grid: int):
    """Host-only: the all-steps forward's items and their cost in KV tiles,
    and the unit lists of a persistent launch over ``grid`` CTAs.  Returns
    ``(tiles, units, cta_off)`` as int32 numpy arrays; unit = item + n_items * head."""
    import numpy as np
    cu = _b.cu_array(cu_seqlens)
    n = ctypes.c_int64(0)
    args = (cu, len(cu_seqlens) - 1, prefix_len, P, H, grid)
    _b.check(_b.lib().cp_plan_unit_lists(*args, ctypes.byref(n), None, None, None))
    tiles = np.zeros(n.value, np.int32)
    units = np.zeros(n.value * H, np.int32)
    off = np.zeros(grid + 1, np.int32)
    p32 = ctypes.POINTER(ctypes.c_int32)
    _b.check(_b.lib().cp_plan_unit_lists(*args, ctypes.byref(n), tiles.ctypes.data_as(p32),
                                         units.ctypes.data_as(p32), off.ctypes.data_as(p32)))
    return tiles, units, off


_side = {}


def _side_streams(dev):
    """Two copy streams per device: host-to-device and device-to-host."""
    key = str(dev)
    if key not in _side:
        _side[key] = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    return _side[key]


_host_bufs = {}


def release_host_buffers():
    """Free the device buffers :func:`attention_host` keeps between calls."""
    _host_bufs.clear()


def host_chunks(T: int, H: int, H_kv: int, d: int, elem: int) -> int:
    """Head chunks of :func:`attention_host`: 4 (or 2) when the problem's
    tensors exceed 256 MB, so that one chunk's copies hide behind another's
    kernels; 1 for smaller problems, whose launches would shrink too far."""
    if T * (2 * H + 2 * H_kv) * d * elem < (256 << 20):
        return 1
    for n in (4, 2):
        if H_kv % n == 0:
            return n
    return 1


def _copy_rows(dst, dst_off, dst_pitch, src, src_off, src_pitch, width, rows, stream):
    _b.check(_b.lib().cp_copy_rows(ctypes.c_void_p(dst.data_ptr() + dst_off), dst_pitch,
                                   ctypes.c_void_p(src.data_ptr() + src_off), src_pitch,
                                   width, rows, ctypes.c_void_p(stream.cuda_stream)))


def attention_host(q, k, v, dout, cu_seqlens, P: int, prefix_len: int, softmax_scale: float,
                   device="cuda", host_out=None, chunks: int = 0):
    """End-to-end call on host tensors (pinned for asynchronous copies): copy the
    inputs to ``device``, run forward (and backward when ``dout`` is given),
    copy results back.  Returns host tensors ``(out, lse[, dq, dk, dv])``;
    ``host_out`` may supply them (pinned).  ``k``, ``v`` may have fewer heads
    than ``q`` (grouped KV heads).

    Heads are independent, so the call streams them through the device in
    ``chunks`` groups of KV heads (default :func:`host_chunks`), each with its
    own device buffers: while the kernels of one group run on the current
    stream, later groups' q, k, v, dO go up on one copy stream and earlier
    groups' results come down on another (strided row copies of the head
    range, ``cp_copy_rows``).  Within a group, dO goes up while the
    forward runs and out, lse come down while the backward runs.  Events order
    every copy against the kernels that write or read its buffers.  The
    device buffers are cached per shape, so concurrent calls from several
    host threads must be serialised by the caller."""
    dev = torch.device(device)
    comp = torch.cuda.current_stream(dev)
    up, down = _side_streams(dev)
    T, H, d = q.shape
    Hkv = k.shape[1]
    dt = q.dtype
    elem = q.element_size()
    bwd = dout is not None
    keep = bwd and dt == torch.bfloat16
    n = chunks or host_chunks(T, H, Hkv, d, elem)
    if Hkv % n != 0:
        raise ValueError("chunks must divide the KV heads")
    Gc, Hc = Hkv // n, H // n          # KV and query heads per chunk
    n_res = 5 if bwd else 2
    if host_out is None:
        shapes = [((T, H, d), dt), ((H, T), torch.float32)]
        if bwd:
            shapes += [((T, H, d), torch.float32), ((T, Hkv, d), torch.float32),
                       ((T, Hkv, d), torch.float32)]
        host_out = [torch.empty(sh, dtype=dt_, pin_memory=True) for sh, dt_ in shapes]
    # device buffers of every chunk (the footprint of the unchunked call), so
    # that no upload waits for an earlier chunk's download: a copy that stalls
    # delays only its own chunk.  Kept for the next call of the same shape
    # (release_host_buffers() frees them).
    nb = n
    key = (str(dev), T, Hc, Gc, d, dt, bwd, keep)
    sets = _host_bufs.get(key)
    if sets is None:
        _host_bufs.clear()
        sets = []
        for _ in range(nb):
            st = {"q": torch.empty((T, Hc, d), dtype=dt, device=dev),
                  "k": torch.empty((T, Gc, d), dtype=dt, device=dev),
                  "v": torch.empty((T, Gc, d), dtype=dt, device=dev),
                  "out": torch.empty((T, Hc, d), dtype=dt, device=dev),
                  "lse": torch.empty((Hc, T), dtype=torch.float32, device=dev)}
            if keep:
                st["lo"] = torch.empty((T, Hc, d), dtype=dt, device=dev)
            if bwd:
                st["do"] = torch.empty((T, Hc, d), dtype=dt, device=dev)
                st["dq"] = torch.empty((T, Hc, d), dtype=torch.float32, device=dev)
                st["dk"] = torch.empty((T, Gc, d), dtype=torch.float32, device=dev)
                st["dv"] = torch.empty((T, Gc, d), dtype=torch.float32, device=dev)
            sets.append(st)
        _host_bufs[key] = sets
    ready = torch.cuda.Event()
    ready.record(comp)               # buffers allocated (and earlier work) on comp
    up.wait_event(ready)
    down.wait_event(ready)
    freed = [None] * nb              # per set: its last results have come down
    qrow, krow = H * d, Hkv * d      # elements per host row
    for c in range(n):
        S = sets[c % nb]
        h0, g0 = c * Hc, c * Gc
        # ---- inputs up
        if freed[c % nb] is not None:
            up.wait_event(freed[c % nb])
        for name, src, row, heads, h in (("q", q, qrow, Hc, h0), ("k", k, krow, Gc, g0),
                                         ("v", v, krow, Gc, g0)):
            _copy_rows(S[name], 0, heads * d * elem, src, h * d * elem, row * elem,
                       heads * d * elem, T, up)
        ev_in = torch.cuda.Event()
        ev_in.record(up)
        if bwd:
            _copy_rows(S["do"], 0, Hc * d * elem, dout, h0 * d * elem, qrow * elem,
                       Hc * d * elem, T, up)
            ev_do = torch.cuda.Event()
            ev_do.record(up)
        # ---- kernels
        comp.wait_event(ev_in)
        cp_attn_fwd_gqa(S["q"], S["k"], S["v"], cu_seqlens, P, prefix_len, softmax_scale,
                        out=S["out"], lse=S["lse"], residual=keep,
                        out_lo=S["lo"] if keep else None)
        ev_fwd = torch.cuda.Event()
        ev_fwd.record(comp)
        if bwd:
            comp.wait_event(ev_do)
            cp_attn_bwd_gqa(S["q"], S["k"], S["v"], S["out"], S["lse"], S["do"], cu_seqlens, P,
                            prefix_len, softmax_scale, grads=(S["dq"], S["dk"], S["dv"]),
                            out_lo=S["lo"] if keep else None)
            ev_bwd = torch.cuda.Event()
            ev_bwd.record(comp)
        # ---- results down
        down.wait_event(ev_fwd)
        _copy_rows(host_out[0], h0 * d * elem, qrow * elem, S["out"], 0, Hc * d * elem,
                   Hc * d * elem, T, down)
        _copy_rows(host_out[1], h0 * T * 4, Hc * T * 4, S["lse"], 0, Hc * T * 4,
                   Hc * T * 4, 1, down)
        if bwd:
            down.wait_event(ev_bwd)
            for i, (name, row, heads, h) in enumerate((("dq", qrow, Hc, h0),
                                                       ("dk", krow, Gc, g0),
                                                       ("dv", krow, Gc, g0))):
                _copy_rows(host_out[2 + i], h * d * 4, row * 4, S[name], 0, heads * d * 4,
                           heads * d * 4, T, down)
        ev = torch.cuda.Event()
        ev.record(down)
        freed[c % nb] = ev
        # the next use of this set's outputs by the kernels waits for the
        # copies down: its inputs go up only after `freed`, and the kernels
        # wait for the inputs
    down.synchronize()
    up.synchronize()
    comp.synchronize()
    return tuple(host_out[:n_res])
