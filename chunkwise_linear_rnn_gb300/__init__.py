"""GB300-native gated linear attention (GLA): chunked prefill, its backward, and the decode step.

The computation ("Gated Linear Attention (GLA): Mathematical Foundations, ..."
(llms.blog), section "The Gated Recurrent Update"):

    S_t = diag(alpha_t) S_{t-1} + k_t^T v_t,      o_t = scale * q_t S_t

runs entirely in the hand-written sm_103a kernels of ``libgla.so``; this module
only checks and marshals PyTorch tensors into the C ABI of ``include/gla.h``
(device pointers, sizes and the current CUDA stream).

Layouts (contiguous, head-first): q, k ``[B,H,T,dk]`` bf16; v ``[B,H,T,dv]``
bf16; log_alpha ``[B,H,T,dk]`` fp32; o ``[B,H,T,dv]`` bf16; h0 / hT
``[B,H,dk,dv]`` fp32.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import GlaChunkOptions, GlaError, status_string  # noqa: F401

__all__ = ["gla_chunk_fwd", "gla_chunk_fwd_varlen", "gla_chunk_fwd_varlen_plan",
           "gla_chunk_fwd_plan", "gla_chunk_bwd", "gla_chunk_bwd_plan", "gla_chunk_bwd_varlen",
           "gla_chunk", "gla_chunk_varlen", "gla_gdn_fwd",
           "gla_recurrent_step", "gla_last_device_status", "GlaError", "status_string",
           "library_path"]

library_path = _lib.LIB_PATH


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple, device) -> None:
    """Checks a tensor argument; `device` is a CUDA device, or the CPU for host entry points."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is not None and device.type == "cpu":
        if t.device.type != "cpu":
            raise ValueError(f"{name} must be a CPU tensor")
    elif t.device.type != "cuda" or (device is not None and t.device != device):
        raise ValueError(f"{name} must be on the CUDA device {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def gla_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                  scale: float | None = None, h0: torch.Tensor | None = None,
                  output_final_state: bool = True, *, out: torch.Tensor | None = None,
                  final_state: torch.Tensor | None = None, segments: int = 0, dv_tile: int = 0,
                  force_exact: bool = False, cta_pair: int = 0):
    """Chunkwise-parallel GLA forward over whole sequences.

    ``log_alpha`` is ``[B, H, T, dk]`` (one gate per key channel) or
    ``[B, H, T]`` (one gate per token and head, used for every channel).
    Returns ``(o, hT)``; ``hT`` is None when ``output_final_state`` is False.
    ``final_state`` may be ``h0`` itself (in-place state update).
    ``segments``, ``dv_tile``, ``force_exact`` and ``cta_pair`` are the C ABI's
    options (0 / False = automatic; ``cta_pair=-1`` keeps the value tiles of a
    head in independent CTAs).
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, dk]")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be on a CUDA device (gla_chunk_fwd_host takes CPU tensors)")
    _need(q, "q", torch.bfloat16, (B, H, T, dk), dev)
    _need(k, "k", torch.bfloat16, (B, H, T, dk), dev)
    _need(v, "v", torch.bfloat16, (B, H, T, dv), dev)
    # a [B, H, T] gate is one decay per token and head, the same for every channel
    per_head = log_alpha.dim() == 3
    _need(log_alpha, "log_alpha", torch.float32, (B, H, T) if per_head else (B, H, T, dk), dev)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (B, H, dk, dv), dev)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, H, T, dv), dev)
    hT = None
    if output_final_state:
        hT = final_state if final_state is not None else torch.empty(
            B, H, dk, dv, dtype=torch.float32, device=dev)
        _need(hT, "final_state", torch.float32, (B, H, dk, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    opts = GlaChunkOptions(segments=int(segments), dv_tile=int(dv_tile),
                           force_exact=1 if force_exact else 0, cta_pair=int(cta_pair),
                           gate_per_head=1 if per_head else 0)
    with torch.cuda.device(dev):
        st = _lib.lib().gla_chunk_fwd_ex(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), log_alpha.data_ptr(), float(scale),
            None if h0 is None else h0.data_ptr(), out.data_ptr(),
            None if hT is None else hT.data_ptr(), B, H, T, dk, dv, ctypes.byref(opts),
            _stream(dev))
    _lib.check(st, "gla_chunk_fwd")
    return out, hT


def gla_chunk_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         log_alpha: torch.Tensor, cu_seqlens, scale: float | None = None,
                         h0: torch.Tensor | None = None, output_final_state: bool = True, *,
                         out: torch.Tensor | None = None, final_state: torch.Tensor | None = None,
                         segments: int = 0, dv_tile: int = 0, force_exact: bool = False,
                         cta_pair: int = 0):
    """Chunkwise-parallel GLA forward over a packed batch of variable-length sequences.

    ``q``, ``k``, ``log_alpha`` are ``[H, T_total, dk]`` and ``v`` is
    ``[H, T_total, dv]`` (a leading batch dimension of 1 is accepted too);
    sequence ``n`` holds rows ``cu_seqlens[n] : cu_seqlens[n+1]`` of every head.
    ``cu_seqlens`` is a host sequence of ``N + 1`` ints (list, tuple or CPU
    tensor).  ``h0`` and the returned ``hT`` are ``[N, H, dk, dv]``.
    Returns ``(o, hT)`` with ``o`` shaped like ``v``.
    """
    squeeze = q.dim() == 4
    if squeeze:
        if q.shape[0] != 1:
            raise ValueError("a packed batch has a leading dimension of 1")
        q, k, v, log_alpha = q[0], k[0], v[0], log_alpha[0]
        if out is not None:
            out = out[0]
    if q.dim() != 3:
        raise ValueError("q must be [H, T_total, dk]")
    H, T_total, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be on a CUDA device")
    cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
    N = len(cu) - 1
    if N < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    _need(q, "q", torch.bfloat16, (H, T_total, dk), dev)
    _need(k, "k", torch.bfloat16, (H, T_total, dk), dev)
    _need(v, "v", torch.bfloat16, (H, T_total, dv), dev)
    _need(log_alpha, "log_alpha", torch.float32, (H, T_total, dk), dev)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (N, H, dk, dv), dev)
    if out is None:
        out = torch.empty(H, T_total, dv, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (H, T_total, dv), dev)
    hT = None
    if output_final_state:
        hT = final_state if final_state is not None else torch.empty(
            N, H, dk, dv, dtype=torch.float32, device=dev)
        _need(hT, "final_state", torch.float32, (N, H, dk, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    opts = GlaChunkOptions(segments=int(segments), dv_tile=int(dv_tile),
                           force_exact=1 if force_exact else 0, cta_pair=int(cta_pair))
    cu_arr = (ctypes.c_int * len(cu))(*cu)
    with torch.cuda.device(dev):
        st = _lib.lib().gla_chunk_fwd_varlen_ex(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), log_alpha.data_ptr(), float(scale),
            None if h0 is None else h0.data_ptr(), out.data_ptr(),
            None if hT is None else hT.data_ptr(), cu_arr, N, H, T_total, dk, dv,
            ctypes.byref(opts), _stream(dev))
    _lib.check(st, "gla_chunk_fwd_varlen")
    return (out.unsqueeze(0) if squeeze else out), hT


def gla_chunk_fwd_varlen_plan(cu_seqlens, H: int, dk: int, dv: int, *, segments: int = 0,
                              dv_tile: int = 0, force_exact: bool = False,
                              cta_pair: int = 0) -> dict:
    """The launch plan gla_chunk_fwd_varlen would use for this packed batch (no GPU work)."""
    cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
    opts = GlaChunkOptions(segments=int(segments), dv_tile=int(dv_tile),
                           force_exact=1 if force_exact else 0, cta_pair=int(cta_pair))
    nseg, tile, launches = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    sb = ctypes.c_ulong()
    st = _lib.lib().gla_chunk_fwd_varlen_plan((ctypes.c_int * len(cu))(*cu), len(cu) - 1, H,
                                               cu[-1], dk, dv, ctypes.byref(opts),
                                               ctypes.byref(nseg), ctypes.byref(tile),
                                               ctypes.byref(launches), ctypes.byref(sb))
    _lib.check(st, "gla_chunk_fwd_varlen_plan")
    return {"segments": nseg.value, "dv_tile": tile.value, "launches": launches.value,
            "scratch_bytes": sb.value}


def gla_chunk_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                       scale: float | None = None, h0: torch.Tensor | None = None,
                       output_final_state: bool = True, *, out: torch.Tensor | None = None,
                       final_state: torch.Tensor | None = None, device: int | None = None):
    """gla_chunk_fwd on CPU tensors, end to end (copies in, forward, copies out).

    The inputs are CPU tensors; pin them (``tensor.pin_memory()``) for the
    copies to overlap the computation.  The outputs are CPU tensors too;
    when not given, they are allocated pinned.  The work is enqueued on the
    current stream of ``device`` (default: the current CUDA device).  The
    results are valid once that stream has completed; call
    ``torch.cuda.synchronize`` or wait on an event before reading them.
    Returns ``(o, hT)``.
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, dk]")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cpu = torch.device("cpu")
    _need(q, "q", torch.bfloat16, (B, H, T, dk), cpu)
    _need(k, "k", torch.bfloat16, (B, H, T, dk), cpu)
    _need(v, "v", torch.bfloat16, (B, H, T, dv), cpu)
    _need(log_alpha, "log_alpha", torch.float32, (B, H, T, dk), cpu)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (B, H, dk, dv), cpu)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=torch.bfloat16, pin_memory=True)
    _need(out, "out", torch.bfloat16, (B, H, T, dv), cpu)
    hT = None
    if output_final_state:
        hT = final_state if final_state is not None else torch.empty(
            B, H, dk, dv, dtype=torch.float32, pin_memory=True)
        _need(hT, "final_state", torch.float32, (B, H, dk, dv), cpu)
    if scale is None:
        scale = dk ** -0.5
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    with torch.cuda.device(dev):
        st = _lib.lib().gla_chunk_fwd_host(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), log_alpha.data_ptr(), float(scale),
            None if h0 is None else h0.data_ptr(), out.data_ptr(),
            None if hT is None else hT.data_ptr(), B, H, T, dk, dv, _stream(dev))
    _lib.check(st, "gla_chunk_fwd_host")
    return out, hT


def gla_chunk_fwd_plan(B: int, H: int, T: int, dk: int, dv: int, *, segments: int = 0,
                       dv_tile: int = 0, force_exact: bool = False, cta_pair: int = 0) -> dict:
    """The launch plan gla_chunk_fwd would use on the current device (no GPU work)."""
    opts = GlaChunkOptions(segments=int(segments), dv_tile=int(dv_tile),
                           force_exact=1 if force_exact else 0, cta_pair=int(cta_pair))
    nseg, tile, launches = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    scratch = ctypes.c_ulong()
    st = _lib.lib().gla_chunk_fwd_plan(B, H, T, dk, dv, ctypes.byref(opts), ctypes.byref(nseg),
                                       ctypes.byref(tile), ctypes.byref(launches),
                                       ctypes.byref(scratch))
    _lib.check(st, "gla_chunk_fwd_plan")
    return {"segments": nseg.value, "dv_tile": tile.value, "launches": launches.value,
            "scratch_bytes": scratch.value}


def gla_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                  d_o: torch.Tensor, scale: float | None = None, h0: torch.Tensor | None = None,
                  dhT: torch.Tensor | None = None, *, need_dh0: bool = True,
                  force_exact: bool = False):
    """Gradients of L = sum <d_o, o> + <dhT, hT> through the chunked forward.

    Inputs as for ``gla_chunk_fwd`` (gates ``[B,H,T,dk]``, or ``[B,H,T]`` for one
    gate per token and head; ``dlog_alpha`` then has the same shape), with
    ``d_o`` ``[B,H,T,dv]`` bf16 and ``dhT`` ``[B,H,dk,dv]`` fp32 or None (zero).
    Returns ``(dq, dk, dv, dlog_alpha, dh0)``: bf16, bf16, bf16, fp32, and fp32
    or None when ``need_dh0`` is False.  The states are recomputed on the GPU.
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, dk]")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be on a CUDA device")
    _need(q, "q", torch.bfloat16, (B, H, T, dk), dev)
    _need(k, "k", torch.bfloat16, (B, H, T, dk), dev)
    _need(v, "v", torch.bfloat16, (B, H, T, dv), dev)
    per_head = log_alpha.dim() == 3
    _need(log_alpha, "log_alpha", torch.float32, (B, H, T) if per_head else (B, H, T, dk), dev)
    _need(d_o, "d_o", torch.bfloat16, (B, H, T, dv), dev)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (B, H, dk, dv), dev)
    if dhT is not None:
        _need(dhT, "dhT", torch.float32, (B, H, dk, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    dq = torch.empty_like(q)
    dkk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    da = torch.empty_like(log_alpha)
    dh0 = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) if need_dh0 else None
    opts = GlaChunkOptions(force_exact=1 if force_exact else 0, gate_per_head=1 if per_head else 0)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    with torch.cuda.device(dev):
        st = _lib.lib().gla_chunk_bwd_ex(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), log_alpha.data_ptr(), float(scale),
            ptr(h0), d_o.data_ptr(), ptr(dhT), dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(),
            da.data_ptr(), ptr(dh0), B, H, T, dk, dv, ctypes.byref(opts), _stream(dev))
    _lib.check(st, "gla_chunk_bwd")
    return dq, dkk, dvv, da, dh0


def gla_chunk_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         log_alpha: torch.Tensor, d_o: torch.Tensor, cu_seqlens,
                         scale: float | None = None, h0: torch.Tensor | None = None,
                         dhT: torch.Tensor | None = None, *, need_dh0: bool = True,
                         force_exact: bool = False):
    """Gradients of gla_chunk_fwd_varlen over a packed batch of sequences.

    ``q``, ``k``, ``log_alpha`` ``[H, T_total, dk]``; ``v``, ``d_o``
    ``[H, T_total, dv]``; ``h0``, ``dhT`` ``[N, H, dk, dv]`` or None (zero);
    ``cu_seqlens`` a host sequence of ``N + 1`` ints.  Returns
    ``(dq, dk, dv, dlog_alpha, dh0)`` shaped like their inputs (``dh0`` None
    when ``need_dh0`` is False).
    """
    if q.dim() != 3:
        raise ValueError("q must be [H, T_total, dk]")
    H, T_total, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be on a CUDA device")
    cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
    N = len(cu) - 1
    if N < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    _need(q, "q", torch.bfloat16, (H, T_total, dk), dev)
    _need(k, "k", torch.bfloat16, (H, T_total, dk), dev)
    _need(v, "v", torch.bfloat16, (H, T_total, dv), dev)
    _need(log_alpha, "log_alpha", torch.float32, (H, T_total, dk), dev)
    _need(d_o, "d_o", torch.bfloat16, (H, T_total, dv), dev)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (N, H, dk, dv), dev)
    if dhT is not None:
        _need(dhT, "dhT", torch.float32, (N, H, dk, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    dq, dkk, dvv, da = (torch.empty_like(t) for t in (q, k, v, log_alpha))
    dh0 = torch.empty(N, H, dk, dv, dtype=torch.float32, device=dev) if need_dh0 else None
    opts = GlaChunkOptions(force_exact=1 if force_exact else 0)
    cu_arr = (ctypes.c_int * len(cu))(*cu)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    with torch.cuda.device(dev):
        st = _lib.lib().gla_chunk_bwd_varlen_ex(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), log_alpha.data_ptr(), float(scale),
            ptr(h0), d_o.data_ptr(), ptr(dhT), dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(),
            da.data_ptr(), ptr(dh0), cu_arr, N, H, T_total, dk, dv, ctypes.byref(opts),
            _stream(dev))
    _lib.check(st, "gla_chunk_bwd_varlen")
    return dq, dkk, dvv, da, dh0


def gla_chunk_bwd_plan(B: int, H: int, T: int, dk: int, dv: int) -> dict:
    """Chunk length, launches and scratch bytes of gla_chunk_bwd for a shape (no GPU work)."""
    chunk, launches, scratch = ctypes.c_int(), ctypes.c_int(), ctypes.c_ulong()
    st = _lib.lib().gla_chunk_bwd_plan(B, H, T, dk, dv, ctypes.byref(chunk),
                                       ctypes.byref(launches), ctypes.byref(scratch))
    _lib.check(st, "gla_chunk_bwd_plan")
    return {"chunk": chunk.value, "launches": launches.value, "scratch_bytes": scratch.value}


class _GlaChunk(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, log_alpha, h0, scale):
        o, hT = gla_chunk_fwd(q, k, v, log_alpha, scale, h0)
        ctx.save_for_backward(q, k, v, log_alpha, h0)
        ctx.scale = scale
        return o, hT

    @staticmethod
    def backward(ctx, d_o, dhT):
        q, k, v, log_alpha, h0 = ctx.saved_tensors
        if d_o is None:
            d_o = torch.zeros(*q.shape[:-1], v.shape[-1], dtype=torch.bfloat16, device=q.device)
        d_o = d_o.to(torch.bfloat16).contiguous()
        dhT = None if dhT is None else dhT.float().contiguous()
        dq, dk, dv, da, dh0 = gla_chunk_bwd(q, k, v, log_alpha, d_o, ctx.scale, h0, dhT,
                                            need_dh0=h0 is not None and ctx.needs_input_grad[4])
        return dq, dk, dv, da, dh0, None


def gla_chunk(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
              scale: float | None = None, h0: torch.Tensor | None = None):
    """Differentiable chunked GLA: ``(o, hT)`` with gradients through ``gla_chunk_bwd``.

    Gates ``[B,H,T,dk]`` or ``[B,H,T]``.  The backward recomputes the states
    from the saved inputs; ``d_o`` is taken in bf16, ``dhT`` in fp32.
    """
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return _GlaChunk.apply(q, k, v, log_alpha, h0, float(scale))


class _GlaChunkVarlen(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, log_alpha, h0, cu, scale):
        o, hT = gla_chunk_fwd_varlen(q, k, v, log_alpha, cu, scale, h0)
        ctx.save_for_backward(q, k, v, log_alpha, h0)
        ctx.cu, ctx.scale = cu, scale
        return o, hT

    @staticmethod
    def backward(ctx, d_o, dhT):
        q, k, v, log_alpha, h0 = ctx.saved_tensors
        if d_o is None:
            d_o = torch.zeros(*q.shape[:-1], v.shape[-1], dtype=torch.bfloat16, device=q.device)
        d_o = d_o.to(torch.bfloat16).contiguous()
        dhT = None if dhT is None else dhT.float().contiguous()
        dq, dk, dv, da, dh0 = gla_chunk_bwd_varlen(
            q, k, v, log_alpha, d_o, ctx.cu, ctx.scale, h0, dhT,
            need_dh0=h0 is not None and ctx.needs_input_grad[4])
        return dq, dk, dv, da, dh0, None, None


def gla_chunk_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                     cu_seqlens, scale: float | None = None, h0: torch.Tensor | None = None):
    """Differentiable packed-batch GLA: ``(o, hT)`` of ``gla_chunk_fwd_varlen`` with gradients
    through ``gla_chunk_bwd_varlen``.  ``q`` etc. are ``[H, T_total, .]``; ``h0`` is
    ``[N, H, dk, dv]`` or None."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    cu = [int(x) for x in (cu_seqlens.tolist() if torch.is_tensor(cu_seqlens) else cu_seqlens)]
    return _GlaChunkVarlen.apply(q, k, v, log_alpha, h0, cu, float(scale))


def gla_gdn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                beta: torch.Tensor, scale: float | None = None, h0: torch.Tensor | None = None,
                output_final_state: bool = True, chunked: bool = False):
    """Gated delta rule (Gated DeltaNet) forward: ``(o, hT)``.

    q, k ``[B,H,T,dk]`` bf16 (k as given: normalise it first); v ``[B,H,T,dv]``
    bf16; g (log alpha) and beta ``[B,H,T]`` fp32; h0 ``[B,H,dk,dv]`` fp32 or None.
    ``chunked=True`` calls gla_gdn_chunk_fwd (the chunk algorithm on the tensor
    cores, dk = 128), else gla_gdn_fwd (token-recurrent).
    """
    if q.dim() != 4:
        raise ValueError("q must be [B, H, T, dk]")
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q must be on a CUDA device")
    _need(q, "q", torch.bfloat16, (B, H, T, dk), dev)
    _need(k, "k", torch.bfloat16, (B, H, T, dk), dev)
    _need(v, "v", torch.bfloat16, (B, H, T, dv), dev)
    _need(g, "g", torch.float32, (B, H, T), dev)
    _need(beta, "beta", torch.float32, (B, H, T), dev)
    if h0 is not None:
        _need(h0, "h0", torch.float32, (B, H, dk, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    o = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev) if output_final_state else None
    with torch.cuda.device(dev):
        fn = _lib.lib().gla_gdn_chunk_fwd if chunked else _lib.lib().gla_gdn_fwd
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                float(scale), None if h0 is None else h0.data_ptr(), o.data_ptr(),
                None if hT is None else hT.data_ptr(), B, H, T, dk, dv, _stream(dev))
    _lib.check(st, "gla_gdn_chunk_fwd" if chunked else "gla_gdn_fwd")
    return o, hT


def gla_recurrent_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, log_alpha: torch.Tensor,
                       h: torch.Tensor, scale: float | None = None, *,
                       out: torch.Tensor | None = None) -> torch.Tensor:
    """One decode token for every (batch, head): ``h`` is updated in place, returns o.

    q, k, log_alpha: ``[B,H,dk]``; v: ``[B,H,dv]``; h: ``[B,H,dk,dv]`` fp32.
    """
    if h.dim() != 4:
        raise ValueError("h must be [B, H, dk, dv]")
    B, H, dk, dv = h.shape
    dev = h.device
    if dev.type != "cuda":
        raise ValueError("h must be on a CUDA device")
    _need(h, "h", torch.float32, (B, H, dk, dv), dev)
    _need(q, "q", torch.bfloat16, (B, H, dk), dev)
    _need(k, "k", torch.bfloat16, (B, H, dk), dev)
    _need(v, "v", torch.bfloat16, (B, H, dv), dev)
    _need(log_alpha, "log_alpha", torch.float32, (B, H, dk), dev)
    if out is None:
        out = torch.empty(B, H, dv, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (B, H, dv), dev)
    if scale is None:
        scale = dk ** -0.5
    with torch.cuda.device(dev):
        st = _lib.lib().gla_recurrent_step(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           log_alpha.data_ptr(), float(scale), h.data_ptr(),
                                           out.data_ptr(), B, H, dk, dv, _stream(dev))
    _lib.check(st, "gla_recurrent_step")
    return out


def gla_last_device_status(device: torch.device | int | None = None) -> int:
    """Synchronise the current stream and read/clear the library's device status word."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else
                       (device if isinstance(device, int) else device.index))
    with torch.cuda.device(dev):
        return int(_lib.lib().gla_last_device_status(_stream(dev)))
