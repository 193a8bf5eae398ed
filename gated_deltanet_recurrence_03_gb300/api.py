"""PyTorch-facing binding of libgdn: argument marshalling only.

Each function checks shapes and dtypes, allocates the outputs (and the scratch
workspace) with PyTorch, and calls the C ABI entry point of the same name on the
current (or given) CUDA stream.  Every step of the recurrence runs in libgdn's
CUDA kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib as L

_DTYPES = {torch.float32: L.GDN_F32, torch.bfloat16: L.GDN_BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(name, t, dtype, device, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def _opts(lib, dtype, scale, chunk, normalize_qk, stream, device, events, raw_gates=None, Hv=None,
          output_gate=None, out_shape=None):
    o = L.default_opts(lib)
    o.dtype = _DTYPES[dtype]
    o.chunk = int(chunk)
    o.scale = float(scale)
    o.flags = L.GDN_NORMALIZE_QK if normalize_qk else 0
    if raw_gates is not None:
        A_log, dt_bias = raw_gates
        _need("A_log", A_log, torch.float32, device, (Hv,))
        _need("dt_bias", dt_bias, torch.float32, device, (Hv,))
        o.flags |= L.GDN_RAW_GATES
        o.A_log = A_log.data_ptr()
        o.dt_bias = dt_bias.data_ptr()
    if output_gate is not None:
        z, weight, eps = output_gate
        _need("z", z, dtype, device, out_shape)
        _need("norm_weight", weight, torch.float32, device, (out_shape[-1],))
        o.flags |= L.GDN_OUTPUT_GATE
        o.z = z.data_ptr()
        o.norm_weight = weight.data_ptr()
        o.norm_eps = float(eps)
    o.stream = _stream_handle(stream, device)
    keep = None
    if events:
        keep = (ctypes.c_void_p * len(events))(*[int(e) for e in events])
        o.events = ctypes.cast(keep, ctypes.POINTER(ctypes.c_void_p))
        o.num_events = len(events)
    return o, keep


def workspace_size(B: int, T: int, Hqk: int, Hv: int, dk: int, dv: int, *, dtype=torch.bfloat16,
                   chunk: int = 64, num_seqs: Optional[int] = None) -> int:
    """Bytes of device scratch gdn_chunk_fwd needs (0 when the selected kernel needs none)."""
    lib = L.load()
    o = L.default_opts(lib)
    o.dtype = _DTYPES[dtype]
    o.chunk = int(chunk)
    if num_seqs is not None:
        o.cu_seqlens = 16  # any non-null value marks the call as packed for the size query
        o.num_seqs = int(num_seqs)
    return int(lib.gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, ctypes.byref(o)))


def gdn_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  S0: Optional[torch.Tensor] = None, *, scale: float = 1.0, chunk: int = 64,
                  normalize_qk: bool = False, cu_seqlens: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, S_final: Optional[torch.Tensor] = None,
                  output_final_state: bool = True, workspace: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None, events: Optional[Sequence[int]] = None,
                  raw_gates=None, output_gate=None):
    """Chunked prefill.  q, k [B, T, Hqk, dk]; v [B, T, Hv, dv]; g, beta [B, T, Hv] (all bf16 or all
    fp32, on one CUDA device); S0 [nseq, Hv, dk, dv] fp32 or None.  With ``cu_seqlens`` (int32 device
    tensor of nseq+1 offsets) B must be 1.  With ``raw_gates=(A_log, dt_bias)`` (fp32 [Hv] each), g and
    beta are the raw projections a and b and the kernels form the gates.  With
    ``output_gate=(z, norm_weight, eps)`` (z like out, norm_weight fp32 [dv]) the outputs pass through
    RMSNorm * norm_weight * silu(z).  Returns (out [B, T, Hv, dv], S_final or None)."""
    lib = L.load()
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, T, H, d]")
    B, T, Hqk, dk = q.shape
    Hv, dv = int(v.shape[2]), int(v.shape[3])
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    _need("q", q, dt, dev, (B, T, Hqk, dk))
    _need("k", k, dt, dev, (B, T, Hqk, dk))
    _need("v", v, dt, dev, (B, T, Hv, dv))
    _need("g", g, dt, dev, (B, T, Hv))
    _need("beta", beta, dt, dev, (B, T, Hv))
    nseq = B
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1:
            raise ValueError("cu_seqlens must be 1-D")
        nseq = int(cu_seqlens.numel()) - 1
        _need("cu_seqlens", cu_seqlens, torch.int32, dev, (nseq + 1,))
    if S0 is not None:
        _need("S0", S0, torch.float32, dev, (nseq, Hv, dk, dv))
    if out is None:
        out = torch.empty_like(v)
    _need("out", out, dt, dev, (B, T, Hv, dv))
    if S_final is None and output_final_state:
        S_final = torch.empty((nseq, Hv, dk, dv), dtype=torch.float32, device=dev)
    if S_final is not None:
        _need("S_final", S_final, torch.float32, dev, (nseq, Hv, dk, dv))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, scale, chunk, normalize_qk, stream, dev, events, raw_gates, Hv,
                        output_gate, (B, T, Hv, dv))
        if cu_seqlens is not None:
            o.cu_seqlens = cu_seqlens.data_ptr()
            o.num_seqs = nseq
        need = int(lib.gdn_chunk_fwd_workspace_size(B, T, Hqk, Hv, dk, dv, ctypes.byref(o)))
        if need:
            if workspace is None or workspace.numel() * workspace.element_size() < need:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
            o.workspace = workspace.data_ptr()
            o.workspace_bytes = workspace.numel() * workspace.element_size()
        st = lib.gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(out),
                               _ptr(S_final), B, T, Hqk, Hv, dk, dv, ctypes.byref(o))
        del keep
        L.check(lib, st)
    return out, S_final


def gdn_recurrent_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                       S: torch.Tensor, *, scale: float = 1.0, normalize_qk: bool = False,
                       out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                       events: Optional[Sequence[int]] = None, raw_gates=None,
                       output_gate=None) -> torch.Tensor:
    """One decode step.  q, k [N, Hqk, dk]; v [N, Hv, dv]; g, beta [N, Hv]; S [N, Hv, dk, dv] fp32 is
    updated in place.  ``raw_gates`` and ``output_gate`` as for gdn_chunk_fwd.  Returns out [N, Hv, dv]."""
    lib = L.load()
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be 3-D [N, H, d]")
    N, Hqk, dk = q.shape
    Hv, dv = int(v.shape[1]), int(v.shape[2])
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    _need("q", q, dt, dev, (N, Hqk, dk))
    _need("k", k, dt, dev, (N, Hqk, dk))
    _need("v", v, dt, dev, (N, Hv, dv))
    _need("g", g, dt, dev, (N, Hv))
    _need("beta", beta, dt, dev, (N, Hv))
    _need("S", S, torch.float32, dev, (N, Hv, dk, dv))
    if out is None:
        out = torch.empty_like(v)
    _need("out", out, dt, dev, (N, Hv, dv))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, scale, 64, normalize_qk, stream, dev, events, raw_gates, Hv,
                        output_gate, (N, Hv, dv))
        st = lib.gdn_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S), _ptr(out),
                                    N, Hqk, Hv, dk, dv, ctypes.byref(o))
        del keep
        L.check(lib, st)
    return out


def check_device_status(stream: Optional[torch.cuda.Stream] = None, device=None) -> None:
    """Synchronise and raise GdnError if a kernel reported a bounded wait that ran out."""
    lib = L.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        L.check(lib, lib.gdn_check_device_status(_stream_handle(stream, dev)))


def version() -> int:
    return int(L.load().gdn_version())


def gdn_causal_conv1d_fwd(x: torch.Tensor, w: torch.Tensor, cache_in: Optional[torch.Tensor] = None, *,
                          cu_seqlens: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                          cache_out: Optional[torch.Tensor] = None, return_cache: bool = True, stream: Optional[torch.cuda.Stream] = None,
                          events: Optional[Sequence[int]] = None):
    """Depthwise causal convolution + SiLU.  x [B, T, C] (bf16 or fp32; may be a channel slice of a
    wider tensor: rows must be evenly strided with the channels contiguous); w [C, K] fp32;
    cache_in [nseq, K-1, C] or None.  ``cache_out`` (or a new tensor when ``return_cache``) receives each
    sequence's last K-1 inputs.  Returns (y [B, T, C], cache_out [nseq, K-1, C] or None)."""
    lib = L.load()
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(0) != x.shape[1] * x.stride(1):
        raise ValueError("x must be [B, T, C] with contiguous channels and evenly strided token rows")
    B, T, C = x.shape
    dev, dt = x.device, x.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    K = int(w.shape[1])
    _need("w", w, torch.float32, dev, (C, K))
    nseq = B
    if cu_seqlens is not None:
        nseq = int(cu_seqlens.numel()) - 1
        _need("cu_seqlens", cu_seqlens, torch.int32, dev, (nseq + 1,))
    if cache_in is not None:
        _need("cache_in", cache_in, dt, dev, (nseq, K - 1, C))
    if out is None:
        out = torch.empty((B, T, C), dtype=dt, device=dev)
    _need("out", out, dt, dev, (B, T, C))
    if cache_out is None and return_cache:
        cache_out = torch.empty((nseq, K - 1, C), dtype=dt, device=dev)
    if cache_out is not None:
        _need("cache_out", cache_out, dt, dev, (nseq, K - 1, C))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, events)
        if cu_seqlens is not None:
            o.cu_seqlens = cu_seqlens.data_ptr()
            o.num_seqs = nseq
        st = lib.gdn_causal_conv1d_fwd(_ptr(x), x.stride(1), _ptr(w), _ptr(cache_in), _ptr(out), _ptr(cache_out),
                                       B, T, C, K, ctypes.byref(o))
        del keep
        L.check(lib, st)
    return out, cache_out


def gdn_causal_conv1d_bwd(x: torch.Tensor, w: torch.Tensor, grad_y: torch.Tensor, cache_in: Optional[torch.Tensor] = None,
                          *, grad_cache_out: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None,
                          want_grad_w: bool = True, want_grad_cache_in: bool = True,
                          stream: Optional[torch.cuda.Stream] = None, events: Optional[Sequence[int]] = None):
    """Gradients through gdn_causal_conv1d_fwd: x, w, cache_in as there; grad_y [B, T, C] like x (dense);
    grad_cache_out [nseq, K-1, C] like x or None.  Returns fp32 (grad_x [B, T, C], grad_w [C, K] or None,
    grad_cache_in [nseq, K-1, C] or None)."""
    lib = L.load()
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(0) != x.shape[1] * x.stride(1):
        raise ValueError("x must be [B, T, C] with contiguous channels and evenly strided token rows")
    B, T, C = x.shape
    dev, dt = x.device, x.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    K = int(w.shape[1])
    _need("w", w, torch.float32, dev, (C, K))
    _need("grad_y", grad_y, dt, dev, (B, T, C))
    nseq = B
    if cu_seqlens is not None:
        nseq = int(cu_seqlens.numel()) - 1
        _need("cu_seqlens", cu_seqlens, torch.int32, dev, (nseq + 1,))
    if cache_in is not None:
        _need("cache_in", cache_in, dt, dev, (nseq, K - 1, C))
    if grad_cache_out is not None:
        _need("grad_cache_out", grad_cache_out, dt, dev, (nseq, K - 1, C))
    f32 = dict(dtype=torch.float32, device=dev)
    gx = torch.empty((B, T, C), **f32)
    gw = torch.empty((C, K), **f32) if want_grad_w else None
    gc = torch.empty((nseq, K - 1, C), **f32) if want_grad_cache_in and K > 1 else None
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, events)
        if cu_seqlens is not None:
            o.cu_seqlens = cu_seqlens.data_ptr()
            o.num_seqs = nseq
        ws = None
        if want_grad_w:
            need = int(lib.gdn_causal_conv1d_bwd_workspace_size(B, T, C, K, ctypes.byref(o)))
            ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
            o.workspace, o.workspace_bytes = ws.data_ptr(), ws.numel()
        st = lib.gdn_causal_conv1d_bwd(_ptr(x), x.stride(1), _ptr(w), _ptr(cache_in), _ptr(grad_y),
                                       _ptr(grad_cache_out), _ptr(gx), _ptr(gw), _ptr(gc), B, T, C, K,
                                       ctypes.byref(o))
        del keep
        L.check(lib, st)
    return gx, gw, gc


def gdn_causal_conv1d_step(x: torch.Tensor, w: torch.Tensor, cache: torch.Tensor, *,
                           out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
                           events: Optional[Sequence[int]] = None) -> torch.Tensor:
    """One decode token per sequence: x [N, C] (channels contiguous, rows evenly strided), w [C, K] fp32,
    cache [N, K-1, C] updated in place.  Returns y [N, C]."""
    lib = L.load()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [N, C] with contiguous channels")
    N, C = x.shape
    dev, dt = x.device, x.dtype
    K = int(w.shape[1])
    _need("w", w, torch.float32, dev, (C, K))
    _need("cache", cache, dt, dev, (N, K - 1, C))
    if out is None:
        out = torch.empty((N, C), dtype=dt, device=dev)
    _need("out", out, dt, dev, (N, C))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, events)
        st = lib.gdn_causal_conv1d_step(_ptr(x), x.stride(0), _ptr(w), _ptr(cache), _ptr(out), N, C, K,
                                        ctypes.byref(o))
        del keep
        L.check(lib, st)
    return out


def gdn_causal_conv1d_fwd_qkv(x: torch.Tensor, w: torch.Tensor, widths: Sequence[int],
                              cache_in: Optional[torch.Tensor] = None, *, cu_seqlens: Optional[torch.Tensor] = None,
                              out: Optional[Sequence[torch.Tensor]] = None, cache_out: Optional[torch.Tensor] = None,
                              return_cache: bool = True, stream: Optional[torch.cuda.Stream] = None,
                              events: Optional[Sequence[int]] = None):
    """The convolution of gdn_causal_conv1d_fwd over the packed q | k | v projection x [B, T, Cq + Ck + Cv]
    in one launch, the three channel ranges (``widths`` = (Cq, Ck, Cv)) written to three dense tensors.
    Returns ((y_q, y_k, y_v), cache_out [nseq, K-1, C] or None)."""
    lib = L.load()
    if x.dim() != 3 or x.stride(2) != 1 or x.stride(0) != x.shape[1] * x.stride(1):
        raise ValueError("x must be [B, T, C] with contiguous channels and evenly strided token rows")
    B, T, C = x.shape
    Cq, Ck, Cv = (int(c) for c in widths)
    if Cq + Ck + Cv != C:
        raise ValueError(f"widths {widths} do not add up to the {C} channels of x")
    dev, dt = x.device, x.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    K = int(w.shape[1])
    _need("w", w, torch.float32, dev, (C, K))
    nseq = B
    if cu_seqlens is not None:
        nseq = int(cu_seqlens.numel()) - 1
        _need("cu_seqlens", cu_seqlens, torch.int32, dev, (nseq + 1,))
    if cache_in is not None:
        _need("cache_in", cache_in, dt, dev, (nseq, K - 1, C))
    if out is None:
        out = tuple(torch.empty((B, T, c), dtype=dt, device=dev) for c in (Cq, Ck, Cv))
    for name, y, c in zip(("y_q", "y_k", "y_v"), out, (Cq, Ck, Cv)):
        _need(name, y, dt, dev, (B, T, c))
    if cache_out is None and return_cache:
        cache_out = torch.empty((nseq, K - 1, C), dtype=dt, device=dev)
    if cache_out is not None:
        _need("cache_out", cache_out, dt, dev, (nseq, K - 1, C))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, events)
        if cu_seqlens is not None:
            o.cu_seqlens = cu_seqlens.data_ptr()
            o.num_seqs = nseq
        st = lib.gdn_causal_conv1d_fwd_qkv(_ptr(x), x.stride(1), _ptr(w), _ptr(cache_in), _ptr(out[0]), _ptr(out[1]),
                                           _ptr(out[2]), _ptr(cache_out), B, T, Cq, Ck, Cv, K, ctypes.byref(o))
        del keep
        L.check(lib, st)
    return tuple(out), cache_out


def gdn_causal_conv1d_step_qkv(x: torch.Tensor, w: torch.Tensor, cache: torch.Tensor, widths: Sequence[int], *,
                               out: Optional[Sequence[torch.Tensor]] = None,
                               stream: Optional[torch.cuda.Stream] = None,
                               events: Optional[Sequence[int]] = None):
    """One decode token per sequence through the convolution of the packed q | k | v projection
    x [N, Cq + Ck + Cv] (``widths`` = (Cq, Ck, Cv)), cache [N, K-1, C] updated in place, in one launch.
    Returns (y_q [N, Cq], y_k [N, Ck], y_v [N, Cv])."""
    lib = L.load()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [N, C] with contiguous channels")
    N, C = x.shape
    Cq, Ck, Cv = (int(c) for c in widths)
    if Cq + Ck + Cv != C:
        raise ValueError(f"widths {widths} do not add up to the {C} channels of x")
    dev, dt = x.device, x.dtype
    K = int(w.shape[1])
    _need("w", w, torch.float32, dev, (C, K))
    _need("cache", cache, dt, dev, (N, K - 1, C))
    if out is None:
        out = tuple(torch.empty((N, c), dtype=dt, device=dev) for c in (Cq, Ck, Cv))
    for name, y, c in zip(("y_q", "y_k", "y_v"), out, (Cq, Ck, Cv)):
        _need(name, y, dt, dev, (N, c))
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, events)
        st = lib.gdn_causal_conv1d_step_qkv(_ptr(x), x.stride(0), _ptr(w), _ptr(cache), _ptr(out[0]), _ptr(out[1]),
                                            _ptr(out[2]), N, Cq, Ck, Cv, K, ctypes.byref(o))
        del keep
        L.check(lib, st)
    return tuple(out)


def backward_workspace_size(B: int, T: int, Hqk: int, Hv: int, dk: int, dv: int, *,
                            num_seqs: Optional[int] = None, front_end: bool = False) -> int:
    """Bytes of device scratch gdn_recurrent_bwd needs (with ``front_end``: through the l2 norm and / or
    the raw gates)."""
    lib = L.load()
    o = L.default_opts(lib)
    if front_end:
        o.flags = L.GDN_NORMALIZE_QK
    if num_seqs is not None:
        o.cu_seqlens = 1   # only tested for NULL
        o.num_seqs = int(num_seqs)
    return int(lib.gdn_recurrent_bwd_workspace_size(B, T, Hqk, Hv, dk, dv, ctypes.byref(o)))


def gdn_recurrent_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                      S0: Optional[torch.Tensor], grad_out: torch.Tensor, grad_S_final: Optional[torch.Tensor] = None,
                      *, scale: float = 1.0, cu_seqlens: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, want_grad_S0: bool = True,
                      stream: Optional[torch.cuda.Stream] = None, events: Optional[Sequence[int]] = None,
                      normalize_qk: bool = False, raw_gates=None):
    """Gradients of a loss on (out, S_final) of gdn_chunk_fwd with respect to q, k, v, g, beta, S0.
    Inputs as for gdn_chunk_fwd; grad_out like v; grad_S_final fp32 like S_final or None.  Returns fp32
    (grad_q, grad_k, grad_v, grad_g, grad_beta, grad_S0 or None).  With normalize_qk and / or
    raw_gates=(A_log, dt_bias) (g and beta then hold the raw projections a and b) the gradients are
    those of the forward with the same front end, with respect to its raw inputs, and two more tensors
    are returned with raw_gates: grad_A_log, grad_dt_bias (fp32 [Hv])."""
    lib = L.load()
    if q.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, T, H, d]")
    B, T, Hqk, dk = q.shape
    Hv, dv = int(v.shape[2]), int(v.shape[3])
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    _need("q", q, dt, dev, (B, T, Hqk, dk))
    _need("k", k, dt, dev, (B, T, Hqk, dk))
    _need("v", v, dt, dev, (B, T, Hv, dv))
    _need("g", g, dt, dev, (B, T, Hv))
    _need("beta", beta, dt, dev, (B, T, Hv))
    _need("grad_out", grad_out, dt, dev, (B, T, Hv, dv))
    nseq = B
    if cu_seqlens is not None:
        nseq = int(cu_seqlens.numel()) - 1
        _need("cu_seqlens", cu_seqlens, torch.int32, dev, (nseq + 1,))
    if S0 is not None:
        _need("S0", S0, torch.float32, dev, (nseq, Hv, dk, dv))
    if grad_S_final is not None:
        _need("grad_S_final", grad_S_final, torch.float32, dev, (nseq, Hv, dk, dv))
    f32 = dict(dtype=torch.float32, device=dev)
    gq, gk = torch.empty((B, T, Hqk, dk), **f32), torch.empty((B, T, Hqk, dk), **f32)
    gv = torch.empty((B, T, Hv, dv), **f32)
    gg, gb = torch.empty((B, T, Hv), **f32), torch.empty((B, T, Hv), **f32)
    gS0 = torch.empty((nseq, Hv, dk, dv), **f32) if want_grad_S0 else None
    gA = gdt = None
    with torch.cuda.device(dev):
        o, keep = _opts(lib, dt, scale, 64, normalize_qk, stream, dev, events)
        if cu_seqlens is not None:
            o.cu_seqlens = cu_seqlens.data_ptr()
            o.num_seqs = nseq
        if raw_gates is not None:
            A_log, dt_bias = raw_gates
            _need("A_log", A_log, torch.float32, dev, (Hv,))
            _need("dt_bias", dt_bias, torch.float32, dev, (Hv,))
            gA, gdt = torch.empty((Hv,), **f32), torch.empty((Hv,), **f32)
            o.flags |= L.GDN_RAW_GATES
            o.A_log, o.dt_bias = A_log.data_ptr(), dt_bias.data_ptr()
            o.grad_A_log, o.grad_dt_bias = gA.data_ptr(), gdt.data_ptr()
        need = int(lib.gdn_recurrent_bwd_workspace_size(B, T, Hqk, Hv, dk, dv, ctypes.byref(o)))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel()
        st = lib.gdn_recurrent_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(grad_out),
                                   _ptr(grad_S_final), _ptr(gq), _ptr(gk), _ptr(gv), _ptr(gg), _ptr(gb), _ptr(gS0),
                                   B, T, Hqk, Hv, dk, dv, ctypes.byref(o))
        del keep
        L.check(lib, st)
    if raw_gates is not None:
        return gq, gk, gv, gg, gb, gS0, gA, gdt
    return gq, gk, gv, gg, gb, gS0


def gdn_output_gate_fwd(o: torch.Tensor, z: torch.Tensor, norm_weight: torch.Tensor, eps: float = 1e-6, *,
                        out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """The shell's output gate on its own: o / sqrt(mean(o^2) + eps) * norm_weight * silu(z) over the last
    axis (dv of 32, 64 or 128).  o, z [..., dv] (bf16 or fp32, contiguous); out like o (may be o)."""
    lib = L.load()
    dev, dt = o.device, o.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    dv = int(o.shape[-1])
    _need("z", z, dt, dev, tuple(o.shape))
    _need("norm_weight", norm_weight, torch.float32, dev, (dv,))
    if not o.is_contiguous():
        raise ValueError("o must be contiguous")
    y = torch.empty_like(o) if out is None else out
    _need("out", y, dt, dev, tuple(o.shape))
    with torch.cuda.device(dev):
        op, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, None)
        op.norm_eps = float(eps)
        st = lib.gdn_output_gate_fwd(_ptr(o), _ptr(z), _ptr(norm_weight), _ptr(y), o.numel() // dv, dv,
                                     ctypes.byref(op))
        del keep
        L.check(lib, st)
    return y


def gdn_output_gate_bwd(o: torch.Tensor, z: torch.Tensor, norm_weight: torch.Tensor, grad_y: torch.Tensor,
                        eps: float = 1e-6, *, stream: Optional[torch.cuda.Stream] = None):
    """Gradients through gdn_output_gate_fwd: returns fp32 (grad_o, grad_z like o, grad_norm_weight [dv])."""
    lib = L.load()
    dev, dt = o.device, o.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}")
    dv = int(o.shape[-1])
    _need("z", z, dt, dev, tuple(o.shape))
    _need("grad_y", grad_y, dt, dev, tuple(o.shape))
    _need("norm_weight", norm_weight, torch.float32, dev, (dv,))
    rows = o.numel() // dv
    f32 = dict(dtype=torch.float32, device=dev)
    go, gz, gw = torch.empty(tuple(o.shape), **f32), torch.empty(tuple(o.shape), **f32), torch.empty((dv,), **f32)
    with torch.cuda.device(dev):
        op, keep = _opts(lib, dt, 1.0, 64, False, stream, dev, None)
        op.norm_eps = float(eps)
        need = int(lib.gdn_output_gate_bwd_workspace_size(rows, dv, ctypes.byref(op)))
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        op.workspace, op.workspace_bytes = ws.data_ptr(), ws.numel()
        st = lib.gdn_output_gate_bwd(_ptr(o), _ptr(z), _ptr(norm_weight), _ptr(grad_y), _ptr(go), _ptr(gz),
                                     _ptr(gw), rows, dv, ctypes.byref(op))
        del keep
        L.check(lib, st)
    return go, gz, gw
