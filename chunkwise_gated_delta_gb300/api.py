"""Python binding of the C ABI: argument marshalling only.

Every step of the computation runs in the CUDA library (``libkda.so``); this
module only turns torch tensors into pointers and sizes, picks the current
stream and keeps a zero-filled workspace per device and stream.  There is no CPU path:
when the library is missing, :func:`_lib.load` raises.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import KdaError

_GATES = {"none": _lib.KDA_GATE_NONE, "scalar": _lib.KDA_GATE_SCALAR, "channel": _lib.KDA_GATE_CHANNEL}
_workspaces: dict = {}
_MAX_WORKSPACES = 16   # cached (device, stream) workspaces; callers that make many streams evict the oldest


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.KDA_BF16
    if t.dtype == torch.float32:
        return _lib.KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_for(device, nbytes: int, stream=None) -> torch.Tensor:
    """A cached, zero-filled workspace of at least ``nbytes`` for calls on ``stream``
    (default: the current stream of ``device``).

    One per (device, stream): calls on different streams may run at the same time on
    the GPU, and two such calls must not share chunk records or a status block.  The
    workspace is allocated on its stream, so a replaced one goes back to the
    allocator in that stream's order.
    """
    dev = torch.device(device)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    if stream is None:
        stream = torch.cuda.current_stream(idx)
    key = (idx, stream.cuda_stream)
    ws = _workspaces.pop(key, None)
    if ws is None or ws.numel() < nbytes:
        with torch.cuda.stream(stream):
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=torch.device("cuda", idx))
    _workspaces[key] = ws                  # most recently used last
    while len(_workspaces) > _MAX_WORKSPACES:
        # the least recently used goes back to the allocator, in its own stream's order
        _workspaces.pop(next(iter(_workspaces)))
    return ws


def make_args(q, k, v, g=None, beta=None, h0=None, o=None, ht=None, *, gate=None, scale_v=True,
              workspace=None, cu_seqlens=None) -> _lib.KdaFwdArgs:
    """Fill the C argument struct from tensors (no validation beyond the C side's).

    With ``cu_seqlens`` (int32 device tensor [N + 1]) the batch is packed:
    q is [1, T, H, dk] and B is the number of sequences N.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
    if gate is None:
        gate = "none" if g is None else ("scalar" if g.dim() == 3 else "channel")
    a = _lib.KdaFwdArgs()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = B, T, H, dk, dv, 64
    a.dtype = _dtype_code(q)
    a.gate_kind = _GATES[gate]
    a.g_dtype = _dtype_code(g) if g is not None else _lib.KDA_BF16
    a.flags = _lib.KDA_FLAG_BETA_SCALES_V if scale_v else 0
    a.q, a.k, a.v, a.g, a.beta = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta)
    a.h0, a.o, a.ht = _ptr(h0), _ptr(o), _ptr(ht)
    a.cu_seqlens = _ptr(cu_seqlens)
    if workspace is not None:
        a.workspace = _ptr(workspace)
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    return a


def kda_chunk_fwd(q, k, v, g=None, beta=None, h0=None, *, gate=None, scale_v=True,
                  output_final_state=True, o=None, ht=None, workspace=None, stream=None, cu_seqlens=None):
    """Chunkwise gated delta-rule forward through ``kda_chunk_fwd`` of the C ABI.

    q, k: [B, T, H, dk]; v: [B, T, H, dv] (bf16 or fp32, same dtype);
    g: log-decay [B, T, H, dk] (per channel), [B, T, H] (scalar) or None;
    beta: [B, T, H] in the dtype of q, or None (beta = 0);
    h0: [B, H, dv, dk] fp32 or None.
    cu_seqlens: int32 CUDA tensor [N + 1] for a packed batch of N sequences
    (then q is [1, T, H, dk], h0 / ht are [N, H, dv, dk]), or None.
    Returns (o [B, T, H, dv] in q's dtype, ht [B, H, dv, dk] fp32 or None).
    """
    lib = _lib.load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (h0, "h0"),
                    (cu_seqlens, "cu_seqlens")):
        _check(t, name)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if ht is None and output_final_state:
        ht = torch.empty(nseq, H, dv, dk, dtype=torch.float32, device=q.device)
    args = make_args(q, k, v, g, beta, h0, o, ht, gate=gate, scale_v=scale_v, cu_seqlens=cu_seqlens)
    need = lib.kda_chunk_fwd_workspace(ctypes.byref(args))
    if need == 0:
        # invalid arguments: let the launch entry point report which status
        rc = lib.kda_chunk_fwd(ctypes.byref(args), None)
        raise KdaError(rc if rc != 0 else _lib.KDA_ERR_INVALID_ARG, "kda_chunk_fwd")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kda_chunk_fwd(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd")
    return o, ht


def kda_chunk_fwd_noalloc(q, k, v, g=None, beta=None, h0=None, *, gate=None, scale_v=True,
                          output_final_state=True, o=None, ht=None, stream=None, cu_seqlens=None):
    """``kda_chunk_fwd_noalloc`` of the C ABI: the forward without a workspace.

    For callers that cannot allocate device memory at the call (an allocator
    that owns all device memory, a host that hands over only the tensors):
    the library uses its own 256-byte array in place of the workspace.
    o / ht may be passed in preallocated; when they
    are not, this binding allocates them with torch before the call (the C
    entry point itself allocates nothing).  Calls sharing the library array
    must not overlap on the GPU.
    """
    lib = _lib.load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (h0, "h0")):
        _check(t, name)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if ht is None and output_final_state:
        ht = torch.empty(nseq, H, dv, dk, dtype=torch.float32, device=q.device)
    args = make_args(q, k, v, g, beta, h0, o, ht, gate=gate, scale_v=scale_v, cu_seqlens=cu_seqlens)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):   # the C entry point uses the current device's array
        rc = lib.kda_chunk_fwd_noalloc(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_noalloc")
    return o, ht


def make_bwd_args(q, k, v, g, beta, h0, do, dht, grads: dict, *, gate=None, scale_v=True,
                  workspace=None, cu_seqlens=None) -> _lib.KdaBwdArgs:
    """Fill the C backward argument struct (grads: dq, dk, dv, dg, dbeta, dh0 tensors or None).

    With ``cu_seqlens`` (int32 device tensor [N + 1]) the batch is packed as in
    :func:`make_args`.
    """
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
    if gate is None:
        gate = "none" if g is None else ("scalar" if g.dim() == 3 else "channel")
    x = _lib.KdaBwdArgs()
    x.B, x.T, x.H, x.dk, x.dv, x.chunk = B, T, H, dk, dv, 0
    x.dtype = _dtype_code(q)
    x.gate_kind = _GATES[gate]
    x.g_dtype = _dtype_code(g) if g is not None else _lib.KDA_BF16
    x.flags = _lib.KDA_FLAG_BETA_SCALES_V if scale_v else 0
    x.q, x.k, x.v, x.g, x.beta, x.h0 = _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0)
    x.grad_o, x.grad_ht = _ptr(do), _ptr(dht)
    x.grad_q, x.grad_k, x.grad_v = _ptr(grads.get("dq")), _ptr(grads.get("dk")), _ptr(grads.get("dv"))
    x.grad_g, x.grad_beta, x.grad_h0 = _ptr(grads.get("dg")), _ptr(grads.get("dbeta")), _ptr(grads.get("dh0"))
    x.cu_seqlens = _ptr(cu_seqlens)
    if workspace is not None:
        x.workspace = _ptr(workspace)
        x.workspace_bytes = workspace.numel() * workspace.element_size()
    return x


def kda_chunk_bwd(q, k, v, g, beta, h0, do, dht=None, *, gate=None, scale_v=True, grads=None,
                  workspace=None, stream=None, cu_seqlens=None):
    """Backward of :func:`kda_chunk_fwd` through ``kda_chunk_bwd`` of the C ABI.

    Inputs are those of the forward plus do [B, T, H, dv] (dtype of q) and dht
    [B, H, dv, dk] fp32 or None.  Returns a dict with dq, dk, dv (dtype of q),
    dg (dtype and layout of g) when g is given, dbeta when beta is given, and
    dh0 (fp32).  ``grads`` may supply preallocated output tensors by those names.
    cu_seqlens: int32 CUDA tensor [N + 1] for a packed batch of N sequences
    (then q is [1, T, H, dk], h0 / dht / dh0 are [N, H, dv, dk]), or None.
    """
    lib = _lib.load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (h0, "h0"), (do, "do"),
                    (dht, "dht"), (cu_seqlens, "cu_seqlens")):
        _check(t, name)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
    out = dict(grads or {})
    out.setdefault("dq", torch.empty_like(q))
    out.setdefault("dk", torch.empty_like(k))
    out.setdefault("dv", torch.empty_like(v))
    if g is not None:
        out.setdefault("dg", torch.empty_like(g))
    if beta is not None:
        out.setdefault("dbeta", torch.empty_like(beta))
    out.setdefault("dh0", torch.empty(B, H, dv, dk, dtype=torch.float32, device=q.device))
    args = make_bwd_args(q, k, v, g, beta, h0, do, dht, out, gate=gate, scale_v=scale_v, cu_seqlens=cu_seqlens)
    need = lib.kda_chunk_bwd_workspace(ctypes.byref(args))
    if need == 0:
        rc = lib.kda_chunk_bwd(ctypes.byref(args), None)
        raise KdaError(rc if rc != 0 else _lib.KDA_ERR_INVALID_ARG, "kda_chunk_bwd")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.kda_chunk_bwd(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "kda_chunk_bwd")
    return out


def make_dplr_args(q, k, v, a, b, g=None, h0=None, o=None, ht=None, *, gate=None, clip=False,
                   workspace=None, cu_seqlens=None) -> _lib.DplrFwdArgs:
    """Fill the C DPLR argument struct from tensors (q, k, v, o may be None for the norm report).

    With ``cu_seqlens`` the batch is packed as in :func:`make_args`.
    """
    B, T, H, dk = a.shape
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
    dv = v.shape[-1] if v is not None else 0
    if gate is None:
        gate = "none" if g is None else ("scalar" if g.dim() == 3 else "channel")
    x = _lib.DplrFwdArgs()
    x.B, x.T, x.H, x.dk, x.dv, x.chunk = B, T, H, dk, dv, 0
    x.dtype = _dtype_code(a)
    x.gate_kind = _GATES[gate]
    x.g_dtype = _dtype_code(g) if g is not None else _lib.KDA_BF16
    x.flags = _lib.DPLR_FLAG_CLIP_GATE if clip else 0
    x.q, x.k, x.v, x.a, x.b, x.g = _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b), _ptr(g)
    x.h0, x.o, x.ht = _ptr(h0), _ptr(o), _ptr(ht)
    x.cu_seqlens = _ptr(cu_seqlens)
    if workspace is not None:
        x.workspace = _ptr(workspace)
        x.workspace_bytes = workspace.numel() * workspace.element_size()
    return x


def dplr_chunk_fwd(q, k, v, a, b, g=None, h0=None, *, gate=None, clip=False, output_final_state=True,
                   o=None, ht=None, workspace=None, stream=None, cu_seqlens=None):
    """General gated DPLR forward through ``dplr_chunk_fwd`` of the C ABI.

    q, k, a, b: [B, T, H, dk]; v: [B, T, H, dv] (bf16 or fp32, one dtype);
    g: log-decay [B, T, H, dk], [B, T, H] or None; h0: [B, H, dv, dk] fp32 or None.
    clip=True applies the eq. (7) gate clip (``DPLR_FLAG_CLIP_GATE``).
    cu_seqlens: int32 CUDA tensor [N + 1] for a packed batch of N sequences
    (then the inputs are [1, T, H, d], h0 / ht [N, H, dv, dk]), or None.
    Returns (o [B, T, H, dv] in q's dtype, ht [B, H, dv, dk] fp32 or None).
    """
    lib = _lib.load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"), (g, "g"), (h0, "h0"),
                    (cu_seqlens, "cu_seqlens")):
        _check(t, name)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(B, T, H, dv, dtype=q.dtype, device=q.device)
    if ht is None and output_final_state:
        ht = torch.empty(nseq, H, dv, dk, dtype=torch.float32, device=q.device)
    args = make_dplr_args(q, k, v, a, b, g, h0, o, ht, gate=gate, clip=clip, cu_seqlens=cu_seqlens)
    need = lib.dplr_chunk_fwd_workspace(ctypes.byref(args))
    if need == 0:
        rc = lib.dplr_chunk_fwd(ctypes.byref(args), None)
        raise KdaError(rc if rc != 0 else _lib.KDA_ERR_INVALID_ARG, "dplr_chunk_fwd")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    args.workspace = _ptr(workspace)
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.dplr_chunk_fwd(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "dplr_chunk_fwd")
    return o, ht


def dplr_factor_norms(a, b, g=None, *, gate=None, clip=False, stream=None):
    """Per-token transition norms through ``dplr_factor_norms`` of the C ABI.

    Returns (rho [B, T, H], norm [B, T, H], maxes [2]) float32 on a's device:
    rho = ||I - b a^T||_2 by the closed form, norm = ||Diag(alpha)(I - b a^T)||_2,
    maxes = (max rho, max norm).
    """
    lib = _lib.load()
    for t, name in ((a, "a"), (b, "b"), (g, "g")):
        _check(t, name)
    B, T, H, _ = a.shape
    rho = torch.empty(B, T, H, dtype=torch.float32, device=a.device)
    nrm = torch.empty_like(rho)
    maxes = torch.empty(4, dtype=torch.float32, device=a.device)
    args = make_dplr_args(None, None, None, a, b, g, gate=gate, clip=clip)
    if stream is None:
        stream = torch.cuda.current_stream(a.device)
    rc = lib.dplr_factor_norms(ctypes.byref(args), _ptr(rho), _ptr(nrm), _ptr(maxes),
                               ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "dplr_factor_norms")
    return rho, nrm, maxes[:2]


def dplr_chunk_bwd(q, k, v, a, b, g, h0, do, dht=None, *, gate=None, clip=False, grads=None,
                   workspace=None, stream=None, cu_seqlens=None):
    """Backward of :func:`dplr_chunk_fwd` through ``dplr_chunk_bwd`` of the C ABI.

    Returns a dict with dq, dk, dv, da, db (dtype of q), dg (dtype and layout
    of g) when g is given, and dh0 (fp32).  ``grads`` may supply preallocated
    outputs by those names.  cu_seqlens as for :func:`dplr_chunk_fwd`.
    """
    lib = _lib.load()
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (a, "a"), (b, "b"), (g, "g"), (h0, "h0"), (do, "do"),
                    (dht, "dht"), (cu_seqlens, "cu_seqlens")):
        _check(t, name)
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is not None:
        B = cu_seqlens.numel() - 1
    out = dict(grads or {})
    for name, like in (("dq", q), ("dk", k), ("dv", v), ("da", a), ("db", b)):
        out.setdefault(name, torch.empty_like(like))
    if g is not None:
        out.setdefault("dg", torch.empty_like(g))
    out.setdefault("dh0", torch.empty(B, H, dv, dk, dtype=torch.float32, device=q.device))
    if gate is None:
        gate = "none" if g is None else ("scalar" if g.dim() == 3 else "channel")
    x = _lib.DplrBwdArgs()
    x.B, x.T, x.H, x.dk, x.dv, x.chunk = B, T, H, dk, dv, 0
    x.dtype = _dtype_code(q)
    x.gate_kind = _GATES[gate]
    x.g_dtype = _dtype_code(g) if g is not None else _lib.KDA_BF16
    x.flags = _lib.DPLR_FLAG_CLIP_GATE if clip else 0
    x.q, x.k, x.v, x.a, x.b, x.g, x.h0 = (_ptr(t) for t in (q, k, v, a, b, g, h0))
    x.grad_o, x.grad_ht = _ptr(do), _ptr(dht)
    x.grad_q, x.grad_k, x.grad_v = _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"])
    x.grad_a, x.grad_b, x.grad_g, x.grad_h0 = _ptr(out["da"]), _ptr(out["db"]), _ptr(out.get("dg")), _ptr(out["dh0"])
    x.cu_seqlens = _ptr(cu_seqlens)
    need = lib.dplr_chunk_bwd_workspace(ctypes.byref(x))
    if need == 0:
        rc = lib.dplr_chunk_bwd(ctypes.byref(x), None)
        raise KdaError(rc if rc != 0 else _lib.KDA_ERR_INVALID_ARG, "dplr_chunk_bwd")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    x.workspace = _ptr(workspace)
    x.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = lib.dplr_chunk_bwd(ctypes.byref(x), ctypes.c_void_p(stream.cuda_stream))
    if rc != _lib.KDA_OK:
        raise KdaError(rc, "dplr_chunk_bwd")
    return out


def status_read(workspace=None, device=None, stream=None) -> int:
    """Device status word of the workspace (waits for the stream, then clears it); by
    default the cached workspace of ``stream`` (default: the current stream of ``device``)."""
    lib = _lib.load()
    if workspace is not None:
        device = workspace.device
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if workspace is None:
        workspace = workspace_for(dev, 256, stream)
    return lib.kda_status_read(_ptr(workspace), ctypes.c_void_p(stream.cuda_stream))


def gdn_fwd(q, k, v, g, beta, h0=None, **kw):
    """GDN: one log-decay per token and head, g [B, T, H]."""
    return kda_chunk_fwd(q, k, v, g, beta, h0, gate="scalar", scale_v=True, **kw)


def deltanet_fwd(q, k, v, beta, h0=None, **kw):
    """DeltaNet: no decay."""
    return kda_chunk_fwd(q, k, v, None, beta, h0, gate="none", scale_v=True, **kw)


def gla_fwd(q, k, v, g, h0=None, **kw):
    """GLA: per-channel decay, no delta term, v unscaled."""
    return kda_chunk_fwd(q, k, v, g, None, h0, gate="channel", scale_v=False, **kw)


class HostRunner:
    """End-to-end calls from pinned host buffers, pipelined across calls.

    Each :meth:`run` copies the inputs host->device, runs the call
    (``kda_chunk_fwd``; ``dplr_chunk_fwd`` when ``kind="dplr"``;
    ``kda_chunk_bwd`` / ``dplr_chunk_bwd`` when ``kind="kda_bwd"`` / ``"dplr_bwd"``) and copies its results back
    device->host (o and ht, or every gradient).  Copies in run on one stream,
    the call on the caller's stream, copies out on a third, and ``depth`` sets
    of device buffers rotate between calls, so the inputs of one call travel
    while the previous call computes and its results drain; events keep each
    set's copies, call and read-back in order.  Bracket a run of calls with
    :meth:`begin` and :meth:`finish` to order the copy streams after, and the
    caller's stream after, everything they do.  Every call still copies all of
    its inputs in and all of its results out.
    """

    _INPUTS = ("q", "k", "v", "g", "beta", "h0", "a", "b", "do", "dht")

    def __init__(self, host: dict, device="cuda", scale_v=True, gate=None, kind="kda", depth=2):
        if kind not in ("kda", "dplr", "kda_bwd", "dplr_bwd"):
            raise ValueError(f"unknown kind {kind}")
        self.host = {k: v.pin_memory() for k, v in host.items() if k in self._INPUTS and isinstance(v, torch.Tensor)}
        self.scale_v, self.gate, self.kind = scale_v, gate, kind
        self.sets = [self._buffers(device) for _ in range(max(1, depth))]
        self.outs_host = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in self.sets[0][1].items()}
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.sets[0][0].values())
        self.d2h_bytes = sum(v.numel() * v.element_size() for v in self.sets[0][1].values())
        self.copy_in = torch.cuda.Stream(device=device)
        self.copy_out = torch.cuda.Stream(device=device)
        ev = lambda: [torch.cuda.Event() for _ in self.sets]
        self.ev_ready, self.ev_done, self.ev_drained = ev(), ev(), ev()
        self.calls = 0

    def _buffers(self, device):
        dev = {k: torch.empty_like(v, device=device) for k, v in self.host.items()}
        q = dev["q"]
        B, T, H, dk = q.shape
        dv = dev["v"].shape[-1]
        if self.kind in ("kda_bwd", "dplr_bwd"):
            outs = {"dq": torch.empty_like(q), "dk": torch.empty_like(dev["k"]), "dv": torch.empty_like(dev["v"]),
                    "dh0": torch.empty(B, H, dv, dk, dtype=torch.float32, device=device)}
            if "g" in dev:
                outs["dg"] = torch.empty_like(dev["g"])
            if "beta" in dev and self.kind == "kda_bwd":
                outs["dbeta"] = torch.empty_like(dev["beta"])
            if self.kind == "dplr_bwd":
                outs["da"], outs["db"] = torch.empty_like(dev["a"]), torch.empty_like(dev["b"])
        else:
            outs = {"o": torch.empty(B, T, H, dv, dtype=q.dtype, device=device),
                    "ht": torch.empty(B, H, dv, dk, dtype=torch.float32, device=device)}
        return dev, outs

    def begin(self, stream=None):
        """Order the copy streams after everything already on ``stream``."""
        stream = stream or torch.cuda.current_stream()
        self.copy_in.wait_stream(stream)
        self.copy_out.wait_stream(stream)

    def finish(self, stream=None):
        """Order ``stream`` after every copy issued so far; returns the host results of the last call."""
        stream = stream or torch.cuda.current_stream()
        stream.wait_stream(self.copy_in)
        stream.wait_stream(self.copy_out)
        return self.outs_host

    def run(self, stream=None):
        stream = stream or torch.cuda.current_stream()
        i = self.calls % len(self.sets)
        reuse = self.calls >= len(self.sets)
        self.calls += 1
        d, outs = self.sets[i]
        with torch.cuda.stream(self.copy_in):
            if reuse:
                self.copy_in.wait_event(self.ev_done[i])         # the last call on this set has read it
            for k, v in d.items():
                v.copy_(self.host[k], non_blocking=True)
            self.ev_ready[i].record(self.copy_in)
        stream.wait_event(self.ev_ready[i])
        if reuse:
            stream.wait_event(self.ev_drained[i])                 # its results have been copied out
        with torch.cuda.stream(stream):
            if self.kind == "dplr":
                dplr_chunk_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d.get("g"), d.get("h0"),
                               gate=self.gate, o=outs["o"], ht=outs["ht"], stream=stream)
            elif self.kind == "dplr_bwd":
                dplr_chunk_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d.get("g"), d.get("h0"), d["do"],
                               d.get("dht"), gate=self.gate, grads=outs, stream=stream)
            elif self.kind == "kda_bwd":
                kda_chunk_bwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d.get("h0"), d["do"],
                              d.get("dht"), gate=self.gate, scale_v=self.scale_v, grads=outs, stream=stream)
            else:
                kda_chunk_fwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d.get("h0"),
                              gate=self.gate, scale_v=self.scale_v, o=outs["o"], ht=outs["ht"],
                              stream=stream)
            self.ev_done[i].record(stream)
        with torch.cuda.stream(self.copy_out):
            self.copy_out.wait_event(self.ev_done[i])
            for k, v in outs.items():
                self.outs_host[k].copy_(v, non_blocking=True)
            self.ev_drained[i].record(self.copy_out)
        return self.outs_host
