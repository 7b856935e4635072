"""kda_chunk_fwd_noalloc: the forward for callers that cannot allocate device memory.

Callers such as frameworks whose caching allocator owns all device memory,
or plugins handed only the input and output tensors, cannot supply the
workspace that kda_chunk_fwd needs; the no-allocation entry point replaces it
with a small array owned by the library.  Its results must equal those of
kda_chunk_fwd on the same inputs, on every call (the library array keeps the
previous call's contents, so two calls in a row are checked).  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from chunkwise_gated_delta_gb300 import _lib, api
from chunkwise_gated_delta_gb300 import build as kbuild
from chunkwise_gated_delta_gb300.inputs import custom, make_inputs

import oracle

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 5e-3, torch.float32: 1e-5}


def _rel(x, ref):
    x, ref = x.double().cpu().numpy(), ref.double().cpu().numpy()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


@pytest.mark.parametrize("dtype,dk,T", [(torch.bfloat16, 128, 200), (torch.float32, 64, 130)])
def test_noalloc_matches_kda_chunk_fwd_on_two_calls(dtype, dk, T):
    kbuild.build()
    lib = _lib.load()
    w = custom("kda", 2, T, 2, dk, dk, dtype=dtype, h0=True)
    x = make_inputs(w, seed=11)
    d = {k: v.to("cuda:0") for k, v in x.items() if isinstance(v, torch.Tensor)}
    o_ref, ht_ref = api.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    stream = torch.cuda.current_stream()
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        args = api.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, ht)
        rc = lib.kda_chunk_fwd_noalloc(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
        assert rc == _lib.KDA_OK, _lib.status_string(rc)
        torch.cuda.synchronize()
        assert _rel(o, o_ref) <= TOL[dtype]
        assert _rel(ht, ht_ref) <= TOL[dtype]


def test_noalloc_rejects_bad_arguments_like_kda_chunk_fwd():
    kbuild.build()
    lib = _lib.load()
    assert lib.kda_chunk_fwd_noalloc(None, None) == _lib.KDA_ERR_INVALID_ARG
    a = _lib.KdaFwdArgs()
    a.B, a.T, a.H, a.dk, a.dv = 1, 64, 1, 96, 128      # dk = 96 is not implemented
    a.q = a.k = a.v = a.o = None
    assert lib.kda_chunk_fwd_noalloc(ctypes.byref(a), None) == _lib.KDA_ERR_INVALID_ARG


def _noalloc(lib, args, stream):
    rc = lib.kda_chunk_fwd_noalloc(ctypes.byref(args), ctypes.c_void_p(stream.cuda_stream))
    assert rc == _lib.KDA_OK, _lib.status_string(rc)


def test_noalloc_matches_the_oracle_for_kda_and_gla():
    """Against the float64 oracle itself, for KDA and for GLA (beta = 0, v unscaled)."""
    kbuild.build()
    lib = _lib.load()
    stream = torch.cuda.current_stream()
    for variant in ("kda", "gla"):
        w = custom(variant, 1, 150, 2, 128, 128, dtype=torch.bfloat16, h0=True)
        x = make_inputs(w, seed=13)
        d = {k: v.to("cuda:0") for k, v in x.items() if isinstance(v, torch.Tensor)}
        o = torch.empty_like(d["v"])
        ht = torch.empty(1, 2, 128, 128, dtype=torch.float32, device="cuda:0")
        args = api.make_args(d["q"], d["k"], d["v"], d["g"], d.get("beta"), d["h0"], o, ht, gate="channel",
                             scale_v=x["scale_v"])
        _noalloc(lib, args, stream)
        torch.cuda.synchronize()
        f = lambda t: None if t is None else t.double().numpy()
        if variant == "kda":
            ro, rh = oracle.kda_fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), h0=f(x["h0"]))
        else:
            ro, rh = oracle.gla_fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), h0=f(x["h0"]))
        assert _rel(o, torch.from_numpy(ro)) <= 5e-3, variant
        assert _rel(ht, torch.from_numpy(rh)) <= 5e-3, variant


def test_noalloc_packed_sequences_match_kda_chunk_fwd():
    """cu_seqlens through the no-allocation entry point: equal to kda_chunk_fwd on the same packing."""
    kbuild.build()
    lib = _lib.load()
    lens = [70, 0, 129, 1]
    w = custom("kda", 1, sum(lens), 2, 128, 128, dtype=torch.bfloat16, h0=False)
    x = make_inputs(w, seed=14)
    d = {k: v.to("cuda:0") for k, v in x.items() if isinstance(v, torch.Tensor)}
    h0 = 0.1 * torch.randn(len(lens), 2, 128, 128, generator=torch.Generator().manual_seed(2)).to("cuda:0")
    cu = torch.tensor([0, 70, 70, 199, 200], dtype=torch.int32, device="cuda:0")
    o_ref, ht_ref = api.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, cu_seqlens=cu)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        ht = torch.full_like(ht_ref, float("nan"))
        args = api.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, o, ht, cu_seqlens=cu)
        _noalloc(lib, args, stream)
        torch.cuda.synchronize()
        assert _rel(o, o_ref) <= 5e-3 and _rel(ht, ht_ref) <= 5e-3


def test_noalloc_allocates_no_device_memory():
    """After the first call, further calls leave the device's free memory unchanged."""
    kbuild.build()
    lib = _lib.load()
    w = custom("kda", 2, 300, 2, 128, 128, dtype=torch.bfloat16, h0=True)
    x = make_inputs(w, seed=15)
    d = {k: v.to("cuda:0") for k, v in x.items() if isinstance(v, torch.Tensor)}
    o = torch.empty_like(d["v"])
    ht = torch.empty_like(d["h0"])
    args = api.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, ht)
    stream = torch.cuda.current_stream()
    _noalloc(lib, args, stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(lib, args, stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
