"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every symbol include/kda.h declares, and rejects bad arguments before
anything is launched."""
import ctypes
import os
import re

import pytest

from chunkwise_gated_delta_gb300 import _lib
from chunkwise_gated_delta_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return _lib.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b((?:kda|dplr)_[a-z_0-9]+)\s*\(", src))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.kda_status_string(code)
    assert _lib.status_string(_lib.KDA_ERR_TIMEOUT) == "device-side wait timed out"
    assert "decay" in _lib.status_string(_lib.KDA_ERR_RANGE)
    assert _lib.status_string(-99) == "unknown status"


def _args(**over):
    a = _lib.KdaFwdArgs()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = 2, 100, 4, 128, 128, 64
    a.dtype, a.gate_kind, a.g_dtype, a.flags = _lib.KDA_BF16, _lib.KDA_GATE_CHANNEL, _lib.KDA_BF16, 1
    base = 1 << 40          # fake, well-separated 16-byte aligned device addresses (never dereferenced)
    for i, f in enumerate(("q", "k", "v", "g", "beta", "h0", "o", "ht", "workspace")):
        setattr(a, f, base + i * (1 << 32))
    a.workspace_bytes = 256
    for k, v in over.items():
        setattr(a, k, v)
    return a


def _call(lib, a):
    return lib.kda_chunk_fwd(ctypes.byref(a), None)


def test_workspace_query(lib):
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args())) >= 4
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args(dk=96))) == 0
    # bf16 with dk = 64 is documented as unsupported (the fp32 path takes it): no workspace size
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args(dk=64))) == 0
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args(dk=64, dtype=_lib.KDA_F32, g_dtype=_lib.KDA_F32))) == 256
    assert lib.kda_chunk_fwd_workspace(None) == 0


@pytest.mark.parametrize("over,code", [
    (dict(q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(o=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(B=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(T=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(H=-1), _lib.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), _lib.KDA_ERR_INVALID_ARG),
    (dict(gate_kind=9), _lib.KDA_ERR_INVALID_ARG),
    (dict(gate_kind=_lib.KDA_GATE_NONE), _lib.KDA_ERR_INVALID_ARG),      # g given with no gate
    (dict(g=None), _lib.KDA_ERR_INVALID_ARG),                            # gate without g
    (dict(flags=6), _lib.KDA_ERR_INVALID_ARG),
    (dict(q=(1 << 40) + 8), _lib.KDA_ERR_INVALID_ARG),                   # misaligned
    (dict(o=(1 << 40) + 1 * (1 << 32)), _lib.KDA_ERR_INVALID_ARG),       # o aliases k
    (dict(dk=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dv=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(chunk=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dk=64), _lib.KDA_ERR_UNSUPPORTED),                             # bf16 needs dk = 128
    (dict(g_dtype=_lib.KDA_F32), _lib.KDA_ERR_UNSUPPORTED),              # bf16 channel gate in fp32
    (dict(workspace=None, workspace_bytes=0), _lib.KDA_ERR_WORKSPACE),
    (dict(workspace_bytes=16), _lib.KDA_ERR_WORKSPACE),
])
def test_rejects_bad_arguments_before_launch(lib, over, code):
    assert _call(lib, _args(**over)) == code


def test_null_args_pointer(lib):
    assert lib.kda_chunk_fwd(None, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_status_read(None, None) == _lib.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- DPLR entry points
def _dplr_args(**over):
    a = _lib.DplrFwdArgs()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = 2, 100, 4, 128, 128, 0
    a.dtype, a.gate_kind, a.g_dtype = _lib.KDA_BF16, _lib.KDA_GATE_CHANNEL, _lib.KDA_BF16
    base = 1 << 40
    for i, f in enumerate(("q", "k", "v", "a", "b", "g", "h0", "o", "ht", "workspace")):
        setattr(a, f, base + i * (1 << 32))
    a.workspace_bytes = 256
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_dplr_workspace_query(lib):
    assert lib.dplr_chunk_fwd_workspace(ctypes.byref(_dplr_args())) >= 4
    assert lib.dplr_chunk_fwd_workspace(ctypes.byref(_dplr_args(dv=48))) == 0
    assert lib.dplr_chunk_fwd_workspace(None) == 0


@pytest.mark.parametrize("over,code", [
    (dict(a=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(b=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(o=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(T=0), _lib.KDA_ERR_INVALID_ARG),
    (dict(dtype=3), _lib.KDA_ERR_INVALID_ARG),
    (dict(g=None), _lib.KDA_ERR_INVALID_ARG),                            # gate without g
    (dict(b=(1 << 40) + 4 * (1 << 32) + 4), _lib.KDA_ERR_INVALID_ARG),   # misaligned
    (dict(o=(1 << 40) + 3 * (1 << 32)), _lib.KDA_ERR_INVALID_ARG),       # o aliases a
    (dict(dk=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dv=48), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dv=288), _lib.KDA_ERR_UNSUPPORTED),
    (dict(chunk=64), _lib.KDA_ERR_UNSUPPORTED),
    (dict(workspace=None, workspace_bytes=0), _lib.KDA_ERR_WORKSPACE),
])
def test_dplr_rejects_bad_arguments_before_launch(lib, over, code):
    assert lib.dplr_chunk_fwd(ctypes.byref(_dplr_args(**over)), None) == code


def test_dplr_factor_norms_rejects_bad_arguments(lib):
    a = _dplr_args()
    out = (1 << 40) + 20 * (1 << 32)
    assert lib.dplr_factor_norms(None, out, None, None, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.dplr_factor_norms(ctypes.byref(_dplr_args(a=None)), out, None, None, None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.dplr_factor_norms(ctypes.byref(a), out + 4, None, None, None) == _lib.KDA_ERR_INVALID_ARG
    # the per-token output may not alias the input a
    assert lib.dplr_factor_norms(ctypes.byref(a), (1 << 40) + 3 * (1 << 32), None, None, None) == \
        _lib.KDA_ERR_INVALID_ARG
    assert lib.dplr_factor_norms(ctypes.byref(_dplr_args(dk=96)), out, None, None, None) == _lib.KDA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- backward entry points
def _bwd_args(**over):
    a = _lib.KdaBwdArgs()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = 2, 100, 4, 128, 128, 0
    a.dtype, a.gate_kind, a.g_dtype, a.flags = _lib.KDA_BF16, _lib.KDA_GATE_CHANNEL, _lib.KDA_BF16, 1
    base = 1 << 40
    names = ("q", "k", "v", "g", "beta", "h0", "grad_o", "grad_ht", "grad_q", "grad_k", "grad_v", "grad_g",
             "grad_beta", "grad_h0", "workspace")
    for i, f in enumerate(names):
        setattr(a, f, base + i * (1 << 32))
    a.workspace_bytes = 1 << 31
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_bwd_workspace_query(lib):
    need = lib.kda_chunk_bwd_workspace(ctypes.byref(_bwd_args()))
    n_chunks = (100 + 31) // 32
    record = 3 * 32 * 32 + 3 * 32 * 128 + 32 * 128 + 128
    assert need == 256 + 4 * 2 * 4 * ((2 * n_chunks + 1) * 128 * 128 + n_chunks * record + 2 * n_chunks * 32 * 128)
    assert lib.kda_chunk_bwd_workspace(ctypes.byref(_bwd_args(dk=96))) == 0
    assert lib.kda_chunk_bwd_workspace(None) == 0


def test_bwd_workspace_query_packed(lib):
    """Packed sequences: B + ceil(T / 32) chunk slots per head, and one more state slot per sequence."""
    cu = (1 << 40) + 20 * (1 << 32)
    need = lib.kda_chunk_bwd_workspace(ctypes.byref(_bwd_args(B=5, cu_seqlens=cu)))
    slots = 5 + (100 + 31) // 32
    record = 3 * 32 * 32 + 3 * 32 * 128 + 32 * 128 + 128
    assert need == 256 + 4 * 4 * ((2 * slots + 5) * 128 * 128 + slots * record + 2 * slots * 32 * 128)
    # a misaligned offsets array, and one that overlaps an output
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd_args(cu_seqlens=cu + 2)), None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd_args(cu_seqlens=(1 << 40) + 8 * (1 << 32))), None) == \
        _lib.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("over,code", [
    (dict(grad_o=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(grad_q=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(grad_g=None), _lib.KDA_ERR_INVALID_ARG),                       # g given, no grad_g
    (dict(grad_beta=None), _lib.KDA_ERR_INVALID_ARG),                    # beta given, no grad_beta
    (dict(beta=None), _lib.KDA_ERR_INVALID_ARG),                         # grad_beta without beta
    (dict(g=None, gate_kind=_lib.KDA_GATE_NONE), _lib.KDA_ERR_INVALID_ARG),
    (dict(grad_k=(1 << 40) + 8 * (1 << 32)), _lib.KDA_ERR_INVALID_ARG),  # grad_k aliases grad_q
    (dict(grad_v=(1 << 40) + 2 * (1 << 32)), _lib.KDA_ERR_INVALID_ARG),  # grad_v aliases v
    (dict(grad_q=(1 << 40) + 8 * (1 << 32) + 2), _lib.KDA_ERR_INVALID_ARG),
    (dict(dk=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dv=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(chunk=64), _lib.KDA_ERR_UNSUPPORTED),
    (dict(workspace_bytes=4096), _lib.KDA_ERR_WORKSPACE),
    (dict(workspace=None, workspace_bytes=0), _lib.KDA_ERR_WORKSPACE),
])
def test_bwd_rejects_bad_arguments_before_launch(lib, over, code):
    assert lib.kda_chunk_bwd(ctypes.byref(_bwd_args(**over)), None) == code


def _dplr_bwd_args(**over):
    a = _lib.DplrBwdArgs()
    a.B, a.T, a.H, a.dk, a.dv, a.chunk = 2, 100, 4, 128, 128, 0
    a.dtype, a.gate_kind, a.g_dtype, a.flags = _lib.KDA_BF16, _lib.KDA_GATE_CHANNEL, _lib.KDA_BF16, 1
    base = 1 << 40
    names = ("q", "k", "v", "a", "b", "g", "h0", "grad_o", "grad_ht", "grad_q", "grad_k", "grad_v", "grad_a",
             "grad_b", "grad_g", "grad_h0", "workspace")
    for i, f in enumerate(names):
        setattr(a, f, base + i * (1 << 32))
    a.workspace_bytes = 1 << 31
    for k, v in over.items():
        setattr(a, k, v)
    return a


def test_dplr_bwd_workspace_query(lib):
    need = lib.dplr_chunk_bwd_workspace(ctypes.byref(_dplr_bwd_args()))
    n_chunks = (100 + 15) // 16
    record = 4 * 16 * 128 + 16 * 128 + 4 * 16 * 16 + 128
    assert need == 256 + 4 * 2 * 4 * ((2 * n_chunks + 1) * 128 * 128 + n_chunks * record + 2 * n_chunks * 16 * 128)
    assert lib.dplr_chunk_bwd_workspace(ctypes.byref(_dplr_bwd_args(dv=32))) == 0


def test_dplr_workspace_queries_packed(lib):
    """Packed sequences: B + ceil(T / C) chunk slots per head (C = 32 forward, 16 backward)."""
    cu = (1 << 40) + 30 * (1 << 32)
    fwd = lib.dplr_chunk_fwd_workspace(ctypes.byref(_dplr_args(B=5, cu_seqlens=cu)))
    assert fwd == 256 + 4 * 4 * (5 + (100 + 31) // 32) * (4 * 32 * 128 + 2 * 32 * 128 + 128)
    need = lib.dplr_chunk_bwd_workspace(ctypes.byref(_dplr_bwd_args(B=5, cu_seqlens=cu)))
    slots = 5 + (100 + 15) // 16
    record = 4 * 16 * 128 + 16 * 128 + 4 * 16 * 16 + 128
    assert need == 256 + 4 * 4 * ((2 * slots + 5) * 128 * 128 + slots * record + 2 * slots * 16 * 128)
    assert lib.dplr_chunk_bwd(ctypes.byref(_dplr_bwd_args(cu_seqlens=cu + 2)), None) == _lib.KDA_ERR_INVALID_ARG
    assert lib.dplr_chunk_fwd(ctypes.byref(_dplr_args(cu_seqlens=cu + 2)), None) == _lib.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("over,code", [
    (dict(grad_a=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(b=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(grad_g=None), _lib.KDA_ERR_INVALID_ARG),
    (dict(flags=2), _lib.KDA_ERR_INVALID_ARG),
    (dict(grad_b=(1 << 40) + 3 * (1 << 32)), _lib.KDA_ERR_INVALID_ARG),    # grad_b aliases a
    (dict(chunk=32), _lib.KDA_ERR_UNSUPPORTED),
    (dict(dk=96), _lib.KDA_ERR_UNSUPPORTED),
    (dict(workspace_bytes=1024), _lib.KDA_ERR_WORKSPACE),
])
def test_dplr_bwd_rejects_bad_arguments_before_launch(lib, over, code):
    assert lib.dplr_chunk_bwd(ctypes.byref(_dplr_bwd_args(**over)), None) == code


def test_dplr_fwd_rejects_unknown_flags(lib):
    assert lib.dplr_chunk_fwd(ctypes.byref(_dplr_args(flags=4)), None) == _lib.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- workspace alignment
MISALIGNED = (1 << 40) + 40 * (1 << 32) + 8       # 8-byte aligned only, clear of every other fake pointer


def test_fwd_records_need_an_aligned_workspace(lib):
    """With room for the chunk records the forward copies them asynchronously: 16-byte alignment."""
    need = lib.kda_chunk_fwd_workspace(ctypes.byref(_args()))
    assert need > 256                                   # bf16 KDA: status word plus records
    assert _call(lib, _args(workspace=MISALIGNED, workspace_bytes=need)) == _lib.KDA_ERR_INVALID_ARG
    # GLA (flags cleared, no beta) takes the same records (Z = [I ; P], A_chain = [0 ; Q<-])
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args(flags=0, beta=None))) == need
    # float32 inputs never do
    assert lib.kda_chunk_fwd_workspace(ctypes.byref(_args(dtype=_lib.KDA_F32, dk=64))) == 256


def test_bwd_and_dplr_need_an_aligned_workspace(lib):
    a = _bwd_args(workspace=MISALIGNED)
    a.workspace_bytes = lib.kda_chunk_bwd_workspace(ctypes.byref(_bwd_args()))
    assert lib.kda_chunk_bwd(ctypes.byref(a), None) == _lib.KDA_ERR_INVALID_ARG
    d = _dplr_args(workspace=MISALIGNED, workspace_bytes=1 << 31)
    assert lib.dplr_chunk_fwd(ctypes.byref(d), None) == _lib.KDA_ERR_INVALID_ARG
    e = _dplr_bwd_args(workspace=MISALIGNED)
    assert lib.dplr_chunk_bwd(ctypes.byref(e), None) == _lib.KDA_ERR_INVALID_ARG


# ---------------------------------------------------------------- no CPU path
def test_missing_library_raises(monkeypatch, tmp_path):
    """Without libkda.so the binding raises instead of computing anything itself."""
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libkda.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(ImportError, match="missing"):
        _lib.load()


@pytest.mark.parametrize("entry", ["kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_chunk_bwd"])
def test_host_tensors_are_rejected(lib, entry):
    """Every compute call takes device tensors only: host tensors raise, they are not run on the CPU."""
    import torch

    from chunkwise_gated_delta_gb300 import api
    q = torch.zeros(1, 64, 1, 128, dtype=torch.bfloat16)
    beta = torch.zeros(1, 64, 1, dtype=torch.bfloat16)
    args = (q, q, q, q, beta)
    if entry == "kda_chunk_bwd":
        args = args + (None, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        getattr(api, entry)(*args)
