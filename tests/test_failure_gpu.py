"""Failure paths of the bf16 forward on the GPU, made without faulting it.

* A bounded wait that runs out: word 7 of the status block sets the polling
  budget of every bounded wait; a budget of one poll is too small for the
  waits of a real launch, so the kernels record KDA_ERR_TIMEOUT, skip the
  rest of their waits, drain every copy and tensor-core product they started
  and exit.  kda_status_read must then report the timeout, and the next call
  (default budget) must match the oracle: the context and the library are
  unharmed.  Both forms (chunk records + scan; the single kernel, with and
  without the two-CTA pair) are covered.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gb300 import _lib, api
from chunkwise_gated_delta_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def _inputs(T, dv, seed, g_scale=1.0):
    w = custom("kda", 2, T, 2, 128, dv, dtype=torch.bfloat16, h0=True)
    x = make_inputs(w, seed=seed)
    if g_scale != 1.0:
        x["g"] = (x["g"].double() * g_scale).to(torch.bfloat16)
    return x


def _call(lib, x, form, budget):
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o = torch.empty_like(d["v"])
    ht = torch.empty_like(d["h0"])
    a = api.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, ht)
    need = lib.kda_chunk_fwd_workspace(ctypes.byref(a)) if form == "records" else 256
    need = max(need, 256)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    ws[:256].view(torch.int32)[7] = budget
    a.workspace, a.workspace_bytes = ctypes.c_void_p(ws.data_ptr()), need
    rc = lib.kda_chunk_fwd(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.KDA_OK, _lib.status_string(rc)
    st = lib.kda_status_read(ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st, o.double().cpu().numpy(), ht.double().cpu().numpy()


def _oracle(x):
    f = lambda t: t.double().numpy()
    return oracle.kda_fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), h0=f(x["h0"]))


@pytest.mark.parametrize("form,dv", [("records", 128), ("single", 128), ("single", 64)])
def test_wait_budget_runs_out_then_next_call_is_correct(form, dv):
    lib = _lib.load()
    x = _inputs(1024, dv, seed=21)
    st, _, _ = _call(lib, x, form, budget=1)
    assert st == _lib.KDA_ERR_TIMEOUT, _lib.status_string(st)
    st, o, ht = _call(lib, x, form, budget=0)
    assert st == _lib.KDA_OK, _lib.status_string(st)
    ro, rh = _oracle(x)
    assert rel(o, ro) <= 5e-3 and rel(ht, rh) <= 5e-3, (rel(o, ro), rel(ht, rh))


def test_generous_budget_changes_nothing():
    """A budget that every wait fits in gives the same outputs as the default, bit for bit."""
    lib = _lib.load()
    x = _inputs(300, 128, seed=22)
    st0, o0, h0 = _call(lib, x, "single", budget=0)
    st1, o1, h1 = _call(lib, x, "single", budget=1 << 26)
    assert st0 == st1 == _lib.KDA_OK
    assert np.array_equal(o0, o1) and np.array_equal(h0, h1)


@pytest.mark.parametrize("form", ["records", "single"])
def test_decay_within_range_matches_oracle(form):
    """Stronger decay than the workloads' (g = -0.6 softplus(N(0, 1)), about -31 per chunk on average),
    still within the one-product Gram's range: no status, and parity with the oracle."""
    lib = _lib.load()
    x = _inputs(512, 128, seed=24, g_scale=6.0)
    chunk_sums = x["g"].double().reshape(2, 8, 64, 2, 128).sum(2)
    assert float(chunk_sums.min()) > -60.0 and float(chunk_sums.mean()) < -20.0
    st, o, ht = _call(lib, x, form, budget=0)
    assert st == _lib.KDA_OK, _lib.status_string(st)
    ro, rh = _oracle(x)
    assert rel(o, ro) <= 5e-3 and rel(ht, rh) <= 5e-3, (rel(o, ro), rel(ht, rh))
