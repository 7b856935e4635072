"""Float64 CPU oracle for the chunkwise gated delta rule -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing from the product.

The forward oracle is the token recurrence itself (page "Diagonal Plus Low
Rank", section 2, opening equation), run in float64 by ``recurrence.c``:

    S_t = S_{t-1} Diag(alpha_t) (I - b_t a_t^T) + vv_t k_t^T,   o_t = S_t q_t

Every variant is a choice of (a, b, vv, alpha):

* KDA: a = k, b = beta k, vv = beta v, alpha = exp(g) per channel
  (DPLR page, "relation to KDA"; page "How to make GDN2 more stable", eq. (1)).
* GDN: as KDA with one scalar log-decay per token (same eq. (1), D = gamma I).
* DeltaNet: as KDA with alpha = 1 (DeltaNet page, section 4.1).
* GLA: b = 0 and vv = v (GLA page, section 5.1).
* DPLR: a, b given, vv = v (DPLR page, section 2).

The reverse mode of the same loop (``recurrence_bwd.c``) gives the gradients
of L = <do, o> + <dht, ht> with respect to every input.

Parity status of each function is listed in ``PINS`` below; each pin is a test
under ``tests/test_oracle_pins.py`` or ``tests/test_oracle_bwd_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .spectral import clip_gate, clip_gate_bwd, factor_norm_exact, rho_closed_form, rho_of  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "recurrence.c")
_SRC_BWD = os.path.join(_HERE, "recurrence_bwd.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

GATE_NONE, GATE_SCALAR, GATE_CHANNEL = 0, 1, 2

# Which test pins each oracle function to something other than itself.
PINS = {
    "recurrence": [
        "linear-attention closed form (g = 0, beta = 0)",
        "GLA parallel closed form with decay (beta = 0, vv = v)",
        "delta-rule write: with unit k and q = k, o_t = (1 - beta) S_{t-1} Diag(alpha) k + beta v",
        "hand-derived worked example, tests/golden/tiny_kda_worked.txt",
        "DeltaNet/KDA/DPLR chunk forms of the pages equal the recurrence for several C",
        "h0 -> ht chaining over split segments equals one call",
    ],
    "rho_closed_form": ["numpy SVD", "eq. (5) lower bound", "eq. (6) equality case",
                        "hand-derived values, tests/golden/spectral_norm_points.txt"],
    "factor_norm_exact": ["explicit 2x2 reduction of eq. (9)", "D = I reduces to rho"],
    "clip_gate": ["after the clip every factor norm (numpy SVD) is at most 1",
                  "eq. (6): the KDA mapping (a = k unit, b = beta k, beta <= 2) leaves g unchanged",
                  "only channels above -log rho change"],
    "clip_gate_bwd / dplr_bwd(clip=True)": ["central finite differences of dplr_fwd(clip=True)"],
    "recurrence_bwd": [
        "central finite differences of the forward oracle on every input entry (T = 64, all five variants)",
        "central finite differences on sampled entries across four checkpoint segments",
        "chunk backward of page 'Kimi Delta Attention backward' restated in numpy, C in {16, 32, 64}",
        "closed-form gradients of the GLA parallel form (page 'Gated Linear Attention', section 6.3)",
        "scalar-gate gradient equals the channel sum at equal decays",
    ],
}


def build(force: bool = False) -> str:
    """Compile ``recurrence.c`` with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_BWD)))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-o", tmp, _SRC, _SRC_BWD, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_recurrence_head.restype = ctypes.c_int
            lib.oracle_recurrence_head.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                dp, dp, ctypes.c_long,
                dp, ctypes.c_long,
                dp, ctypes.c_long, ctypes.c_int,
                dp, dp, ctypes.c_long,
                dp, ctypes.c_long, ctypes.c_int,
                dp, dp, ctypes.c_long, dp]
            lib.oracle_recurrence_head_bwd.restype = ctypes.c_int
            lib.oracle_recurrence_head_bwd.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                dp, dp, ctypes.c_long,
                dp, ctypes.c_long,
                dp, ctypes.c_long, ctypes.c_int,
                dp, dp, ctypes.c_long,
                dp, ctypes.c_long, ctypes.c_int,
                dp,
                dp, ctypes.c_long, dp,
                dp, dp, dp, dp, dp, dp, dp, dp]
            _lib = lib
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x, offset=0):
    if x is None:
        return None
    return ctypes.cast(x.ctypes.data + 8 * offset, ctypes.POINTER(ctypes.c_double))


def recurrence(q, k, v, g=None, gate=GATE_CHANNEL, beta=None, a=None, b=None,
               scale_v=True, h0=None, threads=None, heads=None):
    """Run the token recurrence for every (batch, head) of [B, T, H, d] inputs.

    q, k: [B, T, H, dk]; v: [B, T, H, dv]; g: [B, T, H, dk] (GATE_CHANNEL),
    [B, T, H] (GATE_SCALAR) or None (GATE_NONE); beta: [B, T, H] or None;
    a, b: [B, T, H, dk] or None (None -> KDA mapping a = k, b = beta k);
    h0: [B, H, dv, dk] or None.  ``heads`` optionally restricts the work to a
    list of (b, h) pairs; the other outputs stay zero.
    Returns (o [B, T, H, dv], ht [B, H, dv, dk]) in float64.
    """
    lib = _load()
    q, k, v, g, beta, a, b, h0 = map(_f64, (q, k, v, g, beta, a, b, h0))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if g is None:
        gate = GATE_NONE
    if (a is None) != (b is None):
        raise ValueError("a and b are given together or not at all")
    o = np.zeros((B, T, H, dv), np.float64)
    ht = np.zeros((B, H, dv, dk), np.float64)
    s_qk, s_v, s_o = H * dk, H * dv, H * dv
    s_g = (H * dk) if gate == GATE_CHANNEL else H
    pairs = heads if heads is not None else [(bi, hi) for bi in range(B) for hi in range(H)]

    def one(pair):
        bi, hi = pair
        base_qk = (bi * T * H + hi) * dk
        base_v = (bi * T * H + hi) * dv
        gbase = 0
        if gate == GATE_CHANNEL:
            gbase = (bi * T * H + hi) * dk
        elif gate == GATE_SCALAR:
            gbase = bi * T * H + hi
        rc = lib.oracle_recurrence_head(
            T, dk, dv,
            _ptr(q, base_qk), _ptr(k, base_qk), s_qk,
            _ptr(v, base_v), s_v,
            _ptr(g, gbase) if g is not None else None, s_g, gate,
            _ptr(a, base_qk) if a is not None else None,
            _ptr(b, base_qk) if b is not None else None, s_qk,
            _ptr(beta, bi * T * H + hi) if beta is not None else None, H,
            1 if scale_v else 0,
            _ptr(h0, (bi * H + hi) * dv * dk) if h0 is not None else None,
            _ptr(o, base_v), s_o,
            _ptr(ht, (bi * H + hi) * dv * dk))
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")

    nthreads = threads or len(os.sched_getaffinity(0))
    if nthreads <= 1 or len(pairs) == 1:
        for p in pairs:
            one(p)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(one, pairs))
    return o, ht


def recurrence_bwd(q, k, v, do, g=None, gate=GATE_CHANNEL, beta=None, a=None, b=None,
                   scale_v=True, h0=None, dht=None, threads=None, heads=None):
    """Reverse mode of :func:`recurrence` for L = <do, o> + <dht, ht>.

    Same inputs as :func:`recurrence` plus do [B, T, H, dv] and dht
    [B, H, dv, dk] (None -> 0).  Returns a dict of float64 gradients: dq, dk,
    dv, dh0, and dg (shape of g) when g is given, dbeta when beta is given,
    da and db when a and b are given.  With the KDA mapping (a, b None) the
    a- and b-paths are folded into dk and dbeta.  ``heads`` restricts the work
    to a list of (b, h) pairs; the other entries stay zero.
    """
    lib = _load()
    q, k, v, do, g, beta, a, b, h0, dht = map(_f64, (q, k, v, do, g, beta, a, b, h0, dht))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if g is None:
        gate = GATE_NONE
    if (a is None) != (b is None):
        raise ValueError("a and b are given together or not at all")
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
           "dh0": np.zeros((B, H, dv, dk))}
    if g is not None:
        out["dg"] = np.zeros_like(g)
    if beta is not None:
        out["dbeta"] = np.zeros_like(beta)
    if a is not None:
        out["da"], out["db"] = np.zeros_like(a), np.zeros_like(b)
    s_qk, s_v = H * dk, H * dv
    s_g = (H * dk) if gate == GATE_CHANNEL else H
    pairs = heads if heads is not None else [(bi, hi) for bi in range(B) for hi in range(H)]

    def one(pair):
        bi, hi = pair
        base_qk = (bi * T * H + hi) * dk
        base_v = (bi * T * H + hi) * dv
        base_s = (bi * H + hi) * dv * dk
        gbase = (bi * T * H + hi) * dk if gate == GATE_CHANNEL else bi * T * H + hi
        o_g = (_ptr(g, gbase), _ptr(out.get("dg"), gbase)) if g is not None else (None, None)
        bb = bi * T * H + hi
        rc = lib.oracle_recurrence_head_bwd(
            T, dk, dv,
            _ptr(q, base_qk), _ptr(k, base_qk), s_qk,
            _ptr(v, base_v), s_v,
            o_g[0], s_g, gate,
            _ptr(a, base_qk), _ptr(b, base_qk), s_qk,
            _ptr(beta, bb), H,
            1 if scale_v else 0,
            _ptr(h0, base_s),
            _ptr(do, base_v), s_v, _ptr(dht, base_s),
            _ptr(out["dq"], base_qk), _ptr(out["dk"], base_qk), _ptr(out["dv"], base_v), o_g[1],
            _ptr(out.get("da"), base_qk), _ptr(out.get("db"), base_qk),
            _ptr(out.get("dbeta"), bb), _ptr(out["dh0"], base_s))
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")

    nthreads = threads or len(os.sched_getaffinity(0))
    if nthreads <= 1 or len(pairs) == 1:
        for p in pairs:
            one(p)
    else:
        with ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(one, pairs))
    return out


def kda_bwd(q, k, v, g, beta, do, h0=None, dht=None, **kw):
    """KDA backward: gradients dq, dk, dv, dg, dbeta, dh0."""
    return recurrence_bwd(q, k, v, do, g=g, gate=GATE_CHANNEL, beta=beta, scale_v=True, h0=h0, dht=dht, **kw)


def gdn_bwd(q, k, v, g, beta, do, h0=None, dht=None, **kw):
    """GDN backward (g [B, T, H])."""
    return recurrence_bwd(q, k, v, do, g=g, gate=GATE_SCALAR, beta=beta, scale_v=True, h0=h0, dht=dht, **kw)


def deltanet_bwd(q, k, v, beta, do, h0=None, dht=None, **kw):
    """DeltaNet backward."""
    return recurrence_bwd(q, k, v, do, g=None, gate=GATE_NONE, beta=beta, scale_v=True, h0=h0, dht=dht, **kw)


def gla_bwd(q, k, v, g, do, h0=None, dht=None, **kw):
    """GLA backward."""
    return recurrence_bwd(q, k, v, do, g=g, gate=GATE_CHANNEL, beta=None, scale_v=False, h0=h0, dht=dht, **kw)


def dplr_bwd(q, k, v, a, b, g, do, h0=None, dht=None, clip=False, **kw):
    """General gated DPLR backward: dq, dk, dv, da, db, dg, dh0.

    clip=True differentiates the forward with the eq. (7) clip applied to g
    (page "How to make GDN2 more stable"): the reverse mode runs on the
    clipped gate and the clip's chain rule maps its gate gradient back onto
    g, a and b.
    """
    if not clip:
        return recurrence_bwd(q, k, v, do, g=g, gate=GATE_CHANNEL, a=a, b=b, scale_v=False, h0=h0, dht=dht, **kw)
    gc = clip_gate(g, a, b)
    out = recurrence_bwd(q, k, v, do, g=gc, gate=GATE_CHANNEL, a=a, b=b, scale_v=False, h0=h0, dht=dht, **kw)
    dg, da, db = clip_gate_bwd(g, a, b, out["dg"])
    heads = kw.get("heads")
    if heads is not None:          # keep the untouched heads at zero, as recurrence_bwd does
        mask = np.zeros(np.asarray(g).shape[:3], dtype=bool)
        for bi, hi in heads:
            mask[bi, :, hi] = True
        dg, da, db = (np.where(mask[..., None], x, 0.0) for x in (dg, da, db))
    out["dg"] = dg
    out["da"] = out["da"] + da
    out["db"] = out["db"] + db
    return out


def kda_fwd(q, k, v, g, beta, h0=None, **kw):
    """KDA: per-channel log-decay g [B,T,H,dk], a = k, b = beta k, vv = beta v."""
    return recurrence(q, k, v, g=g, gate=GATE_CHANNEL, beta=beta, scale_v=True, h0=h0, **kw)


def gdn_fwd(q, k, v, g, beta, h0=None, **kw):
    """GDN: one log-decay per token g [B,T,H] broadcast over channels."""
    return recurrence(q, k, v, g=g, gate=GATE_SCALAR, beta=beta, scale_v=True, h0=h0, **kw)


def deltanet_fwd(q, k, v, beta, h0=None, **kw):
    """DeltaNet: alpha = 1."""
    return recurrence(q, k, v, g=None, gate=GATE_NONE, beta=beta, scale_v=True, h0=h0, **kw)


def gla_fwd(q, k, v, g, h0=None, **kw):
    """GLA: beta = 0 and vv = v (no delta correction, values unscaled)."""
    return recurrence(q, k, v, g=g, gate=GATE_CHANNEL, beta=None, scale_v=False, h0=h0, **kw)


def dplr_fwd(q, k, v, a, b, g, h0=None, clip=False, **kw):
    """General gated DPLR: independent a, b [B,T,H,dk]; vv = v.

    clip=True applies the eq. (7) clip of page "How to make GDN2 more stable"
    to the gate first: g -> min(g, -log ||I - b a^T||_2) token by token.
    """
    if clip:
        g = clip_gate(g, a, b)
    return recurrence(q, k, v, g=g, gate=GATE_CHANNEL, a=a, b=b, scale_v=False, h0=h0, **kw)
