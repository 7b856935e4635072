"""The forward on several streams at once, and under CUDA graph capture.

- Calls on different streams may run at the same time on the GPU.  The Python
  binding gives each stream its own cached workspace (chunk records, status
  block), so records-form calls issued on two streams without any ordering
  between them give the results of the same calls run one after the other.
- A captured graph of the single-kernel form (two launches, the second a
  programmatic dependent launch that redoes the call when the first met a
  chunk past the one-product Gram's decay range) replays to the eager results
  bit for bit: on the captured inputs, after they are overwritten with a
  strong-decay chunk (GLA page, section 5.3), and after they are put back
  (the replay then redoes the call with the note of the earlier replay, which
  gives the same bits).
"""
import ctypes

import pytest
import torch

from chunkwise_gated_delta_gb300 import api, kda_chunk_fwd
from chunkwise_gated_delta_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
_INPUTS = ("q", "k", "v", "g", "beta", "h0")


def _dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def test_each_stream_has_its_own_workspace():
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    w1 = api.workspace_for(DEV, 1 << 20, s1)
    w2 = api.workspace_for(DEV, 1 << 20, s2)
    assert w1.data_ptr() != w2.data_ptr()
    assert api.workspace_for(DEV, 1 << 16, s1).data_ptr() == w1.data_ptr()


@pytest.mark.parametrize("variant,gate", [("gdn", "scalar"), ("kda", "channel")])
def test_unordered_streams_match_calls_in_sequence(variant, gate):
    # B1 H2: four CTAs of 64 values, far below half the SMs, so the records form runs
    ds = [_dev(make_inputs(custom(variant, 1, 1024, 2, 128, 128, dtype=torch.bfloat16, h0=True), seed=40 + i))
          for i in range(2)]

    def call(d, stream=None):
        return kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], gate=gate, stream=stream)

    args = api.make_args(*(ds[0][k] for k in _INPUTS), torch.empty_like(ds[0]["v"]),
                         torch.empty_like(ds[0]["h0"]), gate=gate)
    assert api._lib.load().kda_chunk_fwd_workspace(ctypes.byref(args)) > 256   # the records form
    ref = []
    for d in ds:
        o, ht = call(d)
        ref.append((o.clone(), ht.clone()))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = []
    for _ in range(3):
        outs = []
        for d, s in zip(ds, streams):
            with torch.cuda.stream(s):
                outs.append(call(d, stream=s))
    torch.cuda.synchronize()
    for (o, ht), (ro, rht) in zip(outs, ref):
        assert torch.equal(o, ro) and torch.equal(ht, rht)


def test_graph_replay_of_the_single_kernel_form():
    x = make_inputs(custom("kda", 2, 256, 2, 128, 128, dtype=torch.bfloat16, h0=True), seed=41)
    strong = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    g = strong["g"].double()
    g[:, 64:128] *= 30.0                                   # chunk 1: log-decay near -150 per channel
    strong["g"] = g.to(x["g"].dtype)
    assert float(strong["g"].double()[:, 64:128].sum(1).min()) < -100.0
    d = _dev(x)                                            # the captured (static) inputs
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)   # status block only: the single-kernel form

    def call():
        return kda_chunk_fwd(*(d[k] for k in _INPUTS), gate="channel", workspace=ws)

    def load(src):
        for k in _INPUTS:
            d[k].copy_(src[k])

    ref = {}
    for name, src in (("plain", x), ("strong", strong)):
        load(src)
        o, ht = call()
        ref[name] = (o.clone(), ht.clone())
    torch.cuda.synchronize()
    assert not torch.equal(ref["plain"][0], ref["strong"][0])

    load(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                                             # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        o, ht = call()
    for name, src in (("plain", x), ("strong", strong), ("plain", x)):
        load(src)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref[name][0]) and torch.equal(ht, ref[name][1]), name
    assert api.status_read(ws) == 0
