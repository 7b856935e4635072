"""HostRunner: the end-to-end call from pinned host buffers, pipelined across
calls (copies in, the call and copies out on three streams, buffer sets
rotating).  Its results must equal the direct device call on the same inputs
after any number of calls, for the forward and the backward."""
import pytest
import torch

from chunkwise_gated_delta_gb300 import HostRunner, kda_chunk_bwd, kda_chunk_fwd
from chunkwise_gated_delta_gb300.inputs import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("calls", [1, 2, 5])
def test_forward_runner_equals_direct_call(calls):
    w = custom("kda", 2, 300, 2, 128, 128, dtype=torch.bfloat16, h0=True)
    x = make_inputs(w, seed=3)
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o, ht = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], scale_v=x["scale_v"])
    stream = torch.cuda.current_stream()
    runner = HostRunner(x, device=DEV, scale_v=x["scale_v"], gate="channel", kind="kda")
    runner.begin(stream)
    for _ in range(calls):
        runner.run(stream)
    out = runner.finish(stream)
    torch.cuda.synchronize()
    assert runner.h2d_bytes > 0 and runner.d2h_bytes == o.numel() * 2 + ht.numel() * 4
    assert torch.equal(out["o"], o.cpu()) and torch.equal(out["ht"], ht.cpu())


def test_backward_runner_equals_direct_call():
    w = custom("kda", 1, 100, 2, 128, 128, dtype=torch.bfloat16, h0=True, grads=True)
    x = make_inputs(w, seed=4)
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    ref = kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"],
                        scale_v=x["scale_v"])
    stream = torch.cuda.current_stream()
    runner = HostRunner(x, device=DEV, scale_v=x["scale_v"], gate="channel", kind="kda_bwd")
    runner.begin(stream)
    for _ in range(3):
        runner.run(stream)
    out = runner.finish(stream)
    torch.cuda.synchronize()
    for key, r in ref.items():
        assert torch.equal(out[key], r.cpu()), key
