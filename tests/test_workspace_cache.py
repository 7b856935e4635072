"""The Python binding's workspace cache, on the CPU with stand-ins for the CUDA calls.

One zero-filled workspace per (device, stream), grown when a call needs more,
allocated with its own stream current, and at most a bounded number of them
kept (the least recently used is dropped first).
"""
import contextlib

import pytest
import torch

from chunkwise_gated_delta_gb300 import api


class _Stream:
    def __init__(self, handle):
        self.cuda_stream = handle


@pytest.fixture
def fake_cuda(monkeypatch):
    allocs = []                                     # (stream handle current at allocation, bytes)
    current = {"stream": _Stream(1)}

    @contextlib.contextmanager
    def stream_ctx(s):
        prev = current["stream"]
        current["stream"] = s
        try:
            yield
        finally:
            current["stream"] = prev

    real_zeros = torch.zeros

    def zeros(n, dtype=None, device=None):
        allocs.append((current["stream"].cuda_stream, n))
        return real_zeros(n, dtype=dtype)           # a CPU tensor stands in for device memory

    monkeypatch.setattr(api, "_workspaces", {})
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: current["stream"])
    monkeypatch.setattr(torch.cuda, "stream", stream_ctx)
    monkeypatch.setattr(api.torch, "zeros", zeros)
    return allocs


def test_one_workspace_per_stream_grown_on_demand(fake_cuda):
    s1, s2 = _Stream(11), _Stream(12)
    w1 = api.workspace_for("cuda:0", 1000, s1)
    w2 = api.workspace_for("cuda:0", 1000, s2)
    assert w1 is not w2
    assert api.workspace_for("cuda:0", 500, s1) is w1            # big enough: reused
    w1b = api.workspace_for("cuda:0", 5000, s1)                  # too small: replaced
    assert w1b is not w1 and w1b.numel() == 5000
    assert api.workspace_for("cuda:0", 10, s2) is w2
    assert [a for a in fake_cuda] == [(11, 1000), (12, 1000), (11, 5000)]   # each on its own stream
    assert api.workspace_for("cuda:0", 1).numel() == 256       # default stream, at least 256 bytes


def test_least_recently_used_workspace_is_dropped(fake_cuda):
    n = api._MAX_WORKSPACES
    streams = [_Stream(100 + i) for i in range(n + 1)]
    first = [api.workspace_for("cuda:0", 256, s) for s in streams[:n]]
    api.workspace_for("cuda:0", 256, streams[0])                 # stream 0 is now the most recent
    api.workspace_for("cuda:0", 256, streams[n])                 # one over the bound: stream 1 goes
    assert len(api._workspaces) == n
    assert (0, streams[1].cuda_stream) not in api._workspaces
    assert api._workspaces[(0, streams[0].cuda_stream)] is first[0]
    assert api.workspace_for("cuda:0", 256, streams[1]) is not first[1]


def test_devices_are_kept_apart(fake_cuda):
    s = _Stream(7)
    assert api.workspace_for("cuda:0", 256, s) is not api.workspace_for("cuda:1", 256, s)
