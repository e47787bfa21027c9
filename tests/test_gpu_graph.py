"""CUDA graph capture of the forward and backward (persistent launches).

A persistent launch keeps the work-item counter slot it was given when it was
captured for every replay of the graph.  Captured launches take their slots
from a ring of their own, so eager launches on another stream, running while
the graph replays, never share a slot with it.  Checked here: a captured
fa_forward + fa_backward (sizes whose forward and backward both run
persistent CTAs) replayed many times while eager calls run on a second stream
gives, every time, exactly the outputs of an eager call (the kernels are
deterministic), and no device error is recorded.
"""
import pytest
import torch

from fa_inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def buffers(fa, q):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_backward_workspace_size(B, H, N, d), dtype=torch.uint8,
                     device=q.device)
    return o, lse, dq, dk, dv, ws


def step(fa, q, k, v, dO, bufs, stream):
    o, lse, dq, dk, dv, ws = bufs
    fa.fa_forward(q, k, v, causal=True, o=o, lse=lse, stream=stream)
    fa.fa_backward(q, k, v, o, dO, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws,
                   stream=stream)


def test_graph_replay_beside_eager_launches(fa):
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in make_inputs(2, 4, 1000, 128, seed=13))
    main = torch.cuda.current_stream()
    ref = buffers(fa, q)
    step(fa, q, k, v, dO, ref, main)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0

    s_graph, s_eager = torch.cuda.Stream(), torch.cuda.Stream()
    gbufs, ebufs = buffers(fa, q), buffers(fa, q)
    with torch.cuda.stream(s_graph):  # one-time set-up outside the capture
        step(fa, q, k, v, dO, gbufs, s_graph)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s_graph):
        step(fa, q, k, v, dO, gbufs, s_graph)
    torch.cuda.synchronize()

    names = ("o", "lse", "dq", "dk", "dv")
    for rep in range(20):
        for t in gbufs[:5] + ebufs[:5]:
            t.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s_graph):
            graph.replay()
        for _ in range(3):
            step(fa, q, k, v, dO, ebufs, s_eager)
        torch.cuda.synchronize()
        for nm, r, g, e in zip(names, ref[:5], gbufs[:5], ebufs[:5]):
            assert torch.equal(g, r), f"replay {rep}: graph {nm} differs from the eager call"
            assert torch.equal(e, r), f"replay {rep}: eager {nm} differs"
    assert fa.fa_get_device_error()[0] == 0
