"""The library's calls captured in a CUDA graph and replayed.

Every entry point only enqueues work on the caller's stream (host-side
tensor-map encoding, kernel launches, the split merge launched as a
programmatic dependent), so a training or decoding loop can capture it once
and replay it: the persistent forward (its stream's work counters), the
three backward kernels, and the split-key decode forward with its merge.
Replays must give what eager calls give: the forward bit for bit, the
backward (whose dQ sums are reduced in no fixed order) within rounding; and a
replay after the inputs are overwritten in place must follow the new inputs.
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_95_gb300 as pkg

from parity import make, to_dev

pytestmark = pytest.mark.gpu


def _close(a, b, tol=2e-2):
    a, b = a.float(), b.float()
    return (a - b).abs().max().item() <= tol * max(b.abs().max().item(), 1e-6)


def test_forward_backward_graph_replay():
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    t = make(B, Hq, Hkv, N, d, seed=0x6A00)
    t2 = make(B, Hq, Hkv, N, d, seed=0x6A10)
    g = {k: to_dev(v) for k, v in t.items()}
    g2 = {k: to_dev(v) for k, v in t2.items()}
    ws = torch.empty(pkg.attn_bwd_workspace_size(B, Hq, Hkv, N, d), dtype=torch.uint8, device="cuda")
    O = torch.empty_like(g["Q"])
    L = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    dQ, dK, dV = torch.empty_like(g["Q"]), torch.empty_like(g["K"]), torch.empty_like(g["V"])

    def step():
        pkg.attn_fwd(g["Q"], g["K"], g["V"], None, True, O=O, LSE=L)
        pkg.attn_bwd(g["Q"], g["K"], g["V"], O, g["dO"], L, None, True, dQ, dK, dV, ws)

    # Eager results for both input sets.
    ref = []
    for src in (t, t2):
        for k in g:
            g[k].copy_(to_dev(src[k]))
        step()
        torch.cuda.synchronize()
        ref.append([x.clone() for x in (O, L, dQ, dK, dV)])
    for k in g:
        g[k].copy_(to_dev(t[k]))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on the capturing stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for r, src in ((0, g), (1, g2), (0, None)):
        if src is g2:
            for k in g:
                g[k].copy_(g2[k])
        elif src is None:
            for k in g:
                g[k].copy_(to_dev(t[k]))
        graph.replay()
        torch.cuda.synchronize()
        assert pkg.attn_last_device_status() == pkg.ATTN_OK
        assert torch.equal(O, ref[r][0]) and torch.equal(L, ref[r][1])
        for got, want in zip((dQ, dK, dV), ref[r][2:]):
            assert _close(got, want)


def test_split_decode_graph_replay():
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 1, 9000, 128
    q = make(B, Hq, Hkv, Nq, d, seed=0x6B00, names=("Q",))
    kv = make(B, Hq, Hkv, Nk, d, seed=0x6B01, names=("K", "V"))
    Q, K, V = to_dev(q["Q"]), to_dev(kv["K"]), to_dev(kv["V"])
    ws = torch.empty(max(pkg.attn_fwd_split_workspace_size(B, Hq, Hkv, Nq, Nk, d, 0), 1), dtype=torch.uint8,
                     device="cuda")
    O = torch.empty(B, Hq, Nq, d, dtype=torch.bfloat16, device="cuda")
    L = torch.empty(B, Hq, Nq, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(d)

    def call():
        pkg.attn_fwd_split(Q, K, V, scale, True, num_splits=0, O=O, LSE=L, workspace=ws)

    call()
    torch.cuda.synchronize()
    Oref, Lref = O.clone(), L.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    O.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert pkg.attn_last_device_status() == pkg.ATTN_OK
    assert torch.equal(O, Oref) and torch.equal(L, Lref)
