"""The running routing histogram (per-expert pair counts carried across calls).

The pages' engine counts its own routing and moves the experts it calls most to the
fast tier between steps ("bloomery README 0.3.1", opening feature list, MoE models
larger than the card; "bloomery V4.1 README", feature list, "Adaptive residency").
The library keeps that count as a by-product of ordering the pairs: moe_layer adds
each call's per-expert counts to the caller's array on every path (the chained
decode kernels, the GEMV path and the tensor-core path), and moe_expert_counts_add
does it for callers of moe_permute.  Counts are integers: they must equal the
oracle's (oracle.expert_counts over the oracle's routing) bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import quantized_routed_expert_sigmoid_gb300 as moe
import synth
from helpers import make_layer, route_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,path", [(1, "decode_chain"), (3, "decode_chain"), (9, "gemv"), (300, "tensor")])
def test_layer_counts_every_path(T, path):
    tl = make_layer(synth.DECODE, 31, T)
    E = tl.shape.E
    counts = torch.zeros(E, dtype=torch.int64, device="cuda")
    layer = tl.moe_layer(expert_counts=counts)
    assert layer.path(T) == path
    x = tl.x.cuda()
    calls = 3
    for _ in range(calls):
        layer(x)
    torch.cuda.synchronize()
    bias = None if tl.bias is None else tl.bias.numpy()
    ids, _, _ = route_oracle(tl.shape, tl.x.double().numpy(), tl.Wr.numpy(), bias)
    want = None
    for _ in range(calls):
        want = oracle.expert_counts(ids, E, counts=want)
    got = counts.cpu().numpy().astype(np.uint64)
    assert np.array_equal(got, want)
    assert int(got.sum()) == calls * T * tl.shape.k
    assert layer.device_status(T) == 0


def test_layer_counts_graph_replay():
    # one captured decode step replayed: every replay adds the step's counts
    T = 2
    tl = make_layer(synth.DECODE, 32, T)
    E = tl.shape.E
    counts = torch.zeros(E, dtype=torch.int64, device="cuda")
    layer = tl.moe_layer(expert_counts=counts)
    x = tl.x.cuda()
    out = torch.empty(T, tl.shape.H, device="cuda")
    layer.ensure_workspace(T)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x, out=out)                    # warm up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x, out=out)
    torch.cuda.synchronize()
    counts.zero_()
    replays = 5
    for _ in range(replays):
        g.replay()
    torch.cuda.synchronize()
    bias = None if tl.bias is None else tl.bias.numpy()
    ids, _, _ = route_oracle(tl.shape, tl.x.double().numpy(), tl.Wr.numpy(), bias)
    want = None
    for _ in range(replays):
        want = oracle.expert_counts(ids, E, counts=want)
    assert np.array_equal(counts.cpu().numpy().astype(np.uint64), want)


@pytest.mark.parametrize("T,k,E", [(1, 8, 128), (700, 8, 128), (3000, 3, 1000)])
def test_counts_add_after_permute(T, k, E):
    rng = np.random.default_rng(T + 5 * E)
    p = 1.0 / np.arange(1, E + 1)
    p[E // 2] = 0.0                           # one expert never chosen
    p /= p.sum()
    ids_np = np.stack([np.sort(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]).astype(np.int32)
    ids = torch.from_numpy(ids_np).cuda()
    P = T * k
    sp = torch.empty(P, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pp = torch.empty(P, dtype=torch.int32, device="cuda")
    nb = moe.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    counts = torch.zeros(E, dtype=torch.int64, device="cuda")
    for _ in range(2):
        moe.moe_permute(ids, T, k, E, sp, off, pp, ws, nb)
        moe.moe_expert_counts_add(off, E, counts)
    torch.cuda.synchronize()
    want = oracle.expert_counts(ids_np, E)
    want = oracle.expert_counts(ids_np, E, counts=want)
    assert np.array_equal(counts.cpu().numpy().astype(np.uint64), want)


def test_counts_add_rejects_bad_arguments():
    off = torch.zeros(9, dtype=torch.int32, device="cuda")
    counts = torch.zeros(8, dtype=torch.int64, device="cuda")
    with pytest.raises(RuntimeError):
        moe.moe_expert_counts_add(off, 0, counts)
    with pytest.raises(RuntimeError):
        moe.moe_expert_counts_add(None, 8, counts)
