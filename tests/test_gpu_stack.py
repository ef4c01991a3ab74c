"""The 48-layer stack: x <- x + MoE_l(bf16(RMSNorm_l(x))), captured as one CUDA graph.

Each layer is the decode-shaped layer (hidden 2048, 128 experts, top-8, I=768,
Q4_K).  The oracle runs its own chain in fp64 (it never sees a GPU value);
routing ids must match at every layer whose routing the oracle's own reruns
leave unchanged, the first layer must meet the single-layer tolerance, and the
drift after every later layer must stay within a bound the oracle measures for
itself (see the test).  A layer whose routing margin
(measured on the oracle chain) falls below 1e-3 gets its router redrawn from a
new seed before the chain continues.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MIN_GAP, OQ, oracle_mode, rel_l2

pytestmark = pytest.mark.gpu

N_LAYERS = 48
EPS = 1e-6


def _bf16_neighbours(u):
    """The two bf16 values around each element of u (fp64), and the midpoint between them."""
    f = np.abs(u).astype(np.float32)
    lo_bits = f.view(np.uint32) & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = (lo_bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    return lo, hi, 0.5 * (lo + hi)


def _round_other_way(u, rel=1e-6):
    """bf16(u), except that elements within rel of a rounding midpoint take the other
    neighbour: a computation of u in lower precision may land on either side there."""
    r = np.vectorize(oracle.round_bf16)(u)
    lo, hi, mid = _bf16_neighbours(u)
    amb = np.abs(np.abs(u) - mid) <= rel * np.abs(u)
    other = np.where(np.abs(r) == lo, hi, lo) * np.sign(u)
    return np.where(amb, other, r)


def _oracle_chain(layers, shape, x, flip_rel=0.0):
    """The oracle's own chain from x (fp64), returning x and the routing ids after every
    layer.  flip_rel > 0 rounds the RMSNorm outputs that sit within flip_rel of a bf16
    rounding midpoint the other way (the rounding a less precise RMSNorm may legitimately
    take)."""
    xs, ids = [], []
    for L in layers:
        u = oracle.rmsnorm(x, L["gamma"].numpy(), EPS)
        u = _round_other_way(u, flip_rel) if flip_rel > 0 else np.vectorize(oracle.round_bf16)(u)
        r = oracle.moe_layer(L["spec"], u, n_threads=8)
        x = x + r["out"]
        xs.append(x)
        ids.append(r["ids"])
    return xs, ids


def _first_rerouted(layers, *id_chains):
    """First layer at which any rerun of the oracle chain routes differently from the
    reference chain (len(layers) if none does)."""
    for l, L in enumerate(layers):
        if any(not np.array_equal(ch[l], L["ids"]) for ch in id_chains):
            return l
    return len(layers)


def _build_stack(T, seed=5, n_layers=N_LAYERS):
    shape = synth.DECODE
    x0 = synth.activations(T, shape.H, seed, "bf16").float()
    x = x0.double().numpy()
    layers = []
    for l in range(n_layers):
        lseed = 5000 + l
        gamma = synth.gamma(shape.H, lseed, l)
        u = oracle.rmsnorm(x, gamma.numpy(), EPS)
        u = np.vectorize(oracle.round_bf16)(u)
        for attempt in range(50):
            Wr = synth.router_weight(shape, lseed, l, attempt=attempt)
            lg = oracle.router_logits(u, Wr.numpy())
            ids, w, gaps = oracle.route(oracle_mode(shape), lg, shape.k)
            if gaps[:, 0].min() >= MIN_GAP:
                break
        else:
            raise RuntimeError("no router draw met the margin")
        gate = synth.expert_stack(shape, lseed, l, "gate", "cuda")
        up = synth.expert_stack(shape, lseed, l, "up", "cuda")
        down = synth.expert_stack(shape, lseed, l, "down", "cuda")
        used = sorted(set(ids.reshape(-1).tolist()))
        rb_h, rb_i = synth.row_bytes(shape.qtype, shape.H), synth.row_bytes(shape.qtype, shape.I)
        g_np = np.zeros((shape.E, shape.I, rb_h), np.uint8)
        u_np = np.zeros_like(g_np)
        d_np = np.zeros((shape.E, shape.H, rb_i), np.uint8)
        for e in used:
            g_np[e], u_np[e], d_np[e] = gate[e].cpu().numpy(), up[e].cpu().numpy(), down[e].cpu().numpy()
        spec = oracle.LayerSpec(mode=oracle_mode(shape), E=shape.E, k=shape.k, H=shape.H, I=shape.I,
                                qtype=OQ[shape.qtype], gate=g_np, up=u_np, down=d_np, Wr=Wr.numpy())
        y = oracle.moe_layer(spec, u, n_threads=8)["out"]
        x = x + y
        layers.append(dict(gamma=gamma, Wr=Wr, gate=gate, up=up, down=down, ids=ids, spec=spec, x_after=x))
    return shape, x0, layers, x


def _gpu_stack(shape, x0, layers, T):
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    import quantized_routed_expert_sigmoid_gb300 as moe
    mls = [MoeLayer(mode="softmax", E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
                    gate=L["gate"], up=L["up"], down=L["down"], W_router=L["Wr"].cuda(), accumulate=True)
           for L in layers]
    gammas = [L["gamma"].cuda() for L in layers]
    for m in mls:
        m.ensure_workspace(T)
    x = x0.cuda().contiguous()
    u = torch.empty(T, shape.H, dtype=torch.bfloat16, device="cuda")

    def run(stream=None):
        for m, g in zip(mls, gammas):
            moe.moe_rmsnorm_bf16(x, g, T, shape.H, EPS, u, stream)
            m(u, out=x, stream=stream)

    return mls, x, run


@pytest.mark.parametrize("T", [1, 2])
def test_stack_48_layers_graph(T):
    """Ids bit-exact where the oracle's routing is decided; drift within a bound the oracle sets.

    The stack is a deep residual chain whose bf16 rounding of each layer's input
    is a discontinuous step, so tiny differences grow with depth.  The bound on
    the GPU's distance from the oracle after layer l is derived from the oracle
    alone, from two reruns of its chain: one from an input perturbed by 1e-6
    (relative), and one that rounds every RMSNorm output lying within 1e-6 of a
    bf16 rounding midpoint to the other neighbour (the GPU computes RMSNorm in
    fp32, so such elements may round either way).  The larger of the two
    divergences after layer l, times 10, plus the single-layer tolerance, is the
    allowed distance.  The same reruns say how far down the routing is decided: from
    the first layer at which either of them picks other experts than the reference
    chain, a 1e-6 change of the input already reroutes the oracle itself, so from there
    on only the drift bound applies (the reference keeps a 1e-3 margin on its own
    inputs, but the drift of any chain grows with depth).  At least the first 32 layers
    must stay decided, so the test keeps checking ids over two thirds of the stack.
    """
    shape, x0, layers, x_ref = _build_stack(T)
    rng = np.random.default_rng(7)
    x0_64 = x0.double().numpy()
    pert, pert_ids = _oracle_chain(layers, shape, x0_64 * (1.0 + 1e-6 * rng.standard_normal(x0_64.shape)))
    flip, flip_ids = _oracle_chain(layers, shape, x0_64, flip_rel=1e-6)
    decided = _first_rerouted(layers, pert_ids, flip_ids)
    assert decided >= 32, f"the oracle's own reruns reroute at layer {decided}"
    mls, x, run = _gpu_stack(shape, x0, layers, T)
    # eager, layer by layer: the GPU chain next to the oracle chain (never fed into it)
    import quantized_routed_expert_sigmoid_gb300 as moe
    u = torch.empty(T, shape.H, dtype=torch.bfloat16, device="cuda")
    x.copy_(x0.cuda())
    drift = []
    for l, (m, L) in enumerate(zip(mls, layers)):
        moe.moe_rmsnorm_bf16(x, L["gamma"].cuda(), T, shape.H, EPS, u)
        m(u, out=x)
        torch.cuda.synchronize()
        ids, _, _ = m.debug_views(T)
        if l < decided:
            assert np.array_equal(ids.numpy(), L["ids"]), f"layer {l}: routing ids differ"
        err = rel_l2(x.cpu().numpy(), L["x_after"])
        self_div = max(rel_l2(pert[l], L["x_after"]), rel_l2(flip[l], L["x_after"]))
        drift.append((err, self_div))
        assert err <= 1e-4 + 10 * self_div, f"layer {l}: rel-L2 {err:.3e}, oracle self-divergence {self_div:.3e}"
    eager_final = x.clone()
    assert drift[0][0] <= 1e-4                                         # one layer: the single-layer bar
    # the same stack with the RMSNorm inside each layer call (pre-norm; the chain computes it
    # itself): one call per layer on the residual stream, the bits of the separate kernels
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    fused = [MoeLayer(mode="softmax", E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
                      gate=L["gate"], up=L["up"], down=L["down"], W_router=L["Wr"].cuda(), accumulate=True,
                      x_dtype="f32", norm_gamma=L["gamma"].cuda(), norm_eps=EPS)
             for L in layers]
    xf = x0.cuda().contiguous().clone()
    for m in fused:
        m(xf, out=xf)
    torch.cuda.synchronize()
    assert torch.equal(xf, eager_final), "pre-norm layers differ from RMSNorm + layer"
    # capture the 48 layers once, replay from x0: the same bits as the eager chain
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(stream=s)
    x.copy_(x0.cuda())
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(x, eager_final), "graph replay differs from the eager chain"
    for l, (m, L) in enumerate(zip(mls[:decided], layers)):
        ids, _, _ = m.debug_views(T)
        assert np.array_equal(ids.numpy(), L["ids"]), f"replay, layer {l}: routing ids differ"
    print(f"routing decided through layer {decided - 1};",
          "stack drift (gpu vs oracle, oracle self-divergence) per 8 layers:",
          [(f"{a:.1e}", f"{b:.1e}") for a, b in drift[::8]], "final", f"{drift[-1][0]:.2e}")
