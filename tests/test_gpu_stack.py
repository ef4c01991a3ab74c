"""The 48-layer stack: x <- x + MoE_l(bf16(RMSNorm_l(x))), one residual block per layer call.

Each layer is the decode-shaped layer (hidden 2048, 128 experts, top-8, I=768,
Q4_K); every token count of the sweep T in {1, 2, 4, 8, 16, 32, 64} runs all 48
layers.  Layer l's router is drawn so that the oracle's own chain keeps a 1e-3
routing margin (a layer whose margin falls below it on the oracle chain gets its
router redrawn from a new seed before the chain continues).

Parity is checked per layer with teacher forcing in the oracle's direction: the
GPU's layer l runs on the oracle chain's own input to layer l (the oracle's bf16
RMSNorm output, exact bf16 values), so no GPU value ever enters the oracle:
  - routing ids bit-exact at every layer and token (the router draw keeps the
    1e-3 margin on exactly these inputs);
  - the layer's MoE output within rel-L2 1e-4 of the oracle's.
The GPU's own chain (pre-norm inside the call, residual add, 48 calls in one
CUDA graph) is then checked bit for bit against its parts: each residual block
equals x + layer(bf16(RMSNorm(x))) computed by the separate kernels, the pre-norm
call routes like the plain layer, and the graph replays the eager chain.  The
distance of the whole GPU chain from the oracle's own chain is reported beside
the oracle's distance from itself under flipped bf16 roundings; it is not a
pass/fail bar, because past the first layers it measures how depth amplifies
rounding steps, not the GPU.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MIN_GAP, OQ, TOL_GEMV, oracle_mode, rel_l2

pytestmark = pytest.mark.gpu

N_LAYERS = 48
EPS = 1e-6
SHAPE = synth.DECODE
STACK_T = [1, 2, 4, 8, 16, 32, 64]

_WEIGHTS: dict[int, dict] = {}


def _weights(l: int) -> dict:
    """Layer l's RMSNorm weight and expert tensors (GPU), shared by every T of the sweep."""
    if l not in _WEIGHTS:
        lseed = 5000 + l
        _WEIGHTS[l] = dict(gamma=synth.gamma(SHAPE.H, lseed, l),
                           gate=synth.expert_stack(SHAPE, lseed, l, "gate", "cuda"),
                           up=synth.expert_stack(SHAPE, lseed, l, "up", "cuda"),
                           down=synth.expert_stack(SHAPE, lseed, l, "down", "cuda"))
    return _WEIGHTS[l]


def _spec(W: dict, Wr: torch.Tensor, experts) -> oracle.LayerSpec:
    """The oracle's view of one layer; only `experts` carry their bytes (the rest are zero)."""
    s = SHAPE
    rb_h, rb_i = synth.row_bytes(s.qtype, s.H), synth.row_bytes(s.qtype, s.I)
    g = np.zeros((s.E, s.I, rb_h), np.uint8)
    u = np.zeros((s.E, s.I, rb_h), np.uint8)
    d = np.zeros((s.E, s.H, rb_i), np.uint8)
    idx = np.asarray(sorted(set(int(e) for e in np.asarray(experts).reshape(-1))), dtype=np.int64)
    ti = torch.from_numpy(idx).cuda()
    g[idx] = W["gate"].index_select(0, ti).cpu().numpy()
    u[idx] = W["up"].index_select(0, ti).cpu().numpy()
    d[idx] = W["down"].index_select(0, ti).cpu().numpy()
    return oracle.LayerSpec(mode=oracle_mode(s), E=s.E, k=s.k, H=s.H, I=s.I, qtype=OQ[s.qtype],
                            gate=g, up=u, down=d, Wr=Wr.numpy())


def _round_bf16(u):
    return np.vectorize(oracle.round_bf16)(u)


def _bf16_midpoint_flips(u, rel=1e-6):
    """bf16(u), except that elements within rel of a rounding midpoint take the other
    neighbour (a less precise RMSNorm may land on either side there)."""
    r = _round_bf16(u)
    f = np.abs(u).astype(np.float32)
    lo_bits = f.view(np.uint32) & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = (lo_bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    mid = 0.5 * (lo + hi)
    amb = np.abs(np.abs(u) - mid) <= rel * np.abs(u)
    other = np.where(np.abs(r) == lo, hi, lo) * np.sign(u)
    return np.where(amb, other, r)


def _oracle_chain(layers, x, rounding=_round_bf16, n_threads=None):
    """The oracle's chain from x (fp64): the residual stream after every layer and the ids."""
    n_threads = n_threads or oracle.max_threads()
    xs, ids = [], []
    for l, L in enumerate(layers):
        W = _weights(l)
        u = rounding(oracle.rmsnorm(x, W["gamma"].numpy(), EPS))
        lg = oracle.router_logits(u, L["Wr"].numpy())
        sel, _, _ = oracle.route(oracle_mode(SHAPE), lg, SHAPE.k)
        x = x + oracle.moe_layer(_spec(W, L["Wr"], sel), u, logits=lg, n_threads=n_threads)["out"]
        xs.append(x)
        ids.append(sel)
    return xs, ids


def _build_stack(T: int, seed: int = 5):
    """x0 and the 48 layers' routers, each drawn so that the oracle's own chain keeps the
    routing margin at that layer; also the oracle chain's state after every layer."""
    x0 = synth.activations(T, SHAPE.H, seed, "bf16").float()
    x = x0.double().numpy()
    layers = []
    nt = oracle.max_threads()
    for l in range(N_LAYERS):
        W = _weights(l)
        u = _round_bf16(oracle.rmsnorm(x, W["gamma"].numpy(), EPS))
        for attempt in range(50):
            Wr = synth.router_weight(SHAPE, 5000 + l, l, attempt=attempt)
            lg = oracle.router_logits(u, Wr.numpy())
            ids, _, gaps = oracle.route(oracle_mode(SHAPE), lg, SHAPE.k)
            if gaps[:, 0].min() >= MIN_GAP:
                break
        else:
            raise RuntimeError("no router draw met the margin")
        y = oracle.moe_layer(_spec(W, Wr, ids), u, logits=lg, n_threads=nt)["out"]
        x = x + y
        layers.append(dict(Wr=Wr, ids=ids, u=u, y=y, x_after=x))
    return x0, layers


def _gpu_layers(layers):
    """Per layer: the production residual block (pre-norm inside the call, out == x) and the
    plain layer on a bf16 input (no residual add)."""
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    fused, plain = [], []
    for l, L in enumerate(layers):
        W = _weights(l)
        kw = dict(mode="softmax", E=SHAPE.E, k=SHAPE.k, H=SHAPE.H, I=SHAPE.I, qtype=SHAPE.qtype,
                  gate=W["gate"], up=W["up"], down=W["down"], W_router=L["Wr"].cuda())
        fused.append(MoeLayer(**kw, accumulate=True, x_dtype="f32", norm_gamma=W["gamma"].cuda(), norm_eps=EPS))
        plain.append(MoeLayer(**kw, accumulate=False, x_dtype="bf16"))
    return fused, plain


@pytest.mark.parametrize("T", STACK_T)
def test_stack_48_layers(T):
    """Per-layer parity on the oracle chain's inputs over 48 layers, then the GPU chain checked
    bit for bit: the residual block equals x + layer(norm(x)) exactly, the pre-norm call routes
    like the plain layer, and the captured graph of 48 calls replays the eager chain's bits.
    The distance of the whole chain from the oracle's own chain is printed, not bounded."""
    import quantized_routed_expert_sigmoid_gb300 as moe
    x0, layers = _build_stack(T)
    fused, plain = _gpu_layers(layers)
    H = SHAPE.H

    # ---- teacher forcing: the GPU's layer l on the oracle's input to layer l
    worst = 0.0
    for l in range(N_LAYERS):
        ul = torch.from_numpy(layers[l]["u"]).to(torch.bfloat16).cuda()     # exact: bf16 values
        m = plain[l](ul)
        torch.cuda.synchronize()
        ids, _, _ = plain[l].debug_views(T)
        assert np.array_equal(ids.numpy(), layers[l]["ids"]), f"layer {l}: routing ids differ"
        assert plain[l].device_status(T) == 0
        err = rel_l2(m.cpu().double().numpy(), layers[l]["y"])
        worst = max(worst, err)
        assert err <= TOL_GEMV, f"layer {l}: rel-L2 {err:.3e} > {TOL_GEMV}"

    # ---- the GPU's own chain: each residual block against its parts
    x = x0.cuda().contiguous().clone()
    u = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    gpu_ids, after = [], []
    for l in range(N_LAYERS):
        W = _weights(l)
        x_in = x.clone()
        moe.moe_rmsnorm_bf16(x, W["gamma"].cuda(), T, H, EPS, u)
        m = plain[l](u)
        fused[l](x, out=x)
        torch.cuda.synchronize()
        assert torch.equal(x, x_in + m), f"layer {l}: the residual block is not x + layer(norm(x))"
        ids_p, _, _ = plain[l].debug_views(T)
        ids_f, _, _ = fused[l].debug_views(T)
        assert torch.equal(ids_p, ids_f), f"layer {l}: pre-norm call routes differently"
        assert fused[l].device_status(T) == 0 and plain[l].device_status(T) == 0
        gpu_ids.append(ids_p.numpy())
        after.append(x.cpu().double().numpy())

    # ---- the whole stack as one captured graph: the eager chain's bits
    eager_final = x.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def run(stream=None):
        for m in fused:
            m(x, out=x, stream=stream)

    x.copy_(x0.cuda())
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
    for l in range(N_LAYERS):
        ids_f, _, _ = fused[l].debug_views(T)
        assert np.array_equal(ids_f.numpy(), gpu_ids[l]), f"replay, layer {l}: routing ids differ"

    # ---- end-to-end distance from the oracle's own chain: reported, not a pass/fail bar.  The
    # checks above give every GPU layer within 1e-4 of the oracle's on the same input and the
    # GPU chain composed of those layers bit for bit; what separates the two chains after many
    # layers is each chain's response to slightly different inputs (each bf16 rounding of a
    # layer input is a step, and depth amplifies the steps), which the oracle's rerun with
    # midpoint-flipped roundings shows beside it.
    flip, _ = _oracle_chain(layers, x0.double().numpy(), rounding=_bf16_midpoint_flips)
    drift = [(rel_l2(after[l], layers[l]["x_after"]), rel_l2(flip[l], layers[l]["x_after"])) for l in range(N_LAYERS)]
    print(f"T={T}: per-layer worst rel-L2 {worst:.2e}; distance from the oracle chain (gpu, oracle flip rerun) "
          f"every 8 layers:",
          [(f"{a:.1e}", f"{b:.1e}") for a, b in drift[::8]], f"final {drift[-1][0]:.2e}")
