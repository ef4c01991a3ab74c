"""Shared test helpers: seeded layers with a routing margin, oracle specs, tolerances.

The routing margin: selection must be unambiguous between the fp32 GPU path
and the fp64 oracle, so every token's k-th and (k+1)-th scores (and, in the
sigmoid-group mode, the kept and the first dropped group scores) must differ
by at least 1e-3, measured by the oracle in fp64 on the stored activations.
A token that misses the margin is redrawn from its own seed sub-stream.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

MIN_GAP = 1e-3
TOL_GEMV = 1e-4      # rel-L2 bound, fp32-accumulate dequant-GEMV path
TOL_TC = 5e-3        # rel-L2 bound, fp16-operand tensor-core path

OQ = {synth.Q8_0: oracle.Q8_0, synth.Q4_K: oracle.Q4_K, synth.Q5_K: oracle.Q5_K, synth.Q6_K: oracle.Q6_K,
      synth.Q3_K: oracle.Q3_K, synth.MXFP4: oracle.MXFP4}


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def oracle_mode(shape: synth.LayerShape) -> int:
    return oracle.ROUTE_SIGMOID_GROUP if shape.mode == "sigmoid_group" else oracle.ROUTE_SOFTMAX


def route_oracle(shape, x64, Wr, bias):
    lg = oracle.router_logits(x64, Wr)
    return oracle.route(oracle_mode(shape), lg, shape.k, bias=bias, n_groups=shape.n_groups,
                        topk_groups=shape.topk_groups, renormalize=shape.renormalize, scale=shape.scale)


def gapped_activations(shape: synth.LayerShape, seed: int, T: int, Wr: np.ndarray, bias, max_rounds: int = 100):
    """x [T, H] (bf16 or fp32 torch, CPU) whose routing margin is >= MIN_GAP for every token."""
    token_seeds = list(range(T))
    x = synth.activations(T, shape.H, seed, shape.x_dtype, token_seeds=token_seeds)
    for _ in range(max_rounds):
        _, _, gaps = route_oracle(shape, x.double().numpy(), Wr, bias)
        bad = np.where(gaps.min(axis=1) < MIN_GAP)[0]
        if bad.size == 0:
            return x
        for t in bad:
            token_seeds[t] += 1_000_003
            x[t] = synth.activations(1, shape.H, seed, shape.x_dtype, token_seeds=[token_seeds[t]])[0]
    raise RuntimeError("could not reach the routing margin")


class SeededLayer:
    """A seeded layer: weights on the GPU (exact for `exact` experts), oracle view on the host."""

    def __init__(self, shape: synth.LayerShape, seed: int, x: torch.Tensor, exact=None, layer: int = 0,
                 Wr=None, bias=None, device="cuda"):
        self.shape = shape
        self.seed = seed
        self.Wr = synth.router_weight(shape, seed, layer) if Wr is None else Wr
        self.bias = synth.bias(shape, seed, layer) if bias is None else bias
        self.x = x
        self.bank = synth.ExpertBank(shape, seed, layer, exact=exact, fill_device=device, out_device=device)
        self.exact = set(range(shape.E)) if exact is None else set(int(e) for e in exact)

    def spec(self, experts=None) -> oracle.LayerSpec:
        """Oracle view of the layer; only `experts` (default: all exact ones) carry their bytes."""
        s = self.shape
        rb_h, rb_i = synth.row_bytes(s.qtype, s.H), synth.row_bytes(s.qtype, s.I)
        gate = np.zeros((s.E, s.I, rb_h), np.uint8)
        up = np.zeros((s.E, s.I, rb_h), np.uint8)
        down = np.zeros((s.E, s.H, rb_i), np.uint8)
        for e in sorted(self.exact if experts is None else experts):
            gate[e] = self.bank.gate[e].cpu().numpy()
            up[e] = self.bank.up[e].cpu().numpy()
            down[e] = self.bank.down[e].cpu().numpy()
        kw = {}
        if s.I_s > 0:
            kw = dict(shared_qtype=OQ[s.shared_qtype], I_s=s.I_s, s_gate=self.bank.shared[0].cpu().numpy(),
                      s_up=self.bank.shared[1].cpu().numpy(), s_down=self.bank.shared[2].cpu().numpy())
        return oracle.LayerSpec(mode=oracle_mode(s), E=s.E, k=s.k, H=s.H, I=s.I, qtype=OQ[s.qtype], gate=gate,
                                up=up, down=down, Wr=self.Wr.numpy(),
                                bias=None if self.bias is None else self.bias.numpy(),
                                n_groups=s.n_groups, topk_groups=s.topk_groups, renormalize=s.renormalize,
                                scale=s.scale, **kw)

    def moe_layer(self, accumulate=False, tc_min_tokens=0, expert_counts=None):
        from quantized_routed_expert_sigmoid_gb300 import MoeLayer
        s = self.shape
        sh = self.bank.shared
        return MoeLayer(mode=s.mode, E=s.E, k=s.k, H=s.H, I=s.I, qtype=s.qtype, gate=self.bank.gate,
                        up=self.bank.up, down=self.bank.down, W_router=self.Wr.cuda(),
                        bias=None if self.bias is None else self.bias.cuda(), n_groups=s.n_groups,
                        topk_groups=s.topk_groups, scale=s.scale, renormalize=s.renormalize, x_dtype=s.x_dtype,
                        I_s=s.I_s, shared_qtype=s.shared_qtype, s_gate=sh[0] if sh else None,
                        s_up=sh[1] if sh else None, s_down=sh[2] if sh else None, accumulate=accumulate,
                        tc_min_tokens=tc_min_tokens, expert_counts=expert_counts)


def make_layer(shape: synth.LayerShape, seed: int, T: int, exact_all: bool = False, device="cuda"):
    """Seeded layer + gap-enforced x; exact weights for the experts the oracle routes to."""
    Wr = synth.router_weight(shape, seed, 0)
    bias = synth.bias(shape, seed, 0)
    x = gapped_activations(shape, seed, T, Wr.numpy(), None if bias is None else bias.numpy())
    ids, _, _ = route_oracle(shape, x.double().numpy(), Wr.numpy(), None if bias is None else bias.numpy())
    exact = None if exact_all else sorted(set(ids.reshape(-1).tolist()))
    return SeededLayer(shape, seed, x, exact=exact, Wr=Wr, bias=bias, device=device)
