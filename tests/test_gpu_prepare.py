"""Weight preparation (moe_weights_prepare: Q8_0 -> MOE_Q8_0_R) and mixed weight types, on the GPU.

The repack is pure data movement, so it is checked byte for byte against the
layout the header defines, restated here from the GGUF block (fp16 d, 32 int8
q): per row the blocks' 32-byte quant runs, then their 2-byte scales, padded
to 16 bytes.  Layers whose Q8_0 matrices were prepared are checked against the
oracle run on the original, unprepared blocks: same values, so the bar is the
path's usual tolerance.  The mixed case (Q4_K gate/up with a Q8_0 down matrix,
a combination GGUF files use) runs the GEMV path against the oracle's
separate down type.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OQ, TOL_GEMV, TOL_TC, make_layer, oracle_mode, rel_l2
from quantized_routed_expert_sigmoid_gb300 import MoeLayer
from quantized_routed_expert_sigmoid_gb300 import _native as N
from quantized_routed_expert_sigmoid_gb300.layer import prepare_q8_0

pytestmark = pytest.mark.gpu


def _repack_reference(blocks: np.ndarray, K: int) -> np.ndarray:
    """[rows, K/32*34] Q8_0 bytes -> [rows, row_bytes] in the MOE_Q8_0_R layout."""
    rows = blocks.shape[0]
    nb = K // 32
    b = blocks.reshape(rows, nb, 34)
    pad = (2 * nb + 15) // 16 * 16
    out = np.zeros((rows, 32 * nb + pad), np.uint8)
    out[:, :32 * nb] = b[:, :, 2:].reshape(rows, 32 * nb)
    out[:, 32 * nb:32 * nb + 2 * nb] = b[:, :, :2].reshape(rows, 2 * nb)
    return out


@pytest.mark.parametrize("E,rows,K", [(1, 64, 7168), (3, 40, 96), (2, 16, 2048)])
def test_prepare_is_the_documented_byte_layout(E, rows, K):
    w = synth.normal((E * rows, K), 0.02, 91 + K, "cuda")
    q = synth.encode_q8_0(w).view(E, rows, -1)
    before = q.clone()
    r = prepare_q8_0(q, rows, K, n_experts=E)
    torch.cuda.synchronize()
    assert torch.equal(q, before), "the source was modified"
    got = r.cpu().numpy().reshape(E * rows, -1)
    ref = _repack_reference(q.cpu().numpy().reshape(E * rows, -1), K)
    assert np.array_equal(got, ref)


def _shared_layer(tl, prepared: bool, tc_min_tokens: int = 0):
    """tl's layer with its Q8_0 shared expert as stored or prepared."""
    s = tl.shape
    sg, su, sd = tl.bank.shared
    if prepared:
        sg, su, sd = prepare_q8_0(sg, s.I_s, s.H), prepare_q8_0(su, s.I_s, s.H), prepare_q8_0(sd, s.H, s.I_s)
    return MoeLayer(mode=s.mode, E=s.E, k=s.k, H=s.H, I=s.I, qtype=s.qtype, gate=tl.bank.gate, up=tl.bank.up,
                    down=tl.bank.down, W_router=tl.Wr.cuda(), bias=None if tl.bias is None else tl.bias.cuda(),
                    n_groups=s.n_groups, topk_groups=s.topk_groups, scale=s.scale, renormalize=s.renormalize,
                    x_dtype=s.x_dtype, I_s=s.I_s, shared_qtype="q8_0_r" if prepared else "q8_0", s_gate=sg, s_up=su,
                    s_down=sd, tc_min_tokens=tc_min_tokens)


def _against_oracle(tl, layer, T, tol, sample=None):
    out = layer(tl.x.cuda())
    torch.cuda.synchronize()
    ids, _, _ = layer.debug_views(T)
    sample = np.arange(T) if sample is None else np.asarray(sample)
    ref = oracle.moe_layer(tl.spec(), tl.x[sample].double().numpy(), n_threads=oracle.max_threads())
    assert np.array_equal(ids.numpy()[sample], ref["ids"])
    err = rel_l2(out.cpu().numpy()[sample], ref["out"])
    assert err <= tol, f"rel-L2 {err:.3e} > {tol}"
    assert layer.device_status(T) == 0
    return out


def test_prepared_shared_expert_deepseek_shape_T2():
    # hidden 7168, 256 experts, sigmoid-group routing, Q8_0 shared expert I=2048 (GEMV path)
    tl = make_layer(synth.DEEPSEEK, 4, 2)
    plain = _against_oracle(tl, _shared_layer(tl, False), 2, TOL_GEMV)
    prep = _against_oracle(tl, _shared_layer(tl, True), 2, TOL_GEMV)
    # same values in another layout, same summation order: the same bits
    assert torch.equal(plain, prep)


def test_prepared_shared_expert_decode_chain():
    shape = synth.LayerShape(H=2048, E=64, k=4, I=768, qtype=synth.Q4_K, mode="sigmoid_group", n_groups=8,
                             topk_groups=4, scale=2.5, I_s=512, shared_qtype=synth.Q8_0, bias_std=0.1)
    tl = make_layer(shape, 61, 2, exact_all=True)
    layer = _shared_layer(tl, True)
    assert layer.path(2) == "decode_chain"
    prep = _against_oracle(tl, layer, 2, TOL_GEMV)
    assert torch.equal(prep, _shared_layer(tl, False)(tl.x.cuda()))


def test_prepared_shared_expert_tensor_cores():
    shape = synth.LayerShape(H=1024, E=32, k=4, I=512, qtype=synth.Q4_K, mode="sigmoid_group", n_groups=4,
                             topk_groups=2, scale=2.5, I_s=1024, shared_qtype=synth.Q8_0, bias_std=0.1)
    T = 300
    tl = make_layer(shape, 62, T, exact_all=True)
    layer = _shared_layer(tl, True, tc_min_tokens=1)
    assert layer.path(T) == "tensor"
    prep = _against_oracle(tl, layer, T, TOL_TC, sample=np.arange(0, T, 7))
    plain = _shared_layer(tl, False, tc_min_tokens=1)(tl.x.cuda())
    assert torch.equal(prep, plain)


@pytest.mark.parametrize("T", [3, 40])
def test_mixed_q4k_gate_up_with_q8_0_down(T):
    # Q4_K gate/up with the down matrix stored in Q8_0 (and, second, prepared): GEMV path
    shape = synth.LayerShape(H=1024, E=16, k=4, I=512, qtype=synth.Q4_K)
    seed = 63
    tl = make_layer(shape, seed, T, exact_all=True)
    dshape = dataclasses.replace(shape, qtype=synth.Q8_0)
    down8 = torch.stack([synth.expert_matrix(dshape, seed, 0, "down", e, "cuda") for e in range(shape.E)])
    spec = tl.spec()
    spec = oracle.LayerSpec(mode=oracle_mode(shape), E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=OQ[shape.qtype],
                            gate=spec.gate, up=spec.up, down=down8.cpu().numpy(), Wr=tl.Wr.numpy(),
                            qtype_down=oracle.Q8_0)
    ref = oracle.moe_layer(spec, tl.x.double().numpy(), n_threads=oracle.max_threads())
    outs = []
    for qd, dn in (("q8_0", down8), ("q8_0_r", prepare_q8_0(down8, shape.H, shape.I, n_experts=shape.E))):
        layer = MoeLayer(mode="softmax", E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
                         gate=tl.bank.gate, up=tl.bank.up, down=dn, W_router=tl.Wr.cuda(), qtype_down=qd)
        assert layer.path(T) == "gemv"
        out = layer(tl.x.cuda())
        torch.cuda.synchronize()
        ids, _, _ = layer.debug_views(T)
        assert np.array_equal(ids.numpy(), ref["ids"])
        err = rel_l2(out.cpu().numpy(), ref["out"])
        assert err <= TOL_GEMV, f"{qd} down: rel-L2 {err:.3e}"
        assert layer.device_status(T) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
