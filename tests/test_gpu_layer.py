"""GPU parity of the fused layer (moe_layer through the C ABI) against the fp64 oracle.

Routing ids and per-expert offsets must match bit for bit; the layer output
must be within rel-L2 1e-4 of the oracle on the fp32 GEMV path.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL_GEMV, make_layer, rel_l2

pytestmark = pytest.mark.gpu


def _check_layer(tl, T, tol=TOL_GEMV, n_threads=8, tc_min_tokens=0):
    layer = tl.moe_layer(tc_min_tokens=tc_min_tokens)
    x = tl.x.cuda()
    out = layer(x)
    torch.cuda.synchronize()
    ids, gw, offs = layer.debug_views(T)
    spec = tl.spec()
    ref = oracle.moe_layer(spec, tl.x.double().numpy(), n_threads=n_threads)
    assert np.array_equal(ids.numpy(), ref["ids"]), "routing ids differ"
    _, ref_off, _ = oracle.permute(ref["ids"], tl.shape.E)
    assert np.array_equal(offs.numpy(), ref_off), "expert offsets differ"
    assert np.allclose(gw.numpy(), ref["w"], rtol=1e-5, atol=1e-6), "gates differ"
    err = rel_l2(out.cpu().numpy(), ref["out"])
    assert err <= tol, f"rel-L2 {err:.3e} > {tol}"
    assert layer.device_status(T) == 0
    return layer, out, err


@pytest.mark.parametrize("T", [1, 4, 9])
def test_tiny_q8_0(T):
    tl = make_layer(synth.TINY, 0, T, exact_all=True)
    _check_layer(tl, T)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 6, 7])
def test_decode_q4_k(T):
    tl = make_layer(synth.DECODE, 2, T)
    _check_layer(tl, T)


def test_decode_chain_token_range():
    # at hidden 2048 the chain's staged x and its 16 warps' rings fit up to T = 6 tokens; T = 7
    # and 8 take the GEMV kernels
    tl = make_layer(synth.DECODE, 2, 1)
    layer = tl.moe_layer()
    assert [layer.path(T) for T in range(1, 10)] == ["decode_chain"] * 6 + ["gemv"] * 3


@pytest.mark.parametrize("T", [2, 9, 40])
def test_decode_q4_k_fp32_activations(T):
    # fp32 x: the Q4_K kernels stage it as three byte planes (bf16 x takes two); the chained
    # decode kernels take bf16 values only, so T = 2 runs the separate kernels as well
    shape = dataclasses.replace(synth.DECODE, x_dtype="fp32")
    tl = make_layer(shape, 23, T)
    layer, _, _ = _check_layer(tl, T, tc_min_tokens=1 << 30)
    assert layer.path(T) == "gemv"


@pytest.mark.parametrize("qt", [synth.Q5_K, synth.Q6_K, synth.Q3_K, synth.MXFP4])
@pytest.mark.parametrize("T", [1, 3, 9, 70])
def test_decode_shape_q5_k_q6_k(qt, T):
    # the next expert types on the GEMV kernels (every T): gate/up rows of 2048 weights, down rows
    # of 768, so Q6_K's 210-byte and Q3_K's 110-byte blocks start 2 bytes off a 4-byte boundary in
    # every other row and MXFP4's 17-byte blocks at every byte offset
    shape = dataclasses.replace(synth.DECODE, qtype=qt)
    tl = make_layer(shape, 24, T)
    layer, _, _ = _check_layer(tl, T)
    assert layer.path(T) == "gemv"


@pytest.mark.parametrize("qt", [synth.Q5_K, synth.Q6_K, synth.Q3_K, synth.MXFP4])
def test_small_q5_k_q6_k_fp32(qt):
    # one super-block per row (the short-row lane split) and fp32 activations (three planes)
    shape = synth.LayerShape(H=256, E=8, k=2, I=256, qtype=qt, x_dtype="fp32")
    for T in (1, 4, 13):
        tl = make_layer(shape, 25, T, exact_all=True)
        _check_layer(tl, T)


@pytest.mark.parametrize("T", [1, 9, 70])
def test_q3_k_gate_up_with_q4_k_down(T):
    # the large model's routed-expert mix: Q3_K gate and up, Q4_K down (GEMV kernels at every T;
    # the down matrix takes the segmented Q4_K kernel)
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    from helpers import OQ, oracle_mode
    shape = dataclasses.replace(synth.DECODE, qtype=synth.Q3_K)
    seed = 26
    tl = make_layer(shape, seed, T, exact_all=True)
    dshape = dataclasses.replace(shape, qtype=synth.Q4_K)
    down4 = torch.stack([synth.expert_matrix(dshape, seed, 0, "down", e, "cuda") for e in range(shape.E)])
    spec = tl.spec()
    spec = oracle.LayerSpec(mode=oracle_mode(shape), E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=OQ[shape.qtype],
                            gate=spec.gate, up=spec.up, down=down4.cpu().numpy(), Wr=tl.Wr.numpy(),
                            qtype_down=oracle.Q4_K)
    ref = oracle.moe_layer(spec, tl.x.double().numpy(), n_threads=oracle.max_threads())
    layer = MoeLayer(mode="softmax", E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
                     gate=tl.bank.gate, up=tl.bank.up, down=down4, W_router=tl.Wr.cuda(), qtype_down="q4_k")
    assert layer.path(T) == "gemv"
    out = layer(tl.x.cuda())
    torch.cuda.synchronize()
    ids, _, _ = layer.debug_views(T)
    assert np.array_equal(ids.numpy(), ref["ids"])
    err = rel_l2(out.cpu().numpy(), ref["out"])
    assert err <= TOL_GEMV, f"rel-L2 {err:.3e}"
    assert layer.device_status(T) == 0


def test_decode_q4_k_ragged_batch():
    # 37 tokens: several tokens per expert, passes of 8 pairs plus a ragged tail
    tl = make_layer(synth.DECODE, 21, 37)
    _check_layer(tl, 37, tc_min_tokens=1 << 30)


def test_segmented_gemv_zipf_T120():
    # GEMV path just below the tensor-core threshold with Zipf-skewed routing: the popular
    # experts take many passes of 8 tokens (their work spread over many CTAs by cost), some
    # experts get no token at all; the whole output is compared with the oracle
    from helpers import SeededLayer, route_oracle, MIN_GAP
    shape, seed, T = synth.DECODE, 17, 120
    Wr = synth.router_weight(shape, seed, 0)
    L = synth.zipf_target_logits(T, shape.E, shape.k, seed)
    x = synth.activations_for_logits(L, Wr.numpy(), seed)
    ids, _, gaps = route_oracle(shape, x.double().numpy(), Wr.numpy(), None)
    assert gaps[:, 0].min() >= MIN_GAP
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    assert (counts == 0).sum() >= 8 and counts.max() > 40
    tl = SeededLayer(shape, seed, x, exact=None, Wr=Wr, bias=None)
    layer, _, _ = _check_layer(tl, T, tc_min_tokens=1 << 30)
    assert layer.path(T) == "gemv"


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_prenorm_equals_separate_rmsnorm(T):
    # a pre-norm layer on the fp32 residual stream (the chain computes the RMSNorm itself at
    # T <= 4; the GEMV path runs moe_rmsnorm_bf16 into its workspace) gives the bits of
    # moe_rmsnorm_bf16 followed by the layer on its bf16 output
    import quantized_routed_expert_sigmoid_gb300 as moe
    from quantized_routed_expert_sigmoid_gb300 import MoeLayer
    shape, seed = synth.DECODE, 41
    kw = dict(mode="softmax", E=shape.E, k=shape.k, H=shape.H, I=shape.I, qtype=shape.qtype,
              gate=synth.expert_stack(shape, seed, 0, "gate", "cuda"), up=synth.expert_stack(shape, seed, 0, "up", "cuda"),
              down=synth.expert_stack(shape, seed, 0, "down", "cuda"),
              W_router=synth.router_weight(shape, seed, 0).cuda(), accumulate=True)
    gamma = synth.gamma(shape.H, seed, 0).cuda()
    fused = MoeLayer(**kw, x_dtype="f32", norm_gamma=gamma, norm_eps=1e-6)
    plain = MoeLayer(**kw, x_dtype="bf16")
    assert fused.path(T) == plain.path(T) == ("decode_chain" if T <= 4 else "gemv")
    x0 = 3.0 * synth.activations(T, shape.H, seed, "bf16").float().cuda()
    a = x0.clone()
    fused(a, out=a)
    b = x0.clone()
    u = torch.empty(T, shape.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_rmsnorm_bf16(b, gamma, T, shape.H, 1e-6, u)
    plain(u, out=b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert fused.device_status(T) == 0


def test_deepseek_shape_decode_T2():
    tl = make_layer(synth.DEEPSEEK, 4, 2)
    _check_layer(tl, 2)


def test_sigmoid_group_small_with_shared():
    shape = synth.LayerShape(H=512, E=32, k=4, I=256, qtype=synth.Q4_K, mode="sigmoid_group", n_groups=4,
                             topk_groups=2, scale=2.5, I_s=256, shared_qtype=synth.Q8_0, bias_std=0.1)
    tl = make_layer(shape, 40, 11, exact_all=True)
    _check_layer(tl, 11)


def test_k_equals_E_every_expert_hit():
    shape = synth.LayerShape(H=256, E=4, k=4, I=256, qtype=synth.Q4_K)
    tl = make_layer(shape, 41, 5, exact_all=True)
    _check_layer(tl, 5)


def test_deterministic_and_graph_replay_bitwise():
    tl = make_layer(synth.DECODE, 2, 2)
    layer = tl.moe_layer()
    x = tl.x.cuda()
    out1 = layer(x).clone()
    out2 = layer(x).clone()
    assert torch.equal(out1, out2), "two eager runs differ"
    out_g = torch.zeros_like(out1)
    layer.ensure_workspace(2)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x, out=out_g)           # warm up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x, out=out_g)
    out_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out1), "graph replay differs from eager"


def test_accumulate_is_residual_add():
    tl = make_layer(synth.TINY, 0, 4, exact_all=True)
    plain = tl.moe_layer()(tl.x.cuda()).clone()
    acc_layer = tl.moe_layer(accumulate=True)
    base = torch.randn(4, synth.TINY.H, device="cuda")
    out = base.clone()
    acc_layer(tl.x.cuda(), out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, plain + base)


# ---------------------------------------------------------------- tensor-core path (T >= tc_min_tokens)

def tile_sample(ref_ids, E, bn):
    """Tokens that put at least one checked pair in every (expert, token block) tile of the
    tensor-core GEMM -- the first and the last pair of each block of up to bn pairs of an
    expert's sorted run, so every ragged tail's last pair is among them -- and the number of
    tiles.  The blocks follow from the routing alone (the permutation is bit-exact)."""
    k = ref_ids.shape[1]
    sorted_pairs, offsets, _ = oracle.permute(ref_ids, E)
    tokens, n_tiles = set(), 0
    for e in range(E):
        for p0 in range(int(offsets[e]), int(offsets[e + 1]), bn):
            p1 = min(int(offsets[e + 1]), p0 + bn) - 1
            tokens.add(int(sorted_pairs[p0]) // k)
            tokens.add(int(sorted_pairs[p1]) // k)
            n_tiles += 1
    return np.array(sorted(tokens)), n_tiles


def _check_sampled(tl, T, sample, tol, tc_min_tokens=0, n_threads=None):
    """Whole-layer run on the GPU; routing ids of every token and the outputs of the
    sampled tokens against the oracle (tokens are independent, so the oracle runs on
    the sample alone).  sample=None takes tile_sample of the routing."""
    n_threads = n_threads or oracle.max_threads()
    layer = tl.moe_layer(tc_min_tokens=tc_min_tokens)
    x = tl.x.cuda()
    out = layer(x)
    torch.cuda.synchronize()
    ids, gw, offs = layer.debug_views(T)
    from helpers import route_oracle
    ref_ids, ref_w, _ = route_oracle(tl.shape, tl.x.double().numpy(), tl.Wr.numpy(),
                                     None if tl.bias is None else tl.bias.numpy())
    assert np.array_equal(ids.numpy(), ref_ids), "routing ids differ"
    _, ref_off, _ = oracle.permute(ref_ids, tl.shape.E)
    assert np.array_equal(offs.numpy(), ref_off), "expert offsets differ"
    n_tiles = None
    if sample is None:
        sample, n_tiles = tile_sample(ref_ids, tl.shape.E, 256 if tl.shape.qtype == synth.Q4_K else 128)
    sample = np.asarray(sample)
    need = sorted(set(ref_ids[sample].reshape(-1).tolist()))
    assert set(need) <= tl.exact
    ref = oracle.moe_layer(tl.spec(experts=need), tl.x[sample].double().numpy(), n_threads=n_threads)
    err = rel_l2(out.cpu().numpy()[sample], ref["out"])
    assert err <= tol, f"rel-L2 {err:.3e} > {tol}"
    assert layer.device_status(T) == 0
    print(f"T={T}: {len(sample)} tokens checked against the oracle"
          + (f", covering all {n_tiles} (expert, token block) tiles" if n_tiles else "") + f", rel-L2 {err:.2e}")
    return layer, out, err


def test_tc_tiny_q8_0():
    from helpers import TOL_TC
    for T in (4, 9):
        tl = make_layer(synth.TINY, 0, T, exact_all=True)
        _check_sampled(tl, T, np.arange(T), TOL_TC, tc_min_tokens=1)


def test_default_threshold_T64_T65():
    # the default crossover: T <= 64 takes the GEMV kernels, T = 65 the tensor cores (one
    # token block per expert, every block ragged); both against the oracle on every token
    from helpers import TOL_TC
    for T, path, tol in ((64, "gemv", TOL_GEMV), (65, "tensor", TOL_TC)):
        tl = make_layer(synth.DECODE, 34, T, exact_all=True)
        layer, _, _ = _check_sampled(tl, T, np.arange(T), tol)
        assert layer.path(T) == path


def test_tc_decode_shape_ragged():
    from helpers import TOL_TC
    T = 300                                 # 2400 pairs: many token blocks, a ragged tail per expert
    tl = make_layer(synth.DECODE, 30, T, exact_all=True)
    _check_sampled(tl, T, None, TOL_TC)


def test_tc_prefill_zipf_T4096():
    from helpers import TOL_TC, SeededLayer
    shape, seed, T = synth.DECODE, 3, 4096
    Wr = synth.router_weight(shape, seed, 0)
    L = synth.zipf_target_logits(T, shape.E, shape.k, seed)
    x = synth.activations_for_logits(L, Wr.numpy(), seed)
    from helpers import route_oracle, MIN_GAP
    ids, _, gaps = route_oracle(shape, x.double().numpy(), Wr.numpy(), None)
    assert gaps[:, 0].min() >= MIN_GAP
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    assert (counts == 0).sum() >= 8 and counts.max() > 1000          # uneven, some experts empty
    tl = SeededLayer(shape, seed, x, exact=None, Wr=Wr, bias=None)
    layer, o_tc, _ = _check_sampled(tl, T, None, TOL_TC)
    # the whole output against the fp32 GEMV path on the same layer and tokens
    o_gv = tl.moe_layer(tc_min_tokens=1 << 30)(tl.x.cuda())
    torch.cuda.synchronize()
    err = rel_l2(o_tc.cpu().numpy(), o_gv.cpu().double().numpy())
    assert err <= TOL_TC, f"tensor-core vs GEMV path, all {T} tokens: rel-L2 {err:.3e}"


def test_tc_deepseek_shape_verify_T512():
    from helpers import TOL_TC
    T = 512
    tl = make_layer(synth.DEEPSEEK, 4, T, exact_all=True)
    _check_sampled(tl, T, None, TOL_TC)


def test_tc_deterministic_and_graph_replay():
    tl = make_layer(synth.DECODE, 31, 200, exact_all=True)
    layer = tl.moe_layer()
    x = tl.x.cuda()
    o1 = layer(x).clone()
    o2 = layer(x).clone()
    assert torch.equal(o1, o2)
    out_g = torch.zeros_like(o1)
    layer.ensure_workspace(200)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(x, out=out_g)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(x, out=out_g)
    out_g.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g, o1)


def test_tc_matches_gemv_path():
    """Same layer, same tokens: the tensor-core path stays within its tolerance of the GEMV path."""
    from helpers import TOL_TC
    tl = make_layer(synth.DECODE, 32, 160, exact_all=True)
    o_tc = tl.moe_layer()(tl.x.cuda()).cpu().numpy()
    o_gv = tl.moe_layer(tc_min_tokens=1 << 30)(tl.x.cuda()).cpu().numpy()
    assert rel_l2(o_tc, o_gv) <= TOL_TC


# ---------------------------------------------------------------- chained decode kernels (T <= 4)

def _chain_vs_separate(tl, T):
    """The chained decode kernels and the separate kernels: same routing, same pair
    lists; outputs equal up to summation order (both accumulate in fp32)."""
    chain = tl.moe_layer()
    sep = tl.moe_layer()
    sep.desc.decode_chain_off = 1
    sep.rebuild_plan()
    assert chain.path(T) == "decode_chain" and sep.path(T) == "gemv"
    x = tl.x.cuda()
    o_c = chain(x).clone()
    o_s = sep(x).clone()
    torch.cuda.synchronize()
    (ids_c, gw_c, off_c), (ids_s, gw_s, off_s) = chain.debug_views(T), sep.debug_views(T)
    assert torch.equal(ids_c, ids_s) and torch.equal(off_c, off_s)
    # the router logits are summed in another order: gates agree to rounding
    assert torch.allclose(gw_c, gw_s, rtol=1e-5, atol=0)
    err = rel_l2(o_c.cpu().numpy(), o_s.cpu().double().numpy())
    assert err <= 2e-6, f"chain vs separate kernels: rel-L2 {err:.3e}"
    assert chain.device_status(T) == 0


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_decode_chain_matches_separate_kernels(T):
    _chain_vs_separate(make_layer(synth.DECODE, 50 + T, T), T)


def test_decode_chain_q8_shared_expert():
    shape = synth.LayerShape(H=2048, E=64, k=4, I=768, qtype=synth.Q4_K, mode="sigmoid_group", n_groups=8,
                             topk_groups=4, scale=2.5, I_s=512, shared_qtype=synth.Q8_0, bias_std=0.1)
    tl = make_layer(shape, 60, 2, exact_all=True)
    _chain_vs_separate(tl, 2)
    _check_layer(tl, 2)


def test_deepseek_shape_decode_takes_gemv_path():
    # hidden 7168 leaves the gate/up kernel fewer than 16 warps: the layer runs the GEMV kernels
    assert make_layer(synth.DEEPSEEK, 60, 2).moe_layer().path(2) == "gemv"


def test_decode_chain_q4k_shared_expert():
    shape = synth.LayerShape(H=512, E=32, k=4, I=256, qtype=synth.Q4_K, mode="sigmoid_group", n_groups=4,
                             topk_groups=2, scale=2.5, I_s=512, shared_qtype=synth.Q4_K, bias_std=0.1)
    tl = make_layer(shape, 63, 3, exact_all=True)
    _chain_vs_separate(tl, 3)
    _check_layer(tl, 3)


def test_tc_fp16_range_is_reported():
    """The tensor-core path multiplies fp16 operands: an activation or an intermediate value
    beyond the fp16 range is reported in the status word (MOE_ERR_DEVICE_CHECK), not hidden."""
    from quantized_routed_expert_sigmoid_gb300 import _native as N
    T = 160
    tl = make_layer(synth.DECODE, 33, T, exact_all=True)
    layer = tl.moe_layer()
    assert layer.path(T) == "tensor"
    x = tl.x.cuda()
    layer(x)
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_OK
    big = x.clone()
    big[3, 5] = 1.0e5                                 # a bf16 value with no fp16 counterpart
    layer(big)
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_ERR_DEVICE_CHECK
    loud = (x.float() * 400.0).to(torch.bfloat16)     # x in range; silu(gate) * up beyond 65504
    assert loud.float().abs().max().item() < 6e4
    layer(loud)
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_ERR_DEVICE_CHECK
    layer(x)
    torch.cuda.synchronize()
    assert layer.device_status(T) == N.MOE_OK
