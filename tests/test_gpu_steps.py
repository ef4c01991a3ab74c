"""GPU parity of each C-ABI step (route, permute, expert FFN, combine, RMSNorm) against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
import quantized_routed_expert_sigmoid_gb300 as moe
from helpers import TOL_GEMV, gapped_activations, oracle_mode, rel_l2

pytestmark = pytest.mark.gpu


def _route_case(shape, seed, T):
    Wr = synth.router_weight(shape, seed, 0)
    bias = synth.bias(shape, seed, 0)
    x = gapped_activations(shape, seed, T, Wr.numpy(), None if bias is None else bias.numpy())
    return Wr, bias, x


@pytest.mark.parametrize("name,T", [("tiny", 4), ("decode", 3), ("decode", 70), ("deepseek", 5)])
def test_route(name, T):
    shape = {"tiny": synth.TINY, "decode": synth.DECODE, "deepseek": synth.DEEPSEEK}[name]
    Wr, bias, x = _route_case(shape, 7, T)
    E, k = shape.E, shape.k
    cfg = moe.route_cfg(moe.MOE_ROUTE_SIGMOID_GROUP if shape.mode == "sigmoid_group" else moe.MOE_ROUTE_SOFTMAX,
                        E, k, shape.n_groups, shape.topk_groups, shape.scale, shape.renormalize)
    xd, Wd = x.cuda(), Wr.cuda()
    bd = None if bias is None else bias.cuda()
    logits = torch.empty(T, E, device="cuda")
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    xt = moe.MOE_BF16 if shape.x_dtype == "bf16" else moe.MOE_F32
    moe.moe_route(cfg, xd, xt, T, shape.H, Wd, bd, None, logits, ids, w)
    torch.cuda.synchronize()
    ref_l = oracle.router_logits(x.double().numpy(), Wr.numpy())
    ref_ids, ref_w, _ = oracle.route(oracle_mode(shape), ref_l, k, bias=None if bias is None else bias.numpy(),
                                     n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                     renormalize=shape.renormalize, scale=shape.scale)
    assert np.allclose(logits.cpu().numpy(), ref_l, rtol=0, atol=2e-4)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(w.cpu().numpy(), ref_w, rtol=1e-5, atol=1e-6)
    # logits_in path gives the same selection
    ids2 = torch.empty_like(ids)
    w2 = torch.empty_like(w)
    moe.moe_route(cfg, None, xt, T, shape.H, None, bd, logits, None, ids2, w2)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2) and torch.equal(w, w2)


def test_route_without_renormalisation():
    E, k, T = 16, 3, 6
    l = torch.randn(T, E, generator=torch.Generator().manual_seed(3)) * 2
    for mode, om in ((moe.MOE_ROUTE_SOFTMAX, oracle.ROUTE_SOFTMAX), (moe.MOE_ROUTE_SIGMOID_GROUP, oracle.ROUTE_SIGMOID_GROUP)):
        cfg = moe.route_cfg(mode, E, k, 4, 2, 1.5, False)
        ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, k, device="cuda")
        moe.moe_route(cfg, None, moe.MOE_F32, T, 0, None, None, l.cuda(), None, ids, w)
        torch.cuda.synchronize()
        ri, rw, gaps = oracle.route(om, l.double().numpy(), k, n_groups=4, topk_groups=2, renormalize=False, scale=1.5)
        assert gaps.min() > 1e-4
        assert np.array_equal(ids.cpu().numpy(), ri)
        assert np.allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)


def _permute(ids_np, E):
    T, k = ids_np.shape
    ids = torch.from_numpy(ids_np).cuda()
    P = T * k
    sp = torch.empty(max(P, 1), dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pp = torch.empty(max(P, 1), dtype=torch.int32, device="cuda")
    nb = moe.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    moe.moe_permute(ids, T, k, E, sp, off, pp, ws, nb)
    status = moe.moe_permute_read_device_status(T, k, E, ws)
    return sp.cpu().numpy()[:P], off.cpu().numpy(), pp.cpu().numpy()[:P], status


@pytest.mark.parametrize("T,k,E", [(1, 8, 128), (2, 8, 128), (4, 2, 8), (5, 4, 4), (129, 8, 128), (700, 8, 128),
                                   (4096, 8, 128), (512, 8, 256), (3000, 3, 1000)])
def test_permute_bitexact(T, k, E):
    rng = np.random.default_rng(T * 31 + k * 7 + E)
    if k == E:
        ids = np.tile(np.arange(E, dtype=np.int32), (T, 1))
    else:
        # skewed popularity with some experts never chosen
        p = 1.0 / np.arange(1, E + 1)
        p[E // 2: E // 2 + 3] = 0
        p /= p.sum()
        ids = np.stack([np.sort(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]).astype(np.int32)
    sp, off, pp, status = _permute(ids, E)
    rsp, roff, rpp = oracle.permute(ids, E)
    assert status == 0
    assert np.array_equal(off, roff)
    assert np.array_equal(sp, rsp)
    assert np.array_equal(pp, rpp)


def test_permute_flags_bad_ids():
    ids = np.array([[0, 3], [9, 1]], dtype=np.int32)      # 9 is out of range for E = 8
    sp, off, pp, status = _permute(ids, 8)
    assert status == moe.MOE_ERR_DEVICE_CHECK
    assert off[8] == 3 and pp[2] == -1


def test_permute_zero_tokens():
    sp, off, pp, status = _permute(np.zeros((0, 2), dtype=np.int32), 8)
    assert np.all(off == 0) and status == 0


# the Q4_K cases take the segmented kernels; I = 2048 the down kernel's wide-row layout, with
# up to 20 tokens per expert (three passes of 8)
@pytest.mark.parametrize("qt,H,I,E,T,k", [(synth.Q8_0, 256, 128, 8, 6, 2), (synth.Q4_K, 2048, 768, 16, 5, 4),
                                          (synth.Q4_K, 512, 256, 4, 40, 2), (synth.Q8_0, 1024, 512, 4, 9, 2),
                                          (synth.Q4_K, 1024, 2048, 4, 30, 2)])
def test_expert_ffn(qt, H, I, E, T, k):
    shape = synth.LayerShape(H=H, E=E, k=k, I=I, qtype=qt, x_dtype="bf16")
    bank = synth.ExpertBank(shape, 9, 0, exact=None, fill_device="cuda")
    rng = np.random.default_rng(5)
    ids = np.stack([np.sort(rng.choice(E, size=k, replace=False)) for _ in range(T)]).astype(np.int32)
    sp, off, pp = oracle.permute(ids, E)
    x = synth.activations(T, H, 11, "bf16")
    y = torch.empty(T * k, H, device="cuda")
    oq = moe.MOE_Q4_K if qt == synth.Q4_K else moe.MOE_Q8_0
    rb_h, rb_i = synth.row_bytes(qt, H), synth.row_bytes(qt, I)
    g = moe.qmat(oq, bank.gate, I, H, I * rb_h)
    u = moe.qmat(oq, bank.up, I, H, I * rb_h)
    d = moe.qmat(oq, bank.down, H, I, H * rb_i)
    nb = moe.moe_expert_ffn_workspace_size(T, k, E, H, I)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn(g, u, d, E, x.cuda(), moe.MOE_BF16, T, H, I, torch.from_numpy(sp).cuda(),
                       torch.from_numpy(off).cuda(), k, y, ws, nb)
    torch.cuda.synchronize()
    yg = y.cpu().numpy()
    gate, up, down = bank.gate.cpu().numpy(), bank.up.cpu().numpy(), bank.down.cpu().numpy()
    x64 = x.double().numpy()
    oqt = oracle.Q4_K if qt == synth.Q4_K else oracle.Q8_0
    ref = np.empty_like(yg, dtype=np.float64)
    for i, p in enumerate(sp):
        t, e = p // k, ids.reshape(-1)[p]
        ref[i], _ = oracle.expert_ffn(oqt, gate[e], up[e], down[e], H, I, x64[t])
    assert rel_l2(yg, ref) <= TOL_GEMV


def test_expert_ffn_identity_mapping():
    """sorted_pairs = offsets = NULL: one expert over every token (the shared-expert form)."""
    H, I, T = 1024, 512, 7
    shape = synth.LayerShape(H=H, E=1, k=1, I=I, qtype=synth.Q8_0)
    bank = synth.ExpertBank(shape, 13, 0, exact=None, fill_device="cuda")
    x = synth.activations(T, H, 3, "bf16")
    y = torch.empty(T, H, device="cuda")
    rb_h, rb_i = synth.row_bytes(synth.Q8_0, H), synth.row_bytes(synth.Q8_0, I)
    q = moe.MOE_Q8_0
    nb = moe.moe_expert_ffn_workspace_size(T, 1, 1, H, I)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn(moe.qmat(q, bank.gate, I, H, I * rb_h), moe.qmat(q, bank.up, I, H, I * rb_h),
                       moe.qmat(q, bank.down, H, I, H * rb_i), 1, x.cuda(), moe.MOE_BF16, T, H, I, None, None, 1,
                       y, ws, nb)
    torch.cuda.synchronize()
    ref = np.stack([oracle.expert_ffn(oracle.Q8_0, bank.gate[0].cpu().numpy(), bank.up[0].cpu().numpy(),
                                      bank.down[0].cpu().numpy(), H, I, x[t].double().numpy())[0] for t in range(T)])
    assert rel_l2(y.cpu().numpy(), ref) <= TOL_GEMV


def test_combine_matches_plain_sum():
    T, k, H = 5, 3, 256
    g = torch.Generator().manual_seed(2)
    y = torch.randn(T * k, H, generator=g)
    w = torch.rand(T, k, generator=g)
    perm = torch.randperm(T * k, generator=g).to(torch.int32)
    shared = torch.randn(T, H, generator=g)
    old = torch.randn(T, H, generator=g)
    out = old.clone().cuda()
    moe.moe_combine(y.cuda(), w.cuda(), perm.cuda(), T, k, H, shared.cuda(), 1, out)
    torch.cuda.synchronize()
    ref = old.double() + shared.double()
    for t in range(T):
        for j in range(k):
            ref[t] += w[t, j].double() * y[perm[t * k + j]].double()
    assert rel_l2(out.cpu().numpy(), ref.numpy()) < 1e-6


def test_rmsnorm_bf16():
    T, H = 6, 2048
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(4)) * 3
    gamma = synth.gamma(H, 5, 0)
    u = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_rmsnorm_bf16(x.cuda(), gamma.cuda(), T, H, 1e-6, u)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(x.double().numpy(), gamma.numpy(), 1e-6)
    got = u.float().cpu().numpy()
    # each value is the bf16 rounding of the fp32 result: within one bf16 half-ulp (2^-9 relative) + fp32 error
    assert np.all(np.abs(got - ref) <= np.abs(ref) * (2.0 ** -8) + 1e-30)
    assert rel_l2(got, ref) < 2e-3
