"""Host-only checks of the C ABI: the library loads, exports every declared symbol,
and rejects invalid arguments on the host before any launch (no GPU needed)."""
from __future__ import annotations

import re

import pytest

import quantized_routed_expert_sigmoid_gb300 as moe
from quantized_routed_expert_sigmoid_gb300 import _native as N

FAKE = 0x10000          # a 256-aligned address that is never dereferenced on these paths


def declared_functions():
    text = open(N.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = N.load()
    names = declared_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert moe.moe_version().startswith("moe_gb300")


def _expect(status, fn, *args):
    with pytest.raises(N.MoeError) as ei:
        fn(*args)
    assert ei.value.status == status, str(ei.value)
    return str(ei.value)


def test_route_rejects_bad_config():
    cfg = moe.route_cfg(moe.MOE_ROUTE_SOFTMAX, 8, 9)                     # k > E
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_route, cfg, FAKE, moe.MOE_BF16, 4, 256, FAKE, None, None, FAKE,
            FAKE, FAKE, 0)
    cfg = moe.route_cfg(moe.MOE_ROUTE_SIGMOID_GROUP, 12, 2, 5, 2)         # 5 does not divide 12
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_route, cfg, FAKE, moe.MOE_BF16, 4, 256, FAKE, None, None, FAKE,
            FAKE, FAKE, 0)
    cfg = moe.route_cfg(moe.MOE_ROUTE_SIGMOID_GROUP, 16, 9, 4, 2)         # 9 > 2 groups x 4 experts
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_route, cfg, FAKE, moe.MOE_BF16, 4, 256, FAKE, None, None, FAKE,
            FAKE, FAKE, 0)
    cfg = moe.route_cfg(moe.MOE_ROUTE_SOFTMAX, 8, 2)
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_route, cfg, FAKE, moe.MOE_BF16, 4, 100, FAKE, None, None, FAKE,
            FAKE, FAKE, 0)                                               # H not a multiple of 32
    _expect(N.MOE_ERR_UNSUPPORTED, moe.moe_route, cfg, FAKE, moe.MOE_Q4_K, 4, 256, FAKE, None, None, FAKE,
            FAKE, FAKE, 0)
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_route, cfg, FAKE + 2, moe.MOE_BF16, 4, 256, FAKE, None, None,
            FAKE, FAKE, FAKE, 0)                                         # misaligned x


def test_permute_workspace_checks():
    need = moe.moe_permute_workspace_size(4096, 8, 128)
    assert need >= 256 + 32 * 128 * 4
    _expect(N.MOE_ERR_WORKSPACE, moe.moe_permute, FAKE, 4096, 8, 128, FAKE, FAKE, FAKE, FAKE, need - 1, 0)
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_permute, FAKE, 4, 2, 2000, FAKE, FAKE, FAKE, FAKE, 1 << 20, 0)


def _desc(qtype=N.MOE_Q4_K, H=2048, I=768, E=128, data=FAKE, stride=None, mode=N.MOE_ROUTE_SOFTMAX):
    d = N.moe_layer_desc()
    d.route = moe.route_cfg(mode, E, 8, 8 if mode else 1, 4 if mode else 1, 1.0, True)
    d.hidden, d.intermediate, d.x_type = H, I, N.MOE_BF16
    d.W_router = FAKE
    from quantized_routed_expert_sigmoid_gb300.layer import row_bytes
    rb = ((lambda K: row_bytes(qtype, K)) if qtype in (N.MOE_Q4_K, N.MOE_Q8_0, N.MOE_Q8_0_R, N.MOE_Q5_K, N.MOE_Q6_K,
                                                       N.MOE_Q3_K, N.MOE_MXFP4)
          else (lambda K: K // 32 * 34))
    sgu = stride if stride is not None else I * rb(H)
    d.gate = moe.qmat(qtype, data, I, H, sgu)
    d.up = moe.qmat(qtype, data, I, H, sgu)
    d.down = moe.qmat(qtype, data, H, I, H * rb(I))
    return d


def test_plan_validation():
    plan = moe.moe_layer_plan_create(_desc())
    try:
        for T in (1, 2, 64, 4096):
            assert moe.moe_layer_workspace_size(plan, T) > 0
        assert moe.moe_layer_workspace_size(plan, 4096) > moe.moe_layer_workspace_size(plan, 1)
        _expect(N.MOE_ERR_WORKSPACE, moe.moe_layer, plan, FAKE, 4, FAKE, FAKE, 16, 0)
        moe.moe_layer(plan, None, 0, None, None, 0, 0)     # T = 0: a no-op, nothing launched
        _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer, plan, FAKE, -1, FAKE, FAKE, 1 << 30, 0)
        _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer, plan, FAKE + 8, 4, FAKE, FAKE, 1 << 30, 0)
    finally:
        moe.moe_layer_plan_destroy(plan)
    _expect(N.MOE_ERR_UNSUPPORTED, moe.moe_layer_plan_create, _desc(qtype=N.MOE_BF16))
    for other in (9, 10, -1):            # types the library does not decode, and garbage
        _expect(N.MOE_ERR_UNSUPPORTED, moe.moe_layer_plan_create, _desc(qtype=other))
    for qt in (N.MOE_Q5_K, N.MOE_Q6_K, N.MOE_Q3_K, N.MOE_MXFP4):   # beyond Q4_K/Q8_0: GEMV kernels at every T
        plan = moe.moe_layer_plan_create(_desc(qtype=qt))
        try:
            assert all(moe.moe_layer_path(plan, T) == 0 for T in (1, 2, 64, 4096))
        finally:
            moe.moe_layer_plan_destroy(plan)
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, _desc(H=2000))          # not a block multiple
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, _desc(data=FAKE + 4))   # misaligned weights
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, _desc(stride=100))      # stride too small
    d = _desc()
    d.bias = FAKE                                                                      # bias needs sigmoid mode
    msg = _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, d)
    assert "sigmoid" in msg


def test_expert_ffn_validation():
    q = N.MOE_Q4_K
    g = moe.qmat(q, FAKE, 768, 2048, 768 * 1152)
    dn = moe.qmat(q, FAKE, 2048, 768, 2048 * 432)
    # identity mapping (no sorted_pairs) needs E = 1, k = 1
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_expert_ffn, g, g, dn, 4, FAKE, N.MOE_BF16, 2, 2048, 768, None, None,
            1, FAKE, FAKE, 1 << 30, 0)
    _expect(N.MOE_ERR_WORKSPACE, moe.moe_expert_ffn, g, g, dn, 4, FAKE, N.MOE_BF16, 2, 2048, 768, FAKE, FAKE,
            2, FAKE, FAKE, 8, 0)
    bad = moe.qmat(q, FAKE, 768, 2048, 768 * 1152)
    bad.rows = 700
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_expert_ffn, bad, g, dn, 4, FAKE, N.MOE_BF16, 2, 2048, 768, FAKE,
            FAKE, 2, FAKE, FAKE, 1 << 30, 0)


def test_zero_tokens_is_a_noop():
    cfg = moe.route_cfg(moe.MOE_ROUTE_SOFTMAX, 8, 2)
    moe.moe_route(cfg, None, moe.MOE_BF16, 0, 256, None, None, None, None, None, None, 0)
    moe.moe_combine(None, None, None, 0, 2, 256, None, 0, None, 0)
    plan = moe.moe_layer_plan_create(_desc())
    moe.moe_layer(plan, None, 0, None, None, 0, 0)
    moe.moe_layer_plan_destroy(plan)


def test_last_error_is_per_thread_message():
    cfg = moe.route_cfg(moe.MOE_ROUTE_SOFTMAX, 8, 9)
    with pytest.raises(N.MoeError):
        moe.moe_route(cfg, FAKE, moe.MOE_BF16, 4, 256, FAKE, None, None, FAKE, FAKE, FAKE, 0)
    assert "top_k" in moe.moe_last_error()
    import threading
    seen = []
    t = threading.Thread(target=lambda: seen.append(moe.moe_last_error()))
    t.start()
    t.join()
    assert seen == [""]


def test_prenorm_validation():
    # a pre-norm reads the fp32 residual stream: other input types, a misaligned gamma or a
    # negative eps are refused on the host; an accepted one needs room for u in the workspace
    d = _desc()
    d.norm_gamma, d.norm_eps = FAKE, 1e-6
    msg = _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, d)
    assert "fp32" in msg
    d.x_type = N.MOE_F32
    d.norm_gamma = FAKE + 4
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, d)
    d.norm_gamma, d.norm_eps = FAKE, -1.0
    _expect(N.MOE_ERR_INVALID_ARG, moe.moe_layer_plan_create, d)
    d.norm_eps = 1e-6
    plain_d = _desc()
    plain_d.x_type = N.MOE_F32
    pre, plain = moe.moe_layer_plan_create(d), moe.moe_layer_plan_create(plain_d)
    try:
        for T in (8, 64):
            # no GPU here, so no decode chain: the normalized input u (bf16 [T][H]) gets its own region
            assert moe.moe_layer_workspace_size(pre, T) >= moe.moe_layer_workspace_size(plain, T) + T * 2048 * 2
    finally:
        moe.moe_layer_plan_destroy(pre)
        moe.moe_layer_plan_destroy(plain)


def test_debug_waits_setting_is_validated():
    lib = N.load()
    assert lib.moe_debug_set_waits(1000, 2) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_debug_set_waits(0, 0) == N.MOE_OK


def test_weights_prepare_size_and_validation():
    # Q8_0 rows of K weights repack to 32 * K/32 quant bytes + the K/32 fp16 scales padded to 16
    m = N.qmat(N.MOE_Q8_0, FAKE, 2048, 7168, 2048 * 7168 // 32 * 34)
    assert N.moe_weights_prepare_size(m, 1) == 2048 * (7168 + 448)
    assert N.moe_weights_prepare_size(m, 3) == 3 * 2048 * (7168 + 448)
    m2 = N.qmat(N.MOE_Q8_0, FAKE, 4, 96, 4 * 102)         # 3 blocks: scales 6 bytes -> 16
    assert N.moe_weights_prepare_size(m2, 1) == 4 * (96 + 16)
    q4 = N.qmat(N.MOE_Q4_K, FAKE, 768, 2048, 768 * 1152)  # used as stored
    assert N.moe_weights_prepare_size(q4, 128) == 0
    out = N.moe_weights_prepare(q4, 128, None, 0, 0)
    assert out.qtype == N.MOE_Q4_K and out.data == FAKE
    _expect(N.MOE_ERR_UNSUPPORTED, N.moe_weights_prepare_size, N.qmat(N.MOE_Q8_0_R, FAKE, 4, 96, 0), 1)
    _expect(N.MOE_ERR_INVALID_ARG, N.moe_weights_prepare_size, N.qmat(N.MOE_Q8_0, FAKE, 4, 100, 0), 1)
    _expect(N.MOE_ERR_INVALID_ARG, N.moe_weights_prepare_size, m, 0)
    _expect(N.MOE_ERR_WORKSPACE, N.moe_weights_prepare, m2, 1, FAKE * 16, 16, 0)
    _expect(N.MOE_ERR_INVALID_ARG, N.moe_weights_prepare, m2, 1, FAKE + 8, 1 << 20, 0)
    _expect(N.MOE_ERR_INVALID_ARG, N.moe_weights_prepare, m2, 1, FAKE + 16, 1 << 20, 0)   # overlaps the source


def test_layer_accepts_repacked_q8_0():
    from quantized_routed_expert_sigmoid_gb300.layer import row_bytes
    assert row_bytes(N.MOE_Q8_0_R, 256) == 256 + 16
    plan = moe.moe_layer_plan_create(_desc(qtype=N.MOE_Q8_0_R))
    moe.moe_layer_plan_destroy(plan)
