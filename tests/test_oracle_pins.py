"""Pins for the fp64 oracle: checks against things other than the oracle itself.

The bloomery pages print no worked example for this layer, so each oracle
function is pinned by a closed form, a brute force on tiny inputs, an
invariant, or a special case that reduces to a library routine.  Each pin is
a plain function of the oracle library handle, so test_oracle_mutants.py can
run the same pin against deliberately broken oracle builds and show that it
fails ("a gate is shown to fail on the defect it guards": "bloomery early
V4.1 README", verification list).
"""
from __future__ import annotations

import itertools
import math
import os
import sys

import numpy as np
import pytest
import torch

import oracle
import synth

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
import blocks as golden  # noqa: E402


# ---------------------------------------------------------------- fp16 and dequant

def pin_half_to_double(lib):
    for bits in (0x3C00, 0x3400, 0xC000, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0x8000, 0x3555, 0xFBFF):
        ref = float(np.array([bits], dtype=np.uint16).view(np.float16)[0])
        assert oracle.half_to_double(bits, lib=lib) == ref, hex(bits)


def pin_q8_0_handbuilt(lib):
    fx = golden.read_fixture("Q8_0")
    for name, (blk, expected) in golden.q8_0_cases().items():
        assert fx[name] == blk, f"fixture {name} differs from the packer"
        got = oracle.dequant(oracle.Q8_0, np.frombuffer(blk, np.uint8), 1, 32, lib=lib)[0]
        assert np.array_equal(got, np.array(expected)), name


def pin_q4_k_handbuilt(lib):
    fx = golden.read_fixture("Q4_K")
    for name, (blk, expected) in golden.q4_k_cases().items():
        assert fx[name] == blk, f"fixture {name} differs from the packer"
        got = oracle.dequant(oracle.Q4_K, np.frombuffer(blk, np.uint8), 1, 256, lib=lib)[0]
        assert np.array_equal(got, np.array(expected)), name


def pin_q4_k_multiblock_rows(lib):
    # two rows of two super-blocks each: row r, block b uses d = 2^(r+b), sc = 1,
    # q = 1 everywhere, m = 0 -> w = 2^(r+b) over that block's 256 weights.
    d_bits = {0: 0x3C00, 1: 0x4000, 2: 0x4400}
    data = b""
    for r in range(2):
        for b in range(2):
            data += golden.q4_k_block(d_bits[r + b], 0, [1] * 8, [0] * 8, [1] * 256)
    got = oracle.dequant(oracle.Q4_K, np.frombuffer(data, np.uint8), 2, 512, lib=lib)
    for r in range(2):
        for b in range(2):
            assert np.all(got[r, 256 * b:256 * (b + 1)] == 2.0 ** (r + b))


def _pin_handbuilt(lib, kind, qtype):
    weights, nbytes, make = golden.BLOCK_TYPES[kind]
    fx = golden.read_fixture(kind)
    for name, (blk, expected) in make().items():
        assert len(blk) == nbytes, name
        assert fx[name] == blk, f"fixture {name} differs from the packer"
        got = oracle.dequant(qtype, np.frombuffer(blk, np.uint8), 1, weights, lib=lib)[0]
        assert np.array_equal(got, np.array(expected), equal_nan=True), name


def pin_q5_k_handbuilt(lib):
    _pin_handbuilt(lib, "Q5_K", oracle.Q5_K)


def pin_q6_k_handbuilt(lib):
    _pin_handbuilt(lib, "Q6_K", oracle.Q6_K)


def pin_q3_k_handbuilt(lib):
    _pin_handbuilt(lib, "Q3_K", oracle.Q3_K)


def pin_e2m1(lib):
    # the 16 FP4 E2M1 codes against the format's value list, signed zero included
    for code in range(16):
        got = oracle.e2m1_to_double(code, lib=lib)
        assert got == golden.e2m1_value(code), code
        assert np.signbit(got) == bool(code & 8), code


def pin_mxfp4_handbuilt(lib):
    _pin_handbuilt(lib, "MXFP4", oracle.MXFP4)


def pin_mxfp4_multiblock_rows(lib):
    # two rows of three blocks; block (r, b) has e = 127 + r + b and every code 2 (= 1.0)
    data = b"".join(golden.mxfp4_block(127 + r + b, [2] * 32) for r in range(2) for b in range(3))
    got = oracle.dequant(oracle.MXFP4, np.frombuffer(data, np.uint8), 2, 96, lib=lib)
    for r in range(2):
        for b in range(3):
            assert np.all(got[r, 32 * b:32 * (b + 1)] == 2.0 ** (r + b)), (r, b)


def pin_kquant_multiblock_rows(lib):
    # for each of Q5_K, Q6_K, Q3_K: two rows of two super-blocks; block (r, b) has d = 2^(r+b)
    # and every other field chosen so that each weight decodes to d
    d_bits = {0: 0x3C00, 1: 0x4000, 2: 0x4400}
    blocks = {
        oracle.Q5_K: lambda db: golden.q5_k_block(db, 0, [1] * 8, [0] * 8, [1] * 256),
        oracle.Q6_K: lambda db: golden.q6_k_block(db, [1] * 16, [1] * 256),
        oracle.Q3_K: lambda db: golden.q3_k_block(db, [1] * 16, [1] * 256),
    }
    for qtype, make in blocks.items():
        data = b"".join(make(d_bits[r + b]) for r in range(2) for b in range(2))
        assert len(data) == 2 * oracle.row_bytes(qtype, 512)
        got = oracle.dequant(qtype, np.frombuffer(data, np.uint8), 2, 512, lib=lib)
        for r in range(2):
            for b in range(2):
                assert np.all(got[r, 256 * b:256 * (b + 1)] == 2.0 ** (r + b)), (qtype, r, b)


def test_half_to_double(olib):
    pin_half_to_double(olib)


def test_q8_0_handbuilt(olib):
    pin_q8_0_handbuilt(olib)


def test_q4_k_handbuilt(olib):
    pin_q4_k_handbuilt(olib)


def test_q4_k_multiblock_rows(olib):
    pin_q4_k_multiblock_rows(olib)


def test_q5_k_handbuilt(olib):
    pin_q5_k_handbuilt(olib)


def test_q6_k_handbuilt(olib):
    pin_q6_k_handbuilt(olib)


def test_q3_k_handbuilt(olib):
    pin_q3_k_handbuilt(olib)


def test_kquant_multiblock_rows(olib):
    pin_kquant_multiblock_rows(olib)


def test_e2m1(olib):
    pin_e2m1(olib)


def test_mxfp4_handbuilt(olib):
    pin_mxfp4_handbuilt(olib)


def test_mxfp4_multiblock_rows(olib):
    pin_mxfp4_multiblock_rows(olib)


def test_synth_packer_matches_handbuilt_packer():
    """The synthetic-input encoder lays out bytes exactly as the hand packer."""
    rng = np.random.default_rng(1)
    for _ in range(20):
        sc = rng.integers(0, 64, 8).tolist()
        m = rng.integers(0, 64, 8).tolist()
        q = rng.integers(0, 16, 256).tolist()
        ref = golden.q4_k_block(0x3C00, 0x3800, sc, m, q)
        got = synth.pack_q4_k(torch.tensor(1.0), torch.tensor(0.5), torch.tensor(sc),
                              torch.tensor(m), torch.tensor(q)).numpy().tobytes()
        assert got == ref


def test_synth_kquant_packers_match_handbuilt_packers():
    """The Q5_K, Q6_K and Q3_K encoders of the synthetic inputs lay out bytes exactly as the
    hand packers (written separately, byte by byte) on random fields."""
    rng = np.random.default_rng(2)
    one, half = torch.tensor(1.0), torch.tensor(0.5)
    for _ in range(20):
        sc8 = rng.integers(0, 64, 8).tolist()
        m8 = rng.integers(0, 64, 8).tolist()
        q5 = rng.integers(0, 32, 256).tolist()
        ref = golden.q5_k_block(0x3C00, 0x3800, sc8, m8, q5)
        got = synth.pack_q5_k(one, half, torch.tensor(sc8), torch.tensor(m8), torch.tensor(q5))
        assert got.numpy().tobytes() == ref
        s6 = rng.integers(-128, 128, 16).tolist()
        q6 = rng.integers(-32, 32, 256).tolist()
        ref = golden.q6_k_block(0x3800, s6, q6)
        assert synth.pack_q6_k(half, torch.tensor(s6), torch.tensor(q6)).numpy().tobytes() == ref
        s3 = rng.integers(-32, 32, 16).tolist()
        q3 = rng.integers(-4, 4, 256).tolist()
        ref = golden.q3_k_block(0x3C00, s3, q3)
        assert synth.pack_q3_k(one, torch.tensor(s3), torch.tensor(q3)).numpy().tobytes() == ref
        e = int(rng.integers(0, 256))
        c4 = rng.integers(0, 16, 32).tolist()
        ref = golden.mxfp4_block(e, c4)
        assert synth.pack_mxfp4(torch.tensor(e), torch.tensor(c4)).numpy().tobytes() == ref


def test_synth_kquant_encoders_round_trip(olib):
    """Encoded Q5_K / Q6_K / Q3_K blocks decode (oracle) close to the source weights.  The
    bounds are the quantizers' own: half a step per weight plus the rounding of the group
    scales, which for N(0, 0.02) weights gives these relative L2 errors with margin."""
    w = synth.normal((16, 1024), 0.02, 321)
    ref = w.double().numpy()
    for qt, oq, rel_max in ((synth.Q5_K, oracle.Q5_K, 0.06), (synth.Q6_K, oracle.Q6_K, 0.04),
                            (synth.Q3_K, oracle.Q3_K, 0.25), (synth.MXFP4, oracle.MXFP4, 0.15)):
        blk = synth.encode(qt, w).numpy()
        assert blk.shape == (16, oracle.row_bytes(oq, 1024))
        deq = oracle.dequant(oq, blk, 16, 1024, lib=olib)
        rel = np.linalg.norm(deq - ref) / np.linalg.norm(ref)
        assert rel < rel_max, (qt, rel)
    # more bits, less error: Q6_K < Q5_K < Q4_K < Q3_K on the same weights
    errs = [np.linalg.norm(oracle.dequant(oq, synth.encode(qt, w).numpy(), 16, 1024, lib=olib) - ref)
            for qt, oq in ((synth.Q6_K, oracle.Q6_K), (synth.Q5_K, oracle.Q5_K), (synth.Q4_K, oracle.Q4_K),
                           (synth.Q3_K, oracle.Q3_K))]
    assert errs == sorted(errs), errs


def test_synth_encoders_round_trip(olib):
    """Encoders produce blocks whose oracle decode is close to the source weights."""
    w = synth.normal((8, 512), 0.02, 123)
    for qt, oq, tol in ((synth.Q8_0, oracle.Q8_0, 0.02 / 127 * 4), (synth.Q4_K, oracle.Q4_K, 0.02)):
        blk = synth.encode(qt, w).numpy()
        deq = oracle.dequant(oq, blk, 8, 512, lib=olib)
        err = np.abs(deq - w.double().numpy()).max()
        assert err < tol, (qt, err)
        rel = np.linalg.norm(deq - w.double().numpy()) / np.linalg.norm(w.double().numpy())
        assert rel < (0.01 if qt == synth.Q8_0 else 0.12), (qt, rel)


# ---------------------------------------------------------------- router

def pin_router_integer(lib):
    rng = np.random.default_rng(5)
    x = rng.integers(-3, 4, (3, 16)).astype(np.float64)
    W = rng.integers(-2, 3, (5, 16)).astype(np.float32)
    got = oracle.router_logits(x, W, lib=lib)
    expected = np.array([[sum(int(x[t, h]) * int(W[e, h]) for h in range(16)) for e in range(5)]
                         for t in range(3)], dtype=np.float64)
    assert np.array_equal(got, expected)


def test_router_integer(olib):
    pin_router_integer(olib)


# ---------------------------------------------------------------- softmax top-k

def pin_softmax_topk_bruteforce(lib):
    rng = np.random.default_rng(7)
    E, k = 8, 3
    for _ in range(50):
        l = rng.normal(size=(1, E))
        ids, w, gaps = oracle.route(oracle.ROUTE_SOFTMAX, l, k, lib=lib)
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(l[0, list(c)]))
        assert tuple(ids[0]) == best                       # ascending ids, best-sum subset
        assert abs(w[0].sum() - 1.0) < 1e-12
        # order of gates follows the ratio of exponentials of the logits
        assert abs(w[0, 0] / w[0, 1] - math.exp(l[0, ids[0, 0]] - l[0, ids[0, 1]])) < 1e-12
        srt = np.sort(l[0])[::-1]
        assert abs(gaps[0, 0] - (srt[k - 1] - srt[k])) < 1e-15


def pin_softmax_special(lib):
    # equal logits: ties go to the lower ids, gates 1/k
    ids, w, _ = oracle.route(oracle.ROUTE_SOFTMAX, np.zeros((1, 6)), 4, lib=lib)
    assert ids[0].tolist() == [0, 1, 2, 3] and np.allclose(w, 0.25, rtol=0, atol=1e-15)
    # logits differ by ln 2: the gate ratio is exactly 2
    l = np.array([[0.0, math.log(2.0), -5.0, -6.0]])
    ids, w, _ = oracle.route(oracle.ROUTE_SOFTMAX, l, 2, lib=lib)
    assert ids[0].tolist() == [0, 1] and abs(w[0, 1] / w[0, 0] - 2.0) < 1e-14
    assert abs(w[0, 0] - 1 / 3) < 1e-15
    # k = E: the full softmax (scipy), in id order
    from scipy.special import softmax
    l = np.random.default_rng(3).normal(size=(2, 5))
    ids, w, gaps = oracle.route(oracle.ROUTE_SOFTMAX, l, 5, lib=lib)
    assert np.array_equal(ids, np.tile(np.arange(5), (2, 1)))
    assert np.allclose(w, softmax(l, axis=1), rtol=1e-14, atol=0)
    assert np.all(np.isinf(gaps[:, 0]))
    # without renormalisation the gates are the full softmax probabilities of the chosen ids
    ids, w, _ = oracle.route(oracle.ROUTE_SOFTMAX, l, 2, renormalize=False, lib=lib)
    full = softmax(l, axis=1)
    assert np.allclose(w, np.take_along_axis(full, ids, axis=1), rtol=1e-14, atol=0)


def test_softmax_topk_bruteforce(olib):
    pin_softmax_topk_bruteforce(olib)


def test_softmax_special(olib):
    pin_softmax_special(olib)


# ---------------------------------------------------------------- sigmoid + group top-k

def _brute_sigmoid_group(l, b, G, Gk, k):
    """Best groups by the sum of each group's two largest sel, then the best-sum k subset."""
    E = l.size
    s = 1 / (1 + np.exp(-l))
    sel = s + b
    per = E // G
    score = [sum(sorted(sel[g * per:(g + 1) * per])[-2:]) for g in range(G)]
    gbest = max(itertools.combinations(range(G), Gk), key=lambda c: sum(score[g] for g in c))
    members = [g * per + i for g in gbest for i in range(per)]
    best = max(itertools.combinations(members, k), key=lambda c: sum(sel[list(c)]))
    return tuple(sorted(best)), s


def pin_sigmoid_group_bruteforce(lib):
    rng = np.random.default_rng(11)
    E, G, Gk, k = 12, 4, 2, 3
    for _ in range(40):
        l = rng.normal(size=E) * 2
        b = rng.normal(size=E).astype(np.float32) * 0.1
        ids, w, gaps = oracle.route(oracle.ROUTE_SIGMOID_GROUP, l[None, :], k, bias=b, n_groups=G,
                                    topk_groups=Gk, scale=2.5, lib=lib)
        best, s = _brute_sigmoid_group(l, b.astype(np.float64), G, Gk, k)
        assert tuple(ids[0]) == best
        assert abs(w[0].sum() - 2.5) < 1e-12
        # gates are proportional to s, not to s + bias
        assert abs(w[0, 0] / w[0, 1] - s[ids[0, 0]] / s[ids[0, 1]]) < 1e-12


def pin_sigmoid_group_special(lib):
    # all logits 0 -> s = 0.5 everywhere; the bias alone picks experts; gates = scale / k
    E, G, Gk, k = 16, 4, 2, 4
    b = np.zeros(E, dtype=np.float32)
    b[[1, 2, 13, 14]] = 0.3          # groups 0 and 3 each hold two favoured experts
    b[5] = 0.2                       # group 1 has one favoured expert: group score lower
    ids, w, gaps = oracle.route(oracle.ROUTE_SIGMOID_GROUP, np.zeros((1, E)), k, bias=b, n_groups=G,
                                topk_groups=Gk, scale=2.5, lib=lib)
    assert ids[0].tolist() == [1, 2, 13, 14]
    assert np.allclose(w, 2.5 / 4, rtol=0, atol=1e-15)
    # the group gap: (0.8+0.8) - (0.7+0.5) = 0.4 (float32 biases, so compare loosely)
    assert abs(gaps[0, 1] - 0.4) < 1e-6
    # an expert outside the kept groups is never chosen, even with the best score in its group
    b2 = np.zeros(E, dtype=np.float32)
    b2[[0, 1, 4, 5]] = 0.5
    b2[8] = 0.9                      # group 2: 0.9 + 0 < 1.0 of groups 0 and 1
    ids, _, _ = oracle.route(oracle.ROUTE_SIGMOID_GROUP, np.zeros((1, E)), k, bias=b2, n_groups=G,
                             topk_groups=Gk, scale=1.0, lib=lib)
    assert ids[0].tolist() == [0, 1, 4, 5]
    # without renormalisation the gates are scale * s
    l = np.array([[2.0, -1.0, 0.5, 3.0]])
    ids, w, _ = oracle.route(oracle.ROUTE_SIGMOID_GROUP, l, 2, n_groups=2, topk_groups=2, scale=2.0,
                             renormalize=False, lib=lib)
    assert ids[0].tolist() == [0, 3]
    assert np.allclose(w[0], 2.0 / (1 + np.exp(-np.array([2.0, 3.0]))), rtol=1e-15, atol=0)


def test_sigmoid_group_bruteforce(olib):
    pin_sigmoid_group_bruteforce(olib)


def test_sigmoid_group_special(olib):
    pin_sigmoid_group_special(olib)


# ---------------------------------------------------------------- permute

def pin_permute_bruteforce(lib):
    rng = np.random.default_rng(13)
    for T, k, E in ((1, 1, 1), (4, 2, 8), (7, 3, 5), (33, 8, 16), (5, 4, 64)):
        ids = np.stack([np.sort(rng.choice(E, size=k, replace=False)) if k <= E else
                        rng.integers(0, E, k) for _ in range(T)]).astype(np.int32)
        sp, off, pp = oracle.permute(ids, E, lib=lib)
        flat = ids.reshape(-1)
        expected = [p for e in range(E) for p in range(T * k) if flat[p] == e]
        assert sp.tolist() == expected
        assert off[0] == 0 and off[E] == T * k and np.all(np.diff(off) >= 0)
        for e in range(E):
            assert off[e + 1] - off[e] == int(np.sum(flat == e))
        assert np.array_equal(sp[pp], np.arange(T * k))


def test_permute_bruteforce(olib):
    pin_permute_bruteforce(olib)


def test_permute_rejects_bad_ids(olib):
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 9]], dtype=np.int32), 8, lib=olib)


def pin_expert_counts(lib):
    # a hand-counted example: two calls of T=3, k=2 over E=4
    c = oracle.expert_counts(np.array([[0, 2], [2, 3], [0, 2]]), 4, lib=lib)
    assert c.tolist() == [2, 0, 3, 1]
    c = oracle.expert_counts(np.array([[1, 3], [3, 0], [2, 1]]), 4, counts=c, lib=lib)
    assert c.tolist() == [3, 2, 4, 3]
    # brute force over many calls, and the total is the number of pairs routed
    rng = np.random.default_rng(17)
    E = 37
    c = np.zeros(E, dtype=np.uint64)
    want = [0] * E
    pairs = 0
    for T, k in ((1, 8), (5, 3), (64, 8), (9, 1)):
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        c = oracle.expert_counts(ids, E, counts=c, lib=lib)
        for v in ids.reshape(-1):
            want[int(v)] += 1
        pairs += T * k
    assert c.tolist() == want
    assert int(c.sum()) == pairs
    # the permutation's offsets are one call's counts
    ids = rng.integers(0, E, size=(33, 4)).astype(np.int32)
    _, off, _ = oracle.permute(ids, E, lib=lib)
    assert oracle.expert_counts(ids, E, lib=lib).tolist() == np.diff(off).tolist()


def test_expert_counts(olib):
    pin_expert_counts(olib)


def test_expert_counts_rejects_bad_ids(olib):
    with pytest.raises(ValueError):
        oracle.expert_counts(np.array([[0, 4]], dtype=np.int32), 4, lib=olib)


# ---------------------------------------------------------------- expert FFN and layer

def _identity_q8_0(n: int, d_bits: int = 0x3C00) -> np.ndarray:
    rows = []
    for r in range(n):
        row = b""
        for b in range(n // 32):
            q = [1 if b * 32 + i == r else 0 for i in range(32)]
            row += golden.q8_0_block(d_bits, q)
        rows.append(np.frombuffer(row, np.uint8))
    return np.stack(rows)


def pin_ffn_identity(lib):
    n = 64
    eye = _identity_q8_0(n)
    x = np.linspace(-3.0, 3.0, n)
    y, h = oracle.expert_ffn(oracle.Q8_0, eye, eye, eye, n, n, x, lib=lib)
    silu_x = x / (1.0 + np.exp(-x))
    assert np.allclose(h, silu_x * x, rtol=1e-15, atol=1e-300)
    assert np.allclose(y, silu_x * x, rtol=1e-15, atol=1e-300)
    # doubling d of the down projection doubles y exactly (linearity in W_down)
    eye2 = _identity_q8_0(n, 0x4000)
    y2, _ = oracle.expert_ffn(oracle.Q8_0, eye, eye, eye2, n, n, x, lib=lib)
    assert np.array_equal(y2, 2 * y)
    # gate = 2 * identity: h = silu(2x) * x
    y3, h3 = oracle.expert_ffn(oracle.Q8_0, eye2, eye, eye, n, n, x, lib=lib)
    assert np.allclose(h3, (2 * x) / (1 + np.exp(-2 * x)) * x, rtol=1e-15, atol=1e-300)


def test_ffn_identity(olib):
    pin_ffn_identity(olib)


def pin_ffn_identity_kquants(lib):
    # the identity expert stored as Q5_K, Q6_K and Q3_K (n = 512: two super-blocks a row):
    # every weight decodes to 0 except a 1 on the diagonal, so h = y = silu(x) * x
    n = 512
    x = np.linspace(-3.0, 3.0, n)
    silu_x = x / (1.0 + np.exp(-x))

    def eye(make):
        rows = []
        for i in range(n):
            q = [0] * n
            q[i] = 1
            rows.append(b"".join(make(q[256 * b:256 * (b + 1)]) for b in range(n // 256)))
        return np.frombuffer(b"".join(rows), np.uint8)

    makers = {
        oracle.Q5_K: lambda q: golden.q5_k_block(0x3C00, 0, [1] * 8, [0] * 8, q),
        oracle.Q6_K: lambda q: golden.q6_k_block(0x3C00, [1] * 16, q),
        oracle.Q3_K: lambda q: golden.q3_k_block(0x3C00, [1] * 16, q),
    }
    for qtype, make in makers.items():
        m = eye(make)
        assert m.size == n * oracle.row_bytes(qtype, n)
        y, h = oracle.expert_ffn(qtype, m, m, m, n, n, x, lib=lib)
        assert np.allclose(h, silu_x * x, rtol=1e-15, atol=1e-300), qtype
        assert np.allclose(y, silu_x * x, rtol=1e-15, atol=1e-300), qtype


def test_ffn_identity_kquants(olib):
    pin_ffn_identity_kquants(olib)


def _eye_blocks(n: int, make) -> np.ndarray:
    """The n x n identity stored as 256-weight blocks built by make(q[256])."""
    rows = []
    for i in range(n):
        q = [0] * n
        q[i] = 1
        rows.append(b"".join(make(q[256 * b:256 * (b + 1)]) for b in range(n // 256)))
    return np.stack([np.frombuffer(r, np.uint8) for r in rows])


def pin_ffn_mixed_types(lib):
    # gate/up and down stored in different types: identity gate/up, down = c * identity
    n = 256
    x = np.linspace(-3.0, 3.0, n)
    sx = x / (1.0 + np.exp(-x)) * x
    eye3 = _eye_blocks(n, lambda q: golden.q3_k_block(0x3C00, [1] * 16, q))
    down8 = _identity_q8_0(n, 0x4000)                                   # 2 * identity, Q8_0
    y, h = oracle.expert_ffn(oracle.Q3_K, eye3, eye3, down8, n, n, x, lib=lib, qtype_down=oracle.Q8_0)
    assert np.allclose(h, sx, rtol=1e-15, atol=1e-300)
    assert np.allclose(y, 2 * sx, rtol=1e-15, atol=1e-300)
    eye8 = _identity_q8_0(n)
    down6 = _eye_blocks(n, lambda q: golden.q6_k_block(0x4200, [1] * 16, q))   # 3 * identity, Q6_K
    y, _ = oracle.expert_ffn(oracle.Q8_0, eye8, eye8, down6, n, n, x, lib=lib, qtype_down=oracle.Q6_K)
    assert np.allclose(y, 3 * sx, rtol=1e-15, atol=1e-300)


def test_ffn_mixed_types(olib):
    pin_ffn_mixed_types(olib)


def pin_layer_mixed_types(lib):
    # E = 4 experts with Q3_K identity gate/up and Q4_K down = 2^e * identity; the logits are
    # given (0, 1, 2, 3 for every token), so top-2 = {2, 3} with softmax gates over (2, 3):
    # out = (4 g_2 + 8 g_3) * silu(x) x
    n, E = 256, 4
    eye3 = _eye_blocks(n, lambda q: golden.q3_k_block(0x3C00, [1] * 16, q))
    d_bits = [0x3C00, 0x4000, 0x4400, 0x4800]                          # 1, 2, 4, 8
    downs = [_eye_blocks(n, lambda q, db=db: golden.q4_k_block(db, 0, [1] * 8, [0] * 8, q)) for db in d_bits]
    spec = oracle.LayerSpec(mode=oracle.ROUTE_SOFTMAX, E=E, k=2, H=n, I=n, qtype=oracle.Q3_K,
                            qtype_down=oracle.Q4_K, gate=np.stack([eye3] * E), up=np.stack([eye3] * E),
                            down=np.stack(downs), Wr=np.zeros((E, n), np.float32))
    x = np.stack([np.linspace(-3.0, 3.0, n), np.linspace(2.0, -1.0, n)])
    logits = np.tile(np.arange(E, dtype=np.float64), (2, 1))
    res = oracle.moe_layer(spec, x, logits=logits, lib=lib)
    assert np.array_equal(res["ids"], [[2, 3], [2, 3]])
    g2, g3 = np.exp(2.0) / (np.exp(2.0) + np.exp(3.0)), np.exp(3.0) / (np.exp(2.0) + np.exp(3.0))
    expect = (4 * g2 + 8 * g3) * (x / (1.0 + np.exp(-x)) * x)
    assert np.allclose(res["out"], expect, rtol=1e-13, atol=1e-300)


def test_layer_mixed_types(olib):
    pin_layer_mixed_types(olib)


def _tiny_spec(seed=0, shared=False, mode=oracle.ROUTE_SOFTMAX, E=8, k=2, H=256, I=128, G=1, Gk=1,
               identical=False):
    qt = synth.Q8_0
    shape = synth.LayerShape(H=H, E=E, k=k, I=I, qtype=qt, x_dtype="fp32")
    rb_h, rb_i = synth.row_bytes(qt, H), synth.row_bytes(qt, I)
    gate = np.empty((E, I, rb_h), np.uint8)
    up = np.empty((E, I, rb_h), np.uint8)
    down = np.empty((E, H, rb_i), np.uint8)
    for e in range(E):
        src = 0 if identical else e
        gate[e] = synth.expert_matrix(shape, seed, 0, "gate", src).numpy()
        up[e] = synth.expert_matrix(shape, seed, 0, "up", src).numpy()
        down[e] = synth.expert_matrix(shape, seed, 0, "down", src).numpy()
    Wr = synth.router_weight(shape, seed, 0).numpy()
    kw = {}
    if shared:
        sshape = synth.LayerShape(H=H, E=E, k=k, I=I, qtype=qt, I_s=64, shared_qtype=qt)
        kw = dict(shared_qtype=oracle.Q8_0, I_s=64,
                  s_gate=synth.expert_matrix(sshape, seed, 0, "s_gate", 0).numpy(),
                  s_up=synth.expert_matrix(sshape, seed, 0, "s_up", 0).numpy(),
                  s_down=synth.expert_matrix(sshape, seed, 0, "s_down", 0).numpy())
    bias = synth.normal((E,), 0.1, 77).numpy() if mode == oracle.ROUTE_SIGMOID_GROUP else None
    return oracle.LayerSpec(mode=mode, E=E, k=k, H=H, I=I, qtype=oracle.Q8_0, gate=gate, up=up,
                            down=down, Wr=Wr, bias=bias, n_groups=G, topk_groups=Gk,
                            scale=2.5 if mode == oracle.ROUTE_SIGMOID_GROUP else 1.0, **kw)


def _dense_ffn_all(spec, x, lib):
    """FFN of every expert on every token via dequantized matrices and numpy matmuls."""
    H, I, E = spec.H, spec.I, spec.E
    Y = np.empty((E, x.shape[0], H))
    for e in range(E):
        Wg = oracle.dequant(oracle.Q8_0, spec.gate[e], I, H, lib=lib)
        Wu = oracle.dequant(oracle.Q8_0, spec.up[e], I, H, lib=lib)
        Wd = oracle.dequant(oracle.Q8_0, spec.down[e], H, I, lib=lib)
        g = x @ Wg.T
        u = x @ Wu.T
        Y[e] = ((g / (1 + np.exp(-g))) * u) @ Wd.T
    return Y


def pin_dense_masked_equals_sparse(lib):
    for shared, mode, E, k, G, Gk in ((False, oracle.ROUTE_SOFTMAX, 8, 2, 1, 1),
                                      (True, oracle.ROUTE_SIGMOID_GROUP, 8, 2, 4, 2)):
        spec = _tiny_spec(shared=shared, mode=mode, E=E, k=k, G=G, Gk=Gk)
        x = synth.activations(5, spec.H, 0, "fp32").double().numpy()
        res = oracle.moe_layer(spec, x, lib=lib)
        Y = _dense_ffn_all(spec, x, lib)
        # the mask: gate weight of expert e for token t, zero when e is not selected
        mask = np.zeros((x.shape[0], E))
        for t in range(x.shape[0]):
            for j in range(k):
                mask[t, res["ids"][t, j]] = res["w"][t, j]
        dense = np.einsum("te,eth->th", mask, Y)
        if shared:
            Wg = oracle.dequant(oracle.Q8_0, spec.s_gate, 64, spec.H, lib=lib)
            Wu = oracle.dequant(oracle.Q8_0, spec.s_up, 64, spec.H, lib=lib)
            Wd = oracle.dequant(oracle.Q8_0, spec.s_down, spec.H, 64, lib=lib)
            g, u = x @ Wg.T, x @ Wu.T
            dense += ((g / (1 + np.exp(-g))) * u) @ Wd.T
        rel = np.linalg.norm(res["out"] - dense) / np.linalg.norm(dense)
        assert rel < 1e-13, rel
        # routing is computed from x @ Wr^T
        assert np.allclose(res["logits"], x @ spec.Wr.astype(np.float64).T, rtol=1e-13, atol=1e-13)


def pin_identical_experts_ignore_routing(lib):
    spec = _tiny_spec(identical=True)
    x = synth.activations(4, spec.H, 3, "fp32").double().numpy()
    res = oracle.moe_layer(spec, x, lib=lib)
    y0, _ = oracle.expert_ffn(oracle.Q8_0, spec.gate[0], spec.up[0], spec.down[0], spec.H, spec.I,
                              x[2], lib=lib)
    assert np.allclose(res["out"][2], y0, rtol=1e-13, atol=1e-15)


def pin_token_permutation(lib):
    spec = _tiny_spec()
    x = synth.activations(6, spec.H, 4, "fp32").double().numpy()
    perm = np.array([3, 0, 5, 1, 4, 2])
    a = oracle.moe_layer(spec, x, lib=lib)
    b = oracle.moe_layer(spec, x[perm], lib=lib)
    assert np.array_equal(a["out"][perm], b["out"])
    assert np.array_equal(a["ids"][perm], b["ids"])


def test_dense_masked_equals_sparse(olib):
    pin_dense_masked_equals_sparse(olib)


def test_identical_experts_ignore_routing(olib):
    pin_identical_experts_ignore_routing(olib)


def test_token_permutation(olib):
    pin_token_permutation(olib)


def test_layer_threads_agree(olib):
    spec = _tiny_spec(shared=True, mode=oracle.ROUTE_SIGMOID_GROUP, G=4, Gk=2)
    x = synth.activations(9, spec.H, 9, "fp32").double().numpy()
    a = oracle.moe_layer(spec, x, n_threads=1, lib=olib)
    b = oracle.moe_layer(spec, x, n_threads=4, lib=olib)
    assert np.array_equal(a["out"], b["out"])


# ---------------------------------------------------------------- RMSNorm, bf16, stack

def pin_rmsnorm(lib):
    H = 8
    g = np.linspace(0.5, 2.0, H).astype(np.float32)
    x = np.array([[3.0] * H, [-2.0] * H, [0.0] * H])
    u = oracle.rmsnorm(x, g, eps=1e-6, lib=lib)
    for row, c in enumerate((3.0, -2.0, 0.0)):
        expected = g.astype(np.float64) * (c / math.sqrt(c * c + 1e-6))
        assert np.allclose(u[row], expected, rtol=1e-15, atol=0)
    # with eps = 0 the map is scale invariant: rmsnorm(a x) = rmsnorm(x) for a > 0,
    # and every row of rmsnorm(x) / gamma has mean square 1
    xr = np.random.default_rng(2).normal(size=(2, H))
    u0 = oracle.rmsnorm(xr, g, eps=0.0, lib=lib)
    assert np.allclose(oracle.rmsnorm(1000 * xr, g, eps=0.0, lib=lib), u0, rtol=1e-14, atol=0)
    assert np.allclose(np.mean((u0 / g.astype(np.float64)) ** 2, axis=1), 1.0, rtol=1e-14, atol=0)


def pin_round_bf16(lib):
    # against torch's fp32 -> bf16 conversion (round to nearest even) on fp32 inputs
    v = np.concatenate([np.random.default_rng(8).normal(size=2000) * 10.0 ** np.random.default_rng(9)
                        .integers(-30, 30, 2000), [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0]])
    v32 = v.astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).float().double().numpy()
    got = np.array([oracle.round_bf16(float(a), lib=lib) for a in v32])
    assert np.array_equal(got, ref)


def test_rmsnorm(olib):
    pin_rmsnorm(olib)


def test_round_bf16(olib):
    pin_round_bf16(olib)


def test_stack_zero_experts_is_identity(olib):
    """Experts with d = 0 add nothing: the residual stream passes unchanged."""
    spec = _tiny_spec()
    z = lambda a: np.zeros_like(a)  # noqa: E731
    zspec = oracle.LayerSpec(mode=spec.mode, E=spec.E, k=spec.k, H=spec.H, I=spec.I, qtype=oracle.Q8_0,
                             gate=z(spec.gate), up=z(spec.up), down=z(spec.down), Wr=spec.Wr)
    x = synth.activations(3, spec.H, 1, "fp32").double().numpy()
    out, ids, gaps = oracle.moe_stack([zspec, zspec], [np.ones(spec.H, np.float32)] * 2, x, lib=olib)
    assert np.array_equal(out, x)
    assert ids.shape == (2, 3, spec.k)


def test_stack_one_layer_matches_layer(olib):
    spec = _tiny_spec(seed=3)
    g = synth.gamma(spec.H, 5, 0).numpy()
    x = synth.activations(3, spec.H, 2, "fp32").double().numpy()
    out, ids, _ = oracle.moe_stack([spec], [g], x, lib=olib)
    u = oracle.rmsnorm(x, g, lib=olib)
    u = np.vectorize(lambda a: oracle.round_bf16(a, lib=olib))(u)
    ref = oracle.moe_layer(spec, u, lib=olib)
    assert np.array_equal(out, x + ref["out"])
    assert np.array_equal(ids[0], ref["ids"])


PINS = {
    "half_to_double": pin_half_to_double,
    "q8_0_handbuilt": pin_q8_0_handbuilt,
    "q4_k_handbuilt": pin_q4_k_handbuilt,
    "q4_k_multiblock_rows": pin_q4_k_multiblock_rows,
    "q5_k_handbuilt": pin_q5_k_handbuilt,
    "q6_k_handbuilt": pin_q6_k_handbuilt,
    "q3_k_handbuilt": pin_q3_k_handbuilt,
    "kquant_multiblock_rows": pin_kquant_multiblock_rows,
    "e2m1": pin_e2m1,
    "mxfp4_handbuilt": pin_mxfp4_handbuilt,
    "mxfp4_multiblock_rows": pin_mxfp4_multiblock_rows,
    "router_integer": pin_router_integer,
    "softmax_topk_bruteforce": pin_softmax_topk_bruteforce,
    "softmax_special": pin_softmax_special,
    "sigmoid_group_bruteforce": pin_sigmoid_group_bruteforce,
    "sigmoid_group_special": pin_sigmoid_group_special,
    "permute_bruteforce": pin_permute_bruteforce,
    "expert_counts": pin_expert_counts,
    "ffn_identity": pin_ffn_identity,
    "ffn_identity_kquants": pin_ffn_identity_kquants,
    "ffn_mixed_types": pin_ffn_mixed_types,
    "layer_mixed_types": pin_layer_mixed_types,
    "dense_masked_equals_sparse": pin_dense_masked_equals_sparse,
    "identical_experts_ignore_routing": pin_identical_experts_ignore_routing,
    "token_permutation": pin_token_permutation,
    "rmsnorm": pin_rmsnorm,
    "round_bf16": pin_round_bf16,
}
