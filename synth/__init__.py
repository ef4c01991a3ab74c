"""Seeded synthetic inputs for the routed-expert MoE layer.

This module draws the random tensors (activations, router weights, biases,
RMSNorm weights, expert weights) and stores expert weights in the GGUF block
layouts Q8_0, Q4_K, Q5_K, Q6_K, Q3_K and MXFP4.  It is shared by the tests,
the benchmark and the
smoke check, and it holds none of the layer's arithmetic: it never routes,
never dequantizes and never evaluates an expert.  (Encoding a float matrix
into blocks is how the stored inputs are made; decoding them is the oracle's
and the CUDA library's job, each with its own code.)

Every tensor comes from its own seed, derived from (workload seed, layer,
tensor tag, expert) with splitmix64, so any one expert can be regenerated
alone.  Generation runs with torch on any device; the same seed gives
different numbers on CPU and CUDA, so a parity test draws everything it
compares on the CPU and uploads it.

Workload shapes (also used by bench.py):
  tiny      T=4,    H=256,  E=8,   k=2, I=128,  Q8_0, x fp32, softmax
  decode    T=1|2,  H=2048, E=128, k=8, I=768,  Q4_K, x bf16, softmax
  prefill   T=4096, same as decode, Zipf(1) expert popularity
  deepseek  T=2|512, H=7168, E=256, k=8, I=2048 Q4_K, sigmoid + bias,
            8 groups / best 4, scale 2.5, shared expert I_s=2048 in Q8_0
  stack     48 x (RMSNorm -> decode-shaped layer -> residual), T in 1..64
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

Q8_0 = "q8_0"
Q4_K = "q4_k"
Q5_K = "q5_k"
Q6_K = "q6_k"
Q3_K = "q3_k"
MXFP4 = "mxfp4"

# weights and bytes per block of each stored type
BLOCK = {Q8_0: (32, 34), Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210), Q3_K: (256, 110),
         MXFP4: (32, 17)}

TAGS = {"x": 1, "router": 2, "bias": 3, "gate": 4, "up": 5, "down": 6, "gamma": 7,
        "s_gate": 8, "s_up": 9, "s_down": 10, "zipf": 11, "fill": 12}


def splitmix64(v: int) -> int:
    v = (v + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = v
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def derive_seed(*parts: int) -> int:
    s = 0x5EED
    for p in parts:
        s = splitmix64(s ^ (int(p) & 0xFFFFFFFFFFFFFFFF))
    return s & 0x7FFFFFFFFFFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def row_bytes(qtype: str, K: int) -> int:
    weights, nbytes = BLOCK[qtype]
    return K // weights * nbytes


# --------------------------------------------------------------------------- encoders

def _fp16_bits(v: torch.Tensor) -> torch.Tensor:
    """fp32 -> fp16 (round to nearest even) -> little-endian byte pair [..., 2]."""
    h = v.to(torch.float16).view(torch.int16).to(torch.int32) & 0xFFFF
    return torch.stack([h & 0xFF, (h >> 8) & 0xFF], dim=-1).to(torch.uint8)


def encode_q8_0(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/32*34] uint8 Q8_0 blocks.

    Per block of 32: d = max|w|/127 stored as fp16, q = round-half-away(w/d)
    clamped to int8 (q = 0 where d = 0).
    """
    rows, K = w.shape
    assert K % 32 == 0
    b = w.reshape(rows, K // 32, 32).float()
    amax = b.abs().amax(dim=-1)
    d16 = (amax / 127.0).to(torch.float16)
    d = d16.float()
    inv = torch.where(d > 0, 1.0 / torch.where(d > 0, d, torch.ones_like(d)), torch.zeros_like(d))
    v = b * inv.unsqueeze(-1)
    q = (torch.sign(v) * torch.floor(v.abs() + 0.5)).clamp(-128, 127).to(torch.int32)
    qb = (q & 0xFF).to(torch.uint8)
    out = torch.cat([_fp16_bits(d), qb], dim=-1)               # [rows, nb, 34]
    return out.reshape(rows, K // 32 * 34).contiguous()


def pack_q4_k(d: torch.Tensor, dmin: torch.Tensor, sc: torch.Tensor, m: torch.Tensor,
              q: torch.Tensor) -> torch.Tensor:
    """Pack Q4_K fields into 144-byte blocks.

    d, dmin: [..., ] float (stored as fp16); sc, m: [..., 8] ints in [0, 63];
    q: [..., 256] ints in [0, 15].  Returns [..., 144] uint8.
    Scale/min bytes: S[j] = sc_j | (sc_{j+4} >> 4) << 6, S[j+4] = m_j | (m_{j+4} >> 4) << 6,
    S[j+8] = (sc_{j+4} & 15) | (m_{j+4} & 15) << 4 for j < 4.  Quant byte i of group c
    holds q[64c+i] (low nibble) and q[64c+32+i] (high nibble).
    """
    sc = sc.to(torch.int32)
    m = m.to(torch.int32)
    q = q.to(torch.int32)
    lo_sc, hi_sc = sc[..., :4], sc[..., 4:]
    lo_m, hi_m = m[..., :4], m[..., 4:]
    s0 = (lo_sc & 63) | ((hi_sc >> 4) << 6)
    s1 = (lo_m & 63) | ((hi_m >> 4) << 6)
    s2 = (hi_sc & 15) | ((hi_m & 15) << 4)
    S = torch.cat([s0, s1, s2], dim=-1).to(torch.uint8)           # [..., 12]
    qg = q.reshape(*q.shape[:-1], 4, 2, 32)                        # [..., c, half, i]
    qs = (qg[..., 0, :] | (qg[..., 1, :] << 4)).reshape(*q.shape[:-1], 128).to(torch.uint8)
    return torch.cat([_fp16_bits(d.float()), _fp16_bits(dmin.float()), S, qs], dim=-1)


def encode_q4_k(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/256*144] uint8 Q4_K blocks.

    A plain min/max quantizer per 32-weight sub-block (not ggml's iterative
    search): scale_j = (max - min)/15 with min clamped to <= 0, m_j = -min;
    d = max_j scale_j / 63, dmin = max_j m_j / 63 (fp16); 6-bit sc_j, m_j
    rounded; q = clamp(round((w + dmin*m_j)/(d*sc_j)), 0, 15).
    """
    rows, K = w.shape
    assert K % 256 == 0
    b = w.reshape(rows, K // 256, 8, 32).float()
    mn = b.amin(dim=-1).clamp(max=0.0)
    mx = b.amax(dim=-1)
    scale = (mx - mn) / 15.0
    mins = -mn
    d = (scale.amax(dim=-1) / 63.0).to(torch.float16).float()
    dmin = (mins.amax(dim=-1) / 63.0).to(torch.float16).float()
    safe_d = torch.where(d > 0, d, torch.ones_like(d)).unsqueeze(-1)
    safe_dm = torch.where(dmin > 0, dmin, torch.ones_like(dmin)).unsqueeze(-1)
    sc = torch.where(d.unsqueeze(-1) > 0, torch.round(scale / safe_d), torch.zeros_like(scale)).clamp(0, 63)
    m = torch.where(dmin.unsqueeze(-1) > 0, torch.round(mins / safe_dm), torch.zeros_like(mins)).clamp(0, 63)
    step = (d.unsqueeze(-1) * sc).unsqueeze(-1)                    # [rows, nb, 8, 1]
    off = (dmin.unsqueeze(-1) * m).unsqueeze(-1)
    safe_step = torch.where(step > 0, step, torch.ones_like(step))
    q = torch.where(step > 0, torch.round((b + off) / safe_step), torch.zeros_like(b)).clamp(0, 15)
    blocks = pack_q4_k(d, dmin, sc.to(torch.int32), m.to(torch.int32), q.reshape(rows, K // 256, 256))
    return blocks.reshape(rows, K // 256 * 144).contiguous()


def pack_q5_k(d: torch.Tensor, dmin: torch.Tensor, sc: torch.Tensor, m: torch.Tensor,
              q: torch.Tensor) -> torch.Tensor:
    """Pack Q5_K fields into 176-byte blocks: q [..., 256] ints in [0, 31].  The header and
    the low nibbles are laid out as in Q4_K; byte i of the 32 fifth-bit bytes holds bit 4 of
    q[32j + i] in its bit j."""
    q = q.to(torch.int32)
    base = pack_q4_k(d, dmin, sc, m, q & 15)
    bits = ((q >> 4) & 1).reshape(*q.shape[:-1], 8, 32)             # [..., j, i]
    shifts = torch.arange(8, dtype=torch.int32, device=q.device).reshape(8, 1)
    qh = (bits << shifts).sum(dim=-2).to(torch.uint8)                # [..., 32]
    return torch.cat([base[..., :16], qh, base[..., 16:]], dim=-1)


def encode_q5_k(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/256*176] uint8 Q5_K blocks: the Q4_K quantizer with 32
    levels per sub-block instead of 16."""
    rows, K = w.shape
    assert K % 256 == 0
    b = w.reshape(rows, K // 256, 8, 32).float()
    mn = b.amin(dim=-1).clamp(max=0.0)
    mx = b.amax(dim=-1)
    scale = (mx - mn) / 31.0
    mins = -mn
    d = (scale.amax(dim=-1) / 63.0).to(torch.float16).float()
    dmin = (mins.amax(dim=-1) / 63.0).to(torch.float16).float()
    safe_d = torch.where(d > 0, d, torch.ones_like(d)).unsqueeze(-1)
    safe_dm = torch.where(dmin > 0, dmin, torch.ones_like(dmin)).unsqueeze(-1)
    sc = torch.where(d.unsqueeze(-1) > 0, torch.round(scale / safe_d), torch.zeros_like(scale)).clamp(0, 63)
    m = torch.where(dmin.unsqueeze(-1) > 0, torch.round(mins / safe_dm), torch.zeros_like(mins)).clamp(0, 63)
    step = (d.unsqueeze(-1) * sc).unsqueeze(-1)
    off = (dmin.unsqueeze(-1) * m).unsqueeze(-1)
    safe_step = torch.where(step > 0, step, torch.ones_like(step))
    q = torch.where(step > 0, torch.round((b + off) / safe_step), torch.zeros_like(b)).clamp(0, 31)
    blocks = pack_q5_k(d, dmin, sc.to(torch.int32), m.to(torch.int32), q.reshape(rows, K // 256, 256))
    return blocks.reshape(rows, K // 256 * 176).contiguous()


def _signed_group_quant(w: torch.Tensor, qmax: int, smax: int):
    """Symmetric quantizer shared by Q6_K and Q3_K: per 16-weight group a step s_g =
    max|w| / qmax; one fp16 d per 256 = max_g s_g / smax; integer group scales
    sc_g = round(s_g / d) in [0, smax]; q = clamp(round(w / (d sc_g)), -qmax, qmax - 1).
    w: [rows, nb, 16, 16]."""
    s = w.abs().amax(dim=-1) / qmax                                  # [rows, nb, 16]
    d = (s.amax(dim=-1) / smax).to(torch.float16).float()            # [rows, nb]
    safe_d = torch.where(d > 0, d, torch.ones_like(d)).unsqueeze(-1)
    sc = torch.where(d.unsqueeze(-1) > 0, torch.round(s / safe_d), torch.zeros_like(s)).clamp(0, smax)
    step = (d.unsqueeze(-1) * sc).unsqueeze(-1)
    safe_step = torch.where(step > 0, step, torch.ones_like(step))
    q = torch.where(step > 0, torch.round(w / safe_step), torch.zeros_like(w)).clamp(-qmax, qmax - 1)
    return d, sc.to(torch.int32), q.to(torch.int32)


def pack_q6_k(d: torch.Tensor, sc: torch.Tensor, q: torch.Tensor) -> torch.Tensor:
    """Pack Q6_K fields into 210-byte blocks: sc [..., 16] ints in [-128, 127], q [..., 256]
    ints in [-32, 31].  With u = q + 32, weight 128h + 32r + l puts the low nibble of u in
    byte 64h + 32(r % 2) + l of the first 128 bytes (low nibble for r < 2, high for r >= 2)
    and its top two bits in bits 2r..2r+1 of byte 128 + 32h + l; then the 16 scale bytes,
    then fp16 d."""
    u = (q.to(torch.int32) + 32).reshape(*q.shape[:-1], 2, 4, 32)   # [..., h, r, l]
    lo = u & 15
    ql = torch.cat([lo[..., 0, :] | (lo[..., 2, :] << 4), lo[..., 1, :] | (lo[..., 3, :] << 4)], dim=-1)
    shifts = (2 * torch.arange(4, dtype=torch.int32, device=q.device)).reshape(4, 1)
    qh = (((u >> 4) & 3) << shifts).sum(dim=-2)                      # [..., h, 32]
    lead = q.shape[:-1]
    scb = (sc.to(torch.int32) & 0xFF).to(torch.uint8)
    return torch.cat([ql.reshape(*lead, 128).to(torch.uint8), qh.reshape(*lead, 64).to(torch.uint8), scb,
                      _fp16_bits(d.float())], dim=-1)


def encode_q6_k(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/256*210] uint8 Q6_K blocks (symmetric per 16 weights)."""
    rows, K = w.shape
    assert K % 256 == 0
    d, sc, q = _signed_group_quant(w.reshape(rows, K // 256, 16, 16).float(), 32, 127)
    blocks = pack_q6_k(d, sc, q.reshape(rows, K // 256, 256))
    return blocks.reshape(rows, K // 256 * 210).contiguous()


def pack_q3_k(d: torch.Tensor, sc: torch.Tensor, q: torch.Tensor) -> torch.Tensor:
    """Pack Q3_K fields into 110-byte blocks: sc [..., 16] ints in [-32, 31], q [..., 256]
    ints in [-4, 3].  With v = q + 4, weight 128h + 32r + l puts bit 2 of v in bit 4h + r of
    byte l (the 32 mask bytes) and bits 0-1 in bits 2r..2r+1 of byte 32 + 32h + l.  Scale j
    is stored as s = sc_j + 32: bits 0-3 in the low nibble of byte 96 + j (j < 8) or the high
    nibble of byte 96 + j - 8, bits 4-5 in bits 2(j // 4).. of byte 104 + j % 4; then fp16 d."""
    lead = q.shape[:-1]
    v = (q.to(torch.int32) + 4).reshape(*lead, 2, 4, 32)             # [..., h, r, l]
    hbit = ((v >> 2) & 1).reshape(*lead, 8, 32)                      # [..., 4h + r, l]
    hm = (hbit << torch.arange(8, dtype=torch.int32, device=q.device).reshape(8, 1)).sum(dim=-2)
    qs = ((v & 3) << (2 * torch.arange(4, dtype=torch.int32, device=q.device)).reshape(4, 1)).sum(dim=-2)   # [..., h, l]
    s = sc.to(torch.int32) + 32                                      # [..., 16]
    nib = (s[..., :8] & 15) | ((s[..., 8:] & 15) << 4)               # [..., 8]
    top = ((s >> 4) & 3).reshape(*lead, 4, 4)                        # [..., j // 4, j % 4]
    hi = (top << (2 * torch.arange(4, dtype=torch.int32, device=q.device)).reshape(4, 1)).sum(dim=-2)      # [..., 4]
    return torch.cat([hm.to(torch.uint8), qs.reshape(*lead, 64).to(torch.uint8), nib.to(torch.uint8),
                      hi.to(torch.uint8), _fp16_bits(d.float())], dim=-1)


def encode_q3_k(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/256*110] uint8 Q3_K blocks (symmetric per 16 weights)."""
    rows, K = w.shape
    assert K % 256 == 0
    d, sc, q = _signed_group_quant(w.reshape(rows, K // 256, 16, 16).float(), 4, 31)
    blocks = pack_q3_k(d, sc, q.reshape(rows, K // 256, 256))
    return blocks.reshape(rows, K // 256 * 110).contiguous()


def pack_mxfp4(e: torch.Tensor, codes: torch.Tensor) -> torch.Tensor:
    """Pack MXFP4 fields into 17-byte blocks: e [...] E8M0 scale bytes, codes [..., 32] E2M1
    codes in [0, 15]; byte 1 + j holds codes[j] (low nibble) and codes[j + 16] (high)."""
    c = codes.to(torch.int32)
    qs = (c[..., :16] | (c[..., 16:] << 4)).to(torch.uint8)
    return torch.cat([e.to(torch.int32).unsqueeze(-1).to(torch.uint8), qs], dim=-1)


def encode_mxfp4(w: torch.Tensor) -> torch.Tensor:
    """[rows, K] float -> [rows, K/32*17] uint8 MXFP4 blocks.  Per block of 32 the shared scale
    is 2^(floor(log2 max|w|) - 2) (the largest E2M1 magnitude, 6, has exponent 2); each weight
    takes the nearest E2M1 magnitude of w / scale (the lower one on a tie), clamped to 6."""
    rows, K = w.shape
    assert K % 32 == 0
    b = w.reshape(rows, K // 32, 32).float()
    amax = b.abs().amax(dim=-1)
    E = torch.where(amax > 0, torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 2,
                    torch.full_like(amax, -127.0)).clamp(-127, 127)
    v = b / torch.exp2(E).unsqueeze(-1)
    mags = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], device=b.device)
    idx = (v.abs().clamp(max=6.0).unsqueeze(-1) - mags).abs().argmin(dim=-1)
    codes = torch.where((v < 0) & (idx > 0), idx + 8, idx)
    blocks = pack_mxfp4((E + 127).to(torch.int32), codes)
    return blocks.reshape(rows, K // 32 * 17).contiguous()


_ENCODERS = {Q8_0: encode_q8_0, Q4_K: encode_q4_k, Q5_K: encode_q5_k, Q6_K: encode_q6_k, Q3_K: encode_q3_k,
             MXFP4: encode_mxfp4}


def encode(qtype: str, w: torch.Tensor) -> torch.Tensor:
    return _ENCODERS[qtype](w)


# --------------------------------------------------------------------------- layer specs

@dataclasses.dataclass
class LayerShape:
    H: int
    E: int
    k: int
    I: int
    qtype: str
    mode: str = "softmax"            # or "sigmoid_group"
    n_groups: int = 1
    topk_groups: int = 1
    scale: float = 1.0
    renormalize: bool = True
    I_s: int = 0                     # shared expert intermediate (0 = none)
    shared_qtype: str = Q8_0
    router_std: float = 0.05
    bias_std: float = 0.0            # > 0: per-expert selection bias
    weight_std: float = 0.02
    x_dtype: str = "bf16"            # or "fp32"


TINY = LayerShape(H=256, E=8, k=2, I=128, qtype=Q8_0, x_dtype="fp32")
DECODE = LayerShape(H=2048, E=128, k=8, I=768, qtype=Q4_K)
DEEPSEEK = LayerShape(H=7168, E=256, k=8, I=2048, qtype=Q4_K, mode="sigmoid_group", n_groups=8,
                      topk_groups=4, scale=2.5, I_s=2048, shared_qtype=Q8_0, bias_std=0.1)

WORKLOAD_SEEDS = {"tiny": 0, "decode": 2, "prefill": 3, "deepseek": 4, "stack": 5}


def expert_matrix(shape: LayerShape, seed: int, layer: int, which: str, expert: int,
                  device="cpu") -> torch.Tensor:
    """One expert's quantized matrix: gate/up [I, rb(H)], down [H, rb(I)]."""
    if which in ("gate", "up"):
        rows, K, qt = shape.I, shape.H, shape.qtype
    elif which == "down":
        rows, K, qt = shape.H, shape.I, shape.qtype
    elif which in ("s_gate", "s_up"):
        rows, K, qt = shape.I_s, shape.H, shape.shared_qtype
    else:
        rows, K, qt = shape.H, shape.I_s, shape.shared_qtype
    w = normal((rows, K), shape.weight_std, derive_seed(seed, layer, TAGS[which], expert), device)
    return encode(qt, w)


def router_weight(shape: LayerShape, seed: int, layer: int, attempt: int = 0, device="cpu"):
    return normal((shape.E, shape.H), shape.router_std,
                  derive_seed(seed, layer, TAGS["router"], 1000 * attempt), device)


def bias(shape: LayerShape, seed: int, layer: int, device="cpu"):
    if shape.bias_std <= 0:
        return None
    return normal((shape.E,), shape.bias_std, derive_seed(seed, layer, TAGS["bias"]), device)


def gamma(H: int, seed: int, layer: int, device="cpu"):
    return 1.0 + normal((H,), 0.01, derive_seed(seed, layer, TAGS["gamma"]), device)


def activations(T: int, H: int, seed: int, x_dtype: str = "bf16", token_seeds=None,
                device="cpu") -> torch.Tensor:
    """x [T, H] ~ N(0, 1); bf16 values (returned as bf16) or fp32.

    token_seeds (optional list of ints, one per token) redraws individual
    tokens from their own sub-streams (used to enforce a routing margin).
    """
    if token_seeds is None:
        x = normal((T, H), 1.0, derive_seed(seed, TAGS["x"]), device)
    else:
        x = torch.stack([normal((H,), 1.0, derive_seed(seed, TAGS["x"], 7, s), device)
                         for s in token_seeds])
    return x.to(torch.bfloat16) if x_dtype == "bf16" else x


class ExpertBank:
    """All experts of one layer, as uint8 tensors [E, rows, row_bytes].

    `exact` lists the experts drawn from their own seeds on the CPU (what a
    parity test compares); every other expert is drawn on `fill_device` from
    a separate seed (same distribution, never compared).  exact=None draws all
    experts on `fill_device`.
    """

    def __init__(self, shape: LayerShape, seed: int, layer: int = 0, exact=None,
                 fill_device="cpu", out_device=None, chunk: int = 16):
        out_device = out_device or fill_device
        s = shape
        rb_h, rb_i = row_bytes(s.qtype, s.H), row_bytes(s.qtype, s.I)
        self.gate = torch.empty((s.E, s.I, rb_h), dtype=torch.uint8, device=out_device)
        self.up = torch.empty((s.E, s.I, rb_h), dtype=torch.uint8, device=out_device)
        self.down = torch.empty((s.E, s.H, rb_i), dtype=torch.uint8, device=out_device)
        exact_set = set(range(s.E)) if exact is None else set(int(e) for e in exact)
        for e in range(s.E):
            exact_e = e in exact_set
            dev = fill_device if (exact is None or not exact_e) else "cpu"
            tag_layer = layer if exact_e else layer + (1 << 20)
            for name, buf in (("gate", self.gate), ("up", self.up), ("down", self.down)):
                buf[e].copy_(expert_matrix(s, seed, tag_layer, name, e, dev))
        self.shared = None
        if s.I_s > 0:
            self.shared = tuple(expert_matrix(s, seed, layer, n, 0, "cpu").to(out_device)
                                for n in ("s_gate", "s_up", "s_down"))


def expert_stack(shape: LayerShape, seed: int, layer: int, which: str, device="cpu",
                 chunk_rows: int = 1 << 17) -> torch.Tensor:
    """All E experts of one matrix at once (a different stream from expert_matrix):
    gate/up -> [E, I, rb(H)], down -> [E, H, rb(I)].  Drawn and encoded in row
    chunks so the fp32 staging stays small."""
    rows, K = (shape.I, shape.H) if which in ("gate", "up") else (shape.H, shape.I)
    total = shape.E * rows
    out = torch.empty((total, row_bytes(shape.qtype, K)), dtype=torch.uint8, device=device)
    for i, r0 in enumerate(range(0, total, chunk_rows)):
        n = min(chunk_rows, total - r0)
        w = normal((n, K), shape.weight_std, derive_seed(seed, layer, TAGS[which], 1 << 30, i), device)
        out[r0:r0 + n] = encode(shape.qtype, w)
    return out.view(shape.E, rows, -1)


# --------------------------------------------------------------------------- Zipf routing

def zipf_target_logits(T: int, E: int, k: int, seed: int, alpha: float = 1.0, n_zero: int = 8,
                       margin: float = 0.5) -> np.ndarray:
    """Target router logits [T, E] whose top-k follows Zipf(alpha) popularity.

    p_e proportional to 1/rank^alpha over a seeded permutation of the experts,
    with the n_zero least popular ranks at p = 0 (they receive no tokens).
    L[t,e] = log p_e + Gumbel(t,e) (Gumbel-top-k samples k experts without
    replacement with probability proportional to p); the chosen k are then
    lifted so that they stand at least `margin` above the best unchosen one.
    """
    rng = np.random.default_rng(derive_seed(seed, TAGS["zipf"]))
    perm = rng.permutation(E)
    ranks = np.empty(E, dtype=np.int64)
    ranks[perm] = np.arange(1, E + 1)
    logp = -alpha * np.log(ranks.astype(np.float64))
    logp[ranks > E - n_zero] = -40.0
    g = rng.gumbel(size=(T, E))
    L = logp[None, :] + g
    order = np.argsort(-L, axis=1, kind="stable")
    chosen = order[:, :k]
    best_rest = np.take_along_axis(L, order[:, k:k + 1], axis=1)[:, 0]
    worst_chosen = np.take_along_axis(L, order[:, k - 1:k], axis=1)[:, 0]
    lift = np.maximum(0.0, margin - (worst_chosen - best_rest))
    rows = np.arange(T)[:, None]
    L[rows, chosen] += lift[:, None]
    L[:, ranks > E - n_zero] = np.minimum(L[:, ranks > E - n_zero], -40.0)
    return L


def activations_for_logits(L: np.ndarray, Wr: np.ndarray, seed: int) -> torch.Tensor:
    """bf16 activations x [T, H] with x @ Wr^T close to the target logits L.

    x = x0 + Wr^T (Wr Wr^T)^{-1} (L - x0 Wr^T) with x0 ~ N(0, 1): the
    minimum-norm correction of a random draw (fp64), then rounded to bf16.
    """
    T, E = L.shape
    H = Wr.shape[1]
    x0 = normal((T, H), 1.0, derive_seed(seed, TAGS["x"]), "cpu").double().numpy()
    W = Wr.astype(np.float64)
    C = W @ W.T
    resid = L - x0 @ W.T
    coef = np.linalg.solve(C, resid.T).T
    x = x0 + coef @ W
    return torch.from_numpy(x).float().to(torch.bfloat16)


def zipf_expert_popularity(E: int, seed: int, alpha: float = 1.0, n_zero: int = 8) -> np.ndarray:
    rng = np.random.default_rng(derive_seed(seed, TAGS["zipf"]))
    perm = rng.permutation(E)
    ranks = np.empty(E, dtype=np.int64)
    ranks[perm] = np.arange(1, E + 1)
    p = 1.0 / ranks.astype(np.float64) ** alpha
    p[ranks > E - n_zero] = 0.0
    return p / p.sum()


def bytes_per_expert(shape: LayerShape) -> int:
    return 2 * shape.I * row_bytes(shape.qtype, shape.H) + shape.H * row_bytes(shape.qtype, shape.I)


def shared_bytes(shape: LayerShape) -> int:
    if shape.I_s <= 0:
        return 0
    return 2 * shape.I_s * row_bytes(shape.shared_qtype, shape.H) + shape.H * row_bytes(shape.shared_qtype, shape.I_s)


def nbytes_gib(n: int) -> float:
    return n / float(1 << 30)

