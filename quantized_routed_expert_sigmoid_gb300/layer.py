"""Device-resident MoE layer: torch tensors in, one moe_layer call out.

A convenience wrapper over the C ABI for callers that hold their weights in
torch tensors.  It fills a moe_layer_desc from the tensors, creates the plan
once, keeps a workspace buffer (torch memory) sized for the largest T seen,
and calls moe_layer.  All arithmetic runs in the CUDA library.
"""
from __future__ import annotations

import torch

from . import _native as N

_QT = {"q8_0": N.MOE_Q8_0, "q4_k": N.MOE_Q4_K, "q8_0_r": N.MOE_Q8_0_R, "q5_k": N.MOE_Q5_K, "q6_k": N.MOE_Q6_K,
       "q3_k": N.MOE_Q3_K, "mxfp4": N.MOE_MXFP4}


def row_bytes(qtype: int, cols: int) -> int:
    if qtype == N.MOE_Q8_0_R:                     # quants, then fp16 scales padded to 16 bytes
        nb = cols // 32
        return 32 * nb + (2 * nb + 15) // 16 * 16
    if qtype == N.MOE_Q8_0:
        return cols // 32 * 34
    if qtype == N.MOE_MXFP4:
        return cols // 32 * 17
    return cols // 256 * {N.MOE_Q4_K: 144, N.MOE_Q5_K: 176, N.MOE_Q6_K: 210, N.MOE_Q3_K: 110}[qtype]


def prepare_q8_0(t, rows: int, cols: int, n_experts: int = 1):
    """A Q8_0 tensor (uint8, [n_experts, rows, rb] or [rows, rb] on the GPU) repacked by
    moe_weights_prepare into a new uint8 tensor of the MOE_Q8_0_R layout (qtype "q8_0_r")."""
    m = N.qmat(N.MOE_Q8_0, t, rows, cols, rows * row_bytes(N.MOE_Q8_0, cols))
    nbytes = N.moe_weights_prepare_size(m, n_experts)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=t.device)
    N.moe_weights_prepare(m, n_experts, dst, nbytes)
    shape = (n_experts, rows, row_bytes(N.MOE_Q8_0_R, cols)) if t.dim() == 3 else (rows, row_bytes(N.MOE_Q8_0_R, cols))
    return dst.view(*shape)


class MoeLayer:
    """gate/up: uint8 [E, I, rb(H)], down: uint8 [E, H, rb(I)] on the GPU (qtype, or
    qtype_down for down); shared expert matrices in shared_qtype."""

    def __init__(self, *, mode: str, E: int, k: int, H: int, I: int, qtype: str, gate, up, down, W_router,
                 bias=None, n_groups: int = 1, topk_groups: int = 1, scale: float = 1.0,
                 renormalize: bool = True, x_dtype: str = "bf16", I_s: int = 0, shared_qtype: str = "q8_0",
                 s_gate=None, s_up=None, s_down=None, accumulate: bool = False, tc_min_tokens: int = 0,
                 decode_chain: bool = True, norm_gamma=None, norm_eps: float = 1e-6, qtype_down: str | None = None,
                 expert_counts=None):
        self.E, self.k, self.H, self.I = E, k, H, I
        self.x_dtype = x_dtype
        qt = _QT[qtype]
        qd = _QT[qtype_down] if qtype_down else qt      # the down matrix may be stored in another type
        self._keep = [gate, up, down, W_router, bias, s_gate, s_up, s_down, norm_gamma, expert_counts]
        d = N.moe_layer_desc()
        d.route = N.route_cfg(N.MOE_ROUTE_SIGMOID_GROUP if mode == "sigmoid_group" else N.MOE_ROUTE_SOFTMAX,
                              E, k, n_groups, topk_groups, scale, renormalize)
        d.hidden, d.intermediate = H, I
        d.x_type = N.MOE_BF16 if x_dtype == "bf16" else N.MOE_F32
        d.W_router = W_router.data_ptr()
        d.bias = bias.data_ptr() if bias is not None else None
        d.gate = N.qmat(qt, gate, I, H, I * row_bytes(qt, H))
        d.up = N.qmat(qt, up, I, H, I * row_bytes(qt, H))
        d.down = N.qmat(qd, down, H, I, H * row_bytes(qd, I))
        d.shared_intermediate = I_s
        if I_s > 0:
            sq = _QT[shared_qtype]
            d.s_gate = N.qmat(sq, s_gate, I_s, H, 0)
            d.s_up = N.qmat(sq, s_up, I_s, H, 0)
            d.s_down = N.qmat(sq, s_down, H, I_s, 0)
        d.accumulate = int(accumulate)
        d.tc_min_tokens = tc_min_tokens
        d.decode_chain_off = 0 if decode_chain else 1
        if norm_gamma is not None:       # pre-norm: x is the fp32 residual stream
            d.norm_gamma = norm_gamma.data_ptr()
            d.norm_eps = norm_eps
        if expert_counts is not None:    # running routing histogram: int64 [E] on the device
            if expert_counts.dtype != torch.int64 or expert_counts.numel() != E or not expert_counts.is_cuda:
                raise ValueError("expert_counts must be an int64 CUDA tensor of E entries")
            d.expert_counts = expert_counts.data_ptr()
        self.desc = d
        self.plan = N.moe_layer_plan_create(d)
        self.ws = None
        self.ws_T = -1

    def path(self, T: int) -> str:
        """Which kernels a call with T tokens runs: "gemv", "decode_chain" or "tensor"."""
        return N.PATH_NAMES[N.moe_layer_path(self.plan, T)]

    def workspace_bytes(self, T: int) -> int:
        return N.moe_layer_workspace_size(self.plan, T)

    def ensure_workspace(self, T: int, device=None):
        if self.ws is None or T > self.ws_T:
            nbytes = self.workspace_bytes(T)
            self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
            self.ws_T = T
        return self.ws

    def __call__(self, x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.float32, device=x.device)
        ws = self.ensure_workspace(T, x.device)
        N.moe_layer(self.plan, x, T, out, ws, ws.numel(), stream)
        return out

    def debug_views(self, T: int):
        """(ids [T,k] int32, gates [T,k] fp32, offsets [E+1] int32) of the last call, copied to the host."""
        pi, pw, po = N.moe_layer_debug_views(self.plan, T, self.ws)
        base = self.ws.data_ptr()
        def view(ptr, n, dtype):
            off = ptr - base
            return self.ws[off:off + n * 4].view(dtype).clone().cpu()
        return (view(pi, T * self.k, torch.int32).view(T, self.k), view(pw, T * self.k, torch.float32).view(T, self.k),
                view(po, self.E + 1, torch.int32))

    def rebuild_plan(self):
        """Re-create the plan after editing self.desc."""
        N.moe_layer_plan_destroy(self.plan)
        self.plan = N.moe_layer_plan_create(self.desc)
        self.ws, self.ws_T = None, -1   # the workspace layout may have changed

    def device_status(self, T: int) -> int:
        return N.moe_read_device_status(self.plan, T, self.ws)

    def __del__(self):
        try:
            if getattr(self, "plan", None):
                N.moe_layer_plan_destroy(self.plan)
                self.plan = None
        except Exception:
            pass
