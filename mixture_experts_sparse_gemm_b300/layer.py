"""Buffer management around the C ABI: one object per layer shape that owns the
packed expert weights and the workspace, and calls the library's entry points.

Only allocation (torch device memory) and argument marshalling happen here; every
step of the layer runs in libmoe_b300.so.
"""
from __future__ import annotations

import torch

from . import binding as B


class MoELayer:
    """A sparsely-gated MoE SwiGLU FFN layer of fixed shape ``cfg`` on one GPU.

    W1, W3: [E, d, f], W2: [E, f, d]; optional shared experts W1s, W3s: [S, d, fs],
    W2s: [S, fs, d]; all in the run dtype on the device.  The weights are packed
    once here (``moe_pack_weights``); the forward never re-lays them out.
    """

    def __init__(self, cfg: B.moe_config, W1, W3, W2, W1s=None, W3s=None, W2s=None, stream=None):
        self.cfg = cfg
        self.device = W1.device
        self.dtype = torch.float32 if cfg.dtype == B.MOE_F32 else torch.bfloat16
        self.rows_routed, self.rows_total = B.moe_buffer_rows(cfg)
        self.packed = torch.empty(B.moe_packed_weights_size(cfg), dtype=torch.uint8, device=self.device)
        B.moe_pack_weights(cfg, W1, W3, W2, W1s, W3s, W2s, self.packed, stream)
        self._ws = {}

    # ------------------------------------------------------------------ buffers
    def workspace(self, stage=B.MOE_STAGE_FORWARD):
        if stage not in self._ws:
            n = B.moe_workspace_size(self.cfg, stage)
            self._ws[stage] = torch.empty(max(n, 1), dtype=torch.uint8, device=self.device) if n > 0 else None
        return self._ws[stage]

    def n_select(self):
        c = self.cfg
        return (c.E, c.ec_capacity) if c.mode == B.MOE_EXPERT_CHOICE else (c.T, c.k)

    def n_slots(self):
        c = self.cfg
        return (c.T, c.E) if c.mode == B.MOE_EXPERT_CHOICE else (c.T, c.k)

    # ------------------------------------------------------------------ stages
    def route(self, x, W_r, logit_offset=None, sel_bias=None, stream=None, prob_sum=None):
        idx = torch.empty(self.n_select(), dtype=torch.int32, device=self.device)
        w = torch.empty(self.n_select(), dtype=torch.float32, device=self.device)
        B.moe_route(self.cfg, x, W_r, logit_offset, sel_bias, idx, w, self.workspace(B.MOE_STAGE_ROUTE), stream,
                    prob_sum)
        return idx, w

    def load_stats(self, topk_idx, cnt_raw, prob_sum, stream=None):
        """(token_fraction [E], prob_mean [E], summary [5] float64: LIF, CV, router
        entropy, Switch balance E*sum f1*P, expert balance E*sum f*P)."""
        E = self.cfg.E
        frac = torch.empty(E, dtype=torch.float32, device=self.device)
        pmean = torch.empty(E, dtype=torch.float32, device=self.device)
        summary = torch.empty(5, dtype=torch.float64, device=self.device)
        B.moe_load_stats(self.cfg, topk_idx, cnt_raw, prob_sum, frac, pmean, summary, stream)
        return frac, pmean, summary

    def dispatch(self, idx, x, stream=None, topk_w=None):
        c = self.cfg
        off = torch.empty(c.E + 1, dtype=torch.int32, device=self.device)
        cnt_raw = torch.empty(c.E, dtype=torch.int32, device=self.device)
        slot_of = torch.empty(self.n_slots(), dtype=torch.int32, device=self.device)
        x_perm = torch.empty(max(self.rows_routed, 1), c.d, dtype=self.dtype, device=self.device)
        B.moe_dispatch(c, idx, x, off, cnt_raw, slot_of, x_perm, self.workspace(B.MOE_STAGE_DISPATCH), stream, topk_w)
        return off, cnt_raw, slot_of, x_perm

    def grouped_ffn(self, x_perm, off, x=None, stream=None):
        Y = torch.empty(max(self.rows_total, 1), self.cfg.d, dtype=self.dtype, device=self.device)
        B.moe_grouped_ffn(self.cfg, x_perm, off, self.packed, x, Y, self.workspace(B.MOE_STAGE_GROUPED_FFN), stream)
        return Y

    def combine(self, Y, slot_of, w, stream=None):
        y = torch.empty(self.cfg.T, self.cfg.d, dtype=self.dtype, device=self.device)
        B.moe_combine(self.cfg, Y, slot_of, w, y, None, stream)
        return y

    def forward(self, x, W_r, logit_offset=None, sel_bias=None, out=None, stream=None):
        y = out if out is not None else torch.empty(self.cfg.T, self.cfg.d, dtype=self.dtype, device=self.device)
        B.moe_forward(self.cfg, x, W_r, logit_offset, sel_bias, self.packed, y, self.workspace(), stream)
        return y
