"""Device storage of one attention layer's three-segment token pool.

Host-side plumbing only: it allocates the tensors that `oscar_layer_desc`
points at (page pool, page table, lengths, BF16 sink and recent ring,
rotations, device status word) and fills the descriptor.  All computation on
them happens in liboscar.so.
"""
from __future__ import annotations

import torch

from .binding import LayerDesc, oscar_block_bytes

HEAD_DIM = 128
PAGE_TOKENS = 16


class LayerCache:
    """BF16 sink | INT2 paged history | BF16 recent ring for `batch` requests."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, max_pages_per_seq: int,
                 n_pages: int, r_k: torch.Tensor, r_v: torch.Tensor, tau_k: float, tau_v: float,
                 device="cuda", sink_cap: int = 64, recent_cap: int = 256, quant_group_k: int = 128,
                 quant_group_v: int = 128, levels_k=None, levels_v=None):
        self.batch, self.n_q_heads, self.n_kv_heads = batch, n_q_heads, n_kv_heads
        self.quant_group_k, self.quant_group_v = int(quant_group_k), int(quant_group_v)
        self.block_bytes = oscar_block_bytes(self.quant_group_k, self.quant_group_v)
        if self.block_bytes <= 0:
            raise ValueError("quantisation group sizes must be 32, 64 or 128")
        # Lloyd-Max codebook levels (four fp16 values each) or None (uniform)
        self.levels_k = None if levels_k is None else [float(x) for x in levels_k]
        self.levels_v = None if levels_v is None else [float(x) for x in levels_v]
        if (self.levels_k is None) != (self.levels_v is None):
            raise ValueError("codebook levels for both K and V, or for neither")
        self.sink_cap, self.recent_cap = sink_cap, recent_cap
        self.max_pages_per_seq, self.n_pages = max_pages_per_seq, n_pages
        self.tau_k, self.tau_v = float(tau_k), float(tau_v)
        dev = torch.device(device)
        self.pages = torch.zeros(n_pages * n_kv_heads * self.block_bytes, dtype=torch.uint8, device=dev)
        self.page_table = torch.full((batch, max_pages_per_seq), -1, dtype=torch.int32, device=dev)
        self.hist_len = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.sink_len = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.recent_len = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.recent_start = torch.zeros(batch, dtype=torch.int32, device=dev)
        shape_s = (batch, max(sink_cap, 1), n_kv_heads, HEAD_DIM)
        shape_r = (batch, max(recent_cap, 1), n_kv_heads, HEAD_DIM)
        self.sink_k = torch.zeros(shape_s, dtype=torch.bfloat16, device=dev)
        self.sink_v = torch.zeros(shape_s, dtype=torch.bfloat16, device=dev)
        self.recent_k = torch.zeros(shape_r, dtype=torch.bfloat16, device=dev)
        self.recent_v = torch.zeros(shape_r, dtype=torch.bfloat16, device=dev)
        self.r_k = r_k.to(device=dev, dtype=torch.float32).contiguous()
        self.r_v = r_v.to(device=dev, dtype=torch.float32).contiguous()
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_hist = 0

    def desc(self, max_hist: int = None) -> LayerDesc:
        d = LayerDesc()
        d.batch, d.n_q_heads, d.n_kv_heads, d.head_dim = (self.batch, self.n_q_heads,
                                                          self.n_kv_heads, HEAD_DIM)
        d.sink_cap, d.recent_cap = self.sink_cap, self.recent_cap
        d.max_pages_per_seq = self.max_pages_per_seq
        d.max_hist = self.max_hist if max_hist is None else int(max_hist)
        d.n_pages = self.n_pages
        d.tau_k, d.tau_v = self.tau_k, self.tau_v
        d.quant_group_k, d.quant_group_v = self.quant_group_k, self.quant_group_v
        if self.levels_k is not None:
            d.codebook = 1
            for i in range(4):
                d.levels_k[i], d.levels_v[i] = self.levels_k[i], self.levels_v[i]
        for name in ("pages", "page_table", "hist_len", "sink_k", "sink_v", "sink_len", "recent_k",
                     "recent_v", "recent_len", "recent_start", "r_k", "r_v", "dev_status"):
            setattr(d, name, getattr(self, name).data_ptr())
        return d
