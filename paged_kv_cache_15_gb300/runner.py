"""Moves a seeded workload onto the GPU and drives it through the C ABI.

Marshalling only: device copies of the inputs, a context sized for the
workload, and the call sequence of one batch — set_kv_buffer (save_kv_cache),
metadata build, then the ForwardMode-dispatched forward.
"""
from __future__ import annotations

import torch

from . import binding as B
from .workloads import Workload

MODE_OF = {"decode": B.PKV_MODE_DECODE, "extend": B.PKV_MODE_EXTEND, "verify": B.PKV_MODE_TARGET_VERIFY}


def config_for(W: Workload, max_batch=None, max_pages_total=None, max_q_tokens=None, max_qo_len=None):
    G = W.num_q_heads // W.num_kv_heads
    pages = int(((W.seq_lens.astype("int64") + W.page_size - 1) // W.page_size).sum())
    if max_qo_len is None:
        max_qo_len = int(W.qo_lens.max()) if W.mode == "verify" else 1
        max_qo_len = max(1, min(max_qo_len, 128 // G))
    return B.make_config(W.num_q_heads, W.num_kv_heads, W.head_dim, W.page_size,
                         B.PKV_KV_FP8_E4M3 if W.is_fp8 else B.PKV_KV_BF16, W.num_pages,
                         max_batch or max(W.bs, 1), max_pages_total or max(pages, 1),
                         max_q_tokens or max(W.total_q, 1), max_qo_len, head_dim_v=W.head_dim_v)


class DeviceBatch:
    """Device-resident copy of a workload plus a context and output buffers."""

    def __init__(self, W: Workload, device="cuda", cfg=None):
        self.W = W
        dev = torch.device(device)
        self.cfg = cfg or config_for(W)
        self.attn = B.PagedAttention(self.cfg, dev)
        self.q = W.q.to(dev)
        self.k_pool = W.k_pool.to(dev)
        self.v_pool = W.v_pool.to(dev)
        self.k_new = W.k_new.to(dev)
        self.v_new = W.v_new.to(dev)
        self.loc = torch.from_numpy(W.loc).to(dev)
        self.seq_lens = torch.from_numpy(W.seq_lens).to(dev)
        self.qo_lens = None if W.mode == "decode" else torch.from_numpy(W.qo_lens).to(dev)
        self.page_table = torch.from_numpy(W.page_table).to(dev)
        # output rows have the V heads' width
        self.out = torch.empty((W.total_q, W.num_q_heads, W.dv), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((W.total_q, W.num_q_heads), dtype=torch.float32, device=dev)
        self.mode = MODE_OF[W.mode]
        # draft-tree mask words (uint64, carried as int64 bits)
        self.tree = None
        if W.tree_mask is not None:
            self.tree = torch.from_numpy(W.tree_mask.view("int64").copy()).to(dev)
            B.pkv_set_tree_mask(self.ctx, self.tree)
        # attention sinks (fp32 per query head)
        self.sinks = None
        if W.sinks is not None:
            self.sinks = torch.from_numpy(W.sinks.astype("float32")).to(dev)
            B.pkv_set_attention_sinks(self.ctx, self.sinks)

    @property
    def ctx(self):
        return self.attn.ctx

    def set_kv_buffer(self):
        W = self.W
        if W.loc.shape[0]:
            B.pkv_set_kv_buffer(self.ctx, self.k_pool, self.v_pool, self.loc, self.k_new, self.v_new,
                                W.k_inv_scale, W.v_inv_scale)

    def build_metadata(self, mode=None):
        B.pkv_build_metadata(self.ctx, self.mode if mode is None else mode, self.W.bs, self.seq_lens,
                             self.qo_lens, self.page_table)

    def forward(self, spec_mode=B.PKV_SPEC_PREFILL, mode=None, lse=True):
        W = self.W
        B.pkv_forward(self.ctx, self.mode if mode is None else mode, spec_mode, self.q, self.k_pool, self.v_pool,
                      W.sm_scale, self.out, self.lse if lse else None, W.k_scale, W.v_scale)

    def step(self, spec_mode=B.PKV_SPEC_PREFILL):
        self.set_kv_buffer()
        self.build_metadata()
        self.forward(spec_mode)

    def device_error(self) -> int:
        return B.pkv_get_device_error(self.ctx)
