"""Seeded synthetic inputs for paged-KV attention.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic, and both the CUDA path and the CPU oracle read the
same arrays it returns. Every array is a CPU tensor.

Shapes follow the serving cases of "--attention-backend" (SGLang manual,
sections "What an attention backend is" and "What we measured on an L4"):
a paged pool of token slots, ``slot = page * page_size + offset``, laid out
``[slot, kv_head, head_dim]`` with separate K and V pools, and per-batch page
tables. The five named presets are the model-shaped cases that stand in for
the pages' live-serving workloads (no dataset or trained weights are used).

Recipe (seeds are ``torch.Generator`` seeds):
  * seed 0: request lengths (``torch.randint`` with inclusive bounds), then one
    ``torch.randperm`` of the pool pages 1..num_pages-1 whose first pages are
    handed to the requests in order. Page 0 is a sentinel page never handed
    out; unused page-table entries point at it.
  * seed 1: queries, N(0, 1) in fp32 rounded to bf16, ``[T, Hq, D]``.
  * seed 2 / 3: K / V of the cached prefix tokens, N(0, 1) (bf16, or fp8 E4M3
    via torch's float8_e4m3fn cast after dividing by ``max|x| / 448``).
  * seed 4: K then V of the step's new tokens, N(0, 1) bf16, ``[n_new, Hkv, D]``;
    they enter the pool only through ``set_kv_buffer`` at slots ``loc``.
  * K and V heads may differ in width (``head_dim`` for Q and K, ``head_dim_v``
    for V and the output); the draws are the same with each pool's own width.
    The score scale is ``1 / sqrt(head_dim)``.
  * every slot that holds no prefix token (tails of last pages, pages no
    request owns, slots of new tokens before the scatter, the sentinel page)
    is filled with NaN (bf16 0x7FC0, E4M3 0x7F), so a read of an unused slot
    shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    mode: str  # "decode" | "extend" | "verify"
    bs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str  # "bf16" | "fp8_e4m3"
    num_pages: int
    prefix_lens: np.ndarray  # int32 [bs]  tokens already in the pool
    qo_lens: np.ndarray  # int32 [bs]      new tokens (query rows) per request
    seq_lens: np.ndarray  # int32 [bs]     prefix + new
    page_table: np.ndarray  # int32 [bs, max_pages]
    loc: np.ndarray  # int32 [n_new]       slots of the new tokens
    q: torch.Tensor  # bf16 [T, Hq, D]
    k_pool: torch.Tensor  # bf16 or uint8 (E4M3 bits) [slots, Hkv, D]
    v_pool: torch.Tensor
    k_new: torch.Tensor  # bf16 [n_new, Hkv, D]
    v_new: torch.Tensor
    k_scale: float = 1.0
    v_scale: float = 1.0
    sm_scale: float = 1.0
    extra: dict = field(default_factory=dict)
    # draft-tree visibility (verify batches): None for chain drafts, else
    # uint64 [T], bit j of token t's word = it sees the j-th new token of its
    # request (every cached key stays visible)
    tree_mask: Optional[np.ndarray] = None
    # attention sinks: None, or fp32 [Hq], each query head's sink logit
    sinks: Optional[np.ndarray] = None
    # width of the V heads (and of the output rows); 0 means head_dim
    head_dim_v: int = 0

    @property
    def dv(self) -> int:
        return self.head_dim_v or self.head_dim

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size

    @property
    def total_q(self) -> int:
        return int(self.qo_lens.sum())

    @property
    def k_inv_scale(self) -> float:
        return float(np.float32(1.0) / np.float32(self.k_scale))

    @property
    def v_inv_scale(self) -> float:
        return float(np.float32(1.0) / np.float32(self.v_scale))

    @property
    def is_fp8(self) -> bool:
        return self.kv_dtype == "fp8_e4m3"


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 array of its bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def pool_bits(t: torch.Tensor) -> np.ndarray:
    """Pool tensor -> numpy bit array (uint16 for bf16, uint8 for E4M3)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.contiguous().numpy()


def _randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def random_tree_masks(qo_lens, seed: int = 5) -> np.ndarray:
    """Visibility words of random draft trees, one per query token.

    In each request draft 0 hangs off the cached prefix and draft j > 0 off a
    uniformly drawn earlier draft or, with probability 1/(j+1), off the prefix
    as well; every draft sees itself and its ancestors.
    """
    rng = np.random.default_rng(seed)
    words = []
    for n in np.asarray(qo_lens, dtype=np.int64):
        if n > 64:
            raise ValueError("a draft tree holds at most 64 tokens")
        mask = []
        for j in range(int(n)):
            parent = int(rng.integers(-1, j)) if j > 0 else -1
            mask.append((1 << j) | (mask[parent] if parent >= 0 else 0))
        words.extend(mask)
    return np.array(words, dtype=np.uint64)


def random_sinks(num_q_heads: int, seed: int = 6, lo: float = -2.0, hi: float = 4.0) -> np.ndarray:
    """Per-head sink logits drawn uniformly from [lo, hi) (the scores of
    N(0, 1) inputs scaled by 1/sqrt(D) sit around 0), stored as fp32."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, num_q_heads).astype(np.float32)


def chain_tree_masks(qo_lens) -> np.ndarray:
    """The visibility words of chain drafts: token i sees new tokens 0..i."""
    return np.array([(1 << (i + 1)) - 1 for n in np.asarray(qo_lens, dtype=np.int64) for i in range(int(n))],
                    dtype=np.uint64)


def make_workload(name: str, mode: str, bs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  prefix_lens, qo_lens, page_size: int = 16, kv_dtype: str = "bf16",
                  num_pages: Optional[int] = None, pool_slack: float = 0.10,
                  head_dim_v: Optional[int] = None) -> Workload:
    """Build a workload from explicit per-request prefix and new-token counts.
    ``head_dim_v`` is the width of the V heads (default: ``head_dim``)."""
    prefix = np.asarray(prefix_lens, dtype=np.int64).reshape(bs)
    qo = np.asarray(qo_lens, dtype=np.int64).reshape(bs)
    seq = prefix + qo
    pages_needed = (seq + page_size - 1) // page_size
    total_pages = int(pages_needed.sum())
    if num_pages is None:
        # total tokens plus the slack, never fewer than the pages the requests own,
        # plus the sentinel page
        num_pages = max(int(math.ceil((1.0 + pool_slack) * int(seq.sum()) / page_size)), total_pages) + 1
    if num_pages < total_pages + 1:
        raise ValueError("pool too small")
    g0 = torch.Generator().manual_seed(0)
    # lengths were drawn by the caller with the same generator seed; the page
    # permutation continues from a fresh seed-0 stream so explicit lengths and
    # drawn lengths give the same page layout
    perm = torch.randperm(num_pages - 1, generator=g0).numpy().astype(np.int64) + 1
    max_pages = max(int(pages_needed.max()) if bs else 1, 1)
    page_table = np.zeros((bs, max_pages), dtype=np.int32)
    off = 0
    for b in range(bs):
        n = int(pages_needed[b])
        page_table[b, :n] = perm[off:off + n]
        off += n
    num_slots = num_pages * page_size
    # slot of every (request, position)
    def slots_of(b, lo, hi):
        pos = np.arange(lo, hi, dtype=np.int64)
        return page_table[b, pos // page_size].astype(np.int64) * page_size + pos % page_size

    prefix_slots = np.concatenate([slots_of(b, 0, int(prefix[b])) for b in range(bs)] + [np.zeros(0, np.int64)])
    loc = np.concatenate([slots_of(b, int(prefix[b]), int(seq[b])) for b in range(bs)] + [np.zeros(0, np.int64)])
    T = int(qo.sum())
    n_prefix = prefix_slots.shape[0]

    g1 = torch.Generator().manual_seed(1)
    q = _randn_bf16(g1, (T, num_q_heads, head_dim))

    fp8 = kv_dtype == "fp8_e4m3"
    if kv_dtype not in ("bf16", "fp8_e4m3"):
        raise ValueError(kv_dtype)
    pools = []
    scales = []
    idx = torch.from_numpy(prefix_slots)
    dv = head_dim if head_dim_v is None else int(head_dim_v)
    for seed, width in ((2, head_dim), (3, dv)):
        g = torch.Generator().manual_seed(seed)
        data = torch.randn((n_prefix, num_kv_heads, width), generator=g, dtype=torch.float32)
        if fp8:
            amax = float(data.abs().max()) if n_prefix else 1.0
            scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
            pool = torch.full((num_slots, num_kv_heads, width), E4M3_NAN, dtype=torch.uint8)
            codes = (data / scale).to(torch.float8_e4m3fn).view(torch.uint8)
            pool[idx] = codes
        else:
            scale = 1.0
            pool = torch.full((num_slots, num_kv_heads, width), BF16_NAN, dtype=torch.int16)
            pool = pool.view(torch.bfloat16)
            pool[idx] = data.to(torch.bfloat16)
        del data
        pools.append(pool)
        scales.append(scale)

    g4 = torch.Generator().manual_seed(4)
    n_new = loc.shape[0]
    k_new = _randn_bf16(g4, (n_new, num_kv_heads, head_dim))
    v_new = _randn_bf16(g4, (n_new, num_kv_heads, dv))

    return Workload(name=name, mode=mode, bs=bs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, page_size=page_size, kv_dtype=kv_dtype, num_pages=num_pages,
                    prefix_lens=prefix.astype(np.int32), qo_lens=qo.astype(np.int32), seq_lens=seq.astype(np.int32),
                    page_table=page_table, loc=loc.astype(np.int32), q=q, k_pool=pools[0], v_pool=pools[1],
                    k_new=k_new, v_new=v_new, k_scale=scales[0], v_scale=scales[1],
                    sm_scale=1.0 / math.sqrt(head_dim), head_dim_v=0 if dv == head_dim else dv)


def _randint(gen, lo, hi, n):
    """n integers uniform in [lo, hi] (inclusive bounds)."""
    return torch.randint(lo, hi + 1, (n,), generator=gen).numpy().astype(np.int64)


# --------------------------------------------------------------------------
# Named presets (the five model-shaped cases) and scaled-down variants.
# --------------------------------------------------------------------------

PRESETS = ("tiny_decode", "llama3_8b_decode", "prefix_extend", "spec_verify", "long_fp8_decode")
# E4M3 pools on the prefix-cached extend case: the same lengths and values,
# with the cached prefix quantised on the host and the new tokens quantised by
# set_kv_buffer
VARIANTS = ("prefix_extend_fp8",)


def preset(name: str, bs: Optional[int] = None, len_scale: float = 1.0, page_size: int = 16,
           kv_dtype: Optional[str] = None, head_dims: Optional[tuple] = None) -> Workload:
    """The five cases at full size (defaults), or with fewer requests / shorter
    lengths (``len_scale`` multiplies every length bound) for quick parity runs.
    ``page_size`` and ``kv_dtype`` override the case's page size (16) and pool
    element type; ``head_dims = (head_dim, head_dim_v)`` the widths of the Q/K
    and V heads (192/128 is the shape of models whose K and V heads differ);
    the lengths, pages and values are drawn the same way."""
    g = torch.Generator().manual_seed(0)
    ps = page_size
    dk_over, dv_over = head_dims if head_dims is not None else (None, None)

    def make(nm, mode, n, hq, hkv, d, P, N, **kw):
        return make_workload(nm, mode, n, hq, hkv, dk_over or d, P, N, head_dim_v=dv_over, **kw)

    def kvd(default):
        return kv_dtype if kv_dtype is not None else default

    def lens(lo, hi, n):
        lo2 = max(1, int(round(lo * len_scale)))
        hi2 = max(lo2, int(round(hi * len_scale)))
        return _randint(g, lo2, hi2, n)

    if name == "tiny_decode":
        # batch 4, 8/2 heads, head_dim 64, contexts 37/100/211/300, 128-page pool
        L = np.array([37, 100, 211, 300], dtype=np.int64)
        if bs is not None:
            L = L[:bs]
        n = L.shape[0]
        # a 128-page pool of 16-token pages (2,048 slots), the same slots at other page sizes
        return make(name, "decode", n, 8, 2, 64, L - 1, np.ones(n), page_size=ps,
                    num_pages=max(128 * 16 // ps, 1 + int(((L + ps - 1) // ps).sum())), kv_dtype=kvd("bf16"))
    if name == "llama3_8b_decode":
        n = 64 if bs is None else bs
        L = lens(1024, 8192, n)
        return make(name, "decode", n, 32, 8, 128, L - 1, np.ones(n), page_size=ps, kv_dtype=kvd("bf16"))
    if name in ("prefix_extend", "prefix_extend_fp8"):
        n = 8 if bs is None else bs
        P = _randint(g, 0, int(round(4096 * len_scale)), n)
        N = lens(128, 2048, n)
        dt = kvd("fp8_e4m3" if name == "prefix_extend_fp8" else "bf16")
        return make(name, "extend", n, 32, 8, 128, P, N, page_size=ps, kv_dtype=dt)
    if name == "spec_verify":
        n = 32 if bs is None else bs
        ctx = lens(2048, 16384, n)
        N = _randint(g, 4, 8, n)
        return make(name, "verify", n, 64, 4, 128, ctx, N, page_size=ps, kv_dtype=kvd("bf16"))
    if name == "long_fp8_decode":
        n = 8 if bs is None else bs
        L = lens(32768, 131072, n)
        return make(name, "decode", n, 32, 8, 128, L - 1, np.ones(n), page_size=ps, kv_dtype=kvd("fp8_e4m3"))
    raise KeyError(name)
