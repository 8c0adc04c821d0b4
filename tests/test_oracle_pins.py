"""Pins of the fp64 oracle against facts fixed outside it.

Each test ties one oracle function to something other than the oracle itself:
values the source pages print (golden fixtures), closed forms, invariants,
brute force on tiny inputs, and library routines (torch's E4M3 cast, torch
scaled-dot-product attention in fp64).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_15_gb300.workloads import (Workload, bf16_bits, chain_tree_masks, make_workload, pool_bits,
                                               preset, random_sinks, random_tree_masks)
from tests._pipeline import oracle_meta, oracle_pools, oracle_reference

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append(vals)
    return out


def _tiny(mode="extend", kv_dtype="bf16", page_size=4, seed_shift=0, hq=4, hkv=2, d=8, dv=None):
    rng = np.random.default_rng(7 + seed_shift)
    bs = 3
    if mode == "decode":
        prefix = rng.integers(0, 39, bs)
        qo = np.ones(bs, np.int64)
    else:
        prefix = rng.integers(0, 30, bs)
        qo = rng.integers(1, 10, bs)
    return make_workload("tiny", mode, bs, hq, hkv, d, prefix, qo, page_size=page_size, kv_dtype=kv_dtype,
                         head_dim_v=dv)


def _contiguous_kv(W: Workload):
    """Per request, the logical K and V rows 0..L-1 in fp64, read straight from
    the page table (prefix from the pool, new tokens from k_new/v_new)."""
    kp = pool_bits(W.k_pool)
    vp = pool_bits(W.v_pool)
    kn = bf16_bits(W.k_new)
    vn = bf16_bits(W.v_new)
    dec_pool = (lambda a: oracle.e4m3_decode_array(a)) if W.is_fp8 else \
        (lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    dec_new = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = []
    new_off = 0
    for b in range(W.bs):
        P, L = int(W.prefix_lens[b]), int(W.seq_lens[b])
        ks, vs = [], []
        for p in range(L):
            if p < P:
                slot = int(W.page_table[b, p // W.page_size]) * W.page_size + p % W.page_size
                ks.append(dec_pool(kp[slot]) * W.k_scale)
                vs.append(dec_pool(vp[slot]) * W.v_scale)
            else:
                i = new_off + (p - P)
                if W.is_fp8:
                    # the new token enters an E4M3 pool through set_kv_buffer's rounding
                    kq = (W.k_new[i].float() * W.k_inv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    vq = (W.v_new[i].float() * W.v_inv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    ks.append(dec_pool(kq) * W.k_scale)
                    vs.append(dec_pool(vq) * W.v_scale)
                else:
                    ks.append(dec_new(kn[i]))
                    vs.append(dec_new(vn[i]))
        new_off += L - P
        out.append((np.array(ks).reshape(L, W.num_kv_heads, W.head_dim),
                    np.array(vs).reshape(L, W.num_kv_heads, W.dv)))
    return out


def _q64(W):
    return W.q.double().numpy()


# ---------------------------------------------------------------- P1 brute force
@pytest.mark.parametrize("mode", ["decode", "extend"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("dv", [None, 5, 12])
def test_p1_bruteforce_unpaged_loops(mode, kv_dtype, dv):
    """dv: V heads of another width than the Q/K heads (P15; the scores
    contract head_dim columns, the output has dv)."""
    W = _tiny(mode, kv_dtype, dv=dv)
    o, lse = oracle_reference(W)
    q = _q64(W)
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    kv = _contiguous_kv(W)
    worst = 0.0
    for b in range(W.bs):
        K, V = kv[b]
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        for i in range(N):
            t = qo_indptr[b] + i
            for h in range(W.num_q_heads):
                g = h // G
                vis = L - N + i + 1
                s = [W.sm_scale * sum(q[t, h, d] * K[j, g, d] for d in range(W.head_dim)) for j in range(vis)]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                ref_o = [sum(e[j] * V[j, g, d] for j in range(vis)) / z for d in range(W.dv)]
                ref_lse = m + math.log(z)
                worst = max(worst, max(abs(a - r) for a, r in zip(o[t, h], ref_o)), abs(lse[t, h] - ref_lse))
    assert o.shape[-1] == W.dv
    assert worst < 1e-12


@pytest.mark.parametrize("mode", ["decode", "extend"])
@pytest.mark.parametrize("dv", [None, 6])
def test_p1_bruteforce_torch_sdpa_fp64(mode, dv):
    """dv: V heads narrower than the Q/K heads (P15); torch's SDPA takes a
    value width of its own."""
    W = _tiny(mode, "bf16", seed_shift=3, hq=6, hkv=2, d=10 if dv else 8, dv=dv)
    o, lse = oracle_reference(W)
    q = torch.from_numpy(_q64(W))
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        qb = q[qo_indptr[b]:qo_indptr[b + 1]].transpose(0, 1)  # [Hq, N, D]
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, dim=0)  # [Hq, L, D]
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, dim=0)
        # bottom-right alignment: row i sees keys 0 .. L - N + i
        mask = torch.arange(L)[None, :] <= (L - N + torch.arange(N))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kt, Vt, attn_mask=mask, scale=W.sm_scale)
        got = torch.from_numpy(o[qo_indptr[b]:qo_indptr[b + 1]]).transpose(0, 1)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)
        scores = (qb @ Kt.transpose(1, 2)) * W.sm_scale
        ref_lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)  # [Hq, N]
        assert torch.allclose(torch.from_numpy(lse[qo_indptr[b]:qo_indptr[b + 1]]).T, ref_lse, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- P13 draft-tree masks
def _tree_case(seed_shift=0, hq=4, hkv=2):
    W = _tiny("extend", "bf16", seed_shift=seed_shift, hq=hq, hkv=hkv)
    W.tree_mask = random_tree_masks(W.qo_lens, seed=11 + seed_shift)
    return W


def _tree_visible(W, b, i, t):
    """Key positions row i of request b may see: the cached prefix, and the
    drafts up to its own index whose bit is set in its word."""
    P = int(W.prefix_lens[b])
    word = int(W.tree_mask[t])
    return list(range(P)) + [P + j for j in range(i + 1) if (word >> j) & 1]


def test_p13_tree_mask_bruteforce_loops():
    W = _tree_case()
    o, lse = oracle_reference(W)
    q = _q64(W)
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    kv = _contiguous_kv(W)
    worst = 0.0
    seen_branch = False
    for b in range(W.bs):
        K, V = kv[b]
        for i in range(int(W.qo_lens[b])):
            t = qo_indptr[b] + i
            vis = _tree_visible(W, b, i, t)
            seen_branch |= int(W.tree_mask[t]) != (1 << (i + 1)) - 1
            for h in range(W.num_q_heads):
                g = h // G
                s_ = [W.sm_scale * sum(q[t, h, d] * K[p, g, d] for d in range(W.head_dim)) for p in vis]
                m = max(s_)
                e = [math.exp(x - m) for x in s_]
                z = sum(e)
                ref_o = [sum(e[k] * V[p, g, d] for k, p in enumerate(vis)) / z for d in range(W.head_dim)]
                worst = max(worst, max(abs(a - r) for a, r in zip(o[t, h], ref_o)), abs(lse[t, h] - (m + math.log(z))))
    assert seen_branch  # the drawn trees are not all chains
    assert worst < 1e-12


def test_p13_tree_mask_torch_sdpa_fp64():
    W = _tree_case(seed_shift=2, hq=6, hkv=2)
    o, lse = oracle_reference(W)
    q = torch.from_numpy(_q64(W))
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        mask = torch.zeros((N, L), dtype=torch.bool)
        for i in range(N):
            mask[i, _tree_visible(W, b, i, qo_indptr[b] + i)] = True
        qb = q[qo_indptr[b]:qo_indptr[b + 1]].transpose(0, 1)
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, dim=0)
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kt, Vt, attn_mask=mask, scale=W.sm_scale)
        got = torch.from_numpy(o[qo_indptr[b]:qo_indptr[b + 1]]).transpose(0, 1)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)
        scores = (qb @ Kt.transpose(1, 2)) * W.sm_scale
        ref_lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
        assert torch.allclose(torch.from_numpy(lse[qo_indptr[b]:qo_indptr[b + 1]]).T, ref_lse, atol=1e-12, rtol=0)


def test_p13_chain_shaped_tree_equals_causal():
    W = _tiny("extend", "bf16", seed_shift=5)
    o0, l0 = oracle_reference(W)
    W.tree_mask = chain_tree_masks(W.qo_lens)
    o1, l1 = oracle_reference(W)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_p13_bits_above_own_index_ignored():
    """Drafts are ordered parents first, so a row never sees a later draft:
    an all-ones mask is the causal (chain) result."""
    W = _tiny("extend", "bf16", seed_shift=6)
    o0, l0 = oracle_reference(W)
    W.tree_mask = np.full(W.total_q, np.uint64(0xFFFFFFFFFFFFFFFF))
    o1, l1 = oracle_reference(W)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_p13_tree_of_more_than_64_drafts_rejected():
    W = make_workload("t65", "verify", 1, 2, 1, 8, [3], [65], page_size=4)
    W.tree_mask = np.full(65, np.uint64(1))
    with pytest.raises(ValueError):
        oracle_reference(W)
    with pytest.raises(ValueError):
        random_tree_masks([65])


# ---------------------------------------------------------------- P14 attention sinks
def test_p14_minus_inf_sinks_change_nothing():
    W = _tiny("extend", "bf16", seed_shift=8)
    o0, l0 = oracle_reference(W)
    W.sinks = np.full(W.num_q_heads, -np.inf, dtype=np.float32)
    o1, l1 = oracle_reference(W)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


@pytest.mark.parametrize("mode", ["decode", "extend"])
def test_p14_sinks_torch_sdpa_fp64(mode):
    """The sink as one more key: zero key and value rows appended, and an
    additive mask that gives that key head h's sink logit as its score."""
    W = _tiny(mode, "bf16", seed_shift=9, hq=6, hkv=2)
    W.sinks = random_sinks(W.num_q_heads, seed=3)
    o, lse = oracle_reference(W)
    q = torch.from_numpy(_q64(W))
    G = W.num_q_heads // W.num_kv_heads
    sink = torch.from_numpy(W.sinks.astype(np.float64))
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        qb = q[qo_indptr[b]:qo_indptr[b + 1]].transpose(0, 1)  # [Hq, N, D]
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, dim=0)
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, dim=0)
        Kt = torch.cat([Kt, torch.zeros(W.num_q_heads, 1, W.head_dim, dtype=Kt.dtype)], dim=1)
        Vt = torch.cat([Vt, torch.zeros(W.num_q_heads, 1, W.head_dim, dtype=Vt.dtype)], dim=1)
        vis = torch.arange(L)[None, :] <= (L - N + torch.arange(N))[:, None]  # [N, L]
        add = torch.zeros(W.num_q_heads, N, L + 1, dtype=torch.float64)
        add[:, :, :L] = torch.where(vis, 0.0, -math.inf)[None]
        add[:, :, L] = sink[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, Kt, Vt, attn_mask=add, scale=W.sm_scale)
        got = torch.from_numpy(o[qo_indptr[b]:qo_indptr[b + 1]]).transpose(0, 1)
        assert torch.allclose(got, ref, atol=1e-12, rtol=0)
        scores = (qb @ Kt.transpose(1, 2)) * W.sm_scale + add
        ref_lse = torch.logsumexp(scores, dim=-1)
        assert torch.allclose(torch.from_numpy(lse[qo_indptr[b]:qo_indptr[b + 1]]).T, ref_lse, atol=1e-12, rtol=0)


def test_p14_sinks_uniform_scores_closed_form():
    """q = 0: every visible score is 0, so o = (sum of v_j) / (n + e^sink) and
    lse = ln(n + e^sink) with n the visible keys."""
    W = _tiny("extend", "bf16", seed_shift=10)
    W.q = torch.zeros_like(W.q)
    W.sinks = random_sinks(W.num_q_heads, seed=4)
    o, lse = oracle_reference(W)
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        for i in range(N):
            n = L - N + i + 1
            for h in range(W.num_q_heads):
                e = math.exp(float(W.sinks[h]))
                ref = V[:n, h // G].sum(axis=0) / (n + e)
                assert np.allclose(o[qo_indptr[b] + i, h], ref, atol=1e-13, rtol=0)
                assert abs(lse[qo_indptr[b] + i, h] - math.log(n + e)) < 1e-13


def test_p14_sinks_empty_request():
    W = make_workload("sk0", "decode", 2, 4, 2, 8, [0, 5], [1, 1], page_size=4)
    W.seq_lens = np.array([0, 6], dtype=W.seq_lens.dtype)
    W.sinks = random_sinks(4, seed=5)
    o, lse = oracle_reference(W)
    assert np.all(o[0] == 0.0) and np.allclose(lse[0], W.sinks.astype(np.float64), rtol=0, atol=0)


# ---------------------------------------------------------------- P15 K and V heads of different widths
def _pad_k_columns(W: Workload, extra: int) -> Workload:
    """The same workload with `extra` zero columns appended to every Q and K
    head (K pool and new K), V untouched: each score gains only 0 * 0 terms."""
    import copy
    W2 = copy.copy(W)
    pad = lambda t: torch.cat([t, torch.zeros(*t.shape[:-1], extra, dtype=t.dtype)], dim=-1)
    W2.q = pad(W.q)
    W2.k_pool = pad(W.k_pool)
    W2.k_new = pad(W.k_new)
    W2.head_dim = W.head_dim + extra
    W2.head_dim_v = W.dv
    return W2


@pytest.mark.parametrize("mode", ["decode", "extend"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_p15_zero_k_columns_reproduce_equal_widths(mode, kv_dtype):
    """Widening Q and K with zero columns (8 -> 12 while V stays 8) leaves
    every score, hence every output and LSE, bit-identical; the score scale is
    kept, as it is an input."""
    W = _tiny(mode, kv_dtype, seed_shift=12)
    o0, l0 = oracle_reference(W)
    W2 = _pad_k_columns(W, 4)
    assert W2.head_dim == 12 and W2.dv == 8
    o1, l1 = oracle_reference(W2)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_p15_uniform_scores_mean_of_the_narrower_v():
    """q = 0 with K 12 wide and V 5 wide: o is the mean of the visible V rows
    (5 columns) and lse = ln(n)."""
    W = _tiny("extend", "bf16", seed_shift=13, d=12, dv=5)
    W.q = torch.zeros_like(W.q)
    o, lse = oracle_reference(W)
    assert o.shape == (W.total_q, W.num_q_heads, 5)
    G = W.num_q_heads // W.num_kv_heads
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        for i in range(N):
            n = L - N + i + 1
            for h in range(W.num_q_heads):
                assert np.allclose(o[qo_indptr[b] + i, h], V[:n, h // G].mean(axis=0), atol=1e-13, rtol=0)
                assert abs(lse[qo_indptr[b] + i, h] - math.log(n)) < 1e-13


def test_p15_set_kv_buffer_each_pool_its_own_width():
    """K rows land in the 12-wide K pool and V rows in the 5-wide V pool, bit
    for bit, and nothing else of either pool changes."""
    W = _tiny("extend", "bf16", seed_shift=14, d=12, dv=5)
    kp, vp = oracle_pools(W)
    k0, v0 = pool_bits(W.k_pool), pool_bits(W.v_pool)
    kn, vn = bf16_bits(W.k_new), bf16_bits(W.v_new)
    assert kp.shape[-1] == 12 and vp.shape[-1] == 5
    assert np.array_equal(kp[W.loc], kn) and np.array_equal(vp[W.loc], vn)
    rest = np.setdiff1d(np.arange(kp.shape[0]), W.loc)
    assert np.array_equal(kp[rest], k0[rest]) and np.array_equal(vp[rest], v0[rest])


# ---------------------------------------------------------------- P2 / P3 layout invariance
def _relayout(W: Workload, page_map, new_page_size=None):
    """Same logical content, different physical pages (page_map[p] = new page of p)."""
    ps = W.page_size
    kp, vp = pool_bits(W.k_pool), pool_bits(W.v_pool)
    if new_page_size is None:
        nk = np.empty_like(kp)
        nv = np.empty_like(vp)
        for p in range(W.num_pages):
            nk[page_map[p] * ps:(page_map[p] + 1) * ps] = kp[p * ps:(p + 1) * ps]
            nv[page_map[p] * ps:(page_map[p] + 1) * ps] = vp[p * ps:(p + 1) * ps]
        pt = page_map[W.page_table]
        loc = (page_map[W.loc // ps] * ps + W.loc % ps).astype(np.int32)
        return nk, nv, pt.astype(np.int32), loc, ps
    assert new_page_size == 1
    max_len = int(W.seq_lens.max())
    pt = np.zeros((W.bs, max_len), np.int32)
    for b in range(W.bs):
        for p in range(int(W.seq_lens[b])):
            pt[b, p] = W.page_table[b, p // ps] * ps + p % ps
    return kp.copy(), vp.copy(), pt, W.loc.copy(), 1


def _run_layout(W, kp, vp, pt, loc, ps):
    kv = oracle.KV_FP8_E4M3 if W.is_fp8 else oracle.KV_BF16
    oracle.set_kv_buffer(kp, vp, loc, bf16_bits(W.k_new), bf16_bits(W.v_new), kv_dtype=kv,
                         k_inv_scale=W.k_inv_scale, v_inv_scale=W.v_inv_scale)
    meta = oracle.build_metadata(W.seq_lens, pt, ps, qo_lens=None if W.mode == "decode" else W.qo_lens)
    return oracle.attention(bf16_bits(W.q), kp, vp, meta, W.num_q_heads, W.num_kv_heads, ps, W.sm_scale,
                            kv_dtype=kv, k_scale=W.k_scale, v_scale=W.v_scale)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_p2_page_permutation_invariance(kv_dtype):
    W = _tiny("extend", kv_dtype, page_size=4)
    o0, l0 = oracle_reference(W)
    rng = np.random.default_rng(11)
    perm = np.concatenate([[0], rng.permutation(np.arange(1, W.num_pages))])
    o1, l1 = _run_layout(W, *_relayout(W, perm))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_p3_page_size_1_equals_16():
    W = preset("tiny_decode")  # page_size 16
    o0, l0 = oracle_reference(W)
    o1, l1 = _run_layout(W, *_relayout(W, None, new_page_size=1))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


@pytest.mark.parametrize("name", ["tiny_decode", "prefix_extend", "spec_verify"])
def test_p3_page_size_128_equals_16_equals_1(name):
    """The same tokens in 128-token pages, in 16-token pages and in one-token
    pages give the same attention, bit for bit: the presets draw the values of
    every (request, position) in the same order whatever the page size, and
    only the pages that hold them differ."""
    kw = {} if name == "tiny_decode" else dict(bs=3, len_scale=0.05)
    W16 = preset(name, **kw)
    W128 = preset(name, page_size=128, **kw)
    assert W128.page_size == 128 and not np.array_equal(W128.loc, W16.loc)
    o16, l16 = oracle_reference(W16)
    o128, l128 = oracle_reference(W128)
    o1, l1 = _run_layout(W128, *_relayout(W128, None, new_page_size=1))
    assert np.array_equal(o16, o128) and np.array_equal(l16, l128)
    assert np.array_equal(o1, o128) and np.array_equal(l1, l128)


# ---------------------------------------------------------------- P4 / P5 / P6 closed forms
def test_p4_single_key():
    W = make_workload("one", "decode", 2, 4, 2, 8, [0, 0], [1, 1], page_size=4)
    o, lse = oracle_reference(W)
    q = _q64(W)
    kn = W.k_new.double().numpy()
    vn = W.v_new.double().numpy()
    for b in range(2):
        for h in range(4):
            g = h // 2
            assert np.array_equal(o[b, h], vn[b, g])  # softmax of one score is exactly 1
            s = W.sm_scale * float(np.dot(q[b, h], kn[b, g]))
            assert abs(lse[b, h] - s) < 1e-14


def test_p5_uniform_scores():
    W = _tiny("extend", "bf16", seed_shift=5)
    W.q.zero_()
    o, lse = oracle_reference(W)
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    G = W.num_q_heads // W.num_kv_heads
    for b, (K, V) in enumerate(_contiguous_kv(W)):
        L, N = int(W.seq_lens[b]), int(W.qo_lens[b])
        for i in range(N):
            cnt = L - N + i + 1
            t = qo_indptr[b] + i
            for h in range(W.num_q_heads):
                assert np.allclose(o[t, h], V[:cnt, h // G].mean(axis=0), atol=1e-13, rtol=0)
                assert abs(lse[t, h] - math.log(cnt)) < 1e-13


def test_p6_weights_sum_to_one():
    W = _tiny("extend", "bf16", seed_shift=9)
    one = 0x3F80  # bf16 1.0
    vp = pool_bits(W.v_pool)
    used = ~np.isnan((vp.astype(np.uint32) << 16).view(np.float32))
    vp[used] = one
    W.v_new.fill_(1.0)
    o, _ = oracle_reference(W)
    assert np.abs(o - 1.0).max() < 1e-12


# ---------------------------------------------------------------- P7 extend == stacked decodes
def test_p7_extend_equals_stacked_decodes():
    W = _tiny("extend", "bf16", seed_shift=13)
    kp, vp = oracle_pools(W)
    o_ext, l_ext = oracle_reference(W, pools=(kp, vp))
    qo_indptr = np.concatenate([[0], np.cumsum(W.qo_lens)])
    qbits = bf16_bits(W.q)
    for b in range(W.bs):
        P, N = int(W.prefix_lens[b]), int(W.qo_lens[b])
        for i in range(N):
            t = qo_indptr[b] + i
            meta = oracle.build_metadata([P + i + 1], W.page_table[b:b + 1], W.page_size)
            o, l = oracle.attention(qbits[t:t + 1], kp, vp, meta, W.num_q_heads, W.num_kv_heads, W.page_size,
                                    W.sm_scale)
            assert np.array_equal(o[0], o_ext[t]) and np.array_equal(l[0], l_ext[t])


# ---------------------------------------------------------------- P8 LSE merge identity
def test_p8_lse_merge_identity():
    W = make_workload("merge", "decode", 1, 4, 1, 16, [200], [1], page_size=8)
    kp, vp = oracle_pools(W)
    o_all, l_all = oracle_reference(W, pools=(kp, vp))
    L = int(W.seq_lens[0])
    n_pages = (L + 7) // 8
    cuts = [0, 3, 4, 11, n_pages]  # arbitrary chunks of whole pages
    qbits = bf16_bits(W.q)
    for h in range(4):
        parts_o, parts_l = [], []
        for c0, c1 in zip(cuts[:-1], cuts[1:]):
            length = min(L, c1 * 8) - c0 * 8
            meta = oracle.build_metadata([length], W.page_table[:, c0:c1], 8)
            o, l = oracle.attention(qbits, kp, vp, meta, 4, 1, 8, W.sm_scale)
            parts_o.append(o[0, h])
            parts_l.append(l[0, h])
        parts_o.append(np.full(16, 5.0))  # an empty chunk carries no weight
        parts_l.append(-math.inf)
        om, lm = oracle.lse_merge(np.array(parts_o), np.array(parts_l))
        assert np.abs(om - o_all[0, h]).max() < 1e-12 and abs(lm - l_all[0, h]) < 1e-12


# ---------------------------------------------------------------- P9 E4M3 code table
def test_p9_e4m3_table():
    vals = [oracle.e4m3_decode(c) for c in range(256)]
    nans = [c for c, v in enumerate(vals) if math.isnan(v)]
    assert nans == [0x7F, 0xFF]
    fin = [v for v in vals if not math.isnan(v)]
    assert max(fin) == 448.0 and min(fin) == -448.0
    assert min(v for v in fin if v > 0) == 2.0 ** -9
    pos = vals[0:0x7F]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # codes 0x00..0x7E increase strictly
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(vals[c]) == c  # every finite code round-trips
    # torch's float8_e4m3fn widening is a library decode of the same format
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(lib), np.isnan(np.array(vals)))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], np.array(vals)[ok])


def test_p9_e4m3_rounding_vs_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 40, rng.standard_normal(5000) * 0.01,
                        rng.uniform(-447.9, 447.9, 5000)]).astype(np.float32)
    # exact midpoints between neighbouring codes, where ties go to even
    grid = np.array(sorted({oracle.e4m3_decode(c) for c in range(0x7F)}))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # hand-worked ties: 1.0625 lies halfway between 1.0 (m=0) and 1.125 (m=1) -> even -> 1.0;
    # 1.1875 halfway between 1.125 (m=1) and 1.25 (m=2) -> 1.25; 2^-10 halfway 0 and 2^-9 -> 0
    assert oracle.e4m3_encode(1.0625) == 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02
    # saturation of out-of-range magnitudes, canonical NaN
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-math.inf) == 0xFE
    assert oracle.e4m3_encode(460.0) == 0x7E
    assert oracle.e4m3_encode(math.nan) == 0x7F


# ---------------------------------------------------------------- set_kv_buffer
def test_set_kv_buffer_bf16_bits_and_untouched():
    W = _tiny("extend", "bf16")
    before_k = pool_bits(W.k_pool)
    kp, vp = oracle_pools(W)
    kn, vn = bf16_bits(W.k_new), bf16_bits(W.v_new)
    assert np.array_equal(kp[W.loc], kn) and np.array_equal(vp[W.loc], vn)
    mask = np.ones(kp.shape[0], bool)
    mask[W.loc] = False
    assert np.array_equal(kp[mask].view(np.uint16), before_k[mask].view(np.uint16))


def test_set_kv_buffer_fp8_matches_torch_cast():
    W = _tiny("extend", "fp8_e4m3")
    kp, vp = oracle_pools(W)
    ref = (W.k_new.float() * W.k_inv_scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kp[W.loc], ref)


# ---------------------------------------------------------------- metadata
def test_p11_metadata_closed_form():
    g = _golden("tiny_decode_metadata.txt")
    seq = np.array([int(x) for x in g["seq_lens"][0]])
    ps = int(g["page_size"][0][0])
    W = preset("tiny_decode")
    assert np.array_equal(W.seq_lens, seq) and W.page_size == ps
    meta = oracle_meta(W)
    assert meta["kv_indptr"].tolist() == [int(x) for x in g["kv_indptr"][0]]
    assert meta["kv_last_page_len"].tolist() == [int(x) for x in g["kv_last_page_len"][0]]
    assert meta["qo_indptr"].tolist() == [int(x) for x in g["qo_indptr"][0]]
    flat = np.concatenate([W.page_table[b, :n] for b, n in enumerate([3, 7, 14, 19])])
    assert np.array_equal(meta["kv_indices"], flat)


def test_metadata_extend_and_empty_requests():
    seq = np.array([0, 16, 17, 5, 0], np.int32)
    qo = np.array([0, 16, 2, 5, 0], np.int32)
    pt = np.arange(5 * 3, dtype=np.int32).reshape(5, 3) + 100
    meta = oracle.build_metadata(seq, pt, 16, qo_lens=qo)
    assert meta["kv_indptr"].tolist() == [0, 0, 1, 3, 4, 4]
    assert meta["kv_last_page_len"].tolist() == [0, 16, 1, 5, 0]
    assert meta["qo_indptr"].tolist() == [0, 0, 16, 18, 23, 23]
    assert meta["kv_indices"].tolist() == [103, 106, 107, 109]


# ---------------------------------------------------------------- P10 pool sizing
def test_p10_pool_size_matches_server_log():
    g = _golden("l4_pool_log.txt")
    val = lambda k: float(g[k][0][0])
    per_layer = oracle.pool_bytes(int(val("pool_tokens")), int(val("model_kv_heads")), int(val("model_head_dim")),
                                  int(val("pool_dtype_bytes")))
    total = per_layer * int(val("model_layers"))
    assert round(total / 2 ** 30, 2) == val("k_size_gb") == val("v_size_gb")
    assert round(val("decode_tokens") / val("pool_tokens"), 2) == val("decode_token_usage")


# ---------------------------------------------------------------- P12 unused slots
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_p12_nan_unused_slots_never_read(kv_dtype):
    W = _tiny("decode", kv_dtype, seed_shift=2)
    o, lse = oracle_reference(W)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_empty_request_gives_zero_and_neg_inf():
    W = make_workload("pad", "decode", 3, 4, 2, 8, [5, 0, 9], [1, 0, 1], page_size=4)
    meta = oracle.build_metadata(W.seq_lens, W.page_table, 4, qo_lens=np.array([1, 1, 1]))
    kp, vp = oracle_pools(W)
    q = np.zeros((3, 4, 8), np.uint16)
    q[[0, 2]] = bf16_bits(W.q)
    o, lse = oracle.attention(q, kp, vp, meta, 4, 2, 4, W.sm_scale)
    assert np.all(o[1] == 0.0) and np.all(np.isneginf(lse[1]))
    assert np.isfinite(o[[0, 2]]).all()


# ---------------------------------------------------------------- dispatch
_MODES = {"extend": oracle.MODE_EXTEND, "decode": oracle.MODE_DECODE, "idle": oracle.MODE_IDLE,
          "target_verify": oracle.MODE_TARGET_VERIFY, "draft_extend": oracle.MODE_DRAFT_EXTEND}
_SPEC = {"prefill": oracle.SPEC_PREFILL, "decode": oracle.SPEC_DECODE}
_PATH = {"decode": oracle.PATH_DECODE, "extend": oracle.PATH_EXTEND}


def select_backend_table():
    rows = []
    with open(os.path.join(GOLDEN, "select_backend.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                m, s, p = line.split()
                rows.append((_MODES[m], _SPEC[s], _PATH[p]))
    return rows


def test_select_path_truth_table():
    rows = select_backend_table()
    assert len(rows) == 10
    for m, s, p in rows:
        assert oracle.select_path(m, s) == p
    assert oracle.select_path(7, 0) == -1 and oracle.select_path(0, 5) == -1


def test_random_tree_masks_are_trees():
    """The seeded draft trees are valid inputs: each word holds its own bit,
    no later draft, and its parent's word (a tree laid out parents first)."""
    qo = [1, 5, 17, 64, 8]
    words = random_tree_masks(qo, seed=21)
    assert words.dtype == np.uint64 and words.shape == (sum(qo),)
    off = 0
    branched = False
    for n in qo:
        w = [int(x) for x in words[off:off + n]]
        for i in range(n):
            assert (w[i] >> i) & 1
            assert w[i] >> (i + 1) == 0
            below = w[i] & ((1 << i) - 1)
            if below:
                parent = below.bit_length() - 1  # the highest set bit below i is the parent
                assert w[parent] == below
            branched |= w[i] != (1 << (i + 1)) - 1
        off += n
    assert branched
    assert np.array_equal(chain_tree_masks([3]), np.array([1, 3, 7], dtype=np.uint64))
