"""Runs a workload through the CPU oracle: scatter, metadata, attention.

Shared by the oracle pin tests and the GPU parity tests; it calls only
``oracle/`` and the seeded input generator.
"""
import numpy as np

import oracle
from paged_kv_cache_15_gb300.workloads import Workload, bf16_bits, pool_bits


def oracle_pools(W: Workload):
    """Host copies of the pools after the oracle's set_kv_buffer."""
    kp = pool_bits(W.k_pool).copy()
    vp = pool_bits(W.v_pool).copy()
    kv = oracle.KV_FP8_E4M3 if W.is_fp8 else oracle.KV_BF16
    if W.loc.shape[0]:
        oracle.set_kv_buffer(kp, vp, W.loc, bf16_bits(W.k_new), bf16_bits(W.v_new), kv_dtype=kv,
                             k_inv_scale=W.k_inv_scale, v_inv_scale=W.v_inv_scale)
    return kp, vp


def oracle_meta(W: Workload):
    qo = None if W.mode == "decode" else W.qo_lens
    return oracle.build_metadata(W.seq_lens, W.page_table, W.page_size, qo_lens=qo)


def oracle_reference(W: Workload, rows=None, pools=None, nthreads=None):
    """fp64 (o, lse) for every row (rows=None) or for the given (token, head) pairs."""
    kp, vp = pools if pools is not None else oracle_pools(W)
    meta = oracle_meta(W)
    kv = oracle.KV_FP8_E4M3 if W.is_fp8 else oracle.KV_BF16
    return oracle.attention(bf16_bits(W.q), kp, vp, meta, W.num_q_heads, W.num_kv_heads, W.page_size,
                            W.sm_scale, kv_dtype=kv, k_scale=W.k_scale, v_scale=W.v_scale, rows=rows,
                            nthreads=nthreads, tree_mask=W.tree_mask,
                            sinks=None if W.sinks is None else W.sinks.astype(np.float64))
