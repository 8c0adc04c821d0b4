"""fp64 CPU oracle for attention over a paged KV cache — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it: the arithmetic lives in ``pkv_oracle.c`` (plain C,
double precision, one key after another), and this module only marshals numpy
arrays into it.

What each function follows (page titles and sections of the source pages):

* ``build_metadata`` — "--attention-backend", section "What an attention
  backend is": per-batch metadata (page table flattened into ``kv_indices``
  with ``kv_indptr`` offsets, last-page lengths, ``qo_indptr``).
* ``set_kv_buffer`` — "[SGLang] Hybrid Attention", section "forward: 선형
  어텐션까지 지원하는 범용 위임": ``save_kv_cache`` stores the step's K/V into
  the pool before attention; the E4M3 rounding follows the OCP FP8 E4M3FN
  definition.
* ``attention`` — "--attention-backend", same section (forward_decode /
  forward_extend over the paged cache), with the textbook scaled-dot-product
  formula and bottom-right causal alignment.
* ``select_path`` — "[SGLang] Hybrid Attention", section "_select_backend:
  ForwardMode 기반 동적 전환".
* ``lse_merge`` — the identity that combines attention over disjoint key sets.

Pins: tests/test_oracle_pins.py checks every function against facts fixed
outside the oracle itself (brute force, invariants, closed forms, code tables).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1

MODE_EXTEND, MODE_DECODE, MODE_IDLE, MODE_TARGET_VERIFY, MODE_DRAFT_EXTEND = 0, 1, 2, 3, 4
SPEC_PREFILL, SPEC_DECODE = 0, 1
PATH_DECODE, PATH_EXTEND = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off", "-fno-fast-math",
                    "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32p = ctypes.POINTER(ctypes.c_int32)
        vp = ctypes.c_void_p
        lib.oracle_bf16_decode.restype = ctypes.c_double
        lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_select_path.restype = ctypes.c_int
        lib.oracle_select_path.argtypes = [ctypes.c_int, ctypes.c_int]
        lib.oracle_build_metadata.restype = ctypes.c_int
        lib.oracle_build_metadata.argtypes = [ctypes.c_int, ctypes.c_int, i32p, i32p, i32p, ctypes.c_int64,
                                              i32p, i32p, i32p, i32p]
        lib.oracle_set_kv_buffer.restype = None
        lib.oracle_set_kv_buffer.argtypes = [ctypes.c_int, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p,
                                             vp, vp, ctypes.c_int, ctypes.c_float, ctypes.c_float]
        lib.oracle_lse_merge.restype = None
        lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [ctypes.c_int] * 7 + [vp, vp, vp, i32p, i32p, i32p, i32p, vp, vp,
                                                               ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                                               ctypes.c_int64, i32p, i32p, vp, vp, ctypes.c_int]
        lib.oracle_pool_bytes.restype = ctypes.c_int64
        lib.oracle_pool_bytes.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _lib = lib
        return lib


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def bf16_decode(bits: int) -> float:
    return _load().oracle_bf16_decode(int(bits))


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def select_path(mode: int, spec_mode: int) -> int:
    return int(_load().oracle_select_path(int(mode), int(spec_mode)))


def pool_bytes(num_slots: int, num_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return int(_load().oracle_pool_bytes(num_slots, num_kv_heads, head_dim, elem_bytes))


def build_metadata(seq_lens, page_table, page_size, qo_lens=None):
    """Return dict(kv_indptr, kv_indices, kv_last_page_len, qo_indptr) as int32 arrays."""
    lib = _load()
    seq, seq_p = _i32(seq_lens)
    bs = seq.shape[0]
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    if pt.ndim != 2 or pt.shape[0] < bs:
        raise ValueError("page_table must be [bs, max_pages]")
    stride = pt.shape[1]
    pt_p = pt.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    if qo_lens is not None:
        qo, qo_p = _i32(qo_lens)
    else:
        qo, qo_p = None, None
    total_pages = int(sum((int(L) + page_size - 1) // page_size for L in seq))
    kv_indptr, kv_indptr_p = _i32(np.zeros(bs + 1))
    kv_indices, kv_indices_p = _i32(np.zeros(max(total_pages, 1)))
    last, last_p = _i32(np.zeros(max(bs, 1)))
    qo_indptr, qo_indptr_p = _i32(np.zeros(bs + 1))
    st = lib.oracle_build_metadata(bs, page_size, seq_p, qo_p, pt_p, stride, kv_indptr_p, kv_indices_p, last_p,
                                   qo_indptr_p)
    if st != 0:
        raise ValueError(f"oracle_build_metadata failed ({st})")
    return dict(kv_indptr=kv_indptr, kv_indices=kv_indices[:total_pages], kv_last_page_len=last[:bs],
                qo_indptr=qo_indptr)


def set_kv_buffer(k_pool, v_pool, loc, k_new, v_new, kv_dtype=KV_BF16, k_inv_scale=1.0, v_inv_scale=1.0):
    """Scatter in place. Pools: uint16 (bf16 bits) or uint8 (e4m3) arrays [slots, Hkv, D]
    (K) and [slots, Hkv, Dv] (V); k_new/v_new: uint16 bf16 bits [n, Hkv, D] / [n, Hkv, Dv];
    loc: int32 [n]."""
    lib = _load()
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    kn = np.ascontiguousarray(k_new, dtype=np.uint16)
    vn = np.ascontiguousarray(v_new, dtype=np.uint16)
    lc, lc_p = _i32(loc)
    n, hkv, d = kn.shape
    dv = vn.shape[2] if vn.ndim == 3 else d
    assert k_pool.shape[-1] == d and v_pool.shape[-1] == dv
    lib.oracle_set_kv_buffer(int(kv_dtype), _ptr(k_pool), _ptr(v_pool), hkv, d, dv, lc_p, _ptr(kn), _ptr(vn), n,
                             float(k_inv_scale), float(v_inv_scale))


def lse_merge(o_parts, lse_parts):
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.oracle_lse_merge(n, d, _ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse))
    return o, float(lse[0])


def attention(q, k_pool, v_pool, meta, num_q_heads, num_kv_heads, page_size, sm_scale, kv_dtype=KV_BF16,
              k_scale=1.0, v_scale=1.0, rows=None, nthreads=None, tree_mask=None, sinks=None):
    """fp64 attention over the paged pool.

    q: uint16 bf16 bits [T, Hq, D]; pools: uint16 / uint8, K [slots, Hkv, D]
    and V [slots, Hkv, Dv] (Dv = D unless K and V heads differ in width);
    meta: dict from build_metadata. rows: None for every (token, head) row —
    returns o [T, Hq, Dv], lse [T, Hq] — or an int array [n, 2] of (token, head)
    pairs — returns o [n, Dv], lse [n]. tree_mask: None (chain drafts,
    bottom-right causal) or uint64 [T]: bit j of token t's word lets it see
    the j-th new token of its request (every cached key stays visible).
    sinks: None or float [Hq], each head's sink logit (a key with that score
    and a zero value vector).
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    T, hq, d = q.shape
    assert hq == num_q_heads
    dv = v_pool.shape[-1]
    assert k_pool.shape[-1] == d
    bs = meta["kv_indptr"].shape[0] - 1
    kvp, kvp_p = _i32(meta["kv_indptr"])
    kvi, kvi_p = _i32(meta["kv_indices"] if meta["kv_indices"].size else np.zeros(1))
    last, last_p = _i32(meta["kv_last_page_len"] if meta["kv_last_page_len"].size else np.zeros(1))
    qoi, qoi_p = _i32(meta["qo_indptr"])
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    if rows is None:
        n_rows = T * hq
        rt_p = rh_p = None
        out_o = np.zeros((T, hq, dv), dtype=np.float64)
        out_lse = np.zeros((T, hq), dtype=np.float64)
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = rows.shape[0]
        rt, rt_p = _i32(rows[:, 0])
        rh, rh_p = _i32(rows[:, 1])
        out_o = np.zeros((n_rows, dv), dtype=np.float64)
        out_lse = np.zeros((n_rows,), dtype=np.float64)
    tm = None if tree_mask is None else np.ascontiguousarray(tree_mask, dtype=np.uint64)
    if tm is not None:
        assert tm.shape == (T,)
    sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    if sk is not None:
        assert sk.shape == (hq,)
    st = lib.oracle_attention(bs, hq, num_kv_heads, d, dv, page_size, int(kv_dtype), _ptr(q), _ptr(k_pool),
                              _ptr(v_pool), kvp_p, kvi_p, last_p, qoi_p, None if tm is None else _ptr(tm),
                              None if sk is None else _ptr(sk),
                              float(sm_scale), float(k_scale),
                              float(v_scale), n_rows, rt_p, rh_p, _ptr(out_o), _ptr(out_lse), int(nthreads))
    if st != 0:
        raise ValueError(f"oracle_attention failed ({st})")
    return out_o, out_lse
