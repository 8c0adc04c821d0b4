"""ctypes binding of the C ABI in ``include/pkv.h`` — argument marshalling only.

Every function here has the name of the C function it calls and does no
compute: it turns torch tensors into device pointers and the current CUDA
stream into a ``cudaStream_t``, calls the library, and raises ``PkvError`` on a
non-zero status. All attention work runs in the library's CUDA kernels; there
is no CPU or PyTorch fallback, and a missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_CAPACITY, PKV_ERR_CUDA, PKV_ERR_DEVICE = range(6)
(PKV_DEV_OK, PKV_DEV_BAD_LENGTH, PKV_DEV_BAD_PAGE, PKV_DEV_CAPACITY, PKV_DEV_BAD_SLOT, PKV_DEV_QO_TOO_LONG,
 PKV_DEV_TREE_TOO_LONG) = range(7)
PKV_DEV_TIMEOUT = 16
PKV_MODE_EXTEND, PKV_MODE_DECODE, PKV_MODE_IDLE, PKV_MODE_TARGET_VERIFY, PKV_MODE_DRAFT_EXTEND = range(5)
PKV_SPEC_PREFILL, PKV_SPEC_DECODE = 0, 1
PKV_PATH_INVALID, PKV_PATH_DECODE, PKV_PATH_EXTEND = -1, 0, 1
PKV_KV_BF16, PKV_KV_FP8_E4M3 = 0, 1

# every function the header declares (checked against include/pkv.h by the tests)
EXPORTS = ("pkv_status_string", "pkv_workspace_bytes", "pkv_pool_bytes", "pkv_create", "pkv_destroy",
           "pkv_select_backend", "pkv_build_metadata", "pkv_get_metadata", "pkv_set_kv_buffer",
           "pkv_forward_decode", "pkv_forward_extend", "pkv_forward", "pkv_get_device_error", "pkv_describe",
           "pkv_forward_decode_static", "pkv_set_tree_mask", "pkv_set_attention_sinks", "pkv_set_wait_limit",
           "pkv_test_hold_first_load")


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pkv_status_string(status)} (status {status})")


class pkv_config(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "num_q_heads", "num_kv_heads", "head_dim", "page_size", "kv_dtype", "num_pages", "max_batch",
        "max_pages_total", "max_q_tokens", "max_qo_len", "head_dim_v")]


_lock = threading.Lock()
_lib = None


def lib():
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built ({LIB_PATH} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        cfgp = ctypes.POINTER(pkv_config)
        i32pp = ctypes.POINTER(ctypes.c_void_p)
        sig = {
            "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "pkv_workspace_bytes": (ctypes.c_int, [cfgp, ctypes.POINTER(sz)]),
            "pkv_pool_bytes": (ctypes.c_int, [cfgp, ctypes.POINTER(sz)]),
            "pkv_create": (ctypes.c_int, [cfgp, vp, sz, ctypes.POINTER(vp)]),
            "pkv_destroy": (ctypes.c_int, [vp]),
            "pkv_select_backend": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
            "pkv_build_metadata": (ctypes.c_int, [vp, ctypes.c_int, i32, vp, vp, vp, i32, vp]),
            "pkv_get_metadata": (ctypes.c_int, [vp, i32pp, i32pp, i32pp, i32pp]),
            "pkv_set_kv_buffer": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, i32, ctypes.c_float, ctypes.c_float, vp]),
            "pkv_forward_decode": (ctypes.c_int, [vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                  vp, vp, vp]),
            "pkv_forward_extend": (ctypes.c_int, [vp, vp, vp, vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                                  vp, vp, vp]),
            "pkv_forward": (ctypes.c_int, [vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_float, vp, vp, vp]),
            "pkv_set_tree_mask": (ctypes.c_int, [vp, vp]),
            "pkv_set_attention_sinks": (ctypes.c_int, [vp, vp]),
            "pkv_set_wait_limit": (ctypes.c_int, [vp, ctypes.c_uint32, vp]),
            "pkv_test_hold_first_load": (ctypes.c_int, [vp, ctypes.c_int, vp]),
            "pkv_get_device_error": (ctypes.c_int, [vp, ctypes.POINTER(i32), vp]),
            "pkv_describe": (ctypes.c_int, [vp, ctypes.c_char_p, sz]),
            "pkv_forward_decode_static": (ctypes.c_int, [cfgp, i32, vp, vp, i32, vp, vp, vp, ctypes.c_float,
                                                         ctypes.c_float, ctypes.c_float, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def _check(st: int, where: str):
    if st != PKV_OK:
        raise PkvError(st, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def pkv_status_string(status: int) -> str:
    try:
        return lib().pkv_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def make_config(num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, num_pages, max_batch, max_pages_total,
                max_q_tokens, max_qo_len=1, head_dim_v=0) -> pkv_config:
    return pkv_config(num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype, num_pages, max_batch,
                      max_pages_total, max_q_tokens, max_qo_len, head_dim_v)


def pkv_workspace_bytes(cfg: pkv_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().pkv_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "pkv_workspace_bytes")
    return n.value


def pkv_pool_bytes(cfg: pkv_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().pkv_pool_bytes(ctypes.byref(cfg), ctypes.byref(n)), "pkv_pool_bytes")
    return n.value


def pkv_create(cfg: pkv_config, workspace: torch.Tensor) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p()
    _check(lib().pkv_create(ctypes.byref(cfg), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            ctypes.byref(ctx)), "pkv_create")
    return ctx


def pkv_destroy(ctx) -> None:
    _check(lib().pkv_destroy(ctx), "pkv_destroy")


def pkv_select_backend(forward_mode: int, spec_mode: int) -> int:
    return int(lib().pkv_select_backend(int(forward_mode), int(spec_mode)))


def pkv_build_metadata(ctx, forward_mode, batch, seq_lens, qo_lens, page_table, stream=None) -> None:
    stride = page_table.shape[1] if page_table is not None and page_table.dim() == 2 else 0
    _check(lib().pkv_build_metadata(ctx, int(forward_mode), int(batch), _ptr(seq_lens), _ptr(qo_lens),
                                    _ptr(page_table), int(stride), _stream(stream)), "pkv_build_metadata")


def pkv_get_metadata(ctx):
    ptrs = [ctypes.c_void_p() for _ in range(4)]
    _check(lib().pkv_get_metadata(ctx, *[ctypes.byref(p) for p in ptrs]), "pkv_get_metadata")
    return [p.value for p in ptrs]


def pkv_set_kv_buffer(ctx, k_pool, v_pool, loc, k, v, k_inv_scale=1.0, v_inv_scale=1.0, stream=None) -> None:
    _check(lib().pkv_set_kv_buffer(ctx, _ptr(k_pool), _ptr(v_pool), _ptr(loc), _ptr(k), _ptr(v),
                                   int(loc.shape[0]), float(k_inv_scale), float(v_inv_scale), _stream(stream)),
           "pkv_set_kv_buffer")


def pkv_forward_decode(ctx, q, k_pool, v_pool, sm_scale, out, lse=None, k_scale=1.0, v_scale=1.0,
                       stream=None) -> None:
    _check(lib().pkv_forward_decode(ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), float(sm_scale), float(k_scale),
                                    float(v_scale), _ptr(out), _ptr(lse), _stream(stream)), "pkv_forward_decode")


def pkv_forward_extend(ctx, q, k_pool, v_pool, sm_scale, out, lse=None, k_scale=1.0, v_scale=1.0,
                       stream=None) -> None:
    _check(lib().pkv_forward_extend(ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), float(sm_scale), float(k_scale),
                                    float(v_scale), _ptr(out), _ptr(lse), _stream(stream)), "pkv_forward_extend")


def pkv_forward(ctx, forward_mode, spec_mode, q, k_pool, v_pool, sm_scale, out, lse=None, k_scale=1.0,
                v_scale=1.0, stream=None) -> None:
    _check(lib().pkv_forward(ctx, int(forward_mode), int(spec_mode), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                             float(sm_scale), float(k_scale), float(v_scale), _ptr(out), _ptr(lse),
                             _stream(stream)), "pkv_forward")


def pkv_set_tree_mask(ctx, tree_mask) -> None:
    """Draft-tree mask words (uint64 device tensor, one per query token) for
    the verify forwards that follow, or None for chain drafts."""
    _check(lib().pkv_set_tree_mask(ctx, _ptr(tree_mask)), "pkv_set_tree_mask")


def pkv_set_attention_sinks(ctx, sinks) -> None:
    """Per-query-head sink logits (fp32 device tensor [num_q_heads]) for the
    forwards that follow, or None to turn sinks off."""
    _check(lib().pkv_set_attention_sinks(ctx, _ptr(sinks)), "pkv_set_attention_sinks")


def pkv_set_wait_limit(ctx, limit_ns: int, stream=None) -> None:
    """Bound on every wait inside the kernels, in ns (0: the 2 s default)."""
    _check(lib().pkv_set_wait_limit(ctx, int(limit_ns), _stream(stream)), "pkv_set_wait_limit")


def pkv_test_hold_first_load(ctx, enable: bool, stream=None) -> None:
    """Test support: CTA 0 of later forwards never issues its first K/V load,
    so its waits run out after the wait limit."""
    _check(lib().pkv_test_hold_first_load(ctx, 1 if enable else 0, _stream(stream)), "pkv_test_hold_first_load")


def pkv_get_device_error(ctx, stream=None) -> int:
    code = ctypes.c_int32(0)
    st = lib().pkv_get_device_error(ctx, ctypes.byref(code), _stream(stream))
    if st not in (PKV_OK, PKV_ERR_DEVICE):
        raise PkvError(st, "pkv_get_device_error")
    return code.value


def pkv_describe(ctx) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(lib().pkv_describe(ctx, buf, 512), "pkv_describe")
    return buf.value.decode()


def pkv_forward_decode_static(cfg: pkv_config, batch, seq_lens, page_table, q, k_pool, v_pool, sm_scale, out,
                              lse=None, error=None, k_scale=1.0, v_scale=1.0, stream=None) -> None:
    """Decode without a context or workspace (scratch lives in the library's
    fixed device array); see include/pkv.h for who needs this and its limits."""
    stride = page_table.shape[1] if page_table is not None and page_table.dim() == 2 else 0
    _check(lib().pkv_forward_decode_static(ctypes.byref(cfg), int(batch), _ptr(seq_lens), _ptr(page_table),
                                           int(stride), _ptr(q), _ptr(k_pool), _ptr(v_pool), float(sm_scale),
                                           float(k_scale), float(v_scale), _ptr(out), _ptr(lse), _ptr(error),
                                           _stream(stream)), "pkv_forward_decode_static")


class PagedAttention:
    """Owns one context and its workspace (a torch uint8 tensor on the device)."""

    def __init__(self, cfg: pkv_config, device=None):
        self.cfg = cfg
        self.device = torch.device(device or "cuda")
        nbytes = pkv_workspace_bytes(cfg)
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self.workspace = self.workspace[off:off + nbytes]
        self.ctx = pkv_create(cfg, self.workspace)

    def close(self):
        if self.ctx:
            pkv_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
