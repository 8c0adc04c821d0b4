"""The C-ABI library builds, loads and exports every symbol include/pkv.h declares;
host-only calls (dispatch, pool sizing, config checks) behave as documented.
No CUDA device is needed: nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

import oracle
from paged_kv_cache_15_gb300 import binding as B
from paged_kv_cache_15_gb300 import build as pkv_build
from tests.test_oracle_pins import _golden, select_backend_table

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return B.lib()


def header_functions():
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert header_functions() == sorted(B.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(B.LIB_PATH)
    for name in header_functions():
        assert hasattr(raw, name), name


def test_select_backend_matches_pages_and_oracle(lib):
    for m, s, p in select_backend_table():
        assert B.pkv_select_backend(m, s) == p
        assert B.pkv_select_backend(m, s) == oracle.select_path(m, s)
    assert B.pkv_select_backend(9, 0) == B.PKV_PATH_INVALID
    assert B.pkv_select_backend(0, 2) == B.PKV_PATH_INVALID
    assert B.pkv_select_backend(-1, 0) == B.PKV_PATH_INVALID


def test_status_strings(lib):
    for st in range(6):
        assert B.pkv_status_string(st)
    assert "unknown" in B.pkv_status_string(99)


def test_pool_bytes_reproduces_server_log(lib):
    g = _golden("l4_pool_log.txt")
    v = lambda k: float(g[k][0][0])
    tokens = int(v("pool_tokens"))
    cfg = B.make_config(32, int(v("model_kv_heads")), int(v("model_head_dim")), 1, B.PKV_KV_BF16, tokens, 1, 1, 1)
    per_layer = B.pkv_pool_bytes(cfg)
    assert per_layer == oracle.pool_bytes(tokens, int(v("model_kv_heads")), int(v("model_head_dim")), 2)
    assert round(per_layer * int(v("model_layers")) / 2 ** 30, 2) == v("k_size_gb")
    cfg8 = B.make_config(32, 8, 128, 16, B.PKV_KV_FP8_E4M3, 10, 1, 1, 1)
    assert B.pkv_pool_bytes(cfg8) == 10 * 16 * 8 * 128


def _cfg(**kw):
    base = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, kv_dtype=B.PKV_KV_BF16, num_pages=100,
                max_batch=4, max_pages_total=100, max_q_tokens=64, max_qo_len=1)
    base.update(kw)
    return B.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=30), B.PKV_ERR_INVALID_ARG),       # heads not a multiple
    (dict(num_kv_heads=0), B.PKV_ERR_INVALID_ARG),
    (dict(head_dim=96), B.PKV_ERR_UNSUPPORTED),
    (dict(page_size=32), B.PKV_ERR_UNSUPPORTED),
    (dict(page_size=64), B.PKV_ERR_UNSUPPORTED),
    (dict(page_size=256), B.PKV_ERR_UNSUPPORTED),
    (dict(kv_dtype=7), B.PKV_ERR_INVALID_ARG),
    (dict(kv_dtype=B.PKV_KV_FP8_E4M3, head_dim=64), B.PKV_ERR_UNSUPPORTED),
    (dict(num_q_heads=64, num_kv_heads=2), B.PKV_ERR_UNSUPPORTED),  # group 32
    (dict(max_qo_len=9, num_q_heads=64, num_kv_heads=4), B.PKV_ERR_UNSUPPORTED),  # 9 x 16 rows > 128
    (dict(max_batch=0), B.PKV_ERR_INVALID_ARG),
    # K and V heads of different widths: only 192 / 128, bf16 pools
    (dict(head_dim_v=-1), B.PKV_ERR_INVALID_ARG),
    (dict(head_dim=128, head_dim_v=64), B.PKV_ERR_UNSUPPORTED),
    (dict(head_dim=192, head_dim_v=64), B.PKV_ERR_UNSUPPORTED),
    (dict(head_dim=192), B.PKV_ERR_UNSUPPORTED),  # 192-wide V heads
    (dict(head_dim=64, head_dim_v=128), B.PKV_ERR_UNSUPPORTED),
    (dict(kv_dtype=B.PKV_KV_FP8_E4M3, head_dim=192, head_dim_v=128), B.PKV_ERR_UNSUPPORTED),
])
def test_config_rejected_before_any_device_call(lib, kw, status):
    n = ctypes.c_size_t(0)
    st = B.lib().pkv_workspace_bytes(ctypes.byref(_cfg(**kw)), ctypes.byref(n))
    assert st == status


def test_null_arguments_rejected(lib):
    L = B.lib()
    assert L.pkv_workspace_bytes(None, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_create(None, None, 0, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_build_metadata(None, 0, 1, None, None, None, 1, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_set_kv_buffer(None, None, None, None, None, None, 1, 1.0, 1.0, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_forward_decode(None, None, None, None, 1.0, 1.0, 1.0, None, None, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_forward(None, 0, 0, None, None, None, 1.0, 1.0, 1.0, None, None, None) == B.PKV_ERR_INVALID_ARG
    assert L.pkv_destroy(None) == B.PKV_OK
    code = ctypes.c_int32(0)
    assert L.pkv_get_device_error(None, ctypes.byref(code), None) == B.PKV_ERR_INVALID_ARG


@pytest.mark.parametrize("widths", [(64, 0), (128, 0), (128, 128), (192, 128)])
def test_supported_head_widths_accepted(lib, widths):
    """Equal widths (head_dim_v 0 or equal) and 192-wide Q/K heads with
    128-wide V heads pass the configuration checks."""
    n = ctypes.c_size_t(0)
    st = B.lib().pkv_workspace_bytes(ctypes.byref(_cfg(head_dim=widths[0], head_dim_v=widths[1])), ctypes.byref(n))
    assert st in (B.PKV_OK, B.PKV_ERR_CUDA)


def test_pool_bytes_is_the_k_pool(lib):
    cfg = B.make_config(32, 8, 192, 16, B.PKV_KV_BF16, 10, 1, 1, 1, head_dim_v=128)
    assert B.pkv_pool_bytes(cfg) == 10 * 16 * 8 * 192 * 2


@pytest.mark.parametrize("page_size", [16, 128])
def test_supported_page_sizes_accepted(lib, page_size):
    """Both page sizes pass the configuration checks (without a device the
    call then stops at the SM-count query with PKV_ERR_CUDA)."""
    n = ctypes.c_size_t(0)
    st = B.lib().pkv_workspace_bytes(ctypes.byref(_cfg(page_size=page_size)), ctypes.byref(n))
    assert st in (B.PKV_OK, B.PKV_ERR_CUDA)
